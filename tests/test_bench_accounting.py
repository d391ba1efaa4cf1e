"""The algorithmic work the benchmark divides by (CPU): bytes and flops of one decode call,
checked against hand-counted values for the cache layout (per packed C4 token: 256 B of latent
codes, 32 B of k_R codes, 16 B of latent metadata; 256 B of k_R metadata per page; 1152 B per
BF16 token)."""
import math
import os

import bench
import workloads


def test_c4r4_one_sequence_by_hand():
    w = workloads.Workload("acct", 1, 16, 8192, 4, 128)
    protected = 4 + 128
    packed = 8192 - protected
    pages = math.ceil((8192 - 128) / 128)  # pages holding packed tokens: 0 .. 62
    want = packed * (256 + 32 + 16) + pages * 256 + protected * 1152 + 16 * 1152 + 16 * 513 * 4
    assert want == 2_669_696
    assert bench.decode_bytes(w, [8192], 16) == want


def test_c2r4_and_short_sequences():
    w = workloads.Workload("acct2", 3, 16, 1000, 2, 64)
    per_tok = 128 + 32 + 16
    # T = 100: every token protected; T = 0: nothing but the query/output rows
    t1000 = (1000 - 132) * per_tok + math.ceil((1000 - 128) / 64) * 256 + 132 * 1152
    t100 = 100 * 1152
    rows = 3 * (16 * 1152 + 16 * 513 * 4)
    assert bench.decode_bytes(w, [1000, 100, 0], 16) == t1000 + t100 + rows


def test_bf16_bytes_and_flops():
    assert bench.bf16_decode_bytes([1000, 24], 16) == 1024 * 1152 + 2 * 16 * 1152 + 2 * 16 * 513 * 4
    assert bench.decode_flops([1000, 24], 64) == 1024 * 64 * 2 * (576 + 512)


def test_traffic_record_from_ncu_csv(tmp_path, monkeypatch):
    """roofline.traffic comes from a JSON written by --record-traffic out of ncu's CSV (units
    converted, read + write per launch of the matching kernel, other kernels ignored)."""
    import bench
    csv = tmp_path / "t.csv"
    head = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size",'
            '"Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"\n')
    row = lambda i, k, m, u, v: f'"{i}","1","python","h","{k}","1","7","(128, 1, 1)","(32, 1, 14)","0","10.3","s","{m}","{u}","{v}"\n'
    dk = "void mlaq::decode_kernel<4, false, false>(mlaq::DecodeParams)"
    ck = "void mlaq::combine_kernel(mlaq::DecodeParams)"
    csv.write_text("==PROF== Connected\n" + head + row(0, dk, "dram__bytes_read.sum", "Mbyte", "84.85") +
                   row(0, dk, "dram__bytes_write.sum", "Kbyte", "3,110") + row(1, ck, "dram__bytes_read.sum", "Mbyte", "14.7") +
                   row(1, ck, "dram__bytes_write.sum", "byte", "1000") + row(2, dk, "dram__bytes_read.sum", "Gbyte", "0.08485") +
                   row(2, dk, "dram__bytes_write.sum", "byte", "3110000"))
    monkeypatch.setattr(bench, "traffic_path", lambda w: str(tmp_path / f"traffic_{w}.json"))
    rec = bench.record_traffic(str(csv), "v2lite_c4r4_b32_h16_t8k", r"decode_kernel", "ncu ...")
    assert rec["launches"] == 2
    assert abs(rec["dram_bytes_per_launch"] - 87.96e6) < 1.0
    assert bench.profiled_traffic("v2lite_c4r4_b32_h16_t8k") == rec["dram_bytes_per_launch"]


def test_traffic_record_keyed_by_its_own_kernel_sources(tmp_path, monkeypatch):
    """A traffic record holds while the sources of its own kernel are unchanged: an edit of the
    64-head kernel's file leaves a 16-head record valid and voids a 64-head one; an edit of a
    shared header voids both."""
    import json
    import shutil

    import bench
    csrc = tmp_path / "r" / "bit_mla_kv_qcache_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in ("decode.cu", "decode_tc.cu", "kernels.cuh", "ptx.cuh"):
        shutil.copy(os.path.join(bench.ROOT, "bit_mla_kv_qcache_gb300", "csrc", f), csrc / f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path / "r"))
    monkeypatch.setattr(bench, "traffic_path", lambda w: str(tmp_path / f"traffic_{w}.json"))
    for w, k in (("h16", "decode_kernel"), ("h64", "decode_tc_kernel")):
        with open(bench.traffic_path(w), "w") as fh:
            json.dump({"kernel_regex": k, "dram_bytes_per_launch": 1.0, "source_sha": bench.source_sha(k)}, fh)
    assert bench.source_sha("decode_kernel") != bench.source_sha("decode_tc_kernel")
    assert bench.profiled_traffic("h16") == 1.0 and bench.profiled_traffic("h64") == 1.0
    with open(csrc / "decode_tc.cu", "a") as fh:
        fh.write("\n// edited\n")
    assert bench.profiled_traffic("h16") == 1.0 and bench.profiled_traffic("h64") is None
    with open(csrc / "ptx.cuh", "a") as fh:
        fh.write("\n// edited\n")
    assert bench.profiled_traffic("h16") is None
