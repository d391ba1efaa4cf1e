"""Decode-attention parity on the GPU against the fp64 oracle.

Tolerance (stated for the method's output): per (sequence, head) row, max |O - O*| / max |O*|
<= 2e-3, and |LSE - LSE*| <= 2e-3 (fp32 accumulation against fp64).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _run(w, lens, heads=None, extra_pages=0, scale=None):
    inp = workloads.make_inputs(w, seq_lens=np.array(lens, np.int32), extra_pages=extra_pages, heads=heads)
    kw = w.config_kwargs()
    cache = gu.gpu_cache(kw, inp)
    if inp.c.shape[0]:
        gu.write_rows(cache, inp.c, inp.kr, inp.seq_lens, max(1, int(inp.seq_lens.max())))
    sc = w.softmax_scale if scale is None else scale
    out, lse = cache.decode(gu.dev(inp.q_lat), gu.dev(inp.q_rope), sc)
    torch.cuda.synchronize()
    assert cache.error_bits() == 0, cache.error_bits()
    cfg, pool, sink, ring = gu.oracle_cache(kw, inp)
    if inp.c.shape[0]:
        assert oracle.write(cfg, inp.c, inp.kr, inp.cu, np.zeros(len(lens), np.int32),
                            max(1, int(inp.seq_lens.max())), inp.page_table, pool, sink, ring) == 0
    gu.assert_cache_equal(cache, pool, sink, ring)
    o_ref, l_ref, fl = oracle.decode(cfg, inp.q_lat, inp.q_rope, inp.page_table, inp.seq_lens, pool, sink, ring, sc)
    assert fl == 0
    return gu.check_decode(out, lse, o_ref, l_ref, TOL)


C4 = workloads.Workload("c4", 1, 16, 1, 4, 128, random_pages=True, seed=21)
C2 = workloads.Workload("c2", 1, 16, 1, 2, 64, clip_q=0.94, latent_dist="student_t5", n_outliers=8,
                        outlier_scale=20.0, random_pages=True, seed=22)


@pytest.mark.parametrize("T", [0, 1, 2, 4, 5, 131, 132, 133, 127, 128, 129, 259, 1000])
def test_boundaries_c4(T):
    _run(C4, [T, max(0, T - 1)])


@pytest.mark.parametrize("T", [1, 63, 64, 65, 131, 132, 133, 195, 777])
def test_boundaries_c2(T):
    _run(C2, [T, T + 16, 3])


def test_tiny_workload_full():
    w = workloads.WORKLOADS["tiny_c4r4_b1_h16_t1k"]
    _run(w, [w.seq_len])


@pytest.mark.parametrize("heads", [32, 80, 128, 192])
def test_more_heads(heads):
    """16-head blocks (32, 80) and 64-head blocks on the tensor-memory kernel (128, 192)."""
    _run(C4, [700, 300], heads=heads)


def test_no_sink_small_window_small_pages():
    w = workloads.Workload("s0", 1, 16, 1, 4, 32, n_sink=0, n_recent=32, random_pages=True, seed=5)
    _run(w, [500, 33, 32, 31, 65, 64])


def test_wide_window_and_sinks():
    w = workloads.Workload("s16", 1, 16, 1, 2, 32, n_sink=16, n_recent=256, clip_q=0.94, random_pages=True, seed=6)
    _run(w, [900, 272, 271, 40])


def test_ragged_batch_c2r4_serving_shape():
    w = workloads.WORKLOADS["ragged_c2r4_b64_h16_serve"]
    rng = np.random.default_rng(77)
    lens = rng.integers(1, 1500, size=64)
    _run(w, lens)


def test_many_sequences_work_split():
    """More sequences than a CTA has threads (the device-side scan of packed tile counts runs
    over several chunks), with sequences that have no packed tokens, short and long ones: the
    packed CTAs are shared in proportion to each sequence's tiles."""
    rng = np.random.default_rng(5)
    lens = rng.integers(0, 900, size=300)
    lens[::7] = 0
    lens[::11] = 132
    lens[::13] = 133
    _run(C4, lens)


def test_peaked_softmax():
    """A large softmax scale concentrates the weights (stresses the running-max rescaling)."""
    _run(C4, [600, 250], scale=0.5)


def test_full_size_v2lite_decode():
    """The 32 x 8192-token C4R4 decode in the configuration the benchmark times."""
    w = workloads.WORKLOADS["v2lite_c4r4_b32_h16_t8k"]
    rel, dl = _run(w, [w.seq_len] * w.batch, extra_pages=1)
    print(f"full-size rel {rel:.2e} dlse {dl:.2e}")


@pytest.mark.parametrize("w,heads", [(C4, 16), (C4, 32), (C2, 16), (C4, 128), (C2, 64)])
def test_query_alignment_does_not_change_the_result(w, heads):
    """A query that is 4-byte but not 16-byte aligned takes the element-by-element copy instead
    of the bulk copies (16-head blocks, and the 64-head tensor-memory kernel): the same result,
    bit for bit, and within tolerance of the oracle."""
    lens = [1000, 333, 140]
    inp = workloads.make_inputs(w, seq_lens=np.array(lens, np.int32), heads=heads)
    kw = w.config_kwargs()
    cache = gu.gpu_cache(kw, inp)
    gu.write_rows(cache, inp.c, inp.kr, inp.seq_lens, max(lens))
    q_lat, q_rope = gu.dev(inp.q_lat), gu.dev(inp.q_rope)
    out_a, lse_a = cache.decode(q_lat, q_rope, w.softmax_scale)
    # the same values at a 4-byte offset inside larger buffers
    bl = torch.empty(q_lat.numel() + 2, dtype=q_lat.dtype, device=q_lat.device)
    br = torch.empty(q_rope.numel() + 2, dtype=q_rope.dtype, device=q_rope.device)
    bl[2:].copy_(q_lat.reshape(-1))
    br[2:].copy_(q_rope.reshape(-1))
    ql_u, qr_u = bl[2:].view(q_lat.shape), br[2:].view(q_rope.shape)
    assert ql_u.data_ptr() % 16 != 0 and qr_u.data_ptr() % 16 != 0
    out_u, lse_u = cache.decode(ql_u, qr_u, w.softmax_scale)
    torch.cuda.synchronize()
    assert cache.error_bits() == 0
    assert torch.equal(out_a, out_u) and torch.equal(lse_a, lse_u)
    cfg, pool, sink, ring = gu.oracle_cache(kw, inp)
    assert oracle.write(cfg, inp.c, inp.kr, inp.cu, np.zeros(len(lens), np.int32), max(lens), inp.page_table,
                        pool, sink, ring) == 0
    o_ref, l_ref, fl = oracle.decode(cfg, inp.q_lat, inp.q_rope, inp.page_table, inp.seq_lens, pool, sink, ring,
                                     w.softmax_scale)
    assert fl == 0
    gu.check_decode(out_u, lse_u, o_ref, l_ref, TOL)


@pytest.mark.parametrize("heads", [16, 64])
def test_unused_page_table_entries_are_never_checked(heads):
    """Entries of the page table past a sequence's pages may hold anything (the 16-head kernel
    copies short tables whole, before the length is known): no error bit, the same result."""
    lens = [700, 300, 0]
    inp = workloads.make_inputs(C4, seq_lens=np.array(lens, np.int32), extra_pages=3, heads=heads)
    kw = C4.config_kwargs()
    cache = gu.gpu_cache(kw, inp)
    gu.write_rows(cache, inp.c, inp.kr, inp.seq_lens, max(lens))
    pt = inp.page_table.copy()
    for b, T in enumerate(lens):
        used = -(-T // C4.page_size)
        pt[b, used:] = np.where(np.arange(pt.shape[1] - used) % 2 == 0, -7, 10 ** 6)
    cache.page_table.copy_(torch.from_numpy(pt))
    out, lse = cache.decode(gu.dev(inp.q_lat), gu.dev(inp.q_rope), C4.softmax_scale)
    torch.cuda.synchronize()
    assert cache.error_bits() == 0, cache.error_bits()
    cfg, pool, sink, ring = gu.oracle_cache(kw, inp)
    assert oracle.write(cfg, inp.c, inp.kr, inp.cu, np.zeros(len(lens), np.int32), max(lens), inp.page_table,
                        pool, sink, ring) == 0
    o_ref, l_ref, fl = oracle.decode(cfg, inp.q_lat, inp.q_rope, pt, inp.seq_lens, pool, sink, ring,
                                     C4.softmax_scale)
    assert fl == 0
    gu.check_decode(out, lse, o_ref, l_ref, TOL)


def test_bad_page_sets_error_bit():
    inp = workloads.make_inputs(C4, seq_lens=np.array([700], np.int32))
    kw = C4.config_kwargs()
    cache = gu.gpu_cache(kw, inp)
    gu.write_rows(cache, inp.c, inp.kr, inp.seq_lens, 700)
    cache.page_table[0, 2] = 10 ** 6
    out, lse = cache.decode(gu.dev(inp.q_lat), gu.dev(inp.q_rope), C4.softmax_scale)
    torch.cuda.synchronize()
    assert cache.error_bits() & 1
    assert torch.isfinite(out).all()


# ---- 64-head blocks: the packed shares run on the tcgen05 kernel (128-token tiles)

@pytest.mark.parametrize("T", [0, 1, 133, 259, 260, 261, 388, 1000, 2100])
def test_tc_boundaries_c4(T):
    _run(C4, [T, max(0, T - 1)], heads=64)


@pytest.mark.parametrize("T", [1, 131, 132, 133, 260, 777, 1500])
def test_tc_boundaries_c2(T):
    _run(C2, [T, T + 16, 3], heads=64)


def test_tc_small_window_small_pages():
    """A recent window of 32: the last 128-token tile of a share runs past the written
    positions (those rows are neither loaded nor weighted)."""
    w = workloads.Workload("s0", 1, 16, 1, 4, 32, n_sink=0, n_recent=32, random_pages=True, seed=5)
    _run(w, [500, 33, 32, 31, 65, 64, 300], heads=64)


def test_tc_wide_window_and_sinks():
    w = workloads.Workload("s16", 1, 16, 1, 2, 32, n_sink=16, n_recent=256, clip_q=0.94, random_pages=True, seed=6)
    _run(w, [900, 272, 271, 40, 1200], heads=128)


def test_tc_peaked_softmax():
    """Concentrated weights: the running maximum is raised inside a share."""
    _run(C4, [1600, 250], heads=64, scale=0.5)


def test_tc_many_sequences():
    rng = np.random.default_rng(9)
    lens = rng.integers(0, 1300, size=40)
    lens[::5] = 0
    lens[::7] = 132
    _run(C2, lens, heads=64)


def test_tc_bad_page_sets_error_bit():
    inp = workloads.make_inputs(C4, seq_lens=np.array([700], np.int32), heads=64)
    kw = C4.config_kwargs()
    cache = gu.gpu_cache(kw, inp)
    gu.write_rows(cache, inp.c, inp.kr, inp.seq_lens, 700)
    cache.page_table[0, 2] = 10 ** 6
    out, lse = cache.decode(gu.dev(inp.q_lat), gu.dev(inp.q_rope), C4.softmax_scale)
    torch.cuda.synchronize()
    assert cache.error_bits() & 1
    assert torch.isfinite(out).all()


def test_balanced_shares_few_long_many_short():
    """A wide page table with many sequences launches more shares than one wave holds, so the
    16-head kernel takes equal shares sized from the batch: three long sequences among 61 short
    and empty ones (shares past a sequence's end are empty)."""
    w = workloads.WORKLOADS["ragged_c2r4_b64_h16_serve"]
    rng = np.random.default_rng(17)
    lens = rng.integers(0, 2000, size=64)
    lens[[3, 40, 63]] = [12000, 11000, 9000]
    lens[::9] = 0
    _run(w, lens)


@pytest.mark.parametrize("T,bits", [(4000, 4), (5000, 4), (65536, 4), (40000, 2)])
def test_one_sequence_many_splits(T, bits):
    """One sequence over 16 heads spreads its packed tiles over up to a full wave of CTAs; past
    32 partials per head the merge runs as four wide CTAs per (sequence, head)."""
    _run(C4 if bits == 4 else C2, [T])


def test_one_sequence_wide_table_full_wave():
    """A page table far longer than the sequence (5000 tokens in a 5040-page table) still takes
    one wave of shares, most of them empty."""
    _run(C4, [5000], extra_pages=5000)
