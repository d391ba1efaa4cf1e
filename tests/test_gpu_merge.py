"""The split merge inside the decode launch, against the fp64 oracle.

When a decode's CTAs fit on the GPU at once and each (sequence, 16-head block) has 24 partials or
more, the block's CTAs merge their own partials at the end of the launch, counting arrivals in the workspace's first 8192
bytes (a (count, generation) pair of uint32 per block). These tests run one workspace, zeroed
once, through shapes that merge in place and shapes that use the merge launch (64-head blocks),
and check the outputs against the oracle, that every count is zero after every call, and that
the generation words advanced exactly where the merge ran in place (one step per call). An
invalid count (not a possible arrival count) must be reported through the timeout bit at once
and leave the other blocks' outputs correct.

Tolerance as in test_gpu_decode: per (sequence, head) row, max |O - O*| / max |O*| <= 2e-3 and
|LSE - LSE*| <= 2e-3.
"""
import numpy as np
import pytest
import torch

import bit_mla_kv_qcache_gb300 as q
import oracle
import workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
TOL = 2e-3
ARRIVE_BYTES = 8192
DEV_TIMEOUT = 32

C4 = workloads.Workload("c4", 1, 16, 1, 4, 128, random_pages=True, seed=31)
C2 = workloads.Workload("c2", 1, 16, 1, 2, 64, clip_q=0.94, latent_dist="student_t5", n_outliers=8,
                        outlier_scale=20.0, random_pages=True, seed=32)


@pytest.fixture(scope="module")
def ws():
    return torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")


def _setup(w, lens, heads):
    inp = workloads.make_inputs(w, seq_lens=np.array(lens, np.int32), heads=heads)
    kw = w.config_kwargs()
    cache = gu.gpu_cache(kw, inp)
    gu.write_rows(cache, inp.c, inp.kr, inp.seq_lens, max(1, int(inp.seq_lens.max())))
    cfg, pool, sink, ring = gu.oracle_cache(kw, inp)
    assert oracle.write(cfg, inp.c, inp.kr, inp.cu, np.zeros(len(lens), np.int32),
                        max(1, int(inp.seq_lens.max())), inp.page_table, pool, sink, ring) == 0
    o_ref, l_ref, fl = oracle.decode(cfg, inp.q_lat, inp.q_rope, inp.page_table, inp.seq_lens, pool, sink, ring,
                                     w.softmax_scale)
    assert fl == 0
    return inp, cache, o_ref, l_ref


def _decode(w, inp, cache, ws):
    B, H = inp.q_lat.shape[0], inp.q_lat.shape[1]
    assert q.workspace_bytes(cache.cfg, B, H, inp.page_table.shape[1]) <= ws.numel()
    out = torch.full((B, H, 512), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    q.mla_qcache_decode_attn(cache.cfg, gu.dev(inp.q_lat), gu.dev(inp.q_rope), cache.page_table, cache.seq_lens,
                             cache.pool, cache.sink, cache.ring, w.softmax_scale, out, lse, ws, cache.err)
    torch.cuda.synchronize()
    return out, lse


def _counters(ws):
    c = ws[:ARRIVE_BYTES].view(torch.int32).view(-1, 2).cpu().numpy().astype(np.int64)
    return c[:, 0], c[:, 1] & 0xFFFFFFFF


# (workload, lengths, heads, kernel launches of one decode call): 16-head blocks whose partials
# are many (24 or more per block) and fit one wave merge in place (1 launch); fewer partials use
# the merge launch (2); 64-head blocks run the tensor-memory kernel and the merge launch (3)
CASES = [
    (C4, [3000, 1500, 700, 0], 16, 1),
    (C4, [1], 16, 2),
    (C2, [2100, 64, 777], 32, 1),
    (C4, [1200, 1201], 48, 1),
    (C4, [300, 250, 384, 100, 200, 300, 333, 17, 300, 290, 64, 380], 48, 2),
    (C4, [900, 300], 128, 3),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_merge_counters_and_parity(ws, case):
    w, lens, heads, launches = CASES[case]
    inp, cache, o_ref, l_ref = _setup(w, lens, heads)
    assert q.decode_launches(cache.cfg, len(lens), heads, inp.page_table.shape[1]) == launches
    groups = len(lens) * heads // 16
    for call in range(2):
        _, gen0 = _counters(ws)
        out, lse = _decode(w, inp, cache, ws)
        assert cache.error_bits() == 0, cache.error_bits()
        gu.check_decode(out, lse, o_ref, l_ref, TOL)
        count, gen1 = _counters(ws)
        assert not count.any(), f"call {call}: counts left {np.flatnonzero(count)[:8]}"
        step = (gen1 - gen0) & 0xFFFFFFFF
        assert np.all(step[:groups] == (1 if launches == 1 else 0)), step[:groups]
        assert not step[groups:].any()


def test_invalid_count_reports_timeout(ws):
    w, lens, heads = C4, [3000, 2900, 2800], 16
    inp, cache, o_ref, l_ref = _setup(w, lens, heads)
    assert q.decode_launches(cache.cfg, len(lens), heads, inp.page_table.shape[1]) == 1
    ctr = ws[:ARRIVE_BYTES].view(torch.int32)
    ctr[2] = 1 << 20  # block 1 (sequence 1): no arrival count can be this large
    torch.cuda.synchronize()
    out, lse = _decode(w, inp, cache, ws)
    assert cache.error_bits() & DEV_TIMEOUT
    ok = [0, 2]  # the other sequences' blocks merged as usual
    gu.check_decode(out[ok], lse[ok], o_ref[ok], l_ref[ok], TOL)
    count, _ = _counters(ws)
    assert count[0] == 0 and count[2] == 0 and count[1] >= 1 << 20
    # zeroed again, the same workspace serves the call
    ws[:ARRIVE_BYTES].zero_()
    cache.err.zero_()
    out, lse = _decode(w, inp, cache, ws)
    assert cache.error_bits() == 0
    gu.check_decode(out, lse, o_ref, l_ref, TOL)
    count, _ = _counters(ws)
    assert not count.any()


def test_bf16_comparator_merges_in_place(ws):
    """The BF16 comparator uses the same kernel and counters (one wave of shares at batch 2)."""
    from tests.test_gpu_bf16_decode import _pool
    B, H, P = 2, 16, 64
    w = workloads.Workload("bf", 1, H, 1, 4, 128, random_pages=True, seed=9)
    inp = workloads.make_inputs(w, seq_lens=np.array([1500, 700], np.int32), heads=H)
    pt, pool = _pool(inp, P, np.random.default_rng(9))
    assert q.bf16_workspace_bytes(B, H, pt.shape[1], P) <= ws.numel()
    assert q.decode_plan(q.make_config(4, 128), B, H, pt.shape[1], torch.cuda.get_device_properties(0).multi_processor_count)["bf16_parts"] >= 24
    out = torch.empty((B, H, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, gen0 = _counters(ws)
    q.mla_qcache_decode_attn_bf16(gu.dev(inp.q_lat), gu.dev(inp.q_rope), gu.dev(pt), P, gu.dev(inp.seq_lens),
                                  gu.dev(pool.view(np.int16)), 0.072, out, lse, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    count, gen1 = _counters(ws)
    assert not count.any()
    assert np.all(((gen1 - gen0) & 0xFFFFFFFF)[:B] == 1)
    o_ref, l_ref, fl = oracle.decode_bf16(inp.q_lat, inp.q_rope, pt, P, inp.seq_lens, pool, 0.072)
    assert fl == 0
    gu.check_decode(out, lse, o_ref, l_ref, TOL)
