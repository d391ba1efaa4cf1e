"""Multi-token decode on the GPU against the oracle: q_len new tokens per sequence, position i
sees the cache prefix up to itself; rows [position][head]. Same tolerance as the single-token
decode (per row max |O - O*| / max |O*| <= 2e-3, |LSE - LSE*| <= 2e-3)."""
import numpy as np
import pytest
import torch

import bit_mla_kv_qcache_gb300 as q
import oracle
import workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _run(w, lens, heads, q_len, scale=None):
    lens = np.array(lens, np.int32)
    inp = workloads.make_inputs(w, seq_lens=lens, heads=heads)
    kw = w.config_kwargs()
    cache = gu.gpu_cache(kw, inp)
    if inp.c.shape[0]:
        gu.write_rows(cache, inp.c, inp.kr, lens, max(1, int(lens.max())))
    B, R = len(lens), q_len * heads
    ql, qr = workloads.draw_queries(np.random.default_rng(int(lens.sum()) + q_len), B, R)
    out = torch.empty((B, R, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, R), dtype=torch.float32, device="cuda")
    ws = torch.zeros(max(16, q.workspace_bytes(cache.cfg, B, R, inp.page_table.shape[1])), dtype=torch.uint8,
                     device="cuda")
    sc = w.softmax_scale if scale is None else scale
    q.mla_qcache_decode_attn_multi(cache.cfg, q_len, gu.dev(ql), gu.dev(qr), cache.page_table, cache.seq_lens,
                                   cache.pool, cache.sink, cache.ring, sc, out, lse, ws, cache.err)
    torch.cuda.synchronize()
    assert cache.error_bits() == 0
    cfg, pool, sink, ring = gu.oracle_cache(kw, inp)
    if inp.c.shape[0]:
        assert oracle.write(cfg, inp.c, inp.kr, inp.cu, np.zeros(B, np.int32), max(1, int(lens.max())),
                            inp.page_table, pool, sink, ring) == 0
    o_ref, l_ref = oracle.decode_multi(cfg, ql, qr, q_len, inp.page_table, lens, pool, sink, ring, sc)
    return gu.check_decode(out, lse, o_ref, l_ref, TOL), (cache, ql, qr, out, lse, ws)


C4 = workloads.Workload("c4", 1, 16, 1, 4, 128, random_pages=True, seed=31)
C2 = workloads.Workload("c2", 1, 16, 1, 2, 64, clip_q=0.94, latent_dist="student_t5", n_outliers=8,
                        outlier_scale=20.0, random_pages=True, seed=32)
SMALL = workloads.Workload("sm", 1, 16, 1, 4, 32, n_sink=4, n_recent=32, random_pages=True, seed=33)


@pytest.mark.parametrize("q_len", [2, 4])
@pytest.mark.parametrize("T", [1, 3, 5, 131, 133, 300, 1000])
def test_c4_16_heads(q_len, T):
    """32 rows (16-head blocks) and 64 rows (one tensor-memory block holding all positions)."""
    _run(C4, [T, max(0, T - 1), T + 7], 16, q_len)


@pytest.mark.parametrize("q_len,heads", [(4, 16), (2, 32), (3, 64)])
def test_c2_long_and_wide(q_len, heads):
    _run(C2, [2000, 65, 700], heads, q_len)


def test_draft_as_long_as_the_window():
    """q_len = 16 over a 32-token recent window: 256 rows, early positions reach into tokens that
    are read from their packed copies."""
    _run(SMALL, [40, 300, 16], 16, 16)


def test_peaked_scores():
    _run(C4, [900, 260], 16, 4, scale=0.6)


def test_one_position_equals_the_single_token_decode():
    (_, _), (cache, ql, qr, out, lse, ws) = _run(C4, [500, 77], 16, 1)
    out2, lse2 = torch.empty_like(out), torch.empty_like(lse)
    q.mla_qcache_decode_attn(cache.cfg, gu.dev(ql), gu.dev(qr), cache.page_table, cache.seq_lens, cache.pool,
                             cache.sink, cache.ring, C4.softmax_scale, out2, lse2, ws, cache.err)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
