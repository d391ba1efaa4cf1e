"""The unquantized comparator on the GPU (decode over a paged BF16 cache) against the fp64
oracle's exact attention over the same pages. Tolerance as for the quantized decode: per row
max |O - O*| / max |O*| <= 2e-3 and |LSE - LSE*| <= 2e-3."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _pool(inp, P, rng, extra=1):
    B = len(inp.seq_lens)
    max_pages = max(1, int(np.ceil(int(inp.seq_lens.max()) / P))) + extra
    n_pages = B * max_pages
    pt = rng.permutation(n_pages).astype(np.int32).reshape(B, max_pages)
    pool = np.zeros((n_pages, P, 576), dtype=np.uint16)
    for b in range(B):
        rows = np.concatenate([inp.c[inp.cu[b]:inp.cu[b + 1]], inp.kr[inp.cu[b]:inp.cu[b + 1]]], axis=1)
        for t in range(int(inp.seq_lens[b])):
            pool[pt[b, t // P], t % P] = rows[t]
    return pt, pool


def _run(lens, P, heads, seed=3, scale=0.072, bad_page=None):
    import bit_mla_kv_qcache_gb300 as q
    w = workloads.Workload("bf", 1, heads, 1, 4, 128, random_pages=True, seed=seed)
    inp = workloads.make_inputs(w, seq_lens=np.array(lens, np.int32), heads=heads)
    pt, pool = _pool(inp, P, np.random.default_rng(seed))
    if bad_page is not None:
        pt[bad_page] = 10 ** 6
    B, H = len(lens), heads
    d_pt, d_pool = gu.dev(pt), gu.dev(pool.view(np.int16))
    out = torch.empty((B, H, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    ws = torch.zeros(q.bf16_workspace_bytes(B, H, pt.shape[1], P), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q.mla_qcache_decode_attn_bf16(gu.dev(inp.q_lat), gu.dev(inp.q_rope), d_pt, P, gu.dev(inp.seq_lens), d_pool,
                                  scale, out, lse, ws, err)
    torch.cuda.synchronize()
    if bad_page is not None:
        return int(err.item()), out
    assert int(err.item()) == 0
    o_ref, l_ref, fl = oracle.decode_bf16(inp.q_lat, inp.q_rope, pt, P, inp.seq_lens, pool, scale)
    assert fl == 0
    return gu.check_decode(out, lse, o_ref, l_ref, TOL)


@pytest.mark.parametrize("P", [32, 64, 128])
def test_bf16_comparator_boundaries(P):
    _run([0, 1, 15, 16, 17, 31, 32, 33, 200, 1000], P, 16)


def test_bf16_comparator_long_and_64_heads():
    _run([3000, 2049, 5], 64, 64, seed=5)


def test_bf16_comparator_peaked():
    _run([1500, 40], 128, 16, scale=0.5)


def test_bf16_comparator_bad_page_sets_error_bit():
    err, out = _run([300, 100], 64, 16, bad_page=(0, 2))
    assert err & 1
    assert torch.isfinite(out).all()
