"""The allocation-free decode entry point, checked against the workspace entry point.

Some callers cannot call cudaMalloc (a plugin whose host runtime owns all device memory, a
serving loop that must never trigger a device allocation); mla_qcache_decode_attn_noalloc
serves them from a scratch array compiled into the library. This file is collected last so a
stop-at-first-failure run has already run every other test.
"""
import numpy as np
import pytest
import torch

import workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("heads", [16, 64])
def test_noalloc_matches_workspace_entry_point_twice(heads):
    """16 heads run the warp-level kernel, 64 the tensor-memory kernel (both share the scratch)."""
    import bit_mla_kv_qcache_gb300 as q
    from bit_mla_kv_qcache_gb300 import binding as b
    w = workloads.Workload("na", 1, 16, 1, 4, 128, random_pages=True, seed=31)
    inp = workloads.make_inputs(w, seq_lens=np.array([1500, 700, 133, 9], np.int32), heads=heads)
    kw = w.config_kwargs()
    cache = gu.gpu_cache(kw, inp)
    gu.write_rows(cache, inp.c, inp.kr, inp.seq_lens, int(inp.seq_lens.max()))
    ql, qr = gu.dev(inp.q_lat), gu.dev(inp.q_rope)
    ref_o, ref_l = cache.decode(ql, qr, w.softmax_scale)
    torch.cuda.synchronize()
    ref = (ref_o.cpu().double().numpy(), ref_l.cpu().double().numpy())
    assert b.noalloc_scratch_bytes() >= b.workspace_bytes(cache.cfg, 4, heads, inp.page_table.shape[1])
    for _ in range(2):  # the scratch keeps the previous call's contents; both calls must agree
        out = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_l, float("nan"))
        b.mla_qcache_decode_attn_noalloc(cache.cfg, ql, qr, cache.page_table, cache.seq_lens, cache.pool, cache.sink,
                                         cache.ring, w.softmax_scale, out, lse, cache.err)
        torch.cuda.synchronize()
        gu.check_decode(out, lse, *ref, tol=2e-3)
    assert cache.error_bits() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    from bit_mla_kv_qcache_gb300 import binding as b
    cfg = b.make_config(4, 128)
    # B*H*splits partials beyond the built-in scratch: rejected before any launch
    big_B, H, max_pages = 4096, 128, 1024
    assert b.workspace_bytes(cfg, big_B, H, max_pages) > b.noalloc_scratch_bytes()
    dummy = torch.zeros(16, dtype=torch.int16, device="cuda")
    q = torch.zeros((big_B, H, 1), dtype=torch.int16, device="cuda")
    with pytest.raises(b.QCacheError, match="scratch"):
        b.mla_qcache_decode_attn_noalloc(cfg, q, q, torch.zeros((big_B, max_pages), dtype=torch.int32, device="cuda"),
                                         torch.zeros(big_B, dtype=torch.int32, device="cuda"),
                                         torch.zeros((1, 16), dtype=torch.uint8, device="cuda"), dummy, dummy, 0.1,
                                         torch.zeros(16, dtype=torch.float32, device="cuda"),
                                         torch.zeros(16, dtype=torch.float32, device="cuda"),
                                         torch.zeros(1, dtype=torch.int32, device="cuda"))
