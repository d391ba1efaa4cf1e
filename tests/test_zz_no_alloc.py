"""The allocation-free decode entry point, checked against the oracle and the workspace entry point.

Some callers cannot call cudaMalloc (a plugin whose host runtime owns all device memory, a
serving loop that must never trigger a device allocation); mla_qcache_decode_attn_noalloc
serves them from a scratch array compiled into the library. This file is collected last so a
stop-at-first-failure run has already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("heads", [16, 64])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(heads):
    """16 heads run the warp-level kernel, 64 the tensor-memory kernel (both share the scratch).
    Two calls in a row: the scratch keeps the previous call's contents, and both calls must
    agree with the oracle and with the workspace entry point. Neither call may allocate device
    memory: torch's allocator and the driver's free-memory count stay unchanged around them."""
    from bit_mla_kv_qcache_gb300 import binding as b
    w = workloads.Workload("na", 1, 16, 1, 4, 128, random_pages=True, seed=31)
    inp = workloads.make_inputs(w, seq_lens=np.array([1500, 700, 133, 9], np.int32), heads=heads)
    kw = w.config_kwargs()
    cache = gu.gpu_cache(kw, inp)
    gu.write_rows(cache, inp.c, inp.kr, inp.seq_lens, int(inp.seq_lens.max()))
    ql, qr = gu.dev(inp.q_lat), gu.dev(inp.q_rope)
    ref_o, ref_l = cache.decode(ql, qr, w.softmax_scale)
    torch.cuda.synchronize()
    ws_ref = (ref_o.cpu().double().numpy(), ref_l.cpu().double().numpy())

    ocfg, pool, sink, ring = gu.oracle_cache(kw, inp)
    assert oracle.write(ocfg, inp.c, inp.kr, inp.cu, np.zeros(len(inp.seq_lens), np.int32),
                        int(inp.seq_lens.max()), inp.page_table, pool, sink, ring) == 0
    o_or, l_or, _ = oracle.decode(ocfg, inp.q_lat, inp.q_rope, inp.page_table, inp.seq_lens, pool, sink, ring,
                                  w.softmax_scale)

    assert b.noalloc_scratch_bytes() >= b.workspace_bytes(cache.cfg, 4, heads, inp.page_table.shape[1])
    outs = [torch.full_like(ref_o, float("nan")) for _ in range(2)]
    lses = [torch.full_like(ref_l, float("nan")) for _ in range(2)]
    call = lambda k: b.mla_qcache_decode_attn_noalloc(cache.cfg, ql, qr, cache.page_table, cache.seq_lens,
                                                      cache.pool, cache.sink, cache.ring, w.softmax_scale, outs[k],
                                                      lses[k], cache.err)
    call(0)  # warm-up: the first call on a device looks up the scratch address
    torch.cuda.synchronize()
    alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    for k in range(2):
        outs[k].fill_(float("nan"))
        lses[k].fill_(float("nan"))
        call(k)
        torch.cuda.synchronize()
        gu.check_decode(outs[k], lses[k], o_or, l_or, tol=2e-3)
        gu.check_decode(outs[k], lses[k], *ws_ref, tol=2e-3)
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0
    assert cache.error_bits() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    from bit_mla_kv_qcache_gb300 import binding as b
    cfg = b.make_config(4, 128)
    # B*H*splits partials beyond the built-in scratch: rejected before any launch
    B, H, max_pages = 256, 16, 1024
    assert b.workspace_bytes(cfg, B, H, max_pages) > b.noalloc_scratch_bytes()
    i16 = lambda *s: torch.zeros(*s, dtype=torch.int16, device="cuda")
    f32 = lambda *s: torch.zeros(*s, dtype=torch.float32, device="cuda")
    with pytest.raises(b.QCacheError, match="scratch"):
        b.mla_qcache_decode_attn_noalloc(cfg, i16(B, H, 512), i16(B, H, 64),
                                         torch.zeros((B, max_pages), dtype=torch.int32, device="cuda"),
                                         torch.zeros(B, dtype=torch.int32, device="cuda"),
                                         torch.zeros((1, 16), dtype=torch.uint8, device="cuda"), i16(B, 4, 576),
                                         i16(B, 128, 576), 0.1, f32(B, H, 512), f32(B, H),
                                         torch.zeros(1, dtype=torch.int32, device="cuda"))
