"""Decode of a pending write (mla_qcache_decode_attn_pending) on the GPU.

A decode step's write needs to finish before the next step's decode only: because P <= W,
this step's decode reads nothing the write changes except the new rows themselves, which it
takes from the write's inputs. These tests run the writer (with the length update) on a side
stream concurrently with the pending decode, across page fills and window evictions, and check
every step against the oracle (write, then decode): the cache bit-exact, O and LSE within the
decode tolerance; the pending decode also matches the decode after the write.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _wl(bits_c, P, S=4, W=128, seed=5):
    return workloads.Workload("pend", 1, 16, 1, bits_c, P, n_sink=S, n_recent=W,
                              clip_q=0.94 if bits_c == 2 else 0.0,
                              latent_dist="student_t5" if bits_c == 2 else "normal",
                              n_outliers=8 if bits_c == 2 else 4, outlier_scale=20.0 if bits_c == 2 else 10.0,
                              random_pages=True, seed=seed)


@pytest.mark.parametrize("bits_c,P,S,W,heads,steps", [
    (4, 128, 4, 128, 16, 6),   # headline layout: one pending row per sequence
    (2, 64, 4, 128, 16, 70),   # INT2 + clip: page fills every 64 steps, evictions every step
    (4, 32, 4, 32, 16, 40),    # P = W: the page of the evicted token fills exactly W steps earlier
    (4, 128, 4, 128, 64, 5),   # 64-head blocks: packed shares on the tensor-memory kernel
])
def test_pending_decode_with_concurrent_writer(bits_c, P, S, W, heads, steps):
    import bit_mla_kv_qcache_gb300 as q
    w = _wl(bits_c, P, S, W)
    # lengths around the interesting boundaries: empty, inside the sink, all-protected, a page
    # about to fill, a long sequence
    lens = np.array([0, 2, S + W - 1, 3 * P - 1, 1000], np.int32)
    B = len(lens)
    inp = workloads.make_inputs(w, seq_lens=lens, extra_pages=steps // P + 2, heads=heads)
    kw = w.config_kwargs()
    cache = gu.gpu_cache(kw, inp)
    gu.write_rows(cache, inp.c, inp.kr, lens, max(1, int(lens.max())))
    ocfg, pool, sink, ring = gu.oracle_cache(kw, inp)
    assert oracle.write(ocfg, inp.c, inp.kr, inp.cu, np.zeros(B, np.int32), max(1, int(lens.max())), inp.page_table,
                        pool, sink, ring) == 0
    torch.cuda.synchronize()
    ql, qr = gu.dev(inp.q_lat), gu.dev(inp.q_rope)
    cu1 = torch.arange(B + 1, dtype=torch.int32, device="cuda")
    lens_next = torch.empty_like(cache.seq_lens)
    ws = cache.workspace(heads)
    ws2 = torch.zeros_like(ws)
    out = torch.empty((B, heads, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, heads), dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    rng = np.random.default_rng(17)
    cur = lens.copy()
    for step in range(steps):
        c1, k1 = workloads.draw_tokens(rng, B, w.latent_dist, inp.outliers, w.outlier_scale)
        d_c, d_k = gu.dev(c1), gu.dev(k1)
        torch.cuda.synchronize()
        # fork: the writer on the side stream, the pending decode on the main stream
        side.wait_stream(main)
        with torch.cuda.stream(side):
            q.mla_qcache_write_advance(cache.cfg, d_c, d_k, cu1, cache.seq_lens, lens_next, 1, cache.page_table,
                                       cache.pool, cache.sink, cache.ring, cache.err, side)
        q.mla_qcache_decode_attn_pending(cache.cfg, ql, qr, cache.page_table, cache.seq_lens, d_c, d_k, cu1, 1,
                                         cache.pool, cache.sink, cache.ring, w.softmax_scale, out, lse, ws, cache.err)
        main.wait_stream(side)  # join before anything reads the written cache
        torch.cuda.synchronize()
        cache.seq_lens.copy_(lens_next)
        # oracle: write the step's rows, then decode
        cu = np.arange(B + 1, dtype=np.int32)
        assert oracle.write(ocfg, c1, k1, cu, cur, 1, inp.page_table, pool, sink, ring) == 0
        cur = cur + 1
        o_ref, l_ref, fl = oracle.decode(ocfg, inp.q_lat, inp.q_rope, inp.page_table, cur, pool, sink, ring,
                                         w.softmax_scale)
        assert fl == 0
        gu.check_decode(out, lse, o_ref, l_ref, tol=2e-3)
        if step % 8 == 0 or step == steps - 1:
            gu.assert_cache_equal(cache, pool, sink, ring)
            # the decode after the write sees exactly what the pending decode saw
            o2, l2 = torch.empty_like(out), torch.empty_like(lse)
            q.mla_qcache_decode_attn(cache.cfg, ql, qr, cache.page_table, cache.seq_lens, cache.pool, cache.sink,
                                     cache.ring, w.softmax_scale, o2, l2, ws2, cache.err)
            torch.cuda.synchronize()
            assert torch.equal(o2, out) and torch.equal(l2, lse)
    assert np.array_equal(cache.seq_lens.cpu().numpy(), cur)
    assert cache.error_bits() == 0


def test_pending_rows_beyond_max_new_set_the_rows_bit():
    """A sequence whose pending row count exceeds max_new is decoded without its pending rows and
    reports MLA_QCACHE_DEV_ROWS."""
    import bit_mla_kv_qcache_gb300 as q
    w = _wl(4, 32, 4, 64)
    lens = np.array([100, 40], np.int32)
    inp = workloads.make_inputs(w, seq_lens=lens, extra_pages=2)
    cache = gu.gpu_cache(w.config_kwargs(), inp)
    gu.write_rows(cache, inp.c, inp.kr, lens, int(lens.max()))
    ql, qr = gu.dev(inp.q_lat), gu.dev(inp.q_rope)
    c1, k1 = workloads.draw_tokens(np.random.default_rng(1), 3, w.latent_dist, inp.outliers, w.outlier_scale)
    cu = torch.tensor([0, 1, 3], dtype=torch.int32, device="cuda")  # sequence 1 has 2 rows > max_new = 1
    out = torch.empty((2, 16, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((2, 16), dtype=torch.float32, device="cuda")
    q.mla_qcache_decode_attn_pending(cache.cfg, ql, qr, cache.page_table, cache.seq_lens, gu.dev(c1), gu.dev(k1), cu,
                                     1, cache.pool, cache.sink, cache.ring, w.softmax_scale, out, lse,
                                     cache.workspace(16), cache.err)
    torch.cuda.synchronize()
    assert cache.error_bits() & q.DEV_ROWS
    o_ref, l_ref = cache.decode(ql, qr, w.softmax_scale)  # sequence 1 as cached
    torch.cuda.synchronize()
    assert torch.equal(out[1], o_ref[1]) and torch.equal(lse[1], l_ref[1])
