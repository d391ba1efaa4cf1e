"""Writer parity on the GPU: packed pages, metadata, sink and ring are bit-exact with the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _wl(bits_c, P, S=4, W=128, dist=None, random_pages=True, seed=3, clip=None):
    return workloads.Workload("w", 1, 16, 1, bits_c, P, n_sink=S, n_recent=W,
                              clip_q=(0.94 if bits_c == 2 else 0.0) if clip is None else clip,
                              latent_dist=dist or ("student_t5" if bits_c == 2 else "normal"),
                              n_outliers=8 if bits_c == 2 else 4, outlier_scale=20.0 if bits_c == 2 else 10.0,
                              random_pages=random_pages, seed=seed)


CASES = [  # bits_c, P, S, W, lengths
    (4, 128, 4, 128, [1024]),
    (4, 128, 4, 128, [1, 5, 127, 128, 129, 300]),
    (2, 64, 4, 128, [64, 63, 700, 131]),
    (2, 32, 0, 32, [65, 33, 32, 31]),
    (4, 32, 16, 64, [200, 3]),
    (2, 128, 4, 256, [1000]),
]


@pytest.mark.parametrize("bits_c,P,S,W,lens", CASES)
def test_bulk_prefill_bit_exact(bits_c, P, S, W, lens):
    w = _wl(bits_c, P, S, W)
    inp = workloads.make_inputs(w, seq_lens=np.array(lens, np.int32))
    kw = w.config_kwargs()
    cache = gu.gpu_cache(kw, inp)
    gu.write_rows(cache, inp.c, inp.kr, inp.seq_lens, int(inp.seq_lens.max()))
    cfg, pool, sink, ring = gu.oracle_cache(kw, inp)
    assert oracle.write(cfg, inp.c, inp.kr, inp.cu, np.zeros(len(lens), np.int32), int(inp.seq_lens.max()),
                        inp.page_table, pool, sink, ring) == 0
    gu.assert_cache_equal(cache, pool, sink, ring)
    assert cache.error_bits() == 0


@pytest.mark.parametrize("bits_c,P,S,W", [(4, 32, 4, 32), (2, 64, 4, 128), (4, 128, 4, 128)])
def test_decode_steps_fill_pages_and_evict(bits_c, P, S, W):
    """Prefill, then one token per sequence per call across page fills and window evictions
    (the single-launch writer path), checked after every call."""
    w = _wl(bits_c, P, S, W)
    lens = np.array([P - 3, 2 * P + 1, 5], np.int32)
    inp = workloads.make_inputs(w, seq_lens=lens, extra_pages=3)
    kw = w.config_kwargs()
    cache = gu.gpu_cache(kw, inp)
    gu.write_rows(cache, inp.c, inp.kr, lens, int(lens.max()))
    cfg, pool, sink, ring = gu.oracle_cache(kw, inp)
    assert oracle.write(cfg, inp.c, inp.kr, inp.cu, np.zeros(3, np.int32), int(lens.max()), inp.page_table, pool,
                        sink, ring) == 0
    rng = np.random.default_rng(9)
    cur = lens.copy()
    for step in range(min(2 * P + 7, 70)):
        c1, k1 = workloads.draw_tokens(rng, 3, w.latent_dist, inp.outliers, w.outlier_scale)
        gu.write_rows(cache, c1, k1, np.ones(3, np.int32), 1)
        assert oracle.write(cfg, c1, k1, np.arange(4, dtype=np.int32), cur, 1, inp.page_table, pool, sink, ring) == 0
        cur = cur + 1
        if step % 9 == 0 or (cur % P == 0).any():
            gu.assert_cache_equal(cache, pool, sink, ring)
    gu.assert_cache_equal(cache, pool, sink, ring)
    assert np.array_equal(cache.seq_lens.cpu().numpy(), cur)


def test_chunked_prefill_two_launch_path():
    """Chunks larger than W - P + 1 take the page-fill-first path; result equals bulk."""
    w = _wl(4, 64, 4, 128)
    lens = np.array([500, 260], np.int32)
    inp = workloads.make_inputs(w, seq_lens=lens)
    kw = w.config_kwargs()
    cache = gu.gpu_cache(kw, inp)
    done = np.zeros(2, np.int32)
    for chunk in [100, 90, 200, 200]:
        n = np.minimum(chunk, lens - done)
        rows_c = np.concatenate([inp.c[inp.cu[b] + done[b]: inp.cu[b] + done[b] + n[b]] for b in range(2)])
        rows_k = np.concatenate([inp.kr[inp.cu[b] + done[b]: inp.cu[b] + done[b] + n[b]] for b in range(2)])
        gu.write_rows(cache, rows_c, rows_k, n, chunk)
        done += n
    cfg, pool, sink, ring = gu.oracle_cache(kw, inp)
    assert oracle.write(cfg, inp.c, inp.kr, inp.cu, np.zeros(2, np.int32), 500, inp.page_table, pool, sink, ring) == 0
    gu.assert_cache_equal(cache, pool, sink, ring)


def test_full_size_prefill_v2lite_shape():
    """The 32 x 8192-token C4R4 cache the benchmark decodes over, bit-exact."""
    w = workloads.WORKLOADS["v2lite_c4r4_b32_h16_t8k"]
    inp = workloads.make_inputs(w, extra_pages=1)
    kw = w.config_kwargs()
    cache = gu.gpu_cache(kw, inp)
    gu.write_rows(cache, inp.c, inp.kr, inp.seq_lens, int(inp.seq_lens.max()))
    cfg, pool, sink, ring = gu.oracle_cache(kw, inp)
    assert oracle.write(cfg, inp.c, inp.kr, inp.cu, np.zeros(w.batch, np.int32), w.seq_len, inp.page_table, pool,
                        sink, ring) == 0
    gu.assert_cache_equal(cache, pool, sink, ring)
    assert cache.error_bits() == 0


def test_device_error_bits():
    w = _wl(4, 32, 4, 64)
    lens = np.array([40], np.int32)
    inp = workloads.make_inputs(w, seq_lens=lens)
    kw = w.config_kwargs()
    pt = inp.page_table.copy()
    pt[0, 1] = 10 ** 6  # out of the pool
    inp2 = workloads.CacheInputs(**{**inp.__dict__, "page_table": pt})
    cache = gu.gpu_cache(kw, inp2)
    gu.write_rows(cache, inp.c, inp.kr, lens, 40)
    torch.cuda.synchronize()
    assert cache.error_bits() & 1  # bad page
    # overflow of the page table
    cache2 = gu.gpu_cache(kw, inp)
    cache2.seq_lens.fill_(inp.page_table.shape[1] * 32 - 2)
    gu.write_rows(cache2, inp.c[:5], inp.kr[:5], np.array([5], np.int32), 5)
    torch.cuda.synchronize()
    assert cache2.error_bits() & 2


def test_advance_lengths():
    """mla_qcache_advance adds each sequence's new-row count to its length (one kernel)."""
    import bit_mla_kv_qcache_gb300 as q
    lens = torch.tensor([0, 5, 130, 7, 1 << 20], dtype=torch.int32, device="cuda")
    cu = torch.tensor([0, 1, 1, 4, 10, 11], dtype=torch.int32, device="cuda")
    q.mla_qcache_advance(cu, lens)
    torch.cuda.synchronize()
    assert lens.cpu().tolist() == [1, 5, 133, 13, (1 << 20) + 1]


@pytest.mark.parametrize("bits_c,P,S,W,lens", [(4, 128, 4, 128, [1, 5, 127, 128, 129, 300]),
                                              (2, 64, 4, 128, [64, 63, 700, 131]),
                                              (2, 32, 0, 32, [65, 33, 32, 0])])
def test_write_advance_equals_write_then_advance(bits_c, P, S, W, lens):
    """The fused entry stores the same cache bytes as mla_qcache_write and the lengths that
    mla_qcache_advance would produce, into the second length array (prefill, then decode steps
    that cross page fills, and a call without rows)."""
    import bit_mla_kv_qcache_gb300 as q
    w = _wl(bits_c, P, S, W)
    lens = np.array(lens, np.int32)
    inp = workloads.make_inputs(w, seq_lens=lens, extra_pages=3)
    kw = w.config_kwargs()
    a, b = gu.gpu_cache(kw, inp), gu.gpu_cache(kw, inp)
    c, kr, cu = gu.dev(inp.c), gu.dev(inp.kr), gu.dev(inp.cu)
    mx = max(1, int(lens.max()))
    a.write(c, kr, cu, mx)  # write + advance
    nxt = torch.full_like(b.seq_lens, -7)
    q.mla_qcache_write_advance(b.cfg, c, kr, cu, b.seq_lens, nxt, mx, b.page_table, b.pool, b.sink, b.ring, b.err)
    torch.cuda.synchronize()
    assert torch.equal(a.pool, b.pool) and torch.equal(a.sink, b.sink) and torch.equal(a.ring, b.ring)
    assert torch.equal(b.seq_lens.cpu(), torch.zeros(len(lens), dtype=torch.int32))  # input lengths untouched
    assert nxt.cpu().tolist() == a.seq_lens.cpu().tolist() == lens.tolist()
    rng = np.random.default_rng(4)
    cur, alt = nxt, b.seq_lens
    B = len(lens)
    cu1 = torch.arange(B + 1, dtype=torch.int32, device="cuda")
    for step in range(P + 3):
        c1, k1 = workloads.draw_tokens(rng, B, w.latent_dist, inp.outliers, w.outlier_scale)
        d_c, d_k = gu.dev(c1), gu.dev(k1)
        a.write(d_c, d_k, cu1, 1)
        q.mla_qcache_write_advance(b.cfg, d_c, d_k, cu1, cur, alt, 1, b.page_table, b.pool, b.sink, b.ring, b.err)
        cur, alt = alt, cur
    torch.cuda.synchronize()
    assert torch.equal(a.pool, b.pool) and torch.equal(a.sink, b.sink) and torch.equal(a.ring, b.ring)
    assert cur.cpu().tolist() == a.seq_lens.cpu().tolist()
    # no rows: the lengths are copied
    empty_c = torch.zeros((0, 512), dtype=torch.int16, device="cuda")
    empty_k = torch.zeros((0, 64), dtype=torch.int16, device="cuda")
    q.mla_qcache_write_advance(b.cfg, empty_c, empty_k, torch.zeros(B + 1, dtype=torch.int32, device="cuda"),
                               cur, alt, 1, b.page_table, b.pool, b.sink, b.ring, b.err)
    torch.cuda.synchronize()
    assert alt.cpu().tolist() == cur.cpu().tolist()
    assert a.error_bits() == 0 and b.error_bits() == 0
