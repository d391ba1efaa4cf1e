"""The writer over transformed rows (RAQ-MLA page, Figure 4 and appendix Table 9) on the GPU:
the standalone transform, and the fused writer's page bytes, BF16 rows and lengths, bit-exact
with the oracle's transform followed by its writer."""
import numpy as np
import pytest
import torch

import bit_mla_kv_qcache_gb300 as q
import oracle
import workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _mat(d, seed, scale=None):
    rng = np.random.default_rng(seed)
    a = (rng.standard_normal((d, d)) * (scale if scale is not None else d ** -0.5)).astype(np.float32)
    return torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


A_C, A_R = _mat(512, 1), _mat(64, 2)


@pytest.mark.parametrize("d,n", [(512, 1), (512, 300), (64, 77), (64, 1)])
def test_standalone_transform_bit_exact(d, n):
    rng = np.random.default_rng(d + n)
    x = torch.from_numpy(rng.standard_normal((n, d)).astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    a = A_C if d == 512 else A_R
    out = torch.empty((n, d), dtype=torch.int16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q.mla_qcache_row_transform(gu.dev(x), gu.dev(a), out, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _, want = oracle.row_transform(x.view(np.uint16), a)
    assert np.array_equal(out.cpu().numpy().view(np.uint16), want)


def _wl(bits_c, P, S=4, W=128):
    return workloads.Workload("x", 1, 16, 1, bits_c, P, n_sink=S, n_recent=W,
                              clip_q=0.94 if bits_c == 2 else 0.0,
                              latent_dist="student_t5" if bits_c == 2 else "normal",
                              n_outliers=8 if bits_c == 2 else 4, outlier_scale=20.0 if bits_c == 2 else 10.0,
                              random_pages=True, seed=13)


def _write_xf(cache, c, kr, counts, max_new, a_c, a_r, nxt=None):
    cu = np.zeros(len(counts) + 1, np.int32)
    cu[1:] = np.cumsum(counts)
    q.mla_qcache_write_transformed(cache.cfg, gu.dev(c), gu.dev(kr), gu.dev(cu), cache.seq_lens, max_new,
                                   cache.page_table, cache.pool, cache.sink, cache.ring, cache.err,
                                   a_c=None if a_c is None else gu.dev(a_c), a_r=None if a_r is None else gu.dev(a_r),
                                   seq_lens_next=nxt)
    if nxt is None:
        q.mla_qcache_advance(gu.dev(cu), cache.seq_lens)


CASES = [  # bits_c, P, S, W, lengths, (a_c, a_r)
    (4, 128, 4, 128, [1, 127, 128, 129, 300], (True, True)),
    (4, 128, 4, 128, [260, 5], (True, False)),
    (4, 64, 4, 128, [200, 64], (False, True)),
    (2, 64, 4, 128, [64, 63, 700, 131], (True, True)),
    (2, 32, 0, 32, [65, 33, 32, 31], (True, True)),
]


@pytest.mark.parametrize("bits_c,P,S,W,lens,which", CASES)
def test_fused_writer_bit_exact(bits_c, P, S, W, lens, which):
    """Prefill (one launch, or page fills first for long chunks), then decode steps across page
    fills, each checked against the oracle's transform + writer."""
    w = _wl(bits_c, P, S, W)
    lens = np.array(lens, np.int32)
    inp = workloads.make_inputs(w, seq_lens=lens, extra_pages=2)
    kw = w.config_kwargs()
    a_c = A_C if which[0] else None
    a_r = A_R if which[1] else None
    cache = gu.gpu_cache(kw, inp)
    mx = int(lens.max())
    _write_xf(cache, inp.c, inp.kr, lens, mx, a_c, a_r)
    cfg, pool, sink, ring = gu.oracle_cache(kw, inp)
    B = len(lens)
    assert oracle.write_transformed(cfg, inp.c, inp.kr, inp.cu, np.zeros(B, np.int32), mx, inp.page_table, pool,
                                    sink, ring, a_c=a_c, a_r=a_r) == 0
    gu.assert_cache_equal(cache, pool, sink, ring)
    rng = np.random.default_rng(5)
    cur = lens.copy()
    for step in range(P + 2):
        c1, k1 = workloads.draw_tokens(rng, B, w.latent_dist, inp.outliers, w.outlier_scale)
        _write_xf(cache, c1, k1, np.ones(B, np.int32), 1, a_c, a_r)
        assert oracle.write_transformed(cfg, c1, k1, np.arange(B + 1, dtype=np.int32), cur, 1, inp.page_table, pool,
                                        sink, ring, a_c=a_c, a_r=a_r) == 0
        cur = cur + 1
    gu.assert_cache_equal(cache, pool, sink, ring)
    assert np.array_equal(cache.seq_lens.cpu().numpy(), cur)
    assert cache.error_bits() == 0


def test_fused_equals_standalone_then_write_and_advances_lengths():
    """Transforming in the writer (with the length update) stores the bytes that the standalone
    transform followed by the plain writer stores."""
    w = _wl(4, 128)
    lens = np.array([700, 131, 9], np.int32)
    inp = workloads.make_inputs(w, seq_lens=lens, extra_pages=1)
    kw = w.config_kwargs()
    a, b = gu.gpu_cache(kw, inp), gu.gpu_cache(kw, inp)
    nxt = torch.full_like(a.seq_lens, -1)
    _write_xf(a, inp.c, inp.kr, lens, int(lens.max()), A_C, A_R, nxt=nxt)
    c_t = torch.empty((inp.c.shape[0], 512), dtype=torch.int16, device="cuda")
    k_t = torch.empty((inp.c.shape[0], 64), dtype=torch.int16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q.mla_qcache_row_transform(gu.dev(inp.c), gu.dev(A_C), c_t, err)
    q.mla_qcache_row_transform(gu.dev(inp.kr), gu.dev(A_R), k_t, err)
    b.write(c_t, k_t, gu.dev(inp.cu), int(lens.max()))
    torch.cuda.synchronize()
    assert torch.equal(a.pool, b.pool) and torch.equal(a.sink, b.sink) and torch.equal(a.ring, b.ring)
    assert nxt.cpu().tolist() == lens.tolist() and a.seq_lens.cpu().tolist() == [0, 0, 0]


def test_no_transform_is_the_plain_writer():
    w = _wl(2, 64)
    lens = np.array([300, 70], np.int32)
    inp = workloads.make_inputs(w, seq_lens=lens)
    kw = w.config_kwargs()
    a, b = gu.gpu_cache(kw, inp), gu.gpu_cache(kw, inp)
    _write_xf(a, inp.c, inp.kr, lens, 300, None, None)
    gu.write_rows(b, inp.c, inp.kr, lens, 300)
    torch.cuda.synchronize()
    assert torch.equal(a.pool, b.pool) and torch.equal(a.ring, b.ring) and torch.equal(a.sink, b.sink)


def test_overflowing_transform_sets_nonfinite_bit():
    w = _wl(4, 128)
    lens = np.array([3], np.int32)
    inp = workloads.make_inputs(w, seq_lens=lens)
    cache = gu.gpu_cache(w.config_kwargs(), inp)
    huge = _mat(512, 9, scale=3e37)
    _write_xf(cache, inp.c, inp.kr, lens, 3, huge, None)
    torch.cuda.synchronize()
    assert cache.error_bits() & q.DEV_NONFINITE
