"""Full-size parity for the other benchmark configurations (GPU through the C ABI vs the oracle).

Each cache is built by the GPU writer and checked byte for byte against the oracle's writer;
decode outputs are checked on a sample of sequences / heads that the fp64 oracle computes in
seconds (every row of the sample is compared, tolerance as in test_gpu_decode.py).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _prefill_both(w, inp):
    kw = w.config_kwargs()
    cache = gu.gpu_cache(kw, inp)
    gu.write_rows(cache, inp.c, inp.kr, inp.seq_lens, int(inp.seq_lens.max()))
    cfg, pool, sink, ring = gu.oracle_cache(kw, inp)
    B = inp.seq_lens.shape[0]
    assert oracle.write(cfg, inp.c, inp.kr, inp.cu, np.zeros(B, np.int32), int(inp.seq_lens.max()), inp.page_table,
                        pool, sink, ring) == 0
    gu.assert_cache_equal(cache, pool, sink, ring)
    return cache, cfg, pool, sink, ring


def _oracle_sample(cfg, inp, pool, sink, ring, seq_lens, seqs, heads, scale):
    seqs = np.asarray(seqs)
    return oracle.decode(cfg, inp.q_lat[seqs][:, heads], inp.q_rope[seqs][:, heads], inp.page_table[seqs],
                         np.ascontiguousarray(seq_lens[seqs]), pool, np.ascontiguousarray(sink[seqs]),
                         np.ascontiguousarray(ring[seqs]), scale)


def _check_sample(out, lse, seqs, heads, o_ref, l_ref):
    o = out.cpu()[seqs][:, heads]
    l = lse.cpu()[seqs][:, heads]
    return gu.check_decode(o, l, o_ref, l_ref, TOL)


def test_wide_c2r4_h128_t32k():
    w = workloads.WORKLOADS["wide_c2r4_b8_h128_t32k"]
    inp = workloads.make_inputs(w)
    cache, cfg, pool, sink, ring = _prefill_both(w, inp)
    out, lse = cache.decode(gu.dev(inp.q_lat), gu.dev(inp.q_rope), w.softmax_scale)
    torch.cuda.synchronize()
    assert cache.error_bits() == 0
    seqs, heads = [0, 5], list(range(0, 128, 8))
    o_ref, l_ref, fl = _oracle_sample(cfg, inp, pool, sink, ring, inp.seq_lens, seqs, heads, w.softmax_scale)
    assert fl == 0
    _check_sample(out, lse, seqs, heads, o_ref, l_ref)


def test_long_c4r4_h128_t128k():
    w = workloads.WORKLOADS["long_c4r4_b1_h128_t128k"]
    inp = workloads.make_inputs(w)
    cache, cfg, pool, sink, ring = _prefill_both(w, inp)
    out, lse = cache.decode(gu.dev(inp.q_lat), gu.dev(inp.q_rope), w.softmax_scale)
    torch.cuda.synchronize()
    assert cache.error_bits() == 0
    seqs, heads = [0], list(range(3, 128, 6))
    o_ref, l_ref, fl = _oracle_sample(cfg, inp, pool, sink, ring, inp.seq_lens, seqs, heads, w.softmax_scale)
    assert fl == 0
    _check_sample(out, lse, seqs, heads, o_ref, l_ref)


def test_ragged_serving_256_steps():
    """64 ragged sequences, random page table, C2R4: 256 steps of write-one-token + decode.
    The pool stays bit-exact across page fills and window evictions; decode is checked at
    sampled steps on sampled sequences."""
    w = workloads.WORKLOADS["ragged_c2r4_b64_h16_serve"]
    inp = workloads.make_inputs(w, extra_pages=w.steps // w.page_size + 1)
    cache, cfg, pool, sink, ring = _prefill_both(w, inp)
    rng = np.random.default_rng(4242)
    cur = inp.seq_lens.copy()
    B = w.batch
    seqs = [0, 13, 31, 63]
    check_at = {0, 1, 63, 64, 128, 200, w.steps - 1}
    ql, qr = gu.dev(inp.q_lat), gu.dev(inp.q_rope)
    ones = np.ones(B, np.int32)
    for step in range(w.steps):
        c1, k1 = workloads.draw_tokens(rng, B, w.latent_dist, inp.outliers, w.outlier_scale)
        gu.write_rows(cache, c1, k1, ones, 1)
        assert oracle.write(cfg, c1, k1, np.arange(B + 1, dtype=np.int32), cur, 1, inp.page_table, pool, sink,
                            ring) == 0
        cur = cur + 1
        out, lse = cache.decode(ql, qr, w.softmax_scale)
        if step in check_at:
            torch.cuda.synchronize()
            o_ref, l_ref, fl = _oracle_sample(cfg, inp, pool, sink, ring, cur, seqs, list(range(16)), w.softmax_scale)
            assert fl == 0
            _check_sample(out, lse, seqs, list(range(16)), o_ref, l_ref)
    gu.assert_cache_equal(cache, pool, sink, ring)
    assert np.array_equal(cache.seq_lens.cpu().numpy(), cur)
    assert cache.error_bits() == 0
