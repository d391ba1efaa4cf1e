"""Pins of the oracle's decode attention (QuantMLA page, Figure 8; RAQ-MLA page, Figures 3-4).

References: torch.nn.functional.scaled_dot_product_attention in float64 (a library routine) on
values assembled independently (BF16 rows, or the independent layout decoder's dequantized
codes), scipy's logsumexp, and closed forms (uniform scores, one-hot limit, empty sequence).
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import workloads
from tests import cache_util, layout_decode as ld


def _setup(bits_c, P, S, W, T, B=2, H=16, seed=11):
    w = workloads.Workload("a", B, H, T, bits_c, P, n_sink=S, n_recent=W,
                           clip_q=0.94 if bits_c == 2 else 0.0, random_pages=True, seed=seed)
    seq = np.array([max(0, T - 5 * b) for b in range(B)], np.int32)
    inp = workloads.make_inputs(w, seq_lens=seq)
    cfg = oracle.make_config(**w.config_kwargs())
    pool, sink, ring = cache_util.oracle_prefill(cfg, inp)
    return w, cfg, inp, pool, sink, ring


def _values_independent(cfg, inp, pool, b):
    """[T, 576] values attention must use, assembled without the oracle's reader."""
    T = int(inp.seq_lens[b])
    rows = np.concatenate([inp.c[inp.cu[b]:inp.cu[b + 1]], inp.kr[inp.cu[b]:inp.cu[b + 1]]], axis=1)
    bf = workloads.bf16_value(rows).astype(np.float64)
    P, S, W = cfg.page_size, cfg.n_sink, cfg.n_recent
    V = np.empty((T, 576))
    for t in range(T):
        if t < S or t >= T - W:
            V[t] = bf[t]
        else:
            page = pool[inp.page_table[b, t // P]]
            V[t] = ld.dequant_page(page, cfg.bits_c, P)[t % P]
    return V


def _sdpa_ref(q_lat, q_rope, V, scale):
    q = np.concatenate([workloads.bf16_value(q_lat), workloads.bf16_value(q_rope)], axis=-1).astype(np.float64)
    qt = torch.from_numpy(q)[None, :, None, :]  # [1, H, 1, 576]
    kt = torch.from_numpy(V)[None, None].expand(1, q.shape[0], -1, -1)
    vt = torch.from_numpy(V[:, :512])[None, None].expand(1, q.shape[0], -1, -1)
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)[0, :, 0].numpy()
    scores = scale * (q @ V.T)
    lse = scipy.special.logsumexp(scores, axis=-1)
    return out, lse


@pytest.mark.parametrize("bits_c,P,S,W,T", [(4, 16, 4, 32, 30), (4, 128, 4, 128, 132), (2, 64, 4, 128, 100)])
def test_all_protected_equals_bf16_attention(bits_c, P, S, W, T):
    w, cfg, inp, pool, sink, ring = _setup(bits_c, P, S, W, T)
    out, lse, fl = oracle.decode(cfg, inp.q_lat, inp.q_rope, inp.page_table, inp.seq_lens, pool, sink, ring,
                                 w.softmax_scale)
    assert fl == 0
    for b in range(inp.seq_lens.shape[0]):
        rows = slice(inp.cu[b], inp.cu[b + 1])
        V = workloads.bf16_value(np.concatenate([inp.c[rows], inp.kr[rows]], axis=1)).astype(np.float64)
        ref_o, ref_l = _sdpa_ref(inp.q_lat[b], inp.q_rope[b], V, np.float32(w.softmax_scale))
        np.testing.assert_allclose(out[b], ref_o, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[b], ref_l, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("bits_c,P,S,W,T", [(4, 16, 4, 32, 150), (2, 64, 4, 128, 400), (4, 32, 0, 32, 97),
                                           (4, 128, 4, 128, 700)])
def test_mixed_cache_equals_attention_over_dequantized_values(bits_c, P, S, W, T):
    w, cfg, inp, pool, sink, ring = _setup(bits_c, P, S, W, T)
    out, lse, fl = oracle.decode(cfg, inp.q_lat, inp.q_rope, inp.page_table, inp.seq_lens, pool, sink, ring,
                                 w.softmax_scale)
    assert fl == 0
    for b in range(inp.seq_lens.shape[0]):
        V = _values_independent(cfg, inp, pool, b)
        ref_o, ref_l = _sdpa_ref(inp.q_lat[b], inp.q_rope[b], V, np.float32(w.softmax_scale))
        np.testing.assert_allclose(out[b], ref_o, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse[b], ref_l, rtol=1e-12, atol=1e-12)


def test_zero_query_gives_mean_and_log_count():
    w, cfg, inp, pool, sink, ring = _setup(4, 16, 4, 32, 77, B=1)
    ql = np.zeros_like(inp.q_lat)
    qr = np.zeros_like(inp.q_rope)
    out, lse, _ = oracle.decode(cfg, ql, qr, inp.page_table, inp.seq_lens, pool, sink, ring, w.softmax_scale)
    V = _values_independent(cfg, inp, pool, 0)
    T = int(inp.seq_lens[0])
    np.testing.assert_allclose(out[0], np.broadcast_to(V[:, :512].mean(0), out[0].shape), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse[0], math.log(T), rtol=0, atol=1e-12)


def test_one_hot_limit_selects_best_token():
    w, cfg, inp, pool, sink, ring = _setup(4, 16, 4, 32, 90, B=1, H=16)
    V = _values_independent(cfg, inp, pool, 0)
    # queries = BF16 copies of one token's values: with a huge scale the softmax is one-hot on
    # the token with the largest score (checked to be unique)
    ql = np.repeat(workloads.bf16_bits(V[40:41, :512].astype(np.float32)), 16, 0)[None]
    qr = np.repeat(workloads.bf16_bits(V[40:41, 512:].astype(np.float32)), 16, 0)[None]
    out, lse, _ = oracle.decode(cfg, ql, qr, inp.page_table, inp.seq_lens, pool, sink, ring, 1e4)
    q = np.concatenate([workloads.bf16_value(ql[0, 0]), workloads.bf16_value(qr[0, 0])]).astype(np.float64)
    s = V @ q
    best = int(np.argmax(s))
    assert np.sort(s)[-1] - np.sort(s)[-2] > 1e-2
    np.testing.assert_allclose(out[0, 0], V[best, :512], rtol=0, atol=1e-9)


def test_empty_sequence():
    w, cfg, inp, pool, sink, ring = _setup(4, 16, 4, 32, 5, B=2)
    seq = np.array([0, 5], np.int32)
    out, lse, fl = oracle.decode(cfg, inp.q_lat, inp.q_rope, inp.page_table, seq, pool, sink, ring,
                                 w.softmax_scale)
    assert fl == 0
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))
