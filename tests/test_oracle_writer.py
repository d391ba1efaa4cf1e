"""Pins of the oracle's fused writer (QuantMLA page, appendix Figure 8; RAQ-MLA page, Table 5).

Checked against the independent layout decoder, the (separately pinned) quantizer applied to
the token's values, and the retention rules: BF16 rows kept unchanged for the sink and the
recent ring, k_R quantized per channel exactly when a page fills.
"""
import numpy as np
import pytest

import oracle
import workloads
from tests import cache_util, layout_decode as ld


def _small(bits_c, P, S, W, T, B=2, random_pages=True, clip=None):
    w = workloads.Workload("t", B, 16, T, bits_c, P, n_sink=S, n_recent=W,
                           clip_q=(0.94 if bits_c == 2 else 0.0) if clip is None else clip,
                           latent_dist="student_t5" if bits_c == 2 else "normal",
                           random_pages=random_pages, seed=7)
    seq = np.array([T - 3 * b for b in range(B)], np.int32)
    inp = workloads.make_inputs(w, seq_lens=seq)
    return oracle.make_config(**w.config_kwargs()), inp


def _clip(c, q):
    if q <= 0:
        return c
    a = np.sort(np.abs(c))
    tau = a[int(np.ceil(np.float64(np.float32(q)) * 512)) - 1]
    return np.clip(c, -tau, tau)


@pytest.mark.parametrize("bits_c,P,S,W,T", [(4, 16, 4, 32, 70), (2, 64, 4, 128, 200), (4, 128, 4, 128, 300),
                                           (2, 32, 0, 64, 97)])
def test_writer_bytes_against_definition(bits_c, P, S, W, T):
    cfg, inp = _small(bits_c, P, S, W, T)
    pool, sink, ring = cache_util.oracle_prefill(cfg, inp)
    for b in range(inp.seq_lens.shape[0]):
        Tb = int(inp.seq_lens[b])
        rows = slice(inp.cu[b], inp.cu[b + 1])
        cb = workloads.bf16_value(inp.c[rows]).astype(np.float64)
        kb = workloads.bf16_value(inp.kr[rows]).astype(np.float64)
        for p in range((Tb + P - 1) // P):
            page = pool[inp.page_table[b, p]]
            d = ld.decode_page(page, bits_c, P)
            for tp in range(min(P, Tb - p * P)):
                t = p * P + tp
                cc = _clip(cb[t], cfg.clip_q)
                for g in range(4):
                    codes, sb, mb, fl = oracle.quantize(cc[128 * g:128 * (g + 1)], bits_c)
                    assert list(d["latent"][tp, 128 * g:128 * (g + 1)]) == list(codes)
                    assert d["lat_scale"][tp, g] == oracle.f16_to_double(sb)
                    assert d["lat_min"][tp, g] == oracle.f16_to_double(mb)
            full = (p + 1) * P <= Tb
            if full:
                for j in range(0, 64, 5):
                    codes, sb, mb, fl = oracle.quantize(kb[p * P:(p + 1) * P, j], 4)
                    assert list(d["rope"][:, j]) == list(codes)
                    assert d["rope_scale"][j] == oracle.f16_to_double(sb)
            else:  # k_R of a page that has not filled is not written yet
                off = P * 64 * bits_c
                assert not page[off:off + 32 * P].any()
                assert not page[P * (64 * bits_c + 48):].any()
        # BF16 retention: sink rows and the last W rows, bit-for-bit
        full_rows = np.concatenate([inp.c[rows], inp.kr[rows]], axis=1)
        for t in range(min(S, Tb)):
            assert np.array_equal(sink[b, t], full_rows[t])
        for t in range(max(0, Tb - W), Tb):
            assert np.array_equal(ring[b, t % W], full_rows[t])


@pytest.mark.parametrize("chunk", [1, 5, 64])
def test_incremental_equals_bulk(chunk):
    cfg, inp = _small(2, 32, 4, 64, 150)
    a = cache_util.oracle_prefill(cfg, inp)
    b = cache_util.oracle_prefill(cfg, inp, chunk=chunk)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_eviction_switches_to_existing_packed_copy():
    """Figure 8: a token leaving the recent window is read from the packed copy written at its
    arrival; no re-quantization happens (its bytes do not change)."""
    cfg, inp = _small(4, 16, 4, 32, 64, B=1)
    pool, sink, ring = cache_util.oracle_prefill(cfg, inp)
    T = int(inp.seq_lens[0])
    t_ev = T - cfg.n_recent  # next write evicts this token from the window
    v_before, st = oracle.token_values(cfg, 0, t_ev, T, inp.page_table, pool, sink, ring)
    assert st == 1
    page_before = pool[inp.page_table[0, t_ev // cfg.page_size]].copy()
    rng = np.random.default_rng(3)
    c1, k1 = workloads.draw_tokens(rng, 1, "normal", np.zeros(0, int), 1.0)
    fl = oracle.write(cfg, c1, k1, np.array([0, 1], np.int32), np.array([T], np.int32), 1, inp.page_table,
                      pool, sink, ring)
    assert fl == 0
    v_after, st = oracle.token_values(cfg, 0, t_ev, T + 1, inp.page_table, pool, sink, ring)
    assert st == 0
    d = ld.dequant_page(page_before, cfg.bits_c, cfg.page_size)
    assert np.array_equal(v_after, d[t_ev % cfg.page_size])
    # its latent codes/metadata in the page are unchanged by the later write
    after = pool[inp.page_table[0, t_ev // cfg.page_size]]
    P, bc = cfg.page_size, cfg.bits_c
    assert np.array_equal(ld.decode_page(after, bc, P)["latent"][t_ev % P],
                          ld.decode_page(page_before, bc, P)["latent"][t_ev % P])


def test_error_flags():
    cfg, inp = _small(4, 16, 4, 32, 40, B=1)
    B = 1
    pool, sink, ring = cache_util.empty_cache(cfg, B, inp.n_pages)
    pt = inp.page_table.copy()
    pt[0, 1] = 10 ** 6
    fl = oracle.write(cfg, inp.c, inp.kr, inp.cu, np.zeros(1, np.int32), 64, pt, pool, sink, ring)
    assert fl & oracle.ERR_BAD_PAGE
    fl = oracle.write(cfg, inp.c, inp.kr, np.array([0, 39], np.int32), np.zeros(1, np.int32), 64, inp.page_table,
                      pool, sink, ring)
    assert fl & oracle.ERR_ROWS
    fl = oracle.write(cfg, inp.c, inp.kr, inp.cu, np.array([10 ** 5], np.int32), 64, inp.page_table, pool,
                      sink, ring)
    assert fl & oracle.ERR_SEQ_OVERFLOW
