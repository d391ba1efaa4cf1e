"""Pins of the oracle's multi-token decode: one position reduces to the single-token decode;
with every token protected each position is exact softmax attention over its prefix (torch
float64 scaled_dot_product_attention); tokens past a position's prefix do not change its row."""
import numpy as np
import torch

import oracle
import workloads


def _cache(w, lens):
    inp = workloads.make_inputs(w, seq_lens=np.array(lens, np.int32))
    cfg = oracle.make_config(**w.config_kwargs())
    pool = np.zeros((inp.n_pages, oracle.page_bytes(cfg)), np.uint8)
    sink = np.zeros((len(lens), cfg.n_sink, 576), np.uint16)
    ring = np.zeros((len(lens), cfg.n_recent, 576), np.uint16)
    assert oracle.write(cfg, inp.c, inp.kr, inp.cu, np.zeros(len(lens), np.int32), max(lens), inp.page_table,
                        pool, sink, ring) == 0
    return cfg, inp, pool, sink, ring


def _queries(B, R, seed):
    rng = np.random.default_rng(seed)
    return workloads.draw_queries(rng, B, R)


W4 = workloads.Workload("m", 1, 16, 1, 4, 32, n_sink=4, n_recent=32, seed=7)


def test_one_position_is_the_single_token_decode():
    cfg, inp, pool, sink, ring = _cache(W4, [150, 37])
    ql, qr = _queries(2, 16, 1)
    o1, l1 = oracle.decode_multi(cfg, ql, qr, 1, inp.page_table, inp.seq_lens, pool, sink, ring, 0.1)
    o2, l2, fl = oracle.decode(cfg, ql, qr, inp.page_table, inp.seq_lens, pool, sink, ring, 0.1)
    assert fl == 0
    assert np.allclose(o1, o2, rtol=1e-12, atol=1e-12) and np.allclose(l1, l2, rtol=1e-12, atol=1e-12)


def test_all_protected_prefixes_are_exact_attention():
    """T <= S + W: every token is a BF16 row, so position i is plain attention over rows < T_i."""
    T, q_len, H = 30, 3, 16
    cfg, inp, pool, sink, ring = _cache(W4, [T])
    ql, qr = _queries(1, q_len * H, 2)
    o, l = oracle.decode_multi(cfg, ql, qr, q_len, inp.page_table, inp.seq_lens, pool, sink, ring, 0.25)
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).double()
    K = torch.cat([to(inp.c), to(inp.kr)], dim=1)  # [T, 576]
    Q = torch.cat([to(ql[0]), to(qr[0])], dim=1)   # [q_len*H, 576]
    for i in range(q_len):
        Ti = T - (q_len - 1 - i)
        q = Q[i * H:(i + 1) * H][None]
        ref = torch.nn.functional.scaled_dot_product_attention(q, K[None, :Ti], K[None, :Ti, :512],
                                                               scale=float(np.float32(0.25)))
        assert np.allclose(o[0, i * H:(i + 1) * H], ref[0].numpy(), rtol=1e-10, atol=1e-12)


def test_rows_ignore_tokens_past_their_prefix():
    """Changing the cache's newest token changes only the last position's rows."""
    T, q_len, H = 200, 4, 16
    cfg, inp, pool, sink, ring = _cache(W4, [T])
    ql, qr = _queries(1, q_len * H, 3)
    o1, _ = oracle.decode_multi(cfg, ql, qr, q_len, inp.page_table, inp.seq_lens, pool, sink, ring, 0.1)
    ring2 = ring.copy()
    ring2[0, (T - 1) % 32, :] = 0x3f80  # the newest token's BF16 row (it is in the recent window)
    o2, _ = oracle.decode_multi(cfg, ql, qr, q_len, inp.page_table, inp.seq_lens, pool, sink, ring2, 0.1)
    assert np.array_equal(o1[:, :3 * H], o2[:, :3 * H])
    assert not np.allclose(o1[:, 3 * H:], o2[:, 3 * H:])


def test_positions_before_the_first_token_are_empty():
    T, q_len, H = 2, 4, 16
    cfg, inp, pool, sink, ring = _cache(W4, [T])
    ql, qr = _queries(1, q_len * H, 4)
    o, l = oracle.decode_multi(cfg, ql, qr, q_len, inp.page_table, inp.seq_lens, pool, sink, ring, 0.1)
    assert np.all(o[0, :2 * H] == 0) and np.all(np.isneginf(l[0, :2 * H]))
    assert np.all(np.isfinite(l[0, 2 * H:]))
