"""The unquantized comparator of the oracle (exact attention over a paged BF16 cache), pinned to
the quantized-cache oracle decode in its all-protected case: when every token is a sink or
recent token the quantized cache holds the same BF16 rows, so both must agree exactly; and to
a float64 softmax written out here for a tiny case."""
import numpy as np

import oracle
import workloads


def _paged_bf16(inp, P, rng):
    """Scatter the rows of every sequence into a BF16 pool through a random page table."""
    B = len(inp.seq_lens)
    max_pages = max(1, int(np.ceil(int(inp.seq_lens.max()) / P)))
    n_pages = B * max_pages
    perm = rng.permutation(n_pages).astype(np.int32).reshape(B, max_pages)
    pool = np.zeros((n_pages, P, 576), dtype=np.uint16)
    for b in range(B):
        rows = np.concatenate([inp.c[inp.cu[b]:inp.cu[b + 1]], inp.kr[inp.cu[b]:inp.cu[b + 1]]], axis=1)
        for t in range(int(inp.seq_lens[b])):
            pool[perm[b, t // P], t % P] = rows[t]
    return perm, pool


def test_bf16_decode_equals_all_protected_quantized_decode():
    w = workloads.Workload("p", 1, 16, 1, 4, 64, n_sink=4, n_recent=256, random_pages=True, seed=3)
    lens = np.array([200, 1, 0, 257, 64], np.int32)  # all <= S + W: every token protected
    inp = workloads.make_inputs(w, seq_lens=lens)
    cfg = oracle.make_config(4, 64, n_sink=4, n_recent=256)
    pb = oracle.page_bytes(cfg)
    pool_q = np.zeros((inp.n_pages, pb), np.uint8)
    sink = np.zeros((len(lens), 4, 576), np.uint16)
    ring = np.zeros((len(lens), 256, 576), np.uint16)
    assert oracle.write(cfg, inp.c, inp.kr, inp.cu, np.zeros(len(lens), np.int32), int(lens.max()),
                        inp.page_table, pool_q, sink, ring) == 0
    o1, l1, f1 = oracle.decode(cfg, inp.q_lat, inp.q_rope, inp.page_table, lens, pool_q, sink, ring, 0.07)
    pt, pool = _paged_bf16(inp, 32, np.random.default_rng(1))
    o2, l2, f2 = oracle.decode_bf16(inp.q_lat, inp.q_rope, pt, 32, lens, pool, 0.07)
    assert f1 == 0 and f2 == 0
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_bf16_decode_tiny_against_float64_softmax():
    rng = np.random.default_rng(8)
    B, H, T, P = 1, 2, 5, 32
    rows = workloads.bf16_bits(rng.standard_normal((T, 576)).astype(np.float32))
    ql = workloads.bf16_bits(rng.standard_normal((B, H, 512)).astype(np.float32))
    qr = workloads.bf16_bits(rng.standard_normal((B, H, 64)).astype(np.float32))
    pool = np.zeros((3, P, 576), np.uint16)
    pool[2, :T] = rows
    pt = np.array([[2]], np.int32)
    sc = float(np.float32(0.1))  # the scale crosses the C interface as a float
    out, lse, fl = oracle.decode_bf16(ql, qr, pt, P, np.array([T], np.int32), pool, sc)
    assert fl == 0
    v = workloads.bf16_value(rows).astype(np.float64)
    for h in range(H):
        q = np.concatenate([workloads.bf16_value(ql[0, h]), workloads.bf16_value(qr[0, h])]).astype(np.float64)
        s = sc * (v @ q)
        p = np.exp(s - s.max())
        ref = (p[:, None] * v[:, :512]).sum(0) / p.sum()
        assert np.allclose(out[0, h], ref, rtol=1e-13, atol=1e-13)
        assert abs(lse[0, h] - (s.max() + np.log(p.sum()))) < 1e-12


def test_bf16_decode_bad_page_flag():
    pool = np.zeros((1, 32, 576), np.uint16)
    q = np.zeros((1, 1, 512), np.uint16)
    _, _, fl = oracle.decode_bf16(q, np.zeros((1, 1, 64), np.uint16), np.array([[5]], np.int32), 32,
                                  np.array([3], np.int32), pool, 0.1)
    assert fl & 1
