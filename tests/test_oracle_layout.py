"""Layout and effective-bits pins (RAQ-MLA page, appendix Table 5 and Table 1)."""
import os

import numpy as np
import pytest

import oracle
from tests import layout_decode as ld

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_bits():
    out = {}
    with open(os.path.join(GOLDEN, "effective_bits.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v, _ = [x.strip() for x in line.split("|")]
                out[k] = float(v)
    return out


def test_page_bytes_and_effective_bits():
    g = _golden_bits()
    for bits_c, P in [(4, 128), (2, 64), (2, 128), (4, 64), (4, 16)]:
        cfg = oracle.make_config(bits_c=bits_c, page_size=P)
        pb = oracle.page_bytes(cfg)
        assert pb == ld.page_bytes(bits_c, P)
        assert pb % 128 == 0
    assert oracle.page_bytes(oracle.make_config(4, 128)) == 39168
    assert oracle.page_bytes(oracle.make_config(2, 64)) == 11520

    def latent_bits(bits_c, P):  # codes + per-token group metadata, per latent element
        return (P * 64 * bits_c + 16 * P) * 8 / (512 * P)

    def rope_bits(P):  # codes + per-page channel metadata, per k_R element
        return (32 * P + 256) * 8 / (64 * P)

    assert latent_bits(2, 128) == g["latent_int2_bits"]
    assert rope_bits(128) == g["rope_int4_bits_p128"]
    assert rope_bits(64) == g["rope_int4_bits_p64"]
    bpe = (512 * latent_bits(2, 128) + 64 * rope_bits(128)) / 576
    assert round(bpe, 2) == g["bpe_c2r4_p128"]
    assert round(16 / bpe, 1) == g["capacity_vs_bf16"]
    # page bytes decompose exactly into the four regions
    for bits_c, P in [(4, 128), (2, 64)]:
        cfg = oracle.make_config(bits_c=bits_c, page_size=P)
        bits_total = oracle.page_bytes(cfg) * 8
        assert bits_total == P * (512 * latent_bits(bits_c, P) + 64 * rope_bits(P))


@pytest.mark.parametrize("bits_c,P", [(4, 128), (2, 64), (4, 16), (2, 32)])
def test_code_positions_bijective_and_match_spec(bits_c, P):
    lb, ls = ld.latent_positions(bits_c, P)
    rb, rs = ld.rope_positions(bits_c, P)
    # the oracle's positions agree with the independent decoder at every slot
    for t in range(0, P, max(1, P // 16)):
        for c in range(0, 512, 7):
            assert oracle.latent_code_pos(bits_c, t, c) == (int(lb[t, c]), int(ls[t, c]))
        for j in range(64):
            assert oracle.rope_code_pos(bits_c, P, t, j) == (int(rb[t, j]), int(rs[t, j]))
    # bijection onto the code regions: every bit of regions A and B is used exactly once
    lat_bits = (lb * 8 + ls).ravel()
    assert np.unique(lat_bits).size == lat_bits.size
    assert lat_bits.min() == 0 and (lat_bits.max() + bits_c) == P * 64 * bits_c * 8
    assert np.all(lat_bits % bits_c == 0)
    rope_bits = (rb * 8 + rs).ravel()
    assert np.unique(rope_bits).size == rope_bits.size
    base = P * 64 * bits_c * 8
    assert rope_bits.min() == base and rope_bits.max() + 4 == base + 32 * P * 8


@pytest.mark.parametrize("bits_c", [4, 2])
def test_exhaustive_byte_roundtrip(bits_c):
    """unpack(pack(.)) and pack(unpack(.)) over all 256 byte values of one code byte."""
    P = 16
    lb, ls = ld.latent_positions(bits_c, P)
    width = bits_c
    # pick the codes that live in byte 0 of region A
    sel = np.argwhere(lb == 0)
    assert len(sel) == 8 // width
    for v in range(256):
        page = np.zeros(ld.page_bytes(bits_c, P), dtype=np.uint8)
        page[0] = v
        codes = ld.decode_page(page, bits_c, P)["latent"]
        # repack through the oracle's positions
        out = 0
        for t, c in sel:
            byte, shift = oracle.latent_code_pos(bits_c, int(t), int(c))
            assert byte == 0
            out |= int(codes[t, c]) << shift
        assert out == v
    # rope codes, byte 0 of region B
    rb, rs = ld.rope_positions(bits_c, P)
    sel = np.argwhere(rb == P * 64 * bits_c)
    assert len(sel) == 2
    for v in range(256):
        page = np.zeros(ld.page_bytes(bits_c, P), dtype=np.uint8)
        page[P * 64 * bits_c] = v
        codes = ld.decode_page(page, bits_c, P)["rope"]
        out = 0
        for t, j in sel:
            byte, shift = oracle.rope_code_pos(bits_c, P, int(t), int(j))
            out |= int(codes[t, j]) << shift
        assert out == v


@pytest.mark.parametrize("bits_c", [4, 2])
def test_row_chunks_for_matrix_loads(bits_c):
    """The documented purpose of the latent layout. Region A is token-major (one row of
    64*bits_c bytes per token, channels in order inside the row), and the row's 16-byte chunks
    are XOR-permuted by t mod 8. (1) For 8 consecutive tokens starting at a multiple of 8, the
    same logical chunk lands on 8 distinct 16-byte positions modulo 128 bytes, so an 8x8
    matrix load of 16-bit elements (one 16-byte row per token) touches every shared-memory
    bank once. (2) The 16-bit little-endian element e of logical chunk j holds channels
    32j + 4e + s at bits 4s (INT4) or 64j + 8e + i at bits 2i (INT2)."""
    P = 32
    lb, ls = ld.latent_positions(bits_c, P)
    row = 64 * bits_c
    per_chunk = 128 // bits_c          # channels in a 16-byte chunk
    per_elem = 16 // bits_c            # channels in a 16-bit element
    for t0 in range(0, P, 8):
        for j in range(row // 16):
            c = j * per_chunk          # first channel of logical chunk j
            starts = [(int(lb[t, c]) - t * row) for t in range(t0, t0 + 8)]
            assert all(s0 % 16 == 0 for s0 in starts)
            assert len({s0 % 128 for s0 in starts}) == 8
    rng = np.random.default_rng(0)
    codes = rng.integers(0, 1 << bits_c, size=(P, 512))
    page = np.zeros(ld.page_bytes(bits_c, P), dtype=np.uint8)
    for t in range(P):
        for c in range(512):
            page[lb[t, c]] |= codes[t, c] << ls[t, c]
    for t in range(0, P, 5):
        for j in range(row // 16):
            phys = j ^ (t % 8)
            chunk = page[t * row + 16 * phys: t * row + 16 * phys + 16]
            for e in range(8):
                v = int(chunk[2 * e]) | (int(chunk[2 * e + 1]) << 8)
                for s in range(per_elem):
                    ch = j * per_chunk + per_elem * e + s
                    assert (v >> (bits_c * s)) & ((1 << bits_c) - 1) == codes[t, ch]
