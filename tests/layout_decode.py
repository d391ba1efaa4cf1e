"""Independent numpy decoder of the physical page layout documented in include/mla_qcache.h.

Written from the layout's prose description only; it shares nothing with the oracle's C code
or the CUDA kernels, so agreement between them pins the byte layout.
"""
import numpy as np


def page_bytes(bits_c, P):
    return P * (64 * bits_c + 32 + 16) + 256


def latent_positions(bits_c, P):
    """(byte, shift) arrays of shape [P, 512] for every latent code of a page."""
    t = np.arange(P)[:, None]
    c = np.arange(512)[None, :]
    k = c * bits_c // 8                      # byte of the token's row, channels in order
    byte = t * (64 * bits_c) + 16 * ((k // 16) ^ (t % 8)) + k % 16
    shift = (c * bits_c) % 8
    return np.broadcast_to(byte, (P, 512)), np.broadcast_to(shift, (P, 512))


def rope_positions(bits_c, P):
    t = np.arange(P)[:, None]
    j = np.arange(64)[None, :]
    e = j % 16
    q, h, o = (e % 8) // 2, e // 8, e % 2
    n = (t % 16) // 8
    lane = 4 * (t % 8) + q
    bit = 4 * (2 * n + h + 4 * o)
    byte = P * 64 * bits_c + ((t // 16) * 4 + j // 16) * 128 + lane * 4 + bit // 8
    return np.broadcast_to(byte, (P, 64)), np.broadcast_to(bit % 8, (P, 64))


def decode_page(page: np.ndarray, bits_c: int, P: int):
    """-> dict with latent codes [P,512], latent scale/min [P,4] (float64), rope codes [P,64],
    rope scale/min [64] (float64)."""
    page = np.asarray(page, dtype=np.uint8)
    lb, ls = latent_positions(bits_c, P)
    lat = (page[lb] >> ls) & ((1 << bits_c) - 1)
    rb, rs = rope_positions(bits_c, P)
    rope = (page[rb] >> rs) & 0xF
    c_off = P * (64 * bits_c + 32)
    meta = page[c_off:c_off + 16 * P].view(np.uint16).reshape(P, 4, 2)
    d_off = P * (64 * bits_c + 48)
    rmeta = page[d_off:d_off + 256].view(np.uint16).reshape(64, 2)
    f = lambda u: u.view(np.float16).astype(np.float64)
    return dict(latent=lat.astype(np.int64), lat_scale=f(meta[:, :, 0].copy()), lat_min=f(meta[:, :, 1].copy()),
                rope=rope.astype(np.int64), rope_scale=f(rmeta[:, 0].copy()), rope_min=f(rmeta[:, 1].copy()))


def dequant_page(page, bits_c, P):
    """[P, 576] float64 dequantized values (min + code*scale) of every slot of a page."""
    d = decode_page(page, bits_c, P)
    lat = d["lat_min"].repeat(128, axis=1) + d["latent"] * d["lat_scale"].repeat(128, axis=1)
    rope = d["rope_min"][None, :] + d["rope"] * d["rope_scale"][None, :]
    return np.concatenate([lat, rope], axis=1)
