"""Oracle for the low-bit dual-path MLA KV cache (test infrastructure only).

A plain fp64 CPU restatement, in C (``oracle.c``), of the fused cache writer and the decode
attention, following the RAQ-MLA page (appendix Table 5: the quantizer; Figures 3-4: the
dual-path read) and the QuantMLA page (appendix Figure 8: the fused writer, BF16 protection
of sink and recent tokens, one global softmax). See ``oracle.c`` for the readings taken where
the pages are silent.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference legs
may import this package. It shares no code with the CUDA library and never imports it.

Parity status: every function here is pinned by ``tests/test_oracle_*.py`` against values
that do not come from the oracle itself (numpy's float16, exact rational brute force, the
effective-bits figures of Table 5, closed forms of softmax attention,
``torch.nn.functional.scaled_dot_product_attention`` in float64, and for the cached-tensor
transform: identity and signed-permutation closed forms, a hand-worked float32 sum that fixes
the accumulation order, torch's float64 matmul within the float32 summation bound, and torch's
BF16 rounding; for the projections either side of attention: identity, per-head scaled and
single-entry weights, a hand-worked product, and the BF16 rounding of the attention output).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

LATENT, ROPE, ROW, GROUP = 512, 64, 576, 128

ERR_BAD_PAGE, ERR_SEQ_OVERFLOW, ERR_NONFINITE, ERR_RANGE, ERR_ROWS = 1, 2, 4, 8, 16


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (plain gcc, no GPU code)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", "-o", _LIB_PATH, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
    return _LIB_PATH


class Config(ctypes.Structure):
    _fields_ = [("bits_c", ctypes.c_int32), ("bits_r", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("n_sink", ctypes.c_int32),
                ("n_recent", ctypes.c_int32), ("clip_q", ctypes.c_float)]


def make_config(bits_c=4, page_size=128, n_sink=4, n_recent=128, clip_q=None, bits_r=4) -> Config:
    if clip_q is None:
        clip_q = 0.94 if bits_c == 2 else 0.0
    return Config(bits_c, bits_r, page_size, n_sink, n_recent, clip_q)


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.POINTER
        d, i32, u8, u16 = ctypes.c_double, ctypes.c_int32, ctypes.c_uint8, ctypes.c_uint16
        _lib.oracle_bf16_to_double.restype = d
        _lib.oracle_bf16_to_double.argtypes = [u16]
        _lib.oracle_f16_to_double.restype = d
        _lib.oracle_f16_to_double.argtypes = [u16]
        _lib.oracle_f16_bits.restype = u16
        _lib.oracle_f16_bits.argtypes = [d]
        _lib.oracle_f16_round_down.restype = d
        _lib.oracle_f16_round_down.argtypes = [d, P(ctypes.c_int)]
        _lib.oracle_f16_round_up.restype = d
        _lib.oracle_f16_round_up.argtypes = [d, P(ctypes.c_int)]
        _lib.oracle_quantize.restype = ctypes.c_int
        _lib.oracle_quantize.argtypes = [P(d), ctypes.c_int, ctypes.c_int, P(u8), P(u16), P(u16)]
        _lib.oracle_clip_tau.restype = d
        _lib.oracle_clip_tau.argtypes = [P(d), ctypes.c_int, ctypes.c_float]
        _lib.oracle_page_bytes.restype = ctypes.c_size_t
        _lib.oracle_page_bytes.argtypes = [P(Config)]
        _lib.oracle_config_ok.restype = ctypes.c_int
        _lib.oracle_config_ok.argtypes = [P(Config)]
        _lib.oracle_latent_code_pos.restype = None
        _lib.oracle_latent_code_pos.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                P(ctypes.c_size_t), P(ctypes.c_int)]
        _lib.oracle_rope_code_pos.restype = None
        _lib.oracle_rope_code_pos.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              P(ctypes.c_size_t), P(ctypes.c_int)]
        _lib.oracle_write.restype = ctypes.c_int
        _lib.oracle_write.argtypes = [P(Config), ctypes.c_int, ctypes.c_int, P(u16), P(u16), P(i32),
                                      P(i32), ctypes.c_int, P(i32), ctypes.c_int, P(u8),
                                      ctypes.c_int64, P(u16), P(u16)]
        _lib.oracle_token_values.restype = ctypes.c_int
        _lib.oracle_token_values.argtypes = [P(Config), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             P(i32), ctypes.c_int, P(u8), ctypes.c_int64, P(u16),
                                             P(u16), P(d)]
        _lib.oracle_decode.restype = ctypes.c_int
        _lib.oracle_decode.argtypes = [P(Config), ctypes.c_int, ctypes.c_int, P(u16), P(u16), P(i32),
                                       ctypes.c_int, P(i32), P(u8), ctypes.c_int64, P(u16), P(u16),
                                       ctypes.c_float, P(d), P(d)]
        _lib.oracle_decode_bf16.restype = ctypes.c_int
        _lib.oracle_decode_bf16.argtypes = [ctypes.c_int, ctypes.c_int, P(u16), P(u16), P(i32), ctypes.c_int,
                                            ctypes.c_int, P(i32), P(u16), ctypes.c_int64, ctypes.c_float, P(d),
                                            P(d)]
        _lib.oracle_set_threads.restype = None
        _lib.oracle_set_threads.argtypes = [ctypes.c_int]
        _lib.oracle_max_threads.restype = ctypes.c_int
        _lib.oracle_max_threads.argtypes = []
        _lib.oracle_row_transform.restype = None
        _lib.oracle_row_transform.argtypes = [ctypes.c_int, ctypes.c_int, P(u16), P(u16), P(ctypes.c_float),
                                              P(u16)]
    return _lib


def set_threads(n: int) -> int:
    """Threads of the oracle's parallel loops (timing only; results do not depend on it).
    Returns the count now in effect."""
    lib().oracle_set_threads(int(n))
    return int(lib().oracle_max_threads())


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


# ------------------------------------------------------------------ number formats

def bf16_to_double(bits: int) -> float:
    return lib().oracle_bf16_to_double(int(bits))


def f16_to_double(bits: int) -> float:
    return lib().oracle_f16_to_double(int(bits))


def f16_bits(v: float) -> int:
    return int(lib().oracle_f16_bits(float(v)))


def f16_round_down(x: float):
    r = ctypes.c_int(0)
    v = lib().oracle_f16_round_down(float(x), ctypes.byref(r))
    return v, bool(r.value)


def f16_round_up(x: float):
    r = ctypes.c_int(0)
    v = lib().oracle_f16_round_up(float(x), ctypes.byref(r))
    return v, bool(r.value)


# ------------------------------------------------------------------ quantizer

def quantize(x, bits: int):
    """Returns (codes uint8[n], scale_bits, min_bits, flags)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    codes = np.zeros(x.shape[0], dtype=np.uint8)
    sb, mb = ctypes.c_uint16(0), ctypes.c_uint16(0)
    fl = lib().oracle_quantize(_ptr(x, ctypes.c_double), x.shape[0], bits, _ptr(codes, ctypes.c_uint8),
                               ctypes.byref(sb), ctypes.byref(mb))
    return codes, int(sb.value), int(mb.value), int(fl)


def clip_tau(x, clip_q: float) -> float:
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    return lib().oracle_clip_tau(_ptr(x, ctypes.c_double), x.shape[0], ctypes.c_float(clip_q))


# ------------------------------------------------------------------ layout

def page_bytes(cfg: Config) -> int:
    return int(lib().oracle_page_bytes(ctypes.byref(cfg)))


def config_ok(cfg: Config) -> bool:
    return bool(lib().oracle_config_ok(ctypes.byref(cfg)))


def latent_code_pos(bits_c: int, t: int, c: int):
    b, s = ctypes.c_size_t(0), ctypes.c_int(0)
    lib().oracle_latent_code_pos(bits_c, t, c, ctypes.byref(b), ctypes.byref(s))
    return int(b.value), int(s.value)


def rope_code_pos(bits_c: int, page_size: int, t: int, j: int):
    b, s = ctypes.c_size_t(0), ctypes.c_int(0)
    lib().oracle_rope_code_pos(bits_c, page_size, t, j, ctypes.byref(b), ctypes.byref(s))
    return int(b.value), int(s.value)


# ------------------------------------------------------------------ writer / reader / decode

def write(cfg: Config, c_new, kr_new, cu_new, seq_lens, max_new, page_table, pool, sink, ring) -> int:
    """In-place sequential writer over numpy buffers; returns ERR_* flags."""
    c_new = np.ascontiguousarray(c_new, dtype=np.uint16)
    kr_new = np.ascontiguousarray(kr_new, dtype=np.uint16)
    cu_new = np.ascontiguousarray(cu_new, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    page_table = np.ascontiguousarray(page_table, dtype=np.int32)
    for a in (pool, sink, ring):
        assert a.flags["C_CONTIGUOUS"]
    B = seq_lens.shape[0]
    n_rows = c_new.shape[0]
    sink_arg = sink if sink.size else np.zeros(1, dtype=np.uint16)
    return int(lib().oracle_write(ctypes.byref(cfg), B, n_rows, _ptr(c_new, ctypes.c_uint16),
                                  _ptr(kr_new, ctypes.c_uint16), _ptr(cu_new, ctypes.c_int32),
                                  _ptr(seq_lens, ctypes.c_int32), int(max_new),
                                  _ptr(page_table, ctypes.c_int32), page_table.shape[1],
                                  _ptr(pool, ctypes.c_uint8), pool.shape[0],
                                  _ptr(sink_arg, ctypes.c_uint16), _ptr(ring, ctypes.c_uint16)))


def token_values(cfg: Config, b: int, t: int, T: int, page_table, pool, sink, ring):
    """(values float64[576], status): status 1 = BF16 row, 0 = dequantized packed copy."""
    v = np.zeros(ROW, dtype=np.float64)
    page_table = np.ascontiguousarray(page_table, dtype=np.int32)
    sink_arg = sink if sink.size else np.zeros(1, dtype=np.uint16)
    st = lib().oracle_token_values(ctypes.byref(cfg), b, t, T, _ptr(page_table, ctypes.c_int32),
                                   page_table.shape[1], _ptr(pool, ctypes.c_uint8), pool.shape[0],
                                   _ptr(sink_arg, ctypes.c_uint16), _ptr(ring, ctypes.c_uint16),
                                   _ptr(v, ctypes.c_double))
    return v, int(st)


def decode(cfg: Config, q_lat, q_rope, page_table, seq_lens, pool, sink, ring, softmax_scale: float):
    """Returns (out float64[B,H,512], lse float64[B,H], flags)."""
    q_lat = np.ascontiguousarray(q_lat, dtype=np.uint16)
    q_rope = np.ascontiguousarray(q_rope, dtype=np.uint16)
    page_table = np.ascontiguousarray(page_table, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, H = q_lat.shape[0], q_lat.shape[1]
    out = np.zeros((B, H, LATENT), dtype=np.float64)
    lse = np.zeros((B, H), dtype=np.float64)
    sink_arg = sink if sink.size else np.zeros(1, dtype=np.uint16)
    fl = lib().oracle_decode(ctypes.byref(cfg), B, H, _ptr(q_lat, ctypes.c_uint16),
                             _ptr(q_rope, ctypes.c_uint16), _ptr(page_table, ctypes.c_int32),
                             page_table.shape[1], _ptr(seq_lens, ctypes.c_int32),
                             _ptr(pool, ctypes.c_uint8), pool.shape[0], _ptr(sink_arg, ctypes.c_uint16),
                             _ptr(ring, ctypes.c_uint16), ctypes.c_float(softmax_scale),
                             _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double))
    return out, lse, int(fl)


def decode_bf16(q_lat, q_rope, page_table, page_size: int, seq_lens, kv_pool, softmax_scale: float):
    """Exact attention over a paged BF16 cache kv_pool uint16[n_pages, P, 576] (the
    unquantized comparator). Returns (out float64[B,H,512], lse float64[B,H], flags)."""
    q_lat = np.ascontiguousarray(q_lat, dtype=np.uint16)
    q_rope = np.ascontiguousarray(q_rope, dtype=np.uint16)
    page_table = np.ascontiguousarray(page_table, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    kv_pool = np.ascontiguousarray(kv_pool, dtype=np.uint16)
    B, H = q_lat.shape[0], q_lat.shape[1]
    out = np.zeros((B, H, LATENT), dtype=np.float64)
    lse = np.zeros((B, H), dtype=np.float64)
    fl = lib().oracle_decode_bf16(B, H, _ptr(q_lat, ctypes.c_uint16), _ptr(q_rope, ctypes.c_uint16),
                                  _ptr(page_table, ctypes.c_int32), page_table.shape[1], int(page_size),
                                  _ptr(seq_lens, ctypes.c_int32), _ptr(kv_pool, ctypes.c_uint16),
                                  kv_pool.shape[0], ctypes.c_float(softmax_scale), _ptr(out, ctypes.c_double),
                                  _ptr(lse, ctypes.c_double))
    return out, lse, int(fl)


# ------------------------------------------------------------------ cached-tensor transforms

def row_transform(x_bits, a_bits):
    """x A for BF16 rows x [n, d] and a BF16 matrix A [d, d] (RAQ-MLA page, Figure 4: A_c on the
    latent, A_R on the positional key before caching). Float32 sums in index order, then BF16
    round-to-nearest-even. Returns (float32 sums [n, d], BF16 bits [n, d])."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    a = np.ascontiguousarray(a_bits, dtype=np.uint16)
    n, d = x.shape
    assert a.shape == (d, d)
    acc = np.empty((n, d), dtype=np.float32)
    out = np.empty((n, d), dtype=np.uint16)
    if n:
        lib().oracle_row_transform(n, d, _ptr(x, ctypes.c_uint16), _ptr(a, ctypes.c_uint16),
                                   _ptr(acc, ctypes.c_float), _ptr(out, ctypes.c_uint16))
    return acc, out


def write_transformed(cfg: Config, c_new, kr_new, cu_new, seq_lens, max_new, page_table, pool, sink, ring,
                      a_c=None, a_r=None) -> int:
    """The writer over transformed rows: c A_c and k_R A_R (either may be None: unchanged)."""
    c = row_transform(c_new, a_c)[1] if a_c is not None else c_new
    kr = row_transform(kr_new, a_r)[1] if a_r is not None else kr_new
    return write(cfg, c, kr, cu_new, seq_lens, max_new, page_table, pool, sink, ring)


# ------------------------------------------------------------------ projections either side of attention

def _bf16_value(bits) -> np.ndarray:
    """BF16 bit patterns -> float64 values (the upper half of a binary32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def _round_bf16(x) -> np.ndarray:
    """float64 -> BF16 bits, round to nearest even (via the exact binary32 value when it is one;
    the float64 is first rounded to binary32 to nearest, which cannot change the nearest-even
    BF16 result unless it lands exactly on a BF16 midpoint: those cases are resolved on the
    float64 value)."""
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lo = (u >> 16) << 16
    hi = lo + (1 << 16)
    vlo = lo.astype(np.uint32).view(np.float32).astype(np.float64)
    vhi = hi.astype(np.uint32).view(np.float32).astype(np.float64)
    # nearest of the two neighbours by the float64 value; exact ties to the even pattern
    dlo, dhi = np.abs(x - vlo), np.abs(vhi - x)
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (((lo >> 16) & 1) == 1))
    out = np.where(pick_hi, hi >> 16, lo >> 16).astype(np.uint16)
    return out


def project(x, w, x_is_f32: bool = False):
    """Per-head projection Y[b, h, :] = X[b, h, :] W[h] (RAQ-MLA page, Figure 4: the query is
    absorbed into the latent space through W_UK with A_c^-1 folded in, k_R is compensated on the
    query side, and the latent readout leaves through W_UV with A_c^-1 folded in).
    x: BF16 bits [B, H, K] (or float32 values when x_is_f32: they are first rounded to BF16,
    the operand precision of the product); w: BF16 bits [H, K, N] or [K, N] (one matrix for
    every head). Returns the exact products as float64 [B, H, N]."""
    xv = _round_bf16_value(np.asarray(x, np.float32)) if x_is_f32 else _bf16_value(x)
    wv = _bf16_value(w)
    if wv.ndim == 2:
        return np.einsum("bhk,kn->bhn", xv, wv)
    return np.einsum("bhk,hkn->bhn", xv, wv)


def _round_bf16_value(x32) -> np.ndarray:
    return _bf16_value(_round_bf16(np.asarray(x32, np.float64)))


def absorb_query(q_nope, w_uk, q_rope=None, r_comp=None):
    """q_lat = BF16(q_nope W_UK[h]) [B, H, 512] and, with r_comp, q_rope' = BF16(q_rope r_comp)
    [B, H, 64]: the decode's query inputs. Returns (q_lat bits, q_rope' bits or None, exact
    q_lat float64, exact q_rope' float64 or None)."""
    ql = project(q_nope, w_uk)
    qr = project(q_rope, r_comp) if r_comp is not None else None
    return _round_bf16(ql), (_round_bf16(qr) if qr is not None else None), ql, qr


def up_project(o, w_uv):
    """Y = BF16(O) W_UV[h] in float64: O float32 [B, H, 512] (the decode output), W_UV BF16
    [H, 512, d_v]."""
    return project(o, w_uv, x_is_f32=True)


# ------------------------------------------------------------------ multi-token decode

def decode_multi(cfg: Config, q_lat, q_rope, q_len: int, page_table, seq_lens, pool, sink, ring,
                 softmax_scale: float):
    """Decode of q_len new tokens per sequence at once (a draft verified in one step, or a short
    chunk): rows of q_lat [B, q_len * H, 512] / q_rope [B, q_len * H, 64] ordered [position i]
    [head h]. The q_len tokens are the cache's last ones (written before the call); position i
    sees the cache tokens t < T - (q_len - 1 - i), itself included, each with the values the
    cache holds at length T (BF16 rows for t < S or t >= T - W, else the packed copy, as
    token_values reads them). Softmax attention per row in float64, written out from the
    definition. Returns (out float64 [B, q_len * H, 512], lse float64 [B, q_len * H])."""
    q_lat = np.ascontiguousarray(q_lat, dtype=np.uint16)
    q_rope = np.ascontiguousarray(q_rope, dtype=np.uint16)
    B, R = q_lat.shape[0], q_lat.shape[1]
    assert R % q_len == 0
    H = R // q_len
    scale = float(np.float32(softmax_scale))
    out = np.zeros((B, R, LATENT), dtype=np.float64)
    lse = np.full((B, R), -np.inf, dtype=np.float64)
    for b in range(B):
        T = int(seq_lens[b])
        if T <= 0:
            continue
        V = np.stack([token_values(cfg, b, t, T, page_table, pool, sink, ring)[0] for t in range(T)])
        ql = _bf16_value(q_lat[b])
        qr = _bf16_value(q_rope[b])
        for i in range(q_len):
            T_i = T - (q_len - 1 - i)
            if T_i <= 0:
                continue
            for h in range(H):
                r = i * H + h
                sc = scale * (V[:T_i, :LATENT] @ ql[r] + V[:T_i, LATENT:] @ qr[r])
                m = sc.max()
                w = np.exp(sc - m)
                out[b, r] = (w @ V[:T_i, :LATENT]) / w.sum()
                lse[b, r] = m + np.log(w.sum())
    return out, lse
