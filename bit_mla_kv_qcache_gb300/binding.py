"""ctypes binding of the C ABI in include/mla_qcache.h (argument marshalling only).

Every step of the hot path runs in the CUDA kernels of libmla_qcache.so; this module only
checks tensor dtypes/devices and passes raw pointers, sizes and the current CUDA stream.
There is no fallback: if the library is missing the calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmla_qcache.so")

OK, ERR_NULL, ERR_CONFIG, ERR_SHAPE, ERR_ALIGN, ERR_WORKSPACE, ERR_CUDA = 0, -1, -2, -3, -4, -5, -6
ERR_SCRATCH_LIMIT = -7
DEV_BAD_PAGE, DEV_SEQ_OVERFLOW, DEV_NONFINITE, DEV_RANGE, DEV_ROWS, DEV_TIMEOUT = 1, 2, 4, 8, 16, 32

# the entry points declared in include/mla_qcache.h
EXPORTS = ("mla_qcache_page_bytes", "mla_qcache_config_check", "mla_qcache_workspace_bytes",
           "mla_qcache_write", "mla_qcache_decode_attn", "mla_qcache_strerror",
           "mla_qcache_decode_attn_noalloc", "mla_qcache_noalloc_scratch_bytes", "mla_qcache_advance",
           "mla_qcache_write_advance", "mla_qcache_decode_attn_bf16", "mla_qcache_bf16_workspace_bytes",
           "mla_qcache_write_transformed", "mla_qcache_row_transform", "mla_qcache_absorb_query",
           "mla_qcache_up_project", "mla_qcache_decode_attn_multi", "mla_qcache_decode_plan",
           "mla_qcache_selftest_wait_timeout", "mla_qcache_decode_attn_pending", "mla_qcache_decode_launches")


class Config(ctypes.Structure):
    """mla_qcache_config."""
    _fields_ = [("bits_c", ctypes.c_int32), ("bits_r", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("n_sink", ctypes.c_int32), ("n_recent", ctypes.c_int32), ("clip_q", ctypes.c_float)]

    def __repr__(self):
        return (f"Config(bits_c={self.bits_c}, bits_r={self.bits_r}, page_size={self.page_size}, "
                f"n_sink={self.n_sink}, n_recent={self.n_recent}, clip_q={self.clip_q:g})")


def make_config(bits_c=4, page_size=128, n_sink=4, n_recent=128, clip_q=None, bits_r=4) -> Config:
    """C4R4 / C2R4 configuration; the latent clip defaults to 0.94 for INT2 and off for INT4."""
    if clip_q is None:
        clip_q = 0.94 if bits_c == 2 else 0.0
    return Config(bits_c, bits_r, page_size, n_sink, n_recent, clip_q)


class QCacheError(RuntimeError):
    pass


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise QCacheError(f"{_LIB_PATH} is not built (run __graft_entry__.build() or "
                              "python -m bit_mla_kv_qcache_gb300.build)")
        L = ctypes.CDLL(_LIB_PATH)
        P, vp, i32, i64, sz = ctypes.POINTER, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        L.mla_qcache_page_bytes.restype = sz
        L.mla_qcache_page_bytes.argtypes = [P(Config)]
        L.mla_qcache_config_check.restype = ctypes.c_int
        L.mla_qcache_config_check.argtypes = [P(Config)]
        L.mla_qcache_workspace_bytes.restype = sz
        L.mla_qcache_workspace_bytes.argtypes = [P(Config), i32, i32, i32]
        L.mla_qcache_write.restype = ctypes.c_int
        L.mla_qcache_write.argtypes = [P(Config), i32, i32, vp, vp, vp, vp, i32, vp, i32, vp, i64, vp, vp, vp, vp]
        L.mla_qcache_decode_attn.restype = ctypes.c_int
        L.mla_qcache_decode_attn.argtypes = [P(Config), i32, i32, vp, vp, vp, i32, vp, vp, i64, vp, vp,
                                             ctypes.c_float, vp, vp, vp, sz, vp, vp]
        L.mla_qcache_decode_attn_noalloc.restype = ctypes.c_int
        L.mla_qcache_decode_attn_noalloc.argtypes = [P(Config), i32, i32, vp, vp, vp, i32, vp, vp, i64, vp, vp,
                                                     ctypes.c_float, vp, vp, vp, vp]
        L.mla_qcache_noalloc_scratch_bytes.restype = sz
        L.mla_qcache_noalloc_scratch_bytes.argtypes = []
        L.mla_qcache_write_advance.restype = ctypes.c_int
        L.mla_qcache_write_advance.argtypes = [P(Config), i32, i32, vp, vp, vp, vp, vp, i32, vp, i32, vp, i64, vp, vp,
                                               vp, vp]
        L.mla_qcache_write_transformed.restype = ctypes.c_int
        L.mla_qcache_write_transformed.argtypes = [P(Config), i32, i32, vp, vp, vp, vp, vp, i32, vp, vp, vp, i32, vp,
                                                   i64, vp, vp, vp, vp]
        L.mla_qcache_row_transform.restype = ctypes.c_int
        L.mla_qcache_row_transform.argtypes = [i32, i32, vp, vp, vp, vp, vp]
        L.mla_qcache_selftest_wait_timeout.restype = ctypes.c_int
        L.mla_qcache_selftest_wait_timeout.argtypes = [vp, vp]
        L.mla_qcache_decode_plan.restype = ctypes.c_int
        L.mla_qcache_decode_plan.argtypes = [P(Config), i32, i32, i32, i32, P(i32)]
        L.mla_qcache_decode_launches.restype = ctypes.c_int
        L.mla_qcache_decode_launches.argtypes = [P(Config), i32, i32, i32]
        L.mla_qcache_decode_attn_pending.restype = ctypes.c_int
        L.mla_qcache_decode_attn_pending.argtypes = [P(Config), i32, i32, vp, vp, vp, i32, vp, vp, vp, vp, i32, vp, i64,
                                                     vp, vp, ctypes.c_float, vp, vp, vp, sz, vp, vp]
        L.mla_qcache_decode_attn_multi.restype = ctypes.c_int
        L.mla_qcache_decode_attn_multi.argtypes = [P(Config), i32, i32, i32, vp, vp, vp, i32, vp, vp, i64, vp, vp,
                                                   ctypes.c_float, vp, vp, vp, sz, vp, vp]
        L.mla_qcache_absorb_query.restype = ctypes.c_int
        L.mla_qcache_absorb_query.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
        L.mla_qcache_up_project.restype = ctypes.c_int
        L.mla_qcache_up_project.argtypes = [i32, i32, i32, vp, vp, vp, vp]
        L.mla_qcache_bf16_workspace_bytes.restype = sz
        L.mla_qcache_bf16_workspace_bytes.argtypes = [i32, i32, i32, i32]
        L.mla_qcache_decode_attn_bf16.restype = ctypes.c_int
        L.mla_qcache_decode_attn_bf16.argtypes = [i32, i32, vp, vp, vp, i32, i32, vp, vp, i64, ctypes.c_float, vp, vp,
                                                  vp, sz, vp, vp]
        L.mla_qcache_advance.restype = ctypes.c_int
        L.mla_qcache_advance.argtypes = [vp, vp, i32, vp]
        L.mla_qcache_strerror.restype = ctypes.c_char_p
        L.mla_qcache_strerror.argtypes = [i32]
        _lib = L
    return _lib


def strerror(status: int) -> str:
    return lib().mla_qcache_strerror(int(status)).decode()


def _raise(status: int, what: str):
    if status != OK:
        raise QCacheError(f"{what}: {strerror(status)} (status {status})")


def page_bytes(cfg: Config) -> int:
    return int(lib().mla_qcache_page_bytes(ctypes.byref(cfg)))


def workspace_bytes(cfg: Config, B: int, H: int, max_pages: int) -> int:
    return int(lib().mla_qcache_workspace_bytes(ctypes.byref(cfg), B, H, max_pages))


def _ptr(t, name, elem_size=None, dtype=None, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise QCacheError(f"{name} is required")
    if not t.is_cuda:
        raise QCacheError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise QCacheError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise QCacheError(f"{name} must be {dtype}, got {t.dtype}")
    if elem_size is not None and t.element_size() != elem_size:
        raise QCacheError(f"{name} must have {elem_size}-byte elements")
    return ctypes.c_void_p(t.data_ptr())


def _check_decode_shapes(q_lat, q_rope, page_table, seq_lens, out, lse, rows_per_seq=None):
    """Shapes every decode entry point relies on, checked before any library call: a mis-shaped
    output, length or page table would otherwise become an out-of-bounds device access."""
    if q_lat is None or q_lat.dim() != 3 or q_lat.shape[2] != 512:
        raise ValueError(f"q_lat must be [B, H, 512], got {None if q_lat is None else tuple(q_lat.shape)}")
    B, R = q_lat.shape[0], q_lat.shape[1]
    if rows_per_seq is not None and R != rows_per_seq:
        raise ValueError(f"q_lat must have {rows_per_seq} rows per sequence, got {R}")
    if q_rope is None or tuple(q_rope.shape) != (B, R, 64):
        raise ValueError(f"q_rope must be [{B}, {R}, 64], got {None if q_rope is None else tuple(q_rope.shape)}")
    if out is None or tuple(out.shape) != (B, R, 512):
        raise ValueError(f"out must be [{B}, {R}, 512], got {None if out is None else tuple(out.shape)}")
    if lse is None or tuple(lse.shape) != (B, R):
        raise ValueError(f"lse must be [{B}, {R}], got {None if lse is None else tuple(lse.shape)}")
    if seq_lens is None or seq_lens.dim() != 1 or seq_lens.shape[0] != B:
        raise ValueError(f"seq_lens must be [{B}], got {None if seq_lens is None else tuple(seq_lens.shape)}")
    if page_table is None or page_table.dim() != 2 or page_table.shape[0] != B:
        raise ValueError(f"page_table must be [{B}, max_pages], got "
                         f"{None if page_table is None else tuple(page_table.shape)}")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def mla_qcache_write(cfg: Config, c_new, kr_new, cu_new, seq_lens, max_new: int, page_table, pool,
                     sink_buf, recent_buf, err_word, stream=None) -> None:
    """Fused cache writer (see include/mla_qcache.h). BF16 inputs may be bfloat16 or 16-bit ints."""
    B = seq_lens.shape[0]
    n_rows = c_new.shape[0]
    st = lib().mla_qcache_write(
        ctypes.byref(cfg), B, n_rows, _ptr(c_new, "c_new", 2), _ptr(kr_new, "kr_new", 2),
        _ptr(cu_new, "cu_new", dtype=torch.int32), _ptr(seq_lens, "seq_lens", dtype=torch.int32), int(max_new),
        _ptr(page_table, "page_table", dtype=torch.int32), page_table.shape[1], _ptr(pool, "pool", 1),
        pool.shape[0], _ptr(sink_buf, "sink_buf", 2, allow_none=True) if cfg.n_sink else None,
        _ptr(recent_buf, "recent_buf", 2), _ptr(err_word, "err_word", dtype=torch.int32), _stream(stream))
    _raise(st, "mla_qcache_write")


def mla_qcache_write_advance(cfg: Config, c_new, kr_new, cu_new, seq_lens, seq_lens_next, max_new: int,
                             page_table, pool, sink_buf, recent_buf, err_word, stream=None) -> None:
    """mla_qcache_write plus seq_lens_next = seq_lens + rows per sequence in the same launch
    (see include/mla_qcache.h); seq_lens_next must be a separate int32 array."""
    B = seq_lens.shape[0]
    n_rows = c_new.shape[0]
    st = lib().mla_qcache_write_advance(
        ctypes.byref(cfg), B, n_rows, _ptr(c_new, "c_new", 2), _ptr(kr_new, "kr_new", 2),
        _ptr(cu_new, "cu_new", dtype=torch.int32), _ptr(seq_lens, "seq_lens", dtype=torch.int32),
        _ptr(seq_lens_next, "seq_lens_next", dtype=torch.int32), int(max_new),
        _ptr(page_table, "page_table", dtype=torch.int32), page_table.shape[1], _ptr(pool, "pool", 1),
        pool.shape[0], _ptr(sink_buf, "sink_buf", 2, allow_none=True) if cfg.n_sink else None,
        _ptr(recent_buf, "recent_buf", 2), _ptr(err_word, "err_word", dtype=torch.int32), _stream(stream))
    _raise(st, "mla_qcache_write_advance")


def mla_qcache_write_transformed(cfg: Config, c_new, kr_new, cu_new, seq_lens, max_new: int, page_table, pool,
                                 sink_buf, recent_buf, err_word, a_c=None, a_r=None, seq_lens_next=None,
                                 stream=None) -> None:
    """The writer over c A_c and k_R A_R (either transform may be None), with the length update
    when seq_lens_next is given (see include/mla_qcache.h)."""
    B = seq_lens.shape[0]
    n_rows = c_new.shape[0]
    if a_c is not None and tuple(a_c.shape) != (512, 512):
        raise ValueError(f"a_c must be [512, 512], got {tuple(a_c.shape)}")
    if a_r is not None and tuple(a_r.shape) != (64, 64):
        raise ValueError(f"a_r must be [64, 64], got {tuple(a_r.shape)}")
    st = lib().mla_qcache_write_transformed(
        ctypes.byref(cfg), B, n_rows, _ptr(c_new, "c_new", 2), _ptr(kr_new, "kr_new", 2),
        _ptr(cu_new, "cu_new", dtype=torch.int32), _ptr(seq_lens, "seq_lens", dtype=torch.int32),
        _ptr(seq_lens_next, "seq_lens_next", dtype=torch.int32, allow_none=True), int(max_new),
        _ptr(a_c, "a_c", 2, allow_none=True), _ptr(a_r, "a_r", 2, allow_none=True),
        _ptr(page_table, "page_table", dtype=torch.int32), page_table.shape[1], _ptr(pool, "pool", 1),
        pool.shape[0], _ptr(sink_buf, "sink_buf", 2, allow_none=True) if cfg.n_sink else None,
        _ptr(recent_buf, "recent_buf", 2), _ptr(err_word, "err_word", dtype=torch.int32), _stream(stream))
    _raise(st, "mla_qcache_write_transformed")


def mla_qcache_row_transform(x, a, out, err_word, stream=None) -> None:
    """out = x A for BF16 rows x [n, d] (d = 64 or 512) and A [d, d] (see include/mla_qcache.h)."""
    n, d = x.shape
    if tuple(a.shape) != (d, d) or tuple(out.shape) != (n, d):
        raise ValueError("row_transform: x [n, d], a [d, d], out [n, d]")
    st = lib().mla_qcache_row_transform(n, d, _ptr(x, "x", 2), _ptr(a, "a", 2), _ptr(out, "out", 2),
                                        _ptr(err_word, "err_word", dtype=torch.int32), _stream(stream))
    _raise(st, "mla_qcache_row_transform")


def selftest_wait_timeout(err_word, stream=None) -> None:
    """Run the kernel whose bounded wait must give up (see include/mla_qcache.h)."""
    _raise(lib().mla_qcache_selftest_wait_timeout(_ptr(err_word, "err_word", dtype=torch.int32), _stream(stream)),
           "mla_qcache_selftest_wait_timeout")


def decode_plan(cfg: Config, B: int, H: int, max_pages: int, num_sms: int) -> dict:
    """The launch plan of a decode call (see include/mla_qcache.h); needs no GPU."""
    out = (ctypes.c_int32 * 5)()
    _raise(lib().mla_qcache_decode_plan(ctypes.byref(cfg), B, H, max_pages, num_sms, out), "mla_qcache_decode_plan")
    return {"n_split": out[0], "n_protected": out[1], "share_slots": out[2], "tensor_memory": bool(out[3]),
            "bf16_parts": out[4]}


def decode_launches(cfg: Config, B: int, H: int, max_pages: int) -> int:
    """Kernel launches of one decode call of this shape on the current device (see
    include/mla_qcache.h): 1 (merged in place), 2 (with a merge launch) or 3 (64-head blocks)."""
    n = lib().mla_qcache_decode_launches(ctypes.byref(cfg), B, H, max_pages)
    _raise(min(n, 0), "mla_qcache_decode_launches")
    return n


def mla_qcache_decode_attn_multi(cfg: Config, q_len: int, q_lat, q_rope, page_table, seq_lens, pool, sink_buf,
                                 recent_buf, softmax_scale: float, out, lse, workspace, err_word, stream=None) -> None:
    """Decode of q_len new tokens per sequence (rows [B, q_len * H, ...] position-major; see
    include/mla_qcache.h); workspace of workspace_bytes(cfg, B, q_len * H, max_pages)."""
    if q_len < 1 or q_lat is None or q_lat.dim() != 3 or q_lat.shape[1] % q_len:
        raise ValueError("q_lat rows must be q_len x heads")
    _check_decode_shapes(q_lat, q_rope, page_table, seq_lens, out, lse)
    B, R = q_lat.shape[0], q_lat.shape[1]
    st = lib().mla_qcache_decode_attn_multi(
        ctypes.byref(cfg), B, R // q_len, int(q_len), _ptr(q_lat, "q_lat", 2), _ptr(q_rope, "q_rope", 2),
        _ptr(page_table, "page_table", dtype=torch.int32), page_table.shape[1],
        _ptr(seq_lens, "seq_lens", dtype=torch.int32), _ptr(pool, "pool", 1), pool.shape[0],
        _ptr(sink_buf, "sink_buf", 2, allow_none=True) if cfg.n_sink else None, _ptr(recent_buf, "recent_buf", 2),
        ctypes.c_float(softmax_scale), _ptr(out, "out", dtype=torch.float32), _ptr(lse, "lse", dtype=torch.float32),
        _ptr(workspace, "workspace", 1), workspace.numel(), _ptr(err_word, "err_word", dtype=torch.int32),
        _stream(stream))
    _raise(st, "mla_qcache_decode_attn_multi")


def mla_qcache_absorb_query(q_nope, w_uk, q_lat, q_rope=None, r_comp=None, q_rope_out=None, stream=None) -> None:
    """q_lat = q_nope W_UK[h] and, with r_comp, q_rope_out = q_rope r_comp (see include/mla_qcache.h)."""
    B, H, d = q_nope.shape
    if tuple(w_uk.shape) != (H, d, 512) or tuple(q_lat.shape) != (B, H, 512):
        raise ValueError("absorb_query: q_nope [B, H, d], w_uk [H, d, 512], q_lat [B, H, 512]")
    if r_comp is not None and (tuple(r_comp.shape) != (64, 64) or q_rope is None or q_rope_out is None):
        raise ValueError("absorb_query: r_comp [64, 64] needs q_rope and q_rope_out [B, H, 64]")
    st = lib().mla_qcache_absorb_query(
        B, H, d, _ptr(q_nope, "q_nope", 2), _ptr(w_uk, "w_uk", 2), _ptr(q_rope, "q_rope", 2, allow_none=True),
        _ptr(r_comp, "r_comp", 2, allow_none=True), _ptr(q_lat, "q_lat", 2),
        _ptr(q_rope_out, "q_rope_out", 2, allow_none=True), _stream(stream))
    _raise(st, "mla_qcache_absorb_query")


def mla_qcache_up_project(o, w_uv, out, stream=None) -> None:
    """out = BF16(O) W_UV[h] (float32 out, see include/mla_qcache.h)."""
    B, H, _ = o.shape
    d_v = w_uv.shape[2]
    if tuple(w_uv.shape) != (H, 512, d_v) or tuple(out.shape) != (B, H, d_v):
        raise ValueError("up_project: o [B, H, 512], w_uv [H, 512, d_v], out [B, H, d_v]")
    st = lib().mla_qcache_up_project(B, H, d_v, _ptr(o, "o", dtype=torch.float32), _ptr(w_uv, "w_uv", 2),
                                     _ptr(out, "out", dtype=torch.float32), _stream(stream))
    _raise(st, "mla_qcache_up_project")


def bf16_workspace_bytes(B: int, H: int, max_pages: int, page_size: int) -> int:
    return int(lib().mla_qcache_bf16_workspace_bytes(B, H, max_pages, page_size))


def mla_qcache_decode_attn_bf16(q_lat, q_rope, page_table, page_size: int, seq_lens, kv_pool, softmax_scale: float,
                                out, lse, workspace, err_word, stream=None) -> None:
    """Decode attention over a paged BF16 cache kv_pool [n_pages, page_size, 576] (the
    unquantized comparator, see include/mla_qcache.h)."""
    if kv_pool.dim() != 3 or kv_pool.shape[1] != page_size or kv_pool.shape[2] != 576:
        raise ValueError(f"kv_pool must be [n_pages, {page_size}, 576], got {tuple(kv_pool.shape)}")
    _check_decode_shapes(q_lat, q_rope, page_table, seq_lens, out, lse)
    B, H = q_lat.shape[0], q_lat.shape[1]
    st = lib().mla_qcache_decode_attn_bf16(
        B, H, _ptr(q_lat, "q_lat", 2), _ptr(q_rope, "q_rope", 2), _ptr(page_table, "page_table", dtype=torch.int32),
        page_table.shape[1], int(page_size), _ptr(seq_lens, "seq_lens", dtype=torch.int32),
        _ptr(kv_pool, "kv_pool", 2), kv_pool.shape[0], ctypes.c_float(softmax_scale),
        _ptr(out, "out", dtype=torch.float32), _ptr(lse, "lse", dtype=torch.float32), _ptr(workspace, "workspace", 1),
        workspace.numel(), _ptr(err_word, "err_word", dtype=torch.int32), _stream(stream))
    _raise(st, "mla_qcache_decode_attn_bf16")


def mla_qcache_advance(cu_new, seq_lens, stream=None) -> None:
    """seq_lens[b] += cu_new[b+1] - cu_new[b] on the device (see include/mla_qcache.h)."""
    st = lib().mla_qcache_advance(_ptr(cu_new, "cu_new", dtype=torch.int32),
                                  _ptr(seq_lens, "seq_lens", dtype=torch.int32), seq_lens.shape[0], _stream(stream))
    _raise(st, "mla_qcache_advance")


def mla_qcache_decode_attn(cfg: Config, q_lat, q_rope, page_table, seq_lens, pool, sink_buf, recent_buf,
                           softmax_scale: float, out, lse, workspace, err_word, stream=None) -> None:
    """Decode attention over the quantized cache (see include/mla_qcache.h)."""
    _check_decode_shapes(q_lat, q_rope, page_table, seq_lens, out, lse)
    B, H = q_lat.shape[0], q_lat.shape[1]
    st = lib().mla_qcache_decode_attn(
        ctypes.byref(cfg), B, H, _ptr(q_lat, "q_lat", 2), _ptr(q_rope, "q_rope", 2),
        _ptr(page_table, "page_table", dtype=torch.int32), page_table.shape[1],
        _ptr(seq_lens, "seq_lens", dtype=torch.int32), _ptr(pool, "pool", 1), pool.shape[0],
        _ptr(sink_buf, "sink_buf", 2, allow_none=True) if cfg.n_sink else None, _ptr(recent_buf, "recent_buf", 2),
        ctypes.c_float(softmax_scale), _ptr(out, "out", dtype=torch.float32), _ptr(lse, "lse", dtype=torch.float32),
        _ptr(workspace, "workspace", 1), workspace.numel() * workspace.element_size(),
        _ptr(err_word, "err_word", dtype=torch.int32), _stream(stream))
    _raise(st, "mla_qcache_decode_attn")


def mla_qcache_decode_attn_pending(cfg: Config, q_lat, q_rope, page_table, seq_lens, c_new, kr_new, cu_new,
                                   max_new: int, pool, sink_buf, recent_buf, softmax_scale: float, out, lse, workspace,
                                   err_word, stream=None) -> None:
    """Decode of the cache as the pending write of rows c_new / kr_new / cu_new will leave it
    (seq_lens: lengths before that write); the write may run concurrently on another stream
    (see include/mla_qcache.h)."""
    _check_decode_shapes(q_lat, q_rope, page_table, seq_lens, out, lse)
    B, H = q_lat.shape[0], q_lat.shape[1]
    if cu_new is None or cu_new.dim() != 1 or cu_new.shape[0] != B + 1:
        raise ValueError(f"cu_new must be [{B + 1}]")
    if c_new is None or c_new.dim() != 2 or c_new.shape[1] != 512 or kr_new is None or \
            tuple(kr_new.shape) != (c_new.shape[0], 64):
        raise ValueError("c_new must be [rows, 512] and kr_new [rows, 64]")
    st = lib().mla_qcache_decode_attn_pending(
        ctypes.byref(cfg), B, H, _ptr(q_lat, "q_lat", 2), _ptr(q_rope, "q_rope", 2),
        _ptr(page_table, "page_table", dtype=torch.int32), page_table.shape[1],
        _ptr(seq_lens, "seq_lens", dtype=torch.int32), _ptr(c_new, "c_new", 2), _ptr(kr_new, "kr_new", 2),
        _ptr(cu_new, "cu_new", dtype=torch.int32), int(max_new), _ptr(pool, "pool", 1), pool.shape[0],
        _ptr(sink_buf, "sink_buf", 2, allow_none=True) if cfg.n_sink else None, _ptr(recent_buf, "recent_buf", 2),
        ctypes.c_float(softmax_scale), _ptr(out, "out", dtype=torch.float32), _ptr(lse, "lse", dtype=torch.float32),
        _ptr(workspace, "workspace", 1), workspace.numel() * workspace.element_size(),
        _ptr(err_word, "err_word", dtype=torch.int32), _stream(stream))
    _raise(st, "mla_qcache_decode_attn_pending")


def noalloc_scratch_bytes() -> int:
    """Size of the scratch built into the library for mla_qcache_decode_attn_noalloc."""
    return int(lib().mla_qcache_noalloc_scratch_bytes())


def mla_qcache_decode_attn_noalloc(cfg: Config, q_lat, q_rope, page_table, seq_lens, pool, sink_buf, recent_buf,
                                   softmax_scale: float, out, lse, err_word, stream=None) -> None:
    """Decode attention without a workspace argument: for callers that cannot allocate device
    memory, it runs on a scratch buffer compiled into the library (see include/mla_qcache.h)."""
    _check_decode_shapes(q_lat, q_rope, page_table, seq_lens, out, lse)
    B, H = q_lat.shape[0], q_lat.shape[1]
    st = lib().mla_qcache_decode_attn_noalloc(
        ctypes.byref(cfg), B, H, _ptr(q_lat, "q_lat", 2), _ptr(q_rope, "q_rope", 2),
        _ptr(page_table, "page_table", dtype=torch.int32), page_table.shape[1],
        _ptr(seq_lens, "seq_lens", dtype=torch.int32), _ptr(pool, "pool", 1), pool.shape[0],
        _ptr(sink_buf, "sink_buf", 2, allow_none=True) if cfg.n_sink else None, _ptr(recent_buf, "recent_buf", 2),
        ctypes.c_float(softmax_scale), _ptr(out, "out", dtype=torch.float32), _ptr(lse, "lse", dtype=torch.float32),
        _ptr(err_word, "err_word", dtype=torch.int32), _stream(stream))
    _raise(st, "mla_qcache_decode_attn_noalloc")
