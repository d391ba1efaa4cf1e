"""The C ABI library loads and exports every entry point include/mla_qcache.h declares; host-side
validation answers without touching a GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from bit_mla_kv_qcache_gb300 import build
    build.build()
    import bit_mla_kv_qcache_gb300 as q
    return q


def _declared():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names += re.findall(r"\b(mla_qcache_\w+)\s*\(", txt)
    return sorted(set(names))


def test_exports_every_declared_symbol(L):
    declared = _declared()
    assert len(declared) >= 6
    lib = L.lib()
    for name in declared:
        assert hasattr(lib, name), name
    assert set(L.EXPORTS) <= set(declared)


def test_page_bytes_and_config_check(L):
    assert L.page_bytes(L.make_config(4, 128)) == 39168
    assert L.page_bytes(L.make_config(2, 64)) == 11520
    lib = L.lib()
    bad = [L.make_config(3, 128), L.make_config(4, 96), L.make_config(4, 128, n_recent=64),
           L.make_config(4, 64, n_sink=17), L.make_config(4, 64, clip_q=1.5), L.make_config(4, 64, bits_r=2),
           L.make_config(4, 16, n_recent=16)]
    for c in bad:
        assert lib.mla_qcache_config_check(ctypes.byref(c)) == -2
        assert L.page_bytes(c) == 0
    assert lib.mla_qcache_config_check(None) == -1
    assert lib.mla_qcache_config_check(ctypes.byref(L.make_config(2, 64))) == 0


def test_strerror(L):
    for s in range(-6, 1):
        assert isinstance(L.strerror(s), str) and L.strerror(s)
    assert L.strerror(-99) == "unknown status"


def test_host_validation_without_gpu(L):
    lib = L.lib()
    cfg = L.make_config(4, 128)
    p = ctypes.c_void_p(16 * 1024)  # never dereferenced: validation fails first
    # zero rows: nothing to do
    assert lib.mla_qcache_write(ctypes.byref(cfg), 1, 0, None, None, None, None, 1, None, 1, None, 1, None, None,
                                None, None) == 0
    # missing pointers
    assert lib.mla_qcache_write(ctypes.byref(cfg), 1, 4, None, p, p, p, 1, p, 1, p, 1, p, p, p, None) == -1
    # bad sizes
    assert lib.mla_qcache_write(ctypes.byref(cfg), 0, 4, p, p, p, p, 1, p, 1, p, 1, p, p, p, None) == -3
    assert lib.mla_qcache_write(ctypes.byref(cfg), 1, 4, p, p, p, p, 0, p, 1, p, 1, p, p, p, None) == -3
    # more write CTAs than one grid dimension holds (4 per page that may fill, per sequence)
    assert lib.mla_qcache_write(ctypes.byref(cfg), 1 << 20, 4, p, p, p, p, 1 << 20, p, 1, p, 1, p, p, p,
                                None) == -3
    # misaligned pool
    assert lib.mla_qcache_write(ctypes.byref(cfg), 1, 4, p, p, p, p, 1, p, 1, ctypes.c_void_p(16 * 1024 + 4), 1,
                                p, p, p, None) == -4
    f = ctypes.c_float(0.1)
    # decode: H not a multiple of 16, null output, bad config
    assert lib.mla_qcache_decode_attn(ctypes.byref(cfg), 1, 24, p, p, p, 1, p, p, 1, p, p, f, p, p, p, 1 << 20, p,
                                      None) == -3
    assert lib.mla_qcache_decode_attn(ctypes.byref(cfg), 1, 16, p, p, p, 1, p, p, 1, p, p, f, None, p, p, 1 << 20,
                                      p, None) == -1
    bad = L.make_config(4, 128, n_recent=64)
    assert lib.mla_qcache_decode_attn(ctypes.byref(bad), 1, 16, p, p, p, 1, p, p, 1, p, p, f, p, p, p, 1 << 20, p,
                                      None) == -2
    # length update: NULL pointers, B < 1, misaligned arrays are rejected before any launch
    assert lib.mla_qcache_advance(None, p, 4, None) == -1
    assert lib.mla_qcache_advance(p, None, 4, None) == -1
    assert lib.mla_qcache_advance(p, p, 0, None) == -3
    assert lib.mla_qcache_advance(ctypes.c_void_p(16 * 1024 + 2), p, 4, None) == -4
    # unquantized comparator: shapes, page size, pointers, alignment
    f = ctypes.c_float(0.1)
    bf = lambda B, H, P, pool, ws: lib.mla_qcache_decode_attn_bf16(B, H, p, p, p, 4, P, p, pool, 8, f, p, p, ws, 1 << 20,
                                                                   p, None)
    assert bf(0, 16, 64, p, p) == -3 and bf(1, 24, 64, p, p) == -3
    assert bf(1, 16, 48, p, p) == -2
    assert bf(1, 16, 64, None, p) == -1
    assert bf(1, 16, 64, ctypes.c_void_p(16 * 1024 + 4), p) == -4
    assert lib.mla_qcache_bf16_workspace_bytes(1, 24, 4, 64) == 0 and lib.mla_qcache_bf16_workspace_bytes(1, 16, 4, 48) == 0
    # fused write + length update: a second, non-overlapping, aligned length array is required
    p2 = ctypes.c_void_p(32 * 1024)
    args = lambda lens, nxt: (ctypes.byref(cfg), 4, 4, p, p, p, lens, nxt, 1, p, 1, p, 1, p, p, p, None)
    assert lib.mla_qcache_write_advance(*args(p, None)) == -1
    assert lib.mla_qcache_write_advance(*args(p, p)) == -3
    assert lib.mla_qcache_write_advance(*args(p, ctypes.c_void_p(16 * 1024 + 8))) == -3  # overlaps [p, p+16)
    assert lib.mla_qcache_write_advance(*args(p, ctypes.c_void_p(32 * 1024 + 2))) == -4
    # the write's own checks still apply (bad config)
    assert lib.mla_qcache_write_advance(ctypes.byref(L.make_config(4, 128, n_recent=64)), 4, 4, p, p, p, p, p2, 1, p,
                                        1, p, 1, p, p, p, None) == -2


def test_transform_entry_points_validate_on_the_host(L):
    lib = L.lib()
    cfg = L.make_config(4, 128)
    p, p2 = ctypes.c_void_p(16 * 1024), ctypes.c_void_p(64 * 1024)
    odd = ctypes.c_void_p(16 * 1024 + 2)

    def wt(a_c, a_r, nxt=None, B=4, lens=p, n_rows=4):
        return lib.mla_qcache_write_transformed(ctypes.byref(cfg), B, n_rows, p, p, p, lens, nxt, 1, a_c, a_r, p, 1,
                                                p, 1, p, p, p, None)

    assert wt(odd, None) == -4 and wt(None, odd) == -4  # transforms need 16-byte alignment
    assert wt(ctypes.c_void_p(16 * 1024 + 8), None) == -4
    assert wt(p, p, nxt=p) == -3  # overlapping length arrays
    assert wt(p, p, nxt=ctypes.c_void_p(32 * 1024 + 2)) == -4
    assert wt(p, p, B=0) == -3
    # eight CTAs per transformed row count against the grid limit
    assert lib.mla_qcache_write_transformed(ctypes.byref(cfg), 1, (1 << 28) + 8, p, p, p, p, None, 1, p, None, p, 1,
                                            p, 1, p, p, p, None) == -3
    # standalone transform: dim, sizes, pointers, alignment, overlap
    e = ctypes.c_void_p(128 * 1024)
    assert lib.mla_qcache_row_transform(4, 128, p, p, p2, e, None) == -3
    assert lib.mla_qcache_row_transform(-1, 512, p, p, p2, e, None) == -3
    assert lib.mla_qcache_row_transform(0, 512, None, None, None, None, None) == 0
    assert lib.mla_qcache_row_transform(4, 512, None, p, p2, e, None) == -1
    assert lib.mla_qcache_row_transform(4, 512, p, p, p2, None, None) == -1
    assert lib.mla_qcache_row_transform(4, 512, ctypes.c_void_p(16 * 1024 + 1), p, p2, e, None) == -4
    assert lib.mla_qcache_row_transform(4, 512, p, ctypes.c_void_p(16 * 1024 + 4), p2, e, None) == -4  # a: 16 B
    assert lib.mla_qcache_row_transform(4, 512, p, p, ctypes.c_void_p(16 * 1024 + 2048), e, None) == -3  # overlaps x


def test_projection_entry_points_validate_on_the_host(L):
    lib = L.lib()
    p, odd = ctypes.c_void_p(16 * 1024), ctypes.c_void_p(16 * 1024 + 8)
    aq = lambda B, H, d, qr, r, qro, x=p: lib.mla_qcache_absorb_query(B, H, d, x, p, qr, r, p, qro, None)
    assert aq(0, 16, 128, None, None, None) == 0  # nothing to do
    assert aq(4, 16, 100, None, None, None) == -3 and aq(4, 16, 1024, None, None, None) == -3
    assert aq(4, 0, 128, None, None, None) == -3
    assert aq(4, 16, 128, p, p, None) == -1  # r_comp without an output
    assert aq(4, 16, 128, None, p, p) == -1  # r_comp without q_rope
    assert aq(4, 16, 128, None, None, None, x=odd) == -4
    up = lambda B, H, dv, o=p: lib.mla_qcache_up_project(B, H, dv, o, p, p, None)
    assert up(4, 16, 100) == -3 and up(4, 16, 0) == -3 and up(-1, 16, 128) == -3
    assert up(4, 16, 128, o=None) == -1 and up(4, 16, 128, o=odd) == -4
    assert up(0, 16, 128, o=None) == 0


def test_multi_token_decode_validates_on_the_host(L):
    lib = L.lib()
    cfg = L.make_config(4, 128)  # W = 128
    p = ctypes.c_void_p(16 * 1024)
    f = ctypes.c_float(0.1)
    mt = lambda H, ql: lib.mla_qcache_decode_attn_multi(ctypes.byref(cfg), 1, H, ql, p, p, p, 1, p, p, 1, p, p, f, p,
                                                        p, p, 1 << 20, p, None)
    assert mt(16, 0) == -3 and mt(24, 2) == -3  # q_len >= 1, heads a multiple of 16
    assert mt(16, 17) == -3  # at most 256 rows
    assert mt(1, 130) == -3  # q_len - 1 <= W (and heads a multiple of 16)


def test_product_path_has_no_cpu_fallback(L, monkeypatch):
    """Without the built library the binding raises instead of computing anything else."""
    import bit_mla_kv_qcache_gb300.binding as b
    monkeypatch.setattr(b, "_lib", None)
    monkeypatch.setattr(b, "_LIB_PATH", "/nonexistent/libmla_qcache.so")
    with pytest.raises(b.QCacheError):
        b.lib()
    src = open(os.path.join(ROOT, "bit_mla_kv_qcache_gb300", "binding.py")).read()
    src += open(os.path.join(ROOT, "bit_mla_kv_qcache_gb300", "cache.py")).read()
    assert "import oracle" not in src and "from oracle" not in src


def test_decode_plan_shapes(L):
    """The share rules of the decode, checked on the host for a 152-SM GB300 (three 16-head CTAs
    or one 64-head CTA per SM)."""
    sms, wave = 152, 3 * 152
    c4 = L.make_config(4, 128)
    # the 32 x 8K, 16-head configuration: one wave of 13 packed shares + 1 protected CTA
    p = L.decode_plan(c4, 32, 16, 66, sms)
    assert (p["n_split"], p["n_protected"], p["share_slots"], p["tensor_memory"]) == (13, 1, 0, False)
    assert 32 * (p["n_split"] + p["n_protected"]) <= wave
    # one sequence at 16 heads over a long table takes a whole wave of shares (not 64), the
    # protected CTAs included (several of them when the packed work per share is small)
    for mp in (513, 514, 2050, 8194):
        p = L.decode_plan(c4, 1, 16, mp, sms)
        assert p["n_split"] == wave - p["n_protected"] and p["share_slots"] == 0
    assert L.decode_plan(c4, 1, 16, 513, sms)["n_protected"] > 1
    # a one-wave plan never launches more CTAs than one wave holds
    for B in (1, 2, 3, 4, 8, 16, 32):
        for mp in (2, 9, 33, 129, 236, 257, 385, 513, 1025):
            p = L.decode_plan(c4, B, 16, mp, sms)
            if p["share_slots"] == 0:
                assert B * (p["n_split"] + p["n_protected"]) <= wave, (B, mp, p)
    # the minimum share: four 32-token tiles, except for up to 32 sequence-head groups: one
    # tile for short tables (up to 96 tiles), two up to 384, four beyond
    p = L.decode_plan(c4, 33, 16, 6, sms)
    assert p["n_split"] == 6 * 128 // 32 // 4
    p = L.decode_plan(c4, 8, 16, 10, sms)
    assert p["n_split"] == 10 * 128 // 32
    p = L.decode_plan(c4, 4, 16, 30, sms)
    assert p["n_split"] == 30 * 128 // 32 // 2
    p = L.decode_plan(c4, 1, 16, 10, sms)
    assert p["n_split"] == 10 * 128 // 32
    p = L.decode_plan(c4, 1, 16, 66, sms)
    assert p["n_split"] == 66 * 128 // 32 // 2
    p = L.decode_plan(c4, 1, 16, 130, sms)
    assert p["n_split"] == 130 * 128 // 32 // 4
    # eight long sequences: more shares than a wave, in the balanced instance
    p = L.decode_plan(c4, 8, 16, 8194, sms)
    assert p["n_split"] == 64 and p["share_slots"] == wave - 8 * p["n_protected"]
    # 64-head blocks on the tensor-memory kernel: one wave of one CTA per SM
    for B, H in ((1, 128), (8, 128), (2, 64)):
        p = L.decode_plan(c4, B, H, 1026, sms)
        assert p["tensor_memory"] and p["n_split"] == sms // (B * H // 64)
    # the BF16 comparator: one wave of shares, or a whole number of waves when shares would be long
    for B, mp in ((1, 8194), (8, 8194), (32, 2050)):
        parts = L.decode_plan(c4, B, 16, mp, sms)["bf16_parts"]
        per_wave = wave // B
        assert parts <= 8 * per_wave and (parts <= per_wave or parts % per_wave == 0)
    # errors
    assert L.lib().mla_qcache_decode_plan(ctypes.byref(c4), 1, 24, 10, sms, (ctypes.c_int32 * 5)()) == -3
    assert L.lib().mla_qcache_decode_launches(ctypes.byref(c4), 1, 24, 10) == -3
    assert L.lib().mla_qcache_decode_launches(ctypes.byref(c4), 0, 16, 10) == -3
    assert L.lib().mla_qcache_decode_launches(None, 1, 16, 10) == -1
    assert L.lib().mla_qcache_decode_plan(ctypes.byref(c4), 1, 16, 10, sms, None) == -1


def test_binding_rejects_bad_shapes_before_any_call(L):
    """Shape errors surface as ValueError in the binding (CPU tensors suffice: nothing is launched)."""
    import torch
    b = L
    i16 = lambda *s: torch.zeros(*s, dtype=torch.int16)
    f32 = lambda *s: torch.zeros(*s, dtype=torch.float32)
    with pytest.raises(ValueError):
        b.mla_qcache_absorb_query(i16(2, 16, 128), i16(16, 128, 256), i16(2, 16, 512))  # w_uk not [H, d, 512]
    with pytest.raises(ValueError):
        b.mla_qcache_absorb_query(i16(2, 16, 128), i16(16, 128, 512), i16(2, 16, 512), r_comp=i16(64, 64))
    with pytest.raises(ValueError):
        b.mla_qcache_up_project(f32(2, 16, 512), i16(16, 512, 128), f32(2, 16, 64))
    with pytest.raises(ValueError):
        b.mla_qcache_row_transform(i16(4, 512), i16(512, 64), i16(4, 512), torch.zeros(1, dtype=torch.int32))
    cfg = b.make_config(4, 128)
    with pytest.raises(ValueError):
        b.mla_qcache_write_transformed(cfg, i16(1, 512), i16(1, 64), None, torch.zeros(1, dtype=torch.int32), 1,
                                       None, None, None, None, None, a_c=i16(64, 64))
    with pytest.raises(ValueError):
        b.mla_qcache_decode_attn_multi(cfg, 3, i16(1, 16, 512), i16(1, 16, 64), None, None, None, None, None, 0.1,
                                       None, None, None, None)
    with pytest.raises(ValueError):
        b.mla_qcache_decode_attn_bf16(i16(1, 16, 512), i16(1, 16, 64), None, 64, None, i16(4, 32, 576), 0.1,
                                      None, None, None, None)
    from bit_mla_kv_qcache_gb300 import binding
    # the single-token decode wrappers (workspace and allocation-free): every tensor's shape is
    # checked against q_lat's [B, H] before a pointer is taken
    B, H = 2, 16
    good = dict(q_lat=i16(B, H, 512), q_rope=i16(B, H, 64), page_table=torch.zeros((B, 4), dtype=torch.int32),
                seq_lens=torch.zeros(B, dtype=torch.int32), out=f32(B, H, 512), lse=f32(B, H))
    bad = [("q_lat", i16(B, H, 256)), ("q_rope", i16(B, H, 32)), ("q_rope", i16(B + 1, H, 64)),
           ("out", f32(B, H, 256)), ("out", f32(B, H - 1, 512)), ("lse", f32(B)), ("lse", f32(B, H + 16)),
           ("seq_lens", torch.zeros(B + 1, dtype=torch.int32)), ("page_table", torch.zeros((B + 1, 4), dtype=torch.int32)),
           ("page_table", torch.zeros(4, dtype=torch.int32))]
    for name, t in bad:
        a = dict(good, **{name: t})
        with pytest.raises(ValueError):
            b.mla_qcache_decode_attn(cfg, a["q_lat"], a["q_rope"], a["page_table"], a["seq_lens"], None, None, None,
                                     0.1, a["out"], a["lse"], None, None)
        with pytest.raises(ValueError):
            binding.mla_qcache_decode_attn_noalloc(cfg, a["q_lat"], a["q_rope"], a["page_table"], a["seq_lens"], None, None,
                                             None, 0.1, a["out"], a["lse"], None)


def test_pending_decode_validates_on_the_host(L):
    """mla_qcache_decode_attn_pending: max_new beyond W - P + 1, missing or misaligned row
    pointers are rejected before any launch; the decode's own checks still apply."""
    lib = L.lib()
    p, odd = ctypes.c_void_p(16 * 1024), ctypes.c_void_p(16 * 1024 + 8)
    f = ctypes.c_float(0.1)
    call = lambda cfg, H, c, k, cu, mx: lib.mla_qcache_decode_attn_pending(
        ctypes.byref(cfg), 1, H, p, p, p, 1, p, c, k, cu, mx, p, 1, p, p, f, p, p, p, 1 << 20, p, None)
    c4 = L.make_config(4, 128)                 # W - P + 1 = 1
    c32 = L.make_config(4, 32, n_recent=128)   # W - P + 1 = 97
    assert call(c4, 16, p, p, p, 2) == -3 and call(c4, 16, p, p, p, -1) == -3
    assert call(c32, 16, p, p, p, 98) == -3
    assert call(c4, 16, None, p, p, 1) == -1 and call(c4, 16, p, None, p, 1) == -1 and call(c4, 16, p, p, None, 1) == -1
    assert call(c4, 16, odd, p, p, 1) == -4 and call(c4, 16, p, odd, p, 1) == -4
    assert call(c4, 24, p, p, p, 1) == -3  # H not a multiple of 16
    assert call(L.make_config(4, 128, n_recent=64), 16, p, p, p, 1) == -2
