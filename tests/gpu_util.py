"""Helpers for the GPU parity tests: move workload inputs to the device and run the library."""
import numpy as np
import torch

import bit_mla_kv_qcache_gb300 as q
import oracle


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def gpu_cache(cfg_kw, inp):
    cfg = q.make_config(**cfg_kw)
    B = inp.seq_lens.shape[0]
    return q.QuantizedMLACache(cfg, B, inp.page_table.shape[1], inp.n_pages,
                               page_table=torch.from_numpy(inp.page_table), device="cuda")


def write_rows(cache, c, kr, counts, max_new):
    cu = np.zeros(len(counts) + 1, np.int32)
    cu[1:] = np.cumsum(counts)
    cache.write(dev(c), dev(kr), dev(cu), max_new)


def oracle_cache(cfg_kw, inp):
    cfg = oracle.make_config(**cfg_kw)
    B = inp.seq_lens.shape[0]
    pool = np.zeros((inp.n_pages, oracle.page_bytes(cfg)), np.uint8)
    sink = np.zeros((B, cfg.n_sink, 576), np.uint16)
    ring = np.zeros((B, cfg.n_recent, 576), np.uint16)
    return cfg, pool, sink, ring


def assert_cache_equal(cache, pool, sink, ring):
    torch.cuda.synchronize()
    gp = cache.pool.cpu().numpy()
    if not np.array_equal(gp, pool):
        bad = np.argwhere(gp != pool)
        raise AssertionError(f"pool differs at {len(bad)} bytes, first {bad[:5].tolist()}")
    assert np.array_equal(cache.sink.cpu().numpy().view(np.uint16), sink), "sink buffer differs"
    assert np.array_equal(cache.ring.cpu().numpy().view(np.uint16), ring), "recent ring differs"


def rel_err_rows(o, o_ref):
    """Per-(b,h) row: max |O - O*| / max |O*| (rows with O* = 0 use the absolute error)."""
    num = np.abs(o - o_ref).max(-1)
    den = np.abs(o_ref).max(-1)
    return np.where(den > 0, num / np.where(den > 0, den, 1), num)


def check_decode(out, lse, o_ref, l_ref, tol=2e-3):
    o = out.cpu().double().numpy()
    l = lse.cpu().double().numpy()
    rel = rel_err_rows(o, o_ref)
    assert np.all(np.isfinite(o)), "non-finite output"
    assert rel.max() <= tol, f"max row-relative error {rel.max():.3e} > {tol}"
    both_inf = np.isneginf(l) & np.isneginf(l_ref)
    with np.errstate(invalid="ignore"):
        d = np.where(both_inf, 0.0, np.abs(l - l_ref))
    assert d.max() <= tol, f"max |dLSE| {d.max():.3e} > {tol}"
    return rel.max(), d.max()
