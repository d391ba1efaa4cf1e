"""Projections either side of the decode attention (RAQ-MLA page, Figure 4) on the GPU against
the oracle's exact float64 products: query absorption through W_UK (BF16 out), the query-side
k_R compensation, and the W_UV up-projection of the float32 attention output.

Tolerance, from the arithmetic: the tensor cores multiply BF16 operands exactly and add in
float32, so |Y - Y*| <= 2 K 2^-24 sum_k |x_k w_k| (a generous float32 accumulation bound);
a BF16 result adds one rounding, 2^-8 |Y*|."""
import numpy as np
import pytest
import torch

import bit_mla_kv_qcache_gb300 as q
import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _bits(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _vals(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def _acc_bound(x, w, K):
    xa = np.abs(x)
    wa = np.abs(w)
    s = np.einsum("bhk,kn->bhn", xa, wa) if wa.ndim == 2 else np.einsum("bhk,hkn->bhn", xa, wa)
    return 2 * K * 2.0 ** -24 * s


@pytest.mark.parametrize("B,H,d", [(1, 16, 128), (7, 16, 128), (64, 4, 128), (100, 3, 64), (5, 2, 512), (3, 1, 16)])
def test_absorb_query(B, H, d):
    rng = np.random.default_rng(B * 100 + d)
    qn = _bits(rng.standard_normal((B, H, d)))
    w = _bits(rng.standard_normal((H, d, 512)) / np.sqrt(d))
    qr = _bits(rng.standard_normal((B, H, 64)))
    r = _bits(rng.standard_normal((64, 64)) / 8)
    ql = torch.empty((B, H, 512), dtype=torch.int16, device="cuda")
    qro = torch.empty((B, H, 64), dtype=torch.int16, device="cuda")
    q.mla_qcache_absorb_query(gu.dev(qn), gu.dev(w), ql, q_rope=gu.dev(qr), r_comp=gu.dev(r), q_rope_out=qro)
    torch.cuda.synchronize()
    _, _, ql_x, qr_x = oracle.absorb_query(qn, w, qr, r)
    got = _vals(ql.cpu().numpy().view(np.uint16))
    assert np.all(np.abs(got - ql_x) <= 2.0 ** -8 * np.abs(ql_x) + _acc_bound(_vals(qn), _vals(w), d))
    got_r = _vals(qro.cpu().numpy().view(np.uint16))
    assert np.all(np.abs(got_r - qr_x) <= 2.0 ** -8 * np.abs(qr_x) + _acc_bound(_vals(qr), _vals(r), 64))
    # most outputs are the correctly rounded exact products
    assert np.mean(ql.cpu().numpy().view(np.uint16) == oracle._round_bf16(ql_x)) > 0.98


def test_absorb_query_without_compensation_leaves_rope_alone():
    B, H, d = 2, 16, 128
    rng = np.random.default_rng(9)
    qn = _bits(rng.standard_normal((B, H, d)))
    w = _bits(rng.standard_normal((H, d, 512)) / 11)
    ql = torch.empty((B, H, 512), dtype=torch.int16, device="cuda")
    q.mla_qcache_absorb_query(gu.dev(qn), gu.dev(w), ql)
    torch.cuda.synchronize()
    ql_x = oracle.project(qn, w)
    assert np.all(np.abs(_vals(ql.cpu().numpy().view(np.uint16)) - ql_x)
                  <= 2.0 ** -8 * np.abs(ql_x) + _acc_bound(_vals(qn), _vals(w), d))


@pytest.mark.parametrize("B,H,dv", [(1, 16, 128), (32, 16, 128), (65, 2, 256), (3, 5, 32)])
def test_up_project(B, H, dv):
    rng = np.random.default_rng(B + dv)
    o = (rng.standard_normal((B, H, 512)) * 0.3).astype(np.float32)
    w = _bits(rng.standard_normal((H, 512, dv)) / 22.6)
    out = torch.empty((B, H, dv), dtype=torch.float32, device="cuda")
    q.mla_qcache_up_project(torch.from_numpy(o).cuda(), gu.dev(w), out)
    torch.cuda.synchronize()
    want = oracle.up_project(o, w)
    ob = _vals(oracle._round_bf16(o.astype(np.float64)))
    assert np.all(np.abs(out.cpu().double().numpy() - want) <= _acc_bound(ob, _vals(w), 512))
