"""Pins of the oracle's projections either side of attention (RAQ-MLA page, Figure 4): closed
forms with identity, per-head scaled and single-entry weights, a hand-worked product, torch's
BF16 rounding, and the BF16 rounding of the float32 attention output before the product."""
import numpy as np
import torch

import oracle


def _bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _vals(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def test_hand_worked_product():
    x = _bits([[[1.0, 2.0]]])
    w = _bits([[[3.0, 4.0], [5.0, 6.0]]])
    assert np.array_equal(oracle.project(x, w), [[[13.0, 16.0]]])


def test_identity_and_per_head_scaled_identity():
    rng = np.random.default_rng(0)
    B, H, K = 3, 4, 32
    x = _bits(rng.standard_normal((B, H, K)))
    eye = np.stack([np.eye(K) * (h + 1) for h in range(H)])
    y = oracle.project(x, _bits(eye))
    want = _vals(x) * (np.arange(H) + 1)[None, :, None]
    assert np.array_equal(y, want)


def test_row_times_matrix_single_entry():
    B, H, K, N = 2, 3, 16, 32
    w = np.zeros((H, K, N), np.float32)
    w[:, 0, 5] = 1.0
    x = _bits(np.random.default_rng(1).standard_normal((B, H, K)))
    y = oracle.project(x, _bits(w))
    assert np.array_equal(y[:, :, 5], _vals(x)[:, :, 0])
    assert not np.any(np.delete(y, 5, axis=2))


def test_one_matrix_for_every_head_equals_per_head_copies():
    rng = np.random.default_rng(2)
    x = _bits(rng.standard_normal((2, 5, 64)))
    r = _bits(rng.standard_normal((64, 64)) / 8)
    assert np.array_equal(oracle.project(x, r), oracle.project(x, np.broadcast_to(r, (5, 64, 64)).copy()))


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.standard_normal(50000) * 10.0 ** rng.integers(-8, 8, 50000),
                        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 0.0])])
    want = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle._round_bf16(v.astype(np.float32).astype(np.float64)), want)
    # exact ties go to the even pattern: 1 + 2^-8 -> 1, 1 + 3 * 2^-8 -> 1 + 2^-6
    assert _vals(oracle._round_bf16(np.array([1.0 + 2.0 ** -8])))[0] == 1.0
    assert _vals(oracle._round_bf16(np.array([1.0 + 3 * 2.0 ** -8])))[0] == 1.0 + 2.0 ** -6


def test_float32_output_is_rounded_to_bf16_before_the_product():
    o = np.full((1, 1, 512), 1.0 + 2.0 ** -10, np.float32)  # rounds to 1.0 in BF16
    w = np.zeros((1, 512, 128), np.float32)
    w[0, :, 0] = 1.0
    y = oracle.up_project(o, _bits(w))
    assert y[0, 0, 0] == 512.0


def test_absorb_query_rounds_the_exact_products():
    rng = np.random.default_rng(4)
    q = _bits(rng.standard_normal((2, 3, 128)))
    w = _bits(rng.standard_normal((3, 128, 512)) / 11)
    qr = _bits(rng.standard_normal((2, 3, 64)))
    r = _bits(rng.standard_normal((64, 64)) / 8)
    ql_bits, qr_bits, ql, qrx = oracle.absorb_query(q, w, qr, r)
    assert np.all(np.abs(_vals(ql_bits) - ql) <= np.abs(ql) * 2.0 ** -8)
    assert np.all(np.abs(_vals(qr_bits) - qrx) <= np.abs(qrx) * 2.0 ** -8)
