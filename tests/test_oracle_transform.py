"""Pins of the oracle's cached-tensor transform x -> x A (RAQ-MLA page, Figure 4) against
closed forms, hand-worked float32 sums, torch's float64 matmul with the recursive-summation
error bound, and torch's BF16 rounding."""
import numpy as np
import pytest
import torch

import oracle
import workloads


def _bf16(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _val(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).float().numpy()


def _rows(n, d, seed=0):
    rng = np.random.default_rng(seed)
    return _bf16(rng.standard_normal((n, d)).astype(np.float32))


@pytest.mark.parametrize("d", [64, 512])
def test_identity_keeps_rows(d):
    x = _rows(7, d)
    _, out = oracle.row_transform(x, _bf16(np.eye(d, dtype=np.float32)))
    assert np.array_equal(out, x)


@pytest.mark.parametrize("d", [64, 512])
def test_signed_scaled_permutation_is_exact(d):
    """A[i, pi(i)] = s_i 2^k: column pi(i) of the result is s_i 2^k x_i, exactly."""
    rng = np.random.default_rng(3)
    pi = rng.permutation(d)
    s = rng.choice([-1.0, 1.0], d)
    a = np.zeros((d, d), np.float32)
    a[np.arange(d), pi] = s * 0.125
    x = _rows(5, d, 1)
    _, out = oracle.row_transform(x, _bf16(a))
    want = np.zeros((5, d), np.float32)
    want[:, pi] = _val(x) * (s * 0.125)[None, :]
    assert np.array_equal(_val(out), want)


def test_row_times_matrix_not_matrix_times_column():
    """A single entry A[0, 1] = 1 moves channel 0 into channel 1 (x A, not A x)."""
    d = 64
    a = np.zeros((d, d), np.float32)
    a[0, 1] = 1.0
    x = _rows(3, d, 2)
    _, out = oracle.row_transform(x, _bf16(a))
    v = _val(out)
    assert np.array_equal(v[:, 1], _val(x)[:, 0])
    assert not np.any(np.delete(v, 1, axis=1))


def test_accumulation_order_is_channel_order():
    """x = (2^24, 1, 1, -2^24), A = all ones: in channel order 2^24 + 1 rounds back to 2^24
    (a tie, to even) twice and the sum is 0; a pairwise sum would give 2."""
    d = 4
    x = _bf16(np.array([[2.0 ** 24, 1.0, 1.0, -(2.0 ** 24)]], np.float32))
    acc, out = oracle.row_transform(x, _bf16(np.ones((d, d), np.float32)))
    assert np.all(acc == 0.0) and np.all(_val(out) == 0.0)


@pytest.mark.parametrize("d,scale", [(512, 1 / 16), (64, 1 / 4)])
def test_random_matrix_within_float32_summation_bound(d, scale):
    """Against torch float64 (exact products; float64 summation error far below float32's):
    |acc - x A| <= (d - 1) 2^-24 sum_i |x_i A_ij| (recursive summation), and the stored value
    is torch's BF16 rounding of acc."""
    rng = np.random.default_rng(11)
    a = _bf16((rng.standard_normal((d, d)) * scale).astype(np.float32))
    x = _rows(64, d, 4)
    acc, out = oracle.row_transform(x, a)
    xv, av = torch.from_numpy(_val(x)).double(), torch.from_numpy(_val(a)).double()
    exact = (xv @ av).numpy()
    bound = (d - 1) * 2.0 ** -24 * (xv.abs() @ av.abs()).numpy()
    assert np.all(np.abs(acc.astype(np.float64) - exact) <= bound)
    assert np.array_equal(out, _bf16(acc))
    # the float32 sums round to the same BF16 as the exact products almost everywhere
    assert np.mean(out == _bf16(exact.astype(np.float32))) > 0.99


def test_write_transformed_is_write_of_transformed_rows():
    """The writer with A_c / A_R caches exactly what the plain writer caches for the rows x A."""
    w = workloads.Workload("t", 1, 16, 1, 4, 32, n_sink=4, n_recent=32, seed=5)
    inp = workloads.make_inputs(w, seq_lens=np.array([70, 33], np.int32))
    cfg = oracle.make_config(**w.config_kwargs())
    rng = np.random.default_rng(6)
    a_c = _bf16((rng.standard_normal((512, 512)) / 22.6).astype(np.float32))
    a_r = _bf16((rng.standard_normal((64, 64)) / 8).astype(np.float32))
    pb = oracle.page_bytes(cfg)

    def fresh():
        return (np.zeros((inp.n_pages, pb), np.uint8), np.zeros((2, 4, 576), np.uint16),
                np.zeros((2, 32, 576), np.uint16))

    p1, s1, r1 = fresh()
    assert oracle.write_transformed(cfg, inp.c, inp.kr, inp.cu, np.zeros(2, np.int32), 70, inp.page_table,
                                    p1, s1, r1, a_c=a_c, a_r=a_r) == 0
    p2, s2, r2 = fresh()
    c2 = oracle.row_transform(inp.c, a_c)[1]
    k2 = oracle.row_transform(inp.kr, a_r)[1]
    assert oracle.write(cfg, c2, k2, inp.cu, np.zeros(2, np.int32), 70, inp.page_table, p2, s2, r2) == 0
    assert np.array_equal(p1, p2) and np.array_equal(s1, s2) and np.array_equal(r1, r2)
    # the retained BF16 rows are the transformed ones
    assert np.array_equal(s1[0, :, :512], c2[:4]) and np.array_equal(s1[0, :, 512:], k2[:4])
