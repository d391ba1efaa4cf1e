"""Pins of the oracle's number-format helpers against numpy's independent float16/float32 code."""
import math

import numpy as np
import pytest

pytestmark = pytest.mark.usefixtures("oracle_lib")


def test_f16_decode_all_patterns(oracle_lib):
    # numpy's binary16 decoder is an independent implementation of the same IEEE format.
    pats = np.arange(65536, dtype=np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([oracle_lib.f16_to_double(int(p)) for p in pats])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_f16_bits_roundtrip_finite():
    import oracle
    pats = np.arange(65536, dtype=np.uint16)
    vals = pats.view(np.float16).astype(np.float64)
    for p, v in zip(pats, vals):
        if not np.isfinite(v):
            continue
        if v == 0.0:
            assert oracle.f16_bits(v) == 0  # zero is always encoded as +0
            continue
        assert oracle.f16_bits(v) == int(p)


def test_bf16_decode_matches_numpy_view():
    import oracle
    rng = np.random.default_rng(1)
    pats = rng.integers(0, 65536, size=4000).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        ref = (pats.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = np.array([oracle.bf16_to_double(int(p)) for p in pats])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


@pytest.mark.parametrize("seed", [0, 1])
def test_directed_roundings_bracket_numpy_nearest(seed):
    """rd16(x) <= x <= ru16(x), both are FP16 values, adjacent, and numpy's RN is the nearer."""
    import oracle
    rng = np.random.default_rng(seed)
    mags = np.exp(rng.uniform(math.log(1e-9), math.log(60000.0), size=3000))
    xs = mags * rng.choice([-1.0, 1.0], size=mags.size)
    xs = np.concatenate([xs, [0.0, -0.0, 65504.0, -65504.0, 6.103515625e-05, 5.960464477539063e-08,
                              1.0, 1.0 + 2.0 ** -11, 1.0 + 2.0 ** -10]])
    for x in xs:
        lo, r1 = oracle.f16_round_down(float(x))
        hi, r2 = oracle.f16_round_up(float(x))
        assert not r1 and not r2
        assert lo <= x <= hi
        for v in (lo, hi):
            assert np.float16(v).astype(np.float64) == v  # exactly representable
        rn = float(np.float16(x))  # numpy: float64 -> float16, round to nearest even
        assert rn in (lo, hi)
        if lo != hi:
            bits = int(np.float16(lo).view(np.uint16))
            nxt_bits = bits + 1 if lo >= 0 else bits - 1  # next FP16 value above lo
            nxt = float(np.uint16(nxt_bits).view(np.float16))
            assert nxt == hi, (x, lo, hi, nxt)
            assert abs(rn - x) <= min(abs(lo - x), abs(hi - x))


def test_directed_rounding_range_flags():
    import oracle
    _, r = oracle.f16_round_down(-70000.0)
    assert r
    _, r = oracle.f16_round_up(70000.0)
    assert r
    v, r = oracle.f16_round_down(70000.0)
    assert v == 65504.0 and not r
    v, r = oracle.f16_round_up(-70000.0)
    assert v == -65504.0 and not r
