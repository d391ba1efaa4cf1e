"""Pins of the oracle's quantizer (RAQ-MLA page, appendix Table 5) and per-token clip.

The references here do not reuse the oracle's arithmetic: hand-worked golden cases, exact
rational brute force over every finite FP16 value and every level, and the invariants the
definition implies (|dequant - x| <= scale/2, codes in [0, L], extremes hit 0 and L).
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# every finite FP16 value as an exact rational, sorted
with np.errstate(invalid="ignore"):
    _F16 = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float64)
_F16_FINITE = sorted({Fraction(float(v)) for v in _F16 if np.isfinite(v)})


def _parse_values(field):
    out = []
    for tok in field.split(","):
        tok = tok.strip()
        out.append(float.fromhex(tok) if "0x" in tok.lower() else float(tok))
    return out


def _golden_cases():
    cases = []
    with open(os.path.join(GOLDEN, "quantizer_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, bits, vals, mn, sc, codes = [x.strip() for x in line.split("|")]
            cases.append((name, int(bits), _parse_values(vals), int(mn, 16), int(sc, 16),
                          [int(c) for c in codes.split(",")]))
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c[0])
def test_golden_hand_worked_cases(case):
    name, bits, vals, mn_bits, sc_bits, codes = case
    got_codes, sb, mb, flags = oracle.quantize(vals, bits)
    assert flags == 0
    assert mb == mn_bits, f"{name}: min bits {mb:#06x} != {mn_bits:#06x}"
    assert sb == sc_bits, f"{name}: scale bits {sb:#06x} != {sc_bits:#06x}"
    assert list(got_codes) == codes


def _brute_force(vals, bits):
    """Exact rational restatement: search all finite FP16 values and all levels."""
    L = (1 << bits) - 1
    xs = [Fraction(v) for v in vals]
    lo, hi = min(xs), max(xs)
    mn = max(v for v in _F16_FINITE if v <= lo)
    sc = min(v for v in _F16_FINITE if v >= 0 and mn + L * v >= hi)
    codes = []
    for x in xs:
        best = None
        for k in range(L + 1):
            d = abs(x - (mn + k * sc))
            if best is None or d < best[0] or (d == best[0] and k % 2 == 0 and best[1] % 2 == 1):
                best = (d, k)
        codes.append(best[1] if sc > 0 else 0)
    return mn, sc, codes


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("seed", range(6))
def test_matches_exact_brute_force(bits, seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(2, 24))
    scale = 10.0 ** rng.uniform(-6, 3)
    vals = (rng.standard_normal(n) * scale + rng.standard_normal() * scale).astype(np.float32)
    # bf16-representable inputs, as the cache stores
    vals = ((vals.view(np.uint32) + 0x8000) & 0xFFFF0000).view(np.float32).astype(np.float64)
    if seed % 3 == 0:  # plant exact half-level ties
        mn0 = float(np.float16(vals.min()))
        vals = np.concatenate([vals, [vals.min(), mn0 + 0.5 * 2.0 ** -3]])
    mn, sc, codes = _brute_force(list(vals), bits)
    got_codes, sb, mb, flags = oracle.quantize(vals, bits)
    assert flags == 0
    assert Fraction(oracle.f16_to_double(mb)) == mn
    assert Fraction(oracle.f16_to_double(sb)) == sc
    assert list(got_codes) == codes


@pytest.mark.parametrize("bits,n", [(4, 128), (2, 128), (4, 64), (4, 16)])
def test_invariants_random(bits, n):
    """|x_hat - x| <= scale/2 exactly; codes in range; extremes map to 0 and L."""
    rng = np.random.default_rng(bits * 1000 + n)
    L = (1 << bits) - 1
    for trial in range(200):
        x = rng.standard_normal(n) * (10.0 ** rng.uniform(-3, 2))
        if trial % 5 == 0:
            x = rng.standard_t(3, n)
        x = ((x.astype(np.float32).view(np.uint32) + 0x8000) & 0xFFFF0000).view(np.float32).astype(np.float64)
        codes, sb, mb, flags = oracle.quantize(x, bits)
        assert flags == 0
        s, m = oracle.f16_to_double(sb), oracle.f16_to_double(mb)
        assert codes.max() <= L
        xh = m + codes.astype(np.float64) * s
        assert np.all(np.abs(xh - x) <= s / 2)  # exact in double for these magnitudes
        assert m <= x.min()
        if s > 0:
            assert codes[np.argmin(x)] == 0
            assert codes[np.argmax(x)] == L
        # scale is the smallest FP16 that covers the range
        prev = oracle.f16_to_double(sb - 1) if sb > 0 else None
        assert m + L * s >= x.max()
        if prev is not None:
            assert m + L * prev < x.max()


def test_constant_and_zero_groups():
    codes, sb, mb, fl = oracle.quantize(np.zeros(128), 4)
    assert fl == 0 and sb == 0 and mb == 0 and codes.max() == 0
    codes, sb, mb, fl = oracle.quantize(np.full(128, -2.5), 2)
    assert fl == 0 and sb == 0 and oracle.f16_to_double(mb) == -2.5 and codes.max() == 0


def test_range_and_nonfinite_flags():
    _, _, _, fl = oracle.quantize(np.array([0.0, 1e6]), 4)
    assert fl & oracle.ERR_RANGE
    _, _, _, fl = oracle.quantize(np.array([-1e6, 0.0]), 4)
    assert fl & oracle.ERR_RANGE
    _, _, _, fl = oracle.quantize(np.array([0.0, np.nan]), 4)
    assert fl & oracle.ERR_NONFINITE


def test_clip_golden_ramp():
    """Values +-1..+-512: the 0.94 nearest-rank quantile of |x| is the 482nd smallest = 482."""
    rng = np.random.default_rng(5)
    x = np.arange(1, 513, dtype=np.float64) * rng.choice([-1.0, 1.0], 512)
    rng.shuffle(x)
    tau = oracle.clip_tau(x, 0.94)
    assert tau == 482.0
    assert int(np.sum(np.abs(x) > tau)) == 30


@pytest.mark.parametrize("seed", range(5))
def test_clip_order_statistic_properties(seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_t(5, 512).astype(np.float32).astype(np.float64)
    if seed == 3:
        x[:100] = 0.25  # many ties
    tau = oracle.clip_tau(x, 0.94)
    k = int(np.ceil(np.float64(np.float32(0.94)) * 512))
    assert k == 482
    a = np.abs(x)
    assert tau in set(a.tolist())
    assert np.sum(a <= tau) >= k and np.sum(a < tau) < k
    assert tau == np.sort(a)[k - 1]
    assert np.sum(a > tau) <= 512 - k
    assert oracle.clip_tau(x, 1.0) == a.max()
