"""Pins of the oracle's NVFP4 element/scale formats against things other than
the oracle: bit-field formulas, torch's float8 conversion, exact rationals and
the printed format constants in tests/golden/nvfp4_format.txt."""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_format.txt")


def _golden():
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        out[key] = vals
    return out


def test_golden_constants():
    g = _golden()
    assert list(F.E2M1_MAGNITUDES) == [float(v) for v in g["e2m1_grid"]]
    assert F.E4M3_VALUES[int(g["e4m3_max_code"][0], 16)] == float(g["e4m3_max"][0])
    assert np.isnan(F.E4M3_VALUES[int(g["e4m3_nan_code"][0], 16)])
    assert F.E4M3_VALUES[0x08] == float(g["e4m3_min_normal"][0])
    assert F.E4M3_VALUES[0x01] == float(g["e4m3_min_subnormal"][0])


def test_e2m1_all_16_codes_match_bit_fields():
    for code in range(16):
        sign = -1.0 if code & 8 else 1.0
        e = (code >> 1) & 3
        m = code & 1
        expect = sign * (m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1))
        got = F.e2m1_value(code)
        assert got == expect and np.signbit(got) == (code >= 8), code


def test_e4m3_all_codes_match_integer_formula_and_torch():
    # value = N * 2^(E - 10) with N = m (E = 0, read as exponent 1) or 8 + m
    for code in range(127):
        e, m = code >> 3, code & 7
        expect = Fraction(m, 2 ** 9) if e == 0 else Fraction(8 + m) * Fraction(2) ** (e - 10)
        assert Fraction(F.E4M3_VALUES[code]) == expect, hex(code)
    codes = torch.arange(127, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(ref, F.E4M3_VALUES[:127])
    assert np.isnan(F.E4M3_VALUES[0x7F])


def _e4m3_exact_rne(q: Fraction) -> int:
    """Exact-rational E4M3 rounding: nearest finite value, ties to even code,
    saturate at 448 (integer comparisons only)."""
    vals = [Fraction(float(v)) for v in F.E4M3_FINITE]
    if q >= vals[-1]:
        return len(vals) - 1
    lo, hi = 0, len(vals) - 1
    while hi - lo > 1:          # vals[lo] <= q < vals[hi]
        mid = (lo + hi) // 2
        if vals[mid] <= q:
            lo = mid
        else:
            hi = mid
    dl, dh = q - vals[lo], vals[hi] - q
    if dl < dh:
        return lo
    if dh < dl:
        return hi
    return lo if lo % 2 == 0 else hi


def _all_positive_finite_bf16():
    bits = np.arange(0x0001, 0x7F80, dtype=np.uint16)
    return F.f32_from_bf16_bits(bits)


def test_e4m3_encode_exhaustive_over_bf16_against_exact_rationals():
    qs = _all_positive_finite_bf16()
    got = F.e4m3_encode_rne_satfinite(qs)
    expect = np.array([_e4m3_exact_rne(Fraction(float(q))) for q in qs], dtype=np.uint8)
    np.testing.assert_array_equal(got, expect)


def test_e4m3_encode_matches_torch_below_saturation():
    rng = np.random.default_rng(1)
    q = np.concatenate([
        _all_positive_finite_bf16(),
        rng.uniform(0, 448, 200000).astype(np.float32),
        np.exp2(rng.uniform(-14, 8.8, 200000)).astype(np.float32),
    ])
    q = q[q <= 448].astype(np.float32)
    ref = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(F.e4m3_encode_rne_satfinite(q), ref)


def test_e4m3_saturates():
    big = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e6, 3e38], dtype=np.float32)
    assert np.all(F.e4m3_encode_rne_satfinite(big) == 0x7E)


def test_e2m1_midpoints_and_neighbours():
    grid = F.E2M1_MAGNITUDES
    for i in range(7):
        mid = np.float32((grid[i] + grid[i + 1]) / 2)
        even = i if i % 2 == 0 else i + 1
        assert F.e2m1_encode_rne_satfinite(mid) == even
        assert F.e2m1_encode_rne_satfinite(np.nextafter(mid, np.float32(np.inf))) == i + 1
        assert F.e2m1_encode_rne_satfinite(np.nextafter(mid, np.float32(0))) == i
        assert F.e2m1_encode_rne_satfinite(-mid) == (even | 8)
    # the tie table written out: 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for v, r in ties.items():
        assert F.e2m1_value(F.e2m1_encode_rne_satfinite(np.float32(v))) == r


def test_e2m1_saturation_and_signed_zero():
    assert F.e2m1_encode_rne_satfinite(np.float32(6.5)) == 7
    assert F.e2m1_encode_rne_satfinite(np.float32(1e30)) == 7
    assert F.e2m1_encode_rne_satfinite(np.float32(-7.0)) == 15
    assert F.e2m1_encode_rne_satfinite(np.float32(0.0)) == 0
    assert F.e2m1_encode_rne_satfinite(np.float32(-0.0)) == 8
    assert F.e2m1_encode_rne_satfinite(np.float32(-0.2)) == 8
    assert F.e2m1_encode_rne_satfinite(np.float32(0.2)) == 0


def test_e2m1_encode_brute_force_random():
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(20000) * 3).astype(np.float32)
    got = F.e2m1_encode_rne_satfinite(v)
    grid = [Fraction(float(g)) for g in F.E2M1_MAGNITUDES]
    for x, c in zip(v[:4000], got[:4000]):
        a = Fraction(float(abs(x)))
        dists = [abs(a - g) for g in grid]
        best = min(dists)
        cands = [i for i, d in enumerate(dists) if d == best]
        mag = cands[0] if len(cands) == 1 else [i for i in cands if i % 2 == 0][0]
        if a > grid[-1]:
            mag = 7
        assert (c & 7) == mag and bool(c & 8) == bool(np.signbit(x))


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32),
                        (rng.standard_normal(1000) * 1e30).astype(np.float32),
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.0078125 - 2 ** -20], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(F.bf16_bits_from_f32_rne(x), ref)
    back = F.f32_from_bf16_bits(ref)
    np.testing.assert_array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16)
                                  .to(torch.float32).numpy())
