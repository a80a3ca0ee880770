"""Pins of the oracle's NVFP4 quantiser Q: exhaustive round-trips of exactly
representable blocks, tie direction at every midpoint for every scale, the
scale rule on every bf16 block maximum, and scaling / sign invariances."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import formats as F
from oracle import quant as Q

F32 = np.float32


def _pack(nibbles):
    n = np.asarray(nibbles, dtype=np.uint8)
    return (n[..., 0::2] | (n[..., 1::2] << 4)).astype(np.uint8)


@pytest.mark.parametrize("s", [2.0 ** -6, 1.0, 2.0 ** -13, 2.0 ** 7])
def test_round_trip_every_scale_and_code(s):
    """x = e2m1(c) * S * s with a +-6 in the block quantises back to (c, S)."""
    codes = np.arange(16, dtype=np.uint8)  # every code, including +-6 and -0
    rows, expect_scales = [], []
    for S in range(1, 0x7F):
        Sval = F.E4M3_VALUES[S]
        rows.append((F.e2m1_value(codes) * Sval * s).astype(F32))
        expect_scales.append(S)
    x = np.stack(rows)
    got_codes, got_scales = Q.quantize_rows(x, F32(s))
    np.testing.assert_array_equal(got_scales[:, 0], np.array(expect_scales, dtype=np.uint8))
    np.testing.assert_array_equal(got_codes, np.broadcast_to(_pack(codes), got_codes.shape))
    # dequantisation gives the inputs back exactly
    np.testing.assert_array_equal(Q.dequantize_rows(got_codes, got_scales, F32(s)), x)


def test_round_trip_fails_without_a_six():
    """A block whose largest code is 4 picks a smaller scale (4/6 of S rounded),
    so its codes do not round-trip: the rule really is amax/6."""
    x = np.array([[4.0] + [1.0] * 15], dtype=F32)
    _, sc = Q.quantize_rows(x, F32(1.0))
    assert F.e4m3_value(sc[0, 0]) == 0.6875  # RNE(4/6) on the E4M3 grid


@pytest.mark.parametrize("S", list(range(1, 0x7F, 5)) + [0x7E, 0x38, 0x08, 0x01])
def test_midpoints_pin_tie_direction(S):
    Sval = F32(F.E4M3_VALUES[S])
    grid = F.E2M1_MAGNITUDES
    # m == 1 exactly when s = 1/S is a power of two: then v == x and nextafter
    # neighbours are exact one-ulp neighbours of the midpoints.
    pow2 = float(Sval) == 2.0 ** np.floor(np.log2(float(Sval)))
    s = F32(1.0 / float(Sval)) if pow2 else F32(1.0)
    m = F32(Sval * s)
    vals, expect = [], []
    for i in range(7):
        mid = (grid[i] + grid[i + 1]) / 2
        even = i if i % 2 == 0 else i + 1
        if pow2:
            up = np.nextafter(F32(mid), F32(np.inf))
            dn = np.nextafter(F32(mid), F32(0))
        else:
            up, dn = mid + 2.0 ** -10, mid - 2.0 ** -10
        for v, code in ((mid, even), (up, i + 1), (dn, i), (-mid, even | 8)):
            vals.append(F32(F32(v) * m))
            expect.append(code)
    # pad to whole blocks, each block led by 6*m so that the block scale is S
    blocks, codes = [], []
    for b in range(0, len(vals), 15):
        chunk = vals[b:b + 15]
        cc = expect[b:b + 15]
        while len(chunk) < 15:
            chunk.append(F32(0.0))
            cc.append(0)
        blocks.append([F32(6.0 * m)] + chunk)
        codes.append([7] + cc)
    x = np.array(blocks, dtype=F32).reshape(1, -1)
    got_codes, got_scales = Q.quantize_rows(x, s)
    assert np.all(got_scales == S)
    np.testing.assert_array_equal(Q.unpack_codes(got_codes)[0], np.array(codes).reshape(-1))


@pytest.mark.parametrize("s", [1.0, 2.0 ** -6, 0.0123])
def test_scale_rule_every_bf16_block_max(s):
    """For every positive finite bf16 block max a: S = E4M3_RNE(a / (6 s)) with
    the two fp32 operations done in IEEE fp32, E4M3 rounding checked in exact
    rationals."""
    a = F.f32_from_bf16_bits(np.arange(0x0001, 0x7F80, dtype=np.uint16))
    x = np.zeros((a.size, 16), dtype=F32)
    x[:, 3] = a
    _, scales = Q.quantize_rows(x, F32(s))
    d = F32(F32(6.0) * F32(s))
    with np.errstate(over="ignore"):
        q = (a / d).astype(F32)
    finite = [Fraction(float(v)) for v in F.E4M3_FINITE]
    fin = np.array([float(v) for v in F.E4M3_FINITE])
    for qi, got in zip(q[::7], scales[::7, 0]):
        if not np.isfinite(qi) or float(qi) >= float(finite[-1]):
            assert got == 0x7E
            continue
        fq = Fraction(float(qi))
        lo = int(np.searchsorted(fin, float(qi), side="right") - 1)
        hi = lo + 1
        dl, dh = fq - finite[lo], finite[hi] - fq
        exp = lo if dl < dh else hi if dh < dl else (lo if lo % 2 == 0 else hi)
        assert got == exp


def test_zero_scale_block_gives_zero_codes():
    x = np.zeros((1, 32), dtype=F32)
    x[0, 0] = 100.0          # block 0 fine
    x[0, 16:] = -1e-9        # block 1 rounds to scale 0 -> all codes 0 (no sign)
    c, sc = Q.quantize_rows(x, F32(100.0 / 2688))
    assert sc[0, 1] == 0 and np.all(c[0, 8:] == 0)
    assert sc[0, 0] != 0


def test_tensor_scale_rule():
    assert Q.tensor_scale(0.0) == F32(1.0)
    assert Q.tensor_scale(F32(2688.0)) == F32(1.0)
    assert Q.tensor_scale(F32(3.0)) == F32(F32(3.0) / F32(2688.0))


def test_power_of_two_scaling_invariance():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((8, 256)).astype(F32)
    c0, s0, t0 = Q.quantize_tensor(x)
    for n in (-5, -1, 3, 9):
        c1, s1, t1 = Q.quantize_tensor((x * F32(2.0 ** n)).astype(F32))
        np.testing.assert_array_equal(c0, c1)
        np.testing.assert_array_equal(s0, s1)
        assert t1 == F32(t0 * F32(2.0 ** n))


def test_negation_flips_only_sign_bits():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((8, 256)).astype(F32)
    c0, s0, t0 = Q.quantize_tensor(x)
    c1, s1, t1 = Q.quantize_tensor(-x)
    np.testing.assert_array_equal(s0, s1)
    assert t0 == t1
    nz = np.repeat(s0 != 0, 8, axis=1)
    np.testing.assert_array_equal(c1[nz], c0[nz] ^ 0x88)


def test_quantisation_error_bound():
    """Away from saturation every element is within half a grid step of x/m."""
    rng = np.random.default_rng(7)
    x = rng.standard_normal((16, 512)).astype(F32)
    c, sc, s = Q.quantize_tensor(x)
    xh = Q.dequantize_rows(c, sc, s)
    m = np.repeat(F.e4m3_value(sc) * float(s), 16, axis=1)
    step = np.where(np.abs(x) / m < 2, 0.5, np.where(np.abs(x) / m < 4, 1.0, 2.0))
    assert np.all(np.abs(xh - x) <= step / 2 * m * (1 + 1e-6) + 1e-30)
