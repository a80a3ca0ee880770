"""NVFP4 element and scale formats (oracle; test infrastructure only).

NVFP4 is NVIDIA's 4-bit floating-point format that the capy-flash engine was
built around (capy-flash status post, "What it's for"): 4-bit E2M1 elements,
one unsigned E4M3 scale per block of 16 consecutive elements and one fp32
scale per tensor.

E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit, no inf or NaN.
      Codes 0..7 are the magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; bit 3 is the sign.
E4M3: (the "fn" FP8 variant) 4 exponent bits (bias 7), 3 mantissa bits,
      subnormals m * 2^-9, largest finite 448 (code 0x7E), 0x7F is NaN.
      Block scales are non-negative, so their sign bit is always 0.

The encoders round to nearest with ties to the even code and saturate to the
largest finite magnitude ("satfinite").  They work by brute force over the
value grid, in float64 where every difference is exact.
"""
import numpy as np

E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def _e4m3_values() -> np.ndarray:
    vals = np.empty(128, dtype=np.float64)
    for code in range(128):
        e, m = code >> 3, code & 7
        if code == 0x7F:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = m * 2.0 ** -9
        else:
            vals[code] = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


E4M3_VALUES = _e4m3_values()          # indexed by code 0..127 (sign bit clear)
E4M3_FINITE = E4M3_VALUES[:0x7F]      # codes 0..126, ascending
E4M3_MAX = 448.0


def e2m1_value(codes) -> np.ndarray:
    """Value of E2M1 nibbles (0..15) as float64."""
    c = np.asarray(codes, dtype=np.uint8)
    mag = E2M1_MAGNITUDES[c & 7]
    return np.where((c & 8) != 0, -mag, mag)


def e4m3_value(codes) -> np.ndarray:
    """Value of unsigned E4M3 scale bytes as float64 (0x7F is NaN)."""
    c = np.asarray(codes, dtype=np.uint8)
    return E4M3_VALUES[c & 0x7F]


def nearest_index_rne(v, grid: np.ndarray) -> np.ndarray:
    """Index of the grid value nearest to each v >= 0; exact ties go to the even
    index; v at or beyond the last grid value maps to the last index.

    ``grid`` is ascending and its index is the format's code, so "even index"
    is "even mantissa".
    """
    v = np.asarray(v, dtype=np.float64)
    n = len(grid)
    i = np.clip(np.searchsorted(grid, v, side="right") - 1, 0, n - 1)
    j = np.minimum(i + 1, n - 1)
    below = v - grid[i]
    above = grid[j] - v
    take_upper = (above < below) | ((above == below) & (i % 2 == 1))
    return np.where(i == n - 1, n - 1, np.where(take_upper, j, i)).astype(np.int64)


def e4m3_encode_rne_satfinite(q) -> np.ndarray:
    """Unsigned E4M3 code of q >= 0 (round to nearest even, saturate at 448)."""
    return nearest_index_rne(q, E4M3_FINITE).astype(np.uint8)


def e2m1_encode_rne_satfinite(v) -> np.ndarray:
    """E2M1 nibble of v: magnitude rounded to nearest even on the 8-value grid,
    saturated at 6; the sign bit copies the sign of v (so -0.2 -> 0x8)."""
    v = np.asarray(v, dtype=np.float64)
    mag = nearest_index_rne(np.abs(v), E2M1_MAGNITUDES).astype(np.uint8)
    return mag | np.where(np.signbit(v), np.uint8(8), np.uint8(0))


def bf16_bits_from_f32_rne(x32) -> np.ndarray:
    """bf16 bit patterns of finite float32 values, round to nearest even."""
    u = np.asarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def f32_from_bf16_bits(b) -> np.ndarray:
    """float32 values of bf16 bit patterns (exact)."""
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32)
