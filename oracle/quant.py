"""Q: the NVFP4 block quantiser (oracle; test infrastructure only).

The GPU path of the engine is W4A4 ("capy-flash v0.7.1: a 125B MoE on 64 GB of
RAM ...", "Why it matters"), so activations and the SwiGLU output are
quantised to NVFP4 on the fly.  The pages do not print the quantiser; this is
the plainest reading of the NVFP4 recipe, fixed as a sequence of correctly
rounded fp32 operations so that both implementations reach the same codes:

  1. A = max |x| over the tensor (exact).
  2. tensor scale s = A / 2688 (2688 = 6 * 448), or 1 when A == 0; for the
     SwiGLU output the layer's static scale s_h is used instead.
  3. for each block of 16 consecutive elements of a row:
       a = max |x_i| over the block,  d = 6 * s,  q = a / d,
       S = E4M3(q), round to nearest even, saturating at 448.
  4. S == 0: all 16 codes are 0.  Otherwise m = S * s, v_i = x_i / m and
     c_i = E2M1(v_i), round to nearest even, saturating at 6, sign bit = sign
     of x_i.
  5. dequantised value: e2m1(c_i) * S * s.

Every "*" and "/" above is one fp32 operation with round-to-nearest-even (no
fused multiply-add); numpy float32 arithmetic is exactly that.  Packing: the
even element of a pair goes to the low nibble; blocks run along the row, which
is always the contraction axis of the matmul that consumes the codes.
"""
import numpy as np

from .formats import (e2m1_encode_rne_satfinite, e2m1_value, e4m3_encode_rne_satfinite,
                      e4m3_value)

F32 = np.float32
BLOCK = 16
SCALE_DIVISOR = F32(6.0 * 448.0)   # 2688


def tensor_scale(amax) -> np.float32:
    """Q step 2: fp32 tensor scale from the tensor's max magnitude."""
    a = F32(amax)
    if a == 0:
        return F32(1.0)
    return F32(a / SCALE_DIVISOR)


def quantize_rows(x, s) -> tuple:
    """Q steps 3-4 on a float32 matrix [R][K] (K % 16 == 0) with tensor scale s.

    Returns (codes uint8 [R][K/2], scales uint8 [R][K/16]).
    """
    x = np.asarray(x, dtype=np.float32)
    rows, cols = x.shape
    assert cols % BLOCK == 0
    s = F32(s)
    blocks = x.reshape(rows, cols // BLOCK, BLOCK)
    a = np.max(np.abs(blocks), axis=2)
    d = F32(F32(6.0) * s)
    with np.errstate(over="ignore"):   # a / d may exceed fp32: saturates below
        q = (a / d).astype(F32)
    S = e4m3_encode_rne_satfinite(q)
    m = (e4m3_value(S).astype(F32) * s).astype(F32)
    nonzero = S != 0
    m_safe = np.where(nonzero, m, F32(1.0)).astype(F32)
    v = (blocks / m_safe[:, :, None]).astype(F32)
    c = e2m1_encode_rne_satfinite(v)
    c = np.where(nonzero[:, :, None], c, np.uint8(0)).astype(np.uint8)
    flat = c.reshape(rows, cols)
    codes = (flat[:, 0::2] | (flat[:, 1::2] << 4)).astype(np.uint8)
    return codes, S.astype(np.uint8)


def quantize_tensor(x) -> tuple:
    """Q with a dynamic tensor scale: returns (codes, scales, s)."""
    x = np.asarray(x, dtype=np.float32)
    s = tensor_scale(np.max(np.abs(x)) if x.size else F32(0))
    codes, scales = quantize_rows(x.reshape(-1, x.shape[-1]), s)
    return codes, scales, s


def unpack_codes(codes) -> np.ndarray:
    """Nibbles [R][K] from packed bytes [R][K/2] (low nibble = even element)."""
    codes = np.asarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = codes & 0xF
    out[..., 1::2] = codes >> 4
    return out


def dequantize_rows(codes, scales, s) -> np.ndarray:
    """Q step 5: exact float64 values e2m1(c) * S * s of a quantised matrix."""
    vals = e2m1_value(unpack_codes(codes))
    sc = np.repeat(e4m3_value(scales), BLOCK, axis=-1)
    return vals * sc * np.float64(F32(s))
