"""S5/S6: expert SwiGLU FFN on NVFP4 operands and the weighted combine
(oracle; test infrastructure only).

Reading taken (the pages say the GPU expert path is W4A4 -- "capy-flash
v0.7.1: a 125B MoE on 64 GB of RAM ...", "Why it matters" -- and print no
expert formula):
  * g = Wg x_hat, u = Wu x_hat with NVFP4 weights and the NVFP4 activation row,
    products and sums in float64 on the exactly dequantised operands;
  * h = silu(g) * u with silu(z) = z / (1 + exp(-z)), in float64, then rounded
    once to float32 (the precision the quantiser works in);
  * h_hat = Q(h; s_h) with the layer's static tensor scale s_h;
  * o = Wd h_hat in float64;
  * y_t = sum_j w_tj * o_(t, j), summed in slot order j = 0 .. k-1.
"""
import numpy as np

from .quant import dequantize_rows, quantize_rows

F32 = np.float32


class NVFP4Experts:
    """One NVFP4 weight matrix per expert: codes [E][N][K/2], scales [E][N][K/16],
    tensor scales [E].  ``dequant(e)`` gives the exact float64 matrix [N][K]."""

    def __init__(self, codes, scales, tensor_scales):
        self.codes = codes
        self.scales = scales
        self.tensor_scales = np.asarray(tensor_scales, dtype=np.float32)

    @property
    def num_experts(self) -> int:
        return self.codes.shape[0]

    @property
    def rows(self) -> int:
        return self.codes.shape[1]

    def quantized(self, e: int):
        return self.codes[e], self.scales[e], self.tensor_scales[e]

    def dequant(self, e: int) -> np.ndarray:
        return dequantize_rows(self.codes[e], self.scales[e], self.tensor_scales[e])


def silu(z):
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def gate_up(x_hat, wg_hat, wu_hat):
    """g = Wg x_hat and u = Wu x_hat for rows of x_hat [m][H]; float64 [m][I] each."""
    return x_hat @ wg_hat.T, x_hat @ wu_hat.T


def swiglu(g, u) -> np.ndarray:
    """h = silu(g) * u in float64."""
    return silu(g) * u


def gate_up_swiglu(x_hat, wg_hat, wu_hat) -> np.ndarray:
    """h = silu(Wg x_hat) * (Wu x_hat) for rows of x_hat [m][H]; float64 [m][I]."""
    return swiglu(*gate_up(x_hat, wg_hat, wu_hat))


def requantize_h(h64, s_h):
    """h rounded once to float32, then Q with the static scale s_h."""
    h32 = np.asarray(h64, dtype=np.float64).astype(F32)
    codes, scales = quantize_rows(h32, F32(s_h))
    return h32, codes, scales


def down(h_hat, wd_hat) -> np.ndarray:
    """o = Wd h_hat for rows of h_hat [m][I]; float64 [m][H]."""
    return h_hat @ wd_hat.T


def combine(weights, outputs) -> np.ndarray:
    """y = sum_j w_j * o_j in slot order; weights [k], outputs [k][H]."""
    y = np.zeros(outputs.shape[1], dtype=np.float64)
    for j in range(outputs.shape[0]):
        y = y + weights[j] * outputs[j]
    return y
