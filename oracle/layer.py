"""The whole routed-expert MoE layer and a stack of layers (oracle; test
infrastructure only).

Steps, in the order the layer runs them (each implemented in its own module):
  S1/S2  router.py   logits in float64, full-sort top-k, renormalised softmax
  S3     quant.py    x_hat = Q(x) with one dynamic tensor scale per call
  S4     permute.py  pairs grouped by expert, token order inside an expert
  S5     expert.py   h = silu(Wg x_hat) * (Wu x_hat), h_hat = Q(float32(h); s_h)
  S6     expert.py   o = Wd h_hat, y_t = sum_j w_tj o_(t,j) in slot order
  stack  x_next = bf16(float32(x) + float32(y)), round to nearest even

Per-expert work is grouped by expert so that each dequantised weight matrix is
built once; every pair still gets exactly the per-pair result above.
"""
import numpy as np

from .expert import NVFP4Experts, combine, down, gate_up, requantize_h, swiglu
from .formats import bf16_bits_from_f32_rne, f32_from_bf16_bits
from .permute import permute
from .quant import dequantize_rows, quantize_rows, tensor_scale
from .router import route, router_logits

F32 = np.float32


def quantize_weight_matrix(w):
    """One expert matrix [N][K] fp32 -> (codes, scales, tensor scale), with the
    tensor scale taken from this matrix's own max magnitude."""
    w = np.asarray(w, dtype=np.float32)
    s = tensor_scale(np.max(np.abs(w)))
    codes, scales = quantize_rows(w, s)
    return codes, scales, s


def quantize_experts(w) -> NVFP4Experts:
    """All experts [E][N][K] fp32 -> NVFP4Experts (one tensor scale per expert)."""
    w = np.asarray(w, dtype=np.float32)
    e_count, n, k = w.shape
    codes = np.empty((e_count, n, k // 2), dtype=np.uint8)
    scales = np.empty((e_count, n, k // 16), dtype=np.uint8)
    ts = np.empty(e_count, dtype=np.float32)
    for e in range(e_count):
        codes[e], scales[e], ts[e] = quantize_weight_matrix(w[e])
    return NVFP4Experts(codes, scales, ts)


class LazyExperts:
    """Experts quantised by the oracle on first use: ``source(e)`` returns the
    fp32 matrix [N][K] of expert e.  For full-size layers, where quantising
    all 512 experts up front would be slow and only the routed ones matter."""

    def __init__(self, source, num_experts: int, rows: int):
        self.source = source
        self.num_experts = num_experts
        self.rows = rows
        self._cache = {}

    def quantized(self, e: int):
        e = int(e)
        if e not in self._cache:
            self._cache[e] = quantize_weight_matrix(self.source(e))
        return self._cache[e]

    def dequant(self, e: int) -> np.ndarray:
        return dequantize_rows(*self.quantized(e))


def moe_layer(x, router_w, bias, gate: NVFP4Experts, up: NVFP4Experts, down_w: NVFP4Experts,
              top_k: int, s_h: float, tokens=None, residual: bool = False, keep=None,
              resident=None) -> dict:
    """Run one layer.

    x         float32 [T][H] holding bf16 values
    router_w  float32 [E][H];  bias float32 [E] or None
    gate/up   NVFP4Experts with N = I, K = H;  down_w with N = H, K = I (any object
              with num_experts, rows and dequant(e) works, e.g. one that
              quantises an expert only when it is first used)
    tokens    None for every token, else a list of token rows to evaluate
              (the activation tensor scale still covers all T rows)
    residual  also return x_next = bf16(x + y) bit patterns
    keep, resident
              route-tail skip (router.route): None computes every pick

    Returns a dict of the intermediate and final results.  Pairs the skip
    dropped have expert index -1, weight 0, and all-zero h and outputs.
    """
    x = np.asarray(x, dtype=np.float32)
    num_tokens = x.shape[0]
    rows = np.arange(num_tokens) if tokens is None else np.asarray(tokens, dtype=np.int64)
    out = {}

    # S1/S2
    logits = router_logits(x[rows], router_w, bias)
    idx, w = route(logits, top_k, keep=keep, resident=resident)
    out.update(logits=logits, idx=idx, w=w)

    # S3: one tensor scale over all T rows; codes for the evaluated rows
    s_x = tensor_scale(np.max(np.abs(x)) if x.size else F32(0))
    xq_codes, xq_scales = quantize_rows(x[rows], s_x)
    out.update(xq_codes=xq_codes, xq_scales=xq_scales, s_x=s_x)

    # S4 (whole call only: positions depend on every token)
    if tokens is None:
        counts, offsets, perm, inv = permute(idx, gate.num_experts)
        out.update(counts=counts, offsets=offsets, perm=perm, inv=inv)

    # S5/S6 grouped by expert
    n_sel = len(rows)
    inter = gate.rows
    hidden = x.shape[1]
    pair_out = np.zeros((n_sel, top_k, hidden), dtype=np.float64)
    pair_hq = np.zeros((n_sel, top_k, inter // 2), dtype=np.uint8)
    pair_hs = np.zeros((n_sel, top_k, inter // 16), dtype=np.uint8)
    pair_h32 = np.zeros((n_sel, top_k, inter), dtype=np.float32)
    pair_g = np.zeros((n_sel, top_k, inter), dtype=np.float64)
    pair_u = np.zeros((n_sel, top_k, inter), dtype=np.float64)
    for e in np.unique(idx[idx >= 0]):
        r_sel, j_sel = np.nonzero(idx == e)
        x_hat = dequantize_rows(xq_codes[r_sel], xq_scales[r_sel], s_x)
        g, u = gate_up(x_hat, gate.dequant(e), up.dequant(e))
        pair_g[r_sel, j_sel] = g
        pair_u[r_sel, j_sel] = u
        h32, hc, hsc = requantize_h(swiglu(g, u), s_h)
        h_hat = dequantize_rows(hc, hsc, F32(s_h))
        pair_out[r_sel, j_sel] = down(h_hat, down_w.dequant(e))
        pair_hq[r_sel, j_sel] = hc
        pair_hs[r_sel, j_sel] = hsc
        pair_h32[r_sel, j_sel] = h32

    y = np.stack([combine(w[r], pair_out[r]) for r in range(n_sel)]) if n_sel else \
        np.zeros((0, hidden))
    out.update(y=y, pair_h32=pair_h32, pair_hq=pair_hq, pair_hs=pair_hs, pair_g=pair_g,
               pair_u=pair_u)

    if tokens is None:
        flat_hq = pair_hq.reshape(-1, inter // 2)
        flat_hs = pair_hs.reshape(-1, inter // 16)
        out["hq"] = flat_hq[out["perm"]]          # computed pairs only, expert-grouped
        out["hs"] = flat_hs[out["perm"]]

    if residual:
        s = (x[rows] + y.astype(F32)).astype(F32)
        out["x_next_bits"] = bf16_bits_from_f32_rne(s)
    return out


def moe_stack(x, layers, top_k: int, s_h: float) -> list:
    """Run a stack of layers with x_{l+1} = bf16(x_l + y_l).  ``layers`` is a
    list of dicts with keys router_w, bias, gate, up, down.  Returns the list
    of per-layer result dicts (each with x_next_bits)."""
    results = []
    cur = np.asarray(x, dtype=np.float32)
    for p in layers:
        r = moe_layer(cur, p["router_w"], p.get("bias"), p["gate"], p["up"], p["down"],
                      top_k, s_h, residual=True)
        results.append(r)
        cur = f32_from_bf16_bits(r["x_next_bits"])
    return results
