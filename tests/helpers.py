"""Test harness: build a layer on the GPU through the C ABI, run the CPU
oracle on the same seeded inputs, and compare them.

Inputs come from ``synth`` (random draws only).  The CUDA side quantises the
fp32 weights with the library (moe_quantize_weights); the oracle quantises the
same fp32 weights with its own quantiser; the codes are compared bit for bit
before any layer output is.
"""
import numpy as np
import torch

import synth
from oracle import formats as OF
from oracle import layer as OL
from oracle import quant as OQ
from oracle import router as OR

TAU = 2.0 ** -12          # near-tie threshold on fp64 logits (top-k parity)
LOGIT_TOL = TAU / 4       # required |l_gpu - l_fp64|
MIDPOINT_REL = 2.0 ** -16  # h elements / blocks this close to a rounding boundary may flip
Y_REL_L2 = 2e-3           # layer output tolerance (relative L2 over the tensor)
# with identical codes the output differs from the oracle only by fp32
# accumulation order (CUDA-core and fused decode paths) or, on the
# tensor-core prefill path, by the fp16 rounding of each per-pair output
# (relative <= 2^-12 per element, so <= 2^-11 over the tensor with margin)
TIGHT_FP32 = 1e-5
TIGHT_FP16_PARTIALS = 2.0 ** -11

E2M1_BOUNDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
E4M3_MIDS = (OF.E4M3_FINITE[:-1] + OF.E4M3_FINITE[1:]) / 2


def layer_weights(cfg, layer=0, device="cpu"):
    """fp32 weights of one layer from the seeded generator."""
    H, E, I = cfg.hidden, cfg.experts, cfg.inter
    return dict(
        router_w=synth.make_router(E, H, cfg.seed, layer, device=device),
        bias=synth.make_router_bias(E, cfg.seed, layer, device=device) if cfg.zipf_bias else None,
        gate=synth.make_expert_weights(layer, "gate", E, I, H, cfg.seed, device=device),
        up=synth.make_expert_weights(layer, "up", E, I, H, cfg.seed, device=device),
        down=synth.make_expert_weights(layer, "down", E, H, I, cfg.seed, device=device),
    )


class GpuLayer:
    """A layer on cuda:0 built through the C ABI from fp32 weights."""

    def __init__(self, cfg, w, max_tokens, keep_fp32=False, flags=0, route_keep=0, resident=None):
        import nvfp4_routed_expert_gb300 as nv
        self.nv = nv
        self.cfg = cfg
        dev = torch.device("cuda", 0)
        self.router_w = w["router_w"].to(dev).contiguous()
        self.bias = w["bias"].to(dev).contiguous() if w["bias"] is not None else None
        self.gate = nv.quantize_weights(w["gate"].to(dev).contiguous())
        self.up = nv.quantize_weights(w["up"].to(dev).contiguous())
        self.down = nv.quantize_weights(w["down"].to(dev).contiguous())
        self.desc = nv.make_desc(cfg.hidden, cfg.experts, cfg.top_k, cfg.inter, max_tokens,
                                 cfg.h_tensor_scale, flags=flags, route_keep=route_keep)
        self.layer = nv.Layer(self.desc, self.router_w, self.bias, self.gate, self.up, self.down)
        self.resident = None
        if resident is not None:
            self.resident = torch.as_tensor(resident, dtype=torch.uint8).to(dev).contiguous()
            nv.moe_layer_set_resident(self.layer, self.resident)
        self.ws = self.layer.workspace(dev)
        self.fp32 = w if keep_fp32 else None

    def with_flags(self, flags):
        """Another handle on the same weights with other desc flags."""
        other = GpuLayer.__new__(GpuLayer)
        other.__dict__.update(self.__dict__)
        d = self.desc
        other.desc = self.nv.make_desc(d.hidden, d.num_experts, d.top_k, d.inter, d.max_tokens,
                                       d.h_tensor_scale, flags=flags, route_keep=d.route_keep)
        other.layer = self.nv.Layer(other.desc, self.router_w, self.bias, self.gate, self.up,
                                    self.down)
        if self.resident is not None:
            self.nv.moe_layer_set_resident(other.layer, self.resident)
        other.ws = other.layer.workspace(self.router_w.device)
        return other

    def with_bias(self, bias):
        """Another handle on the same quantised weights with a different router bias."""
        other = GpuLayer.__new__(GpuLayer)
        other.__dict__.update(self.__dict__)
        other.bias = bias.contiguous()
        other.layer = self.nv.Layer(self.desc, self.router_w, other.bias, self.gate, self.up,
                                    self.down)
        if self.resident is not None:
            self.nv.moe_layer_set_resident(other.layer, self.resident)
        return other

    def forward(self, x_dev, residual=False, debug=True, xq=None):
        cfg, dev = self.cfg, x_dev.device
        T, P = x_dev.shape[0], x_dev.shape[0] * cfg.top_k
        y = torch.empty(T, cfg.hidden, dtype=torch.float32, device=dev)
        x_next = torch.empty(T, cfg.hidden, dtype=torch.bfloat16, device=dev) if residual else None
        dbg = None
        if debug:
            dbg = dict(
                logits=torch.empty(T, cfg.experts, dtype=torch.float32, device=dev),
                idx=torch.empty(T, cfg.top_k, dtype=torch.int32, device=dev),
                weights=torch.empty(T, cfg.top_k, dtype=torch.float32, device=dev),
                counts=torch.empty(cfg.experts, dtype=torch.int32, device=dev),
                offsets=torch.empty(cfg.experts + 1, dtype=torch.int32, device=dev),
                perm=torch.empty(P, dtype=torch.int32, device=dev),
                inv=torch.empty(P, dtype=torch.int32, device=dev),
                hq=torch.empty(P, cfg.inter // 2, dtype=torch.uint8, device=dev),
                hs=torch.empty(P, cfg.inter // 16, dtype=torch.uint8, device=dev),
                xq_codes=torch.empty(T, cfg.hidden // 2, dtype=torch.uint8, device=dev),
                xq_scales=torch.empty(T, cfg.hidden // 16, dtype=torch.uint8, device=dev),
                xq_tensor_scale=torch.empty(1, dtype=torch.float32, device=dev),
            )
        self.nv.moe_forward(self.layer, x_dev, y, self.ws, xq=xq,
                            residual=x_dev if residual else None, x_next=x_next, debug=dbg)
        torch.cuda.synchronize()
        st = self.nv.moe_layer_status(self.layer)
        assert st == 0, self.nv.status_string(st)
        out = {"y": y.cpu().numpy()}
        if x_next is not None:
            out["x_next_bits"] = x_next.view(torch.int16).cpu().numpy().view(np.uint16)
        if dbg is not None:
            out.update({k: v.cpu().numpy() for k, v in dbg.items()})
        return out

    def quantize_act(self, x_dev):
        T, H = x_dev.shape
        codes = torch.empty(T, H // 2, dtype=torch.uint8, device=x_dev.device)
        scales = torch.empty(T, H // 16, dtype=torch.uint8, device=x_dev.device)
        ts = torch.empty(1, dtype=torch.float32, device=x_dev.device)
        self.nv.moe_quantize_act(self.layer, x_dev, codes, scales, ts, self.ws)
        torch.cuda.synchronize()
        return codes, scales, ts


def oracle_experts(w_fp32):
    """Lazily quantised oracle experts from an fp32 tensor [E][N][K] (any device)."""
    E, N, _ = w_fp32.shape
    return OL.LazyExperts(lambda e: w_fp32[e].float().cpu().numpy(), E, N)


def run_oracle(cfg, x_bf16, w, tokens=None, residual=False, experts=None, keep=None,
               resident=None):
    x = x_bf16.float().cpu().numpy()
    if experts is None:
        experts = {m: oracle_experts(w[m]) for m in ("gate", "up", "down")}
    b = w["bias"].cpu().numpy() if w["bias"] is not None else None
    out = OL.moe_layer(x, w["router_w"].cpu().numpy(), b, experts["gate"], experts["up"],
                       experts["down"], cfg.top_k, cfg.h_tensor_scale, tokens=tokens,
                       residual=residual, keep=keep,
                       resident=None if resident is None else np.asarray(resident))
    out["experts"] = experts
    return out


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    d = np.linalg.norm(a - b)
    n = np.linalg.norm(b)
    return d / n if n > 0 else d


ACC_ULPS = 64  # allowance for an fp32 dot product: ACC_ULPS * 2^-24 * sum |x_i w_i|


def _abs_sums(orc, pairs):
    """sum_i |x_hat_i| |w_i| over every gate and up row of each pair (r, j)."""
    experts, idx = orc["experts"], orc["idx"]
    xh = np.abs(OQ.dequantize_rows(orc["xq_codes"], orc["xq_scales"], orc["s_x"]))
    inter = experts["gate"].rows
    a_g = np.zeros((len(pairs), inter))
    a_u = np.zeros((len(pairs), inter))
    e_of = idx[pairs[:, 0], pairs[:, 1]]
    for e in np.unique(e_of):
        sel = np.nonzero(e_of == e)[0]
        rows = xh[pairs[sel, 0]]
        a_g[sel] = rows @ np.abs(experts["gate"].dequant(e)).T
        a_u[sel] = rows @ np.abs(experts["up"].dequant(e)).T
    return a_g, a_u


def h_flip_candidates(orc, pairs, s_h):
    """Boolean [len(pairs)][I]: elements whose NVFP4 code may legitimately differ
    between the oracle (fp64 g, u rounded once) and an fp32 evaluation of h.

    |h_fp32 - h| is bounded through SwiGLU from the dot-product error bound
    ACC_ULPS * 2^-24 * sum |x_i w_i| of g and u plus a few roundings; an element
    is a candidate if its scaled value lies within that bound of an E2M1
    decision boundary (or of 0, where only the sign bit of a zero code can
    change), and a whole block is if its scale decision q lies within the
    bound of an E4M3 midpoint."""
    r, j = pairs[:, 0], pairs[:, 1]
    g, u = orc["pair_g"][r, j], orc["pair_u"][r, j]
    h32 = orc["pair_h32"][r, j].astype(np.float64)
    a_g, a_u = _abs_sums(orc, pairs)
    eps = 2.0 ** -24
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = sig * (1.0 + g * (1.0 - sig))
    dh = (np.abs(dsilu) * ACC_ULPS * eps * a_g * np.abs(u) + np.abs(g * sig) * ACC_ULPS * eps * a_u
          + 16 * eps * np.abs(h32))
    rows_, inter = h32.shape
    hb = np.abs(h32).reshape(rows_, inter // 16, 16)
    db = dh.reshape(rows_, inter // 16, 16)
    a = hb.max(axis=2)
    q = a / (6.0 * s_h)
    dq = db.max(axis=2) / (6.0 * s_h)
    near_mid = np.min(np.abs(q[..., None] - E4M3_MIDS[None, None, :]), axis=2) <= dq
    S = OF.e4m3_encode_rne_satfinite(q.astype(np.float32))
    m = OF.e4m3_value(S) * s_h
    with np.errstate(divide="ignore", invalid="ignore"):
        v = hb / m[..., None]
        dv = db / m[..., None]
    near_b = np.min(np.abs(v[..., None] - E2M1_BOUNDS), axis=-1) <= dv
    near_b = np.where(np.isfinite(v), near_b, False)
    # |h| within its error bound of 0: the sign bit of a zero-magnitude code
    # (0x0 / 0x8, both dequantising to 0) is not determined
    sign_open = hb <= db
    return (near_b | sign_open | near_mid[..., None]).reshape(rows_, inter)


def weight_tol(w, logit_err):
    """Bound on the error of the renormalised top-k softmax weights w given a
    logit error of at most logit_err.  The softmax over the selected logits has
    dw_i = w_i (dl_i - sum_j w_j dl_j), so |dw_i| <= 2 w_i max|dl| to first
    order (the factor 1.01 covers the second-order term at these tiny dl);
    1e-6 covers the fp32 exp, sum and divide of the weights themselves."""
    return 2.0 * 1.01 * logit_err * np.asarray(w, dtype=np.float64) + 1e-6


def compare_routing(cfg, gpu, orc, rows=None):
    """Logits within LOGIT_TOL; top-k identical except near-tie tokens; weights
    within the error the measured logit error allows (weight_tol).  Returns the
    number of near-tie tokens."""
    l_orc = orc["logits"]
    l_gpu = gpu["logits"] if rows is None else gpu["logits"][rows]
    err = np.max(np.abs(l_gpu.astype(np.float64) - l_orc)) if l_orc.size else 0.0
    assert err < LOGIT_TOL, f"router logits differ by {err}"
    ties = OR.near_tie_tokens(l_orc, cfg.top_k, TAU)
    idx_gpu = gpu["idx"] if rows is None else gpu["idx"][rows]
    w_gpu = gpu["weights"] if rows is None else gpu["weights"][rows]
    ok = ~ties
    np.testing.assert_array_equal(idx_gpu[ok], orc["idx"][ok])
    dw = np.abs(w_gpu[ok].astype(np.float64) - orc["w"][ok])
    assert np.all(dw <= weight_tol(orc["w"][ok], err)), np.max(dw)
    # near-tie tokens: the GPU picks must be valid top-k under its own logits
    # (picks a route-tail skip dropped read -1 and are not checked)
    for t in np.nonzero(ties)[0]:
        lg = l_gpu[t].astype(np.float64)
        sel = idx_gpu[t][idx_gpu[t] >= 0]
        rest = np.setdiff1d(np.arange(cfg.experts), idx_gpu[t])
        if (idx_gpu[t] >= 0).all():
            assert lg[sel].min() >= lg[rest].max()
    return int(ties.sum())


def compare_h(cfg, gpu_hq, gpu_hs, orc, pairs):
    """GPU hq/hs rows for the oracle pairs (r, j) (one row per pair, same order):
    identical except at flip candidates.  Returns the number of differing
    elements."""
    pairs = np.asarray(pairs, dtype=np.int64)
    g = OQ.unpack_codes(gpu_hq)
    o = OQ.unpack_codes(orc["pair_hq"][pairs[:, 0], pairs[:, 1]])
    gs = np.repeat(gpu_hs, 16, axis=1)
    os_ = np.repeat(orc["pair_hs"][pairs[:, 0], pairs[:, 1]], 16, axis=1)
    diff = (g != o) | (gs != os_)
    if not diff.any():
        return 0
    flags = h_flip_candidates(orc, pairs, cfg.h_tensor_scale)
    bad = diff & ~flags
    if bad.any():
        for pi, f in np.argwhere(bad)[:8]:
            r, j = pairs[pi]
            b = f // 16
            h = orc["pair_h32"][r, j, f]
            hb = orc["pair_h32"][r, j, 16 * b:16 * b + 16]
            print(f"h mismatch pair (row {r}, slot {j}) feature {f}: h32 {h!r} g {orc['pair_g'][r, j, f]!r} "
                  f"u {orc['pair_u'][r, j, f]!r} gpu code {g[pi, f]} scale {gs[pi, f]} | oracle "
                  f"code {o[pi, f]} scale {os_[pi, f]} | block max {np.abs(hb).max()!r}")
    assert not bad.any(), f"{int(bad.sum())} h codes differ away from rounding boundaries"
    return int(diff.sum())


def assert_flip_ceiling(cfg, flips, orc, pairs):
    """An h code may differ only where the oracle flags a rounding boundary
    (compare_h), and at most a quarter of the flagged elements may differ
    (at least 4 allowed): a GPU evaluation of h that has drifted by more than
    rounding noise flips many of the flagged elements, not a few."""
    if flips == 0:
        return
    flagged = int(h_flip_candidates(orc, np.asarray(pairs, dtype=np.int64), cfg.h_tensor_scale).sum())
    ceiling = max(4, flagged // 4)
    assert flips <= ceiling, f"{flips} h codes differ, ceiling {ceiling} ({flagged} flagged)"


def perm_pairs(perm, k):
    """(token, slot) of each expert-grouped position."""
    perm = np.asarray(perm, dtype=np.int64)
    return np.stack([perm // k, perm % k], axis=1)


def check_x_next(gpu_bits, orc_bits, y_gpu, y_orc):
    """bf16(x + y): GPU and oracle may differ by one bf16 rounding of each and by
    the difference of their y (which near x + y = 0 can flip a tiny value's
    sign, so compare values, not bit patterns)."""
    from oracle.formats import f32_from_bf16_bits
    a = f32_from_bf16_bits(gpu_bits).astype(np.float64)
    b = f32_from_bf16_bits(orc_bits).astype(np.float64)
    dy = np.abs(np.asarray(y_gpu, np.float64) - np.asarray(y_orc, np.float64))
    bound = 2.0 ** -7 * np.maximum(np.abs(a), np.abs(b)) + 2.0 * dy + 1e-30  # one bf16 ulp
    bad = np.abs(a - b) > bound
    assert not bad.any(), f"{int(bad.sum())} x_next values differ beyond rounding"
