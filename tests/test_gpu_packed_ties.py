"""GPU checks with closed-form expectations (no oracle run):

* the packed buffer moe_layer_create fills: the router weights split into
  bf16 hi = RN(Wr) and lo = RN(Wr - hi), then the gate, up and down block
  scales rearranged into the grouped GEMM's tiles (for each 128 rows g and
  256-element stage kb, four 512-byte k-steps [lane i][row quarter j][4 scale
  bytes of row 128 g + 32 j + i]) -- a permutation checked byte for byte;
* exact ties in the router: with Wr = 0 every logit is 0, so top-k must pick
  experts 0 .. k-1 (ties go to the lower index) with weights RN(1/k), on the
  fused decode kernel, the per-step kernels and the tensor-core path."""
import numpy as np
import pytest
import torch

import synth
from tests import helpers as Hp

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def nv():
    import nvfp4_routed_expert_gb300 as m
    m.load()
    return m


def bf16_rn_bits(f32):
    """Round-to-nearest-even fp32 -> bf16 bits (finite inputs)."""
    u = np.ascontiguousarray(f32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def tiled(scales, K):
    """[rows][K/16] scale bytes -> the tiled layout, flattened."""
    rows = scales.shape[0]
    g, kb = rows // 128, K // 256
    t = scales.reshape(g, 4, 32, kb, 4, 4)          # (g, j, i, kb, ks, c)
    return np.ascontiguousarray(t.transpose(0, 3, 4, 2, 1, 5)).ravel()


def test_packed_buffer_layout(nv):
    cfg = synth.get_config("mid_tc")
    H, E, I = cfg.hidden, cfg.experts, cfg.inter
    assert H % 256 == 0 and I % 256 == 0
    w = Hp.layer_weights(cfg)
    gl = Hp.GpuLayer(cfg, w, cfg.tokens)
    torch.cuda.synchronize()
    packed = gl.layer.packed.cpu().numpy()
    assert packed.size == nv.moe_packed_weight_bytes(gl.desc)
    wr = w["router_w"].numpy().astype(np.float32)
    hi = bf16_rn_bits(wr)
    hi_f = (hi.astype(np.uint32) << 16).view(np.float32)
    lo = bf16_rn_bits(wr - hi_f)
    n = E * H
    np.testing.assert_array_equal(packed[:2 * n].view(np.uint16).reshape(E, H), hi)
    np.testing.assert_array_equal(packed[2 * n:4 * n].view(np.uint16).reshape(E, H), lo)
    off = 4 * n
    for name, rows, K in (("gate", E * I, H), ("up", E * I, H), ("down", E * H, I)):
        sc = getattr(gl, name)[1].cpu().numpy().reshape(rows, K // 16)
        got = packed[off:off + rows * K // 16]
        np.testing.assert_array_equal(got, tiled(sc, K), err_msg=name)
        off += rows * K // 16
    assert off == packed.size


@pytest.mark.parametrize("tokens,flags", [(3, 0), (3, 1), (40, 0), (40, 1)],
                         ids=["fused-decode", "per-step-small", "tensor-core", "per-step-large"])
def test_exact_ties_pick_lower_indices(nv, tokens, flags):
    cfg = synth.get_config("mid_tc")
    w = Hp.layer_weights(cfg)
    w["router_w"] = torch.zeros_like(w["router_w"])
    w["bias"] = None
    gl = Hp.GpuLayer(cfg, w, 64, flags=flags)
    x = synth.make_x(tokens, cfg.hidden, cfg.seed)
    out = gl.forward(x.to(DEV))
    k, E = cfg.top_k, cfg.experts
    assert np.all(out["logits"] == 0.0)
    np.testing.assert_array_equal(out["idx"], np.tile(np.arange(k, dtype=np.int32), (tokens, 1)))
    np.testing.assert_array_equal(out["weights"], np.full((tokens, k), np.float32(1) / np.float32(k)))
    counts = np.zeros(E, dtype=np.int32)
    counts[:k] = tokens
    np.testing.assert_array_equal(out["counts"], counts)
    assert np.all(np.isfinite(out["y"]))


@pytest.mark.parametrize("tokens,flags", [(3, 0), (40, 0), (40, 1)],
                         ids=["fused-decode", "tensor-core", "per-step"])
def test_partial_ties_at_the_kth_pick(nv, tokens, flags):
    """Wr = 0 and a bias with a tie across the k-th pick: the logits are the
    bias exactly, the top k are the k - 2 larger values in value order and then
    the two lowest indices of the five experts tied at 1.0 (spread over the
    lanes that hold experts l and l + 32), whatever x is.  Few enough keys
    reach the k-th lane maximum that the per-step top-k takes its threshold
    pass; the weights are the renormalised softmax of the picks."""
    cfg = synth.get_config("mid_tc").with_(experts=64, top_k=8)
    E, k = cfg.experts, cfg.top_k
    w = Hp.layer_weights(cfg)
    w["router_w"] = torch.zeros_like(w["router_w"])
    bias = np.array([-1.0 - e / 128.0 for e in range(E)], dtype=np.float32)
    larger = [5, 40, 17, 63, 2, 33]
    for r, e in enumerate(larger):
        bias[e] = np.float32(2.0 - 0.1 * r)
    tied = [50, 9, 36, 21, 58]
    bias[tied] = np.float32(1.0)
    w["bias"] = torch.from_numpy(bias)
    gl = Hp.GpuLayer(cfg, w, 64, flags=flags)
    x = synth.make_x(tokens, cfg.hidden, cfg.seed)
    out = gl.forward(x.to(DEV))
    np.testing.assert_array_equal(out["logits"], np.tile(bias, (tokens, 1)))
    want = np.array(larger + sorted(tied)[:2], dtype=np.int32)
    np.testing.assert_array_equal(out["idx"], np.tile(want, (tokens, 1)))
    sel = bias[want].astype(np.float64)
    z = np.exp(sel - sel[0])
    np.testing.assert_allclose(out["weights"], np.tile(z / z.sum(), (tokens, 1)), rtol=1e-6, atol=0)
    assert np.all(np.isfinite(out["y"]))
