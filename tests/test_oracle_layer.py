"""Pins of the whole oracle layer (S1..S6 and the residual):
  * identical experts reduce the layer to one dense NVFP4 FFN (sum of weights 1);
  * E = 1, k = 1 is a plain dense NVFP4 FFN, restated with torch.float64;
  * the tiny layer restated with torch library routines (stable sort, softmax,
    silu, float8 scale conversion, float64 matmul) agrees to fp64 round-off;
  * k = 1 combine gives y = o;
  * the residual is the bf16 rounding of x + y;
  * a stack chains every layer on the previous layer's bf16(x + y);
  * experts quantised on first use equal the eagerly quantised ones."""
import numpy as np
import pytest
import torch

import synth
from oracle import layer as L
from oracle import quant as Q
from oracle.expert import NVFP4Experts

F32 = np.float32


def _tiny_inputs(cfg, identical=False, device="cpu"):
    x = synth.make_x(cfg.tokens, cfg.hidden, cfg.seed).float().numpy()
    Wr = synth.make_router(cfg.experts, cfg.hidden, cfg.seed).numpy()
    b = synth.make_router_bias(cfg.experts, cfg.seed).numpy() if cfg.zipf_bias else None
    mats = {}
    for name, (n, kk) in (("gate", (cfg.inter, cfg.hidden)), ("up", (cfg.inter, cfg.hidden)),
                          ("down", (cfg.hidden, cfg.inter))):
        w = synth.make_expert_weights(0, name, cfg.experts, n, kk, cfg.seed).numpy()
        if identical:
            w = np.broadcast_to(w[:1], w.shape).copy()
        mats[name] = L.quantize_experts(w)
    return x, Wr, b, mats


def _torch_dequant(codes, scales, s):
    """Independent dequantisation: E2M1 from its bit fields, E4M3 by torch."""
    c = torch.from_numpy(np.asarray(codes)).to(torch.int64)
    nib = torch.stack([c & 15, c >> 4], dim=-1).reshape(*c.shape[:-1], -1)
    sign = 1.0 - 2.0 * ((nib >> 3) & 1).double()
    e = ((nib >> 1) & 3).double()
    m = (nib & 1).double()
    mag = torch.where(e == 0, m * 0.5, (1 + m / 2) * torch.pow(2.0, e - 1))
    sc = torch.from_numpy(np.asarray(scales)).view(torch.float8_e4m3fn).double()
    return sign * mag * sc.repeat_interleave(16, dim=-1) * float(s)


def test_identical_experts_reduce_to_one_ffn():
    cfg = synth.get_config("tiny").with_(tokens=9)
    x, Wr, b, m = _tiny_inputs(cfg, identical=True)
    out = L.moe_layer(x, Wr, b, m["gate"], m["up"], m["down"], cfg.top_k, cfg.h_tensor_scale)
    xc, xs, sx = Q.quantize_tensor(x)
    xh = Q.dequantize_rows(xc, xs, sx)
    wg, wu, wd = m["gate"].dequant(0), m["up"].dequant(0), m["down"].dequant(0)
    g = torch.from_numpy(xh) @ torch.from_numpy(wg).T
    u = torch.from_numpy(xh) @ torch.from_numpy(wu).T
    h = (torch.nn.functional.silu(g) * u).numpy().astype(F32)
    hc, hs = Q.quantize_rows(h, F32(cfg.h_tensor_scale))
    o = (torch.from_numpy(Q.dequantize_rows(hc, hs, F32(cfg.h_tensor_scale)))
         @ torch.from_numpy(wd).T).numpy()
    np.testing.assert_allclose(out["y"], o, rtol=1e-12, atol=1e-12)


def test_single_expert_dense_ffn_torch_restatement():
    cfg = synth.get_config("tiny").with_(experts=1, top_k=1, tokens=6)
    x, Wr, b, m = _tiny_inputs(cfg)
    out = L.moe_layer(x, Wr, b, m["gate"], m["up"], m["down"], 1, cfg.h_tensor_scale)
    assert np.all(out["idx"] == 0) and np.all(out["w"] == 1.0)
    xh = _torch_dequant(out["xq_codes"], out["xq_scales"], out["s_x"])
    g = xh @ _torch_dequant(m["gate"].codes[0], m["gate"].scales[0], m["gate"].tensor_scales[0]).T
    u = xh @ _torch_dequant(m["up"].codes[0], m["up"].scales[0], m["up"].tensor_scales[0]).T
    h = torch.nn.functional.silu(g) * u
    np.testing.assert_allclose(out["pair_h32"][:, 0], h.float().numpy(), rtol=0, atol=0)
    hh = _torch_dequant(out["pair_hq"][:, 0], out["pair_hs"][:, 0], F32(cfg.h_tensor_scale))
    y = hh @ _torch_dequant(m["down"].codes[0], m["down"].scales[0], m["down"].tensor_scales[0]).T
    np.testing.assert_allclose(out["y"], y.numpy(), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("name", ["tiny", "mid_ragged"])
def test_whole_layer_torch_float64_restatement(name):
    cfg = synth.get_config(name)
    x, Wr, b, m = _tiny_inputs(cfg)
    out = L.moe_layer(x, Wr, b, m["gate"], m["up"], m["down"], cfg.top_k, cfg.h_tensor_scale)
    xt = torch.from_numpy(x).double()
    logits = xt @ torch.from_numpy(Wr).double().T
    if b is not None:
        logits = logits + torch.from_numpy(b).double()
    np.testing.assert_allclose(out["logits"], logits.numpy(), rtol=1e-12, atol=1e-12)
    # top-k by a stable descending sort: equal logits keep the lower index first
    order = torch.sort(logits, dim=1, descending=True, stable=True).indices[:, :cfg.top_k]
    np.testing.assert_array_equal(out["idx"], order.numpy())
    w = torch.softmax(torch.gather(logits, 1, order), dim=1)
    np.testing.assert_allclose(out["w"], w.numpy(), rtol=1e-13, atol=1e-15)
    xh = _torch_dequant(out["xq_codes"], out["xq_scales"], out["s_x"])
    y = torch.zeros(cfg.tokens, cfg.hidden, dtype=torch.float64)
    for t in range(cfg.tokens):
        for j in range(cfg.top_k):
            e = int(order[t, j])
            wg = _torch_dequant(m["gate"].codes[e], m["gate"].scales[e], m["gate"].tensor_scales[e])
            wu = _torch_dequant(m["up"].codes[e], m["up"].scales[e], m["up"].tensor_scales[e])
            wd = _torch_dequant(m["down"].codes[e], m["down"].scales[e], m["down"].tensor_scales[e])
            h = torch.nn.functional.silu(wg @ xh[t]) * (wu @ xh[t])
            np.testing.assert_allclose(out["pair_h32"][t, j], h.float().numpy(), rtol=0, atol=0)
            hh = _torch_dequant(out["pair_hq"][t, j], out["pair_hs"][t, j], F32(cfg.h_tensor_scale))
            y[t] += w[t, j] * (wd @ hh)
    np.testing.assert_allclose(out["y"], y.numpy(), rtol=1e-12, atol=1e-12)
    # hq/hs rows are stored in expert-grouped order
    flat_hq = out["pair_hq"].reshape(-1, cfg.inter // 2)
    np.testing.assert_array_equal(out["hq"], flat_hq[out["perm"]])


def test_k1_combine_is_the_expert_output():
    cfg = synth.get_config("tiny").with_(top_k=1)
    x, Wr, b, m = _tiny_inputs(cfg)
    out = L.moe_layer(x, Wr, b, m["gate"], m["up"], m["down"], 1, cfg.h_tensor_scale)
    assert np.all(out["w"] == 1.0)
    for t in range(cfg.tokens):
        e = int(out["idx"][t, 0])
        hh = Q.dequantize_rows(out["pair_hq"][t], out["pair_hs"][t], F32(cfg.h_tensor_scale))
        np.testing.assert_allclose(out["y"][t], (hh @ m["down"].dequant(e).T)[0], rtol=1e-13)


def test_residual_is_bf16_of_sum():
    cfg = synth.get_config("tiny")
    x, Wr, b, m = _tiny_inputs(cfg)
    out = L.moe_layer(x, Wr, b, m["gate"], m["up"], m["down"], cfg.top_k, cfg.h_tensor_scale,
                      residual=True)
    ref = (torch.from_numpy(x) + torch.from_numpy(out["y"].astype(F32))).to(torch.bfloat16)
    np.testing.assert_array_equal(out["x_next_bits"], ref.view(torch.int16).numpy().view(np.uint16))


def test_sampled_tokens_match_full_call():
    cfg = synth.get_config("mid_zipf")
    x, Wr, b, m = _tiny_inputs(cfg)
    full = L.moe_layer(x, Wr, b, m["gate"], m["up"], m["down"], cfg.top_k, cfg.h_tensor_scale)
    rows = [0, 17, 299, 150]
    part = L.moe_layer(x, Wr, b, m["gate"], m["up"], m["down"], cfg.top_k, cfg.h_tensor_scale,
                       tokens=rows)
    np.testing.assert_array_equal(part["idx"], full["idx"][rows])
    np.testing.assert_allclose(part["y"], full["y"][rows], rtol=1e-13, atol=1e-14)


def _stack_layers(cfg, n):
    layers = []
    for layer in range(n):
        mats = {}
        for name, (rows, cols) in (("gate", (cfg.inter, cfg.hidden)), ("up", (cfg.inter, cfg.hidden)),
                                   ("down", (cfg.hidden, cfg.inter))):
            mats[name] = L.quantize_experts(
                synth.make_expert_weights(layer, name, cfg.experts, rows, cols).numpy())
        layers.append(dict(router_w=synth.make_router(cfg.experts, cfg.hidden, layer=layer).numpy(),
                           **mats))
    return layers


def test_stack_chains_each_layer_on_the_previous_residual_output():
    """Three stacked layers, each checked against an explicit one-layer call
    whose input is the previous layer's bf16(x + y) (decoded from its bit
    patterns); layer 0 sees x itself.  A chain that fed every layer the
    original x, skipped the residual or reused a layer's weights fails here:
    the inputs of layers 1 and 2 differ from x, and the three layers' routings
    differ from each other."""
    cfg = synth.get_config("tiny")
    layers = _stack_layers(cfg, 3)
    x = synth.make_x(cfg.tokens, cfg.hidden).float().numpy()
    res = L.moe_stack(x, layers, cfg.top_k, cfg.h_tensor_scale)
    assert len(res) == 3
    cur = x
    for l, p in enumerate(layers):
        one = L.moe_layer(cur, p["router_w"], None, p["gate"], p["up"], p["down"], cfg.top_k,
                          cfg.h_tensor_scale, residual=True)
        np.testing.assert_array_equal(res[l]["idx"], one["idx"])
        np.testing.assert_array_equal(res[l]["y"], one["y"])
        np.testing.assert_array_equal(res[l]["x_next_bits"], one["x_next_bits"])
        # x_next is the bf16 rounding of (layer input + y), restated with torch
        ref = (torch.from_numpy(cur) + torch.from_numpy(one["y"].astype(F32))).to(torch.bfloat16)
        np.testing.assert_array_equal(one["x_next_bits"],
                                      ref.view(torch.int16).numpy().view(np.uint16))
        nxt = ref.float().numpy()
        assert not np.array_equal(nxt, cur)          # each layer moves the residual stream
        cur = nxt
    assert not np.array_equal(res[1]["idx"], res[0]["idx"])
    assert not np.array_equal(res[2]["idx"], res[1]["idx"])
    # the chain's layer inputs are not the stack's input: feeding x to layer 2
    # instead of its residual input gives another output
    wrong = L.moe_layer(x, layers[2]["router_w"], None, layers[2]["gate"], layers[2]["up"],
                        layers[2]["down"], cfg.top_k, cfg.h_tensor_scale)
    assert not np.allclose(wrong["y"], res[2]["y"])


def test_lazy_experts_match_eager_quantisation():
    """LazyExperts quantises expert e from source(e) on first use and keeps it:
    codes, scales, tensor scale and the dequantised matrix equal those of
    quantize_experts on the full weight tensor, for several experts and for a
    repeated id (whose source is read once)."""
    cfg = synth.get_config("tiny")
    w = synth.make_expert_weights(0, "gate", cfg.experts, cfg.inter, cfg.hidden).numpy()
    eager = L.quantize_experts(w)
    reads = []

    def source(e):
        reads.append(e)
        return w[e]

    lazy = L.LazyExperts(source, cfg.experts, cfg.inter)
    for e in (3, 0, 15, 3, 7, 3):
        c, s, ts = lazy.quantized(e)
        np.testing.assert_array_equal(c, eager.codes[e])
        np.testing.assert_array_equal(s, eager.scales[e])
        assert np.float32(ts) == eager.tensor_scales[e]
        np.testing.assert_array_equal(lazy.dequant(e), eager.dequant(e))
    assert sorted(reads) == [0, 3, 7, 15]
    assert lazy.num_experts == eager.num_experts and lazy.rows == eager.rows
    # a layer run on lazy experts gives the same result as on eager ones
    x = synth.make_x(cfg.tokens, cfg.hidden).float().numpy()
    Wr = synth.make_router(cfg.experts, cfg.hidden).numpy()
    up = L.quantize_experts(synth.make_expert_weights(0, "up", cfg.experts, cfg.inter,
                                                      cfg.hidden).numpy())
    dn = L.quantize_experts(synth.make_expert_weights(0, "down", cfg.experts, cfg.hidden,
                                                      cfg.inter).numpy())
    a = L.moe_layer(x, Wr, None, eager, up, dn, cfg.top_k, cfg.h_tensor_scale)
    b = L.moe_layer(x, Wr, None, lazy, up, dn, cfg.top_k, cfg.h_tensor_scale)
    np.testing.assert_array_equal(a["y"], b["y"])


def test_zipf_bias_skews_loads():
    cfg = synth.get_config("mid_zipf")
    x, Wr, b, m = _tiny_inputs(cfg)
    out = L.moe_layer(x, Wr, b, m["gate"], m["up"], m["down"], cfg.top_k, cfg.h_tensor_scale)
    counts = np.sort(out["counts"])[::-1]
    assert counts[0] > 3 * np.median(counts[counts > 0])


def test_route_tail_skip_layer():
    """Route-tail skip in the whole layer: keeping every rank (or marking every
    expert resident) reproduces the layer; keeping only rank 0 makes y the top
    pick's expert output alone, computed here directly from the dequantised
    matrices; a partial skip is the weighted sum over the kept picks only."""
    cfg = synth.get_config("tiny").with_(tokens=7, top_k=4)
    x, Wr, b, m = _tiny_inputs(cfg)
    args = (x, Wr, b, m["gate"], m["up"], m["down"], cfg.top_k, cfg.h_tensor_scale)
    full = L.moe_layer(*args)
    for keep, res in ((cfg.top_k, None), (1, np.ones(cfg.experts, np.uint8))):
        same = L.moe_layer(*args, keep=keep, resident=res)
        np.testing.assert_array_equal(same["idx"], full["idx"])
        np.testing.assert_array_equal(same["y"], full["y"])
    top1 = L.moe_layer(*args, keep=1)
    assert np.all(top1["idx"][:, 1:] == -1) and np.all(top1["w"][:, 0] == 1.0)
    np.testing.assert_array_equal(top1["idx"][:, 0], full["idx"][:, 0])
    xh = Q.dequantize_rows(top1["xq_codes"], top1["xq_scales"], top1["s_x"])
    for t in range(cfg.tokens):
        e = int(full["idx"][t, 0])
        g = xh[t] @ m["gate"].dequant(e).T
        u = xh[t] @ m["up"].dequant(e).T
        h = (torch.nn.functional.silu(torch.from_numpy(g)) * torch.from_numpy(u)).numpy()
        hc, hs = Q.quantize_rows(h.astype(F32)[None], F32(cfg.h_tensor_scale))
        o = Q.dequantize_rows(hc, hs, F32(cfg.h_tensor_scale))[0] @ m["down"].dequant(e).T
        np.testing.assert_allclose(top1["y"][t], o, rtol=1e-12, atol=1e-14)
    # keep 2 with expert idx[0, 3] resident: token 0 keeps ranks 0, 1, 3
    res = np.zeros(cfg.experts, np.uint8)
    res[full["idx"][0, 3]] = 1
    part = L.moe_layer(*args, keep=2, resident=res)
    kept = [j for j in range(cfg.top_k) if j < 2 or res[full["idx"][0, j]]]
    assert kept[:2] == [0, 1] and 3 in kept
    wk = full["w"][0, kept] / full["w"][0, kept].sum()
    y0 = np.zeros(cfg.hidden)
    for wi, j in zip(wk, kept):
        hh = Q.dequantize_rows(full["pair_hq"][0, j][None], full["pair_hs"][0, j][None],
                               F32(cfg.h_tensor_scale))[0]
        y0 = y0 + wi * (hh @ m["down"].dequant(int(full["idx"][0, j])).T)
    np.testing.assert_allclose(part["y"][0], y0, rtol=1e-12, atol=1e-14)
    assert part["offsets"][-1] == int((part["idx"] >= 0).sum())
