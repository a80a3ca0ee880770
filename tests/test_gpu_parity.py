"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on
the same seeded inputs.

Bar: bit-exact activation / weight codes and scales, router top-k (except
tokens whose fp64 logits have a near tie, where the pick must still be a valid
top-k), permutation, and h codes (except elements the oracle flags as lying on
a rounding boundary); layer output within relative L2 2e-3."""
import numpy as np
import pytest
import torch

import synth
from oracle import layer as OL
from oracle import permute as OP
from oracle import quant as OQ
from tests import helpers as Hp

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def nv():
    import nvfp4_routed_expert_gb300 as m
    m.load()
    return m


# ------------------------------------------------------------------ quantisers

@pytest.mark.parametrize("shape", [(3, 64, 128), (5, 192, 256), (2, 512, 2048), (1, 2048, 512)])
def test_weight_quantiser_bit_exact(nv, shape):
    g = torch.Generator().manual_seed(sum(shape))
    w = torch.randn(*shape, generator=g) * 0.02
    w[0, 0, :16] = 0.0                        # an all-zero block
    w[-1, -1, 5] = 0.5                        # one large outlier sets the tensor scale
    codes, scales, ts = nv.quantize_weights(w.to(DEV))
    for m in range(shape[0]):
        oc, os_, ot = OL.quantize_weight_matrix(w[m].numpy())
        assert np.float32(ts[m].item()) == ot
        np.testing.assert_array_equal(codes[m].cpu().numpy(), oc)
        np.testing.assert_array_equal(scales[m].cpu().numpy(), os_)


def _act_layer(nv, H, max_tokens):
    cfg = synth.get_config("tiny").with_(hidden=H, tokens=max_tokens)
    return Hp.GpuLayer(cfg, Hp.layer_weights(cfg), max_tokens)


@pytest.mark.parametrize("T,H", [(1, 256), (7, 512), (300, 1024), (4096, 2048)])
def test_activation_quantiser_bit_exact(nv, T, H):
    gl = _act_layer(nv, H, T)
    x = synth.make_x(T, H, seed=T)
    codes, scales, ts = gl.quantize_act(x.to(DEV))
    oc, os_, ot = OQ.quantize_tensor(x.float().numpy())
    assert np.float32(ts.item()) == ot
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)
    np.testing.assert_array_equal(scales.cpu().numpy(), os_)


def test_activation_quantiser_ties_and_edges(nv):
    """Every E2M1 midpoint at many block scales, signed zeros, zero blocks,
    subnormal block scales and saturation -- decided by the hardware converts."""
    H = 256
    rows = []
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    for S in range(1, 0x7F):
        Sv = float(OQ.e4m3_value(np.uint8(S)))
        blk = [6.0 * Sv] + [m * Sv for m in mids] + [-m * Sv for m in mids] + [-0.0]
        rows.append(blk)
    flat = np.array(rows, dtype=np.float32).reshape(-1)
    n = (len(flat) + H - 1) // H * H
    x = np.zeros(n, dtype=np.float32)
    x[:len(flat)] = flat
    x = x.reshape(-1, H)
    x[0, 16] = 2688.0                      # tensor amax: s = 1 exactly
    x[1, 16:32] = -1e-30                   # rounds to a zero scale
    xb = torch.from_numpy(x).to(torch.bfloat16)
    gl = _act_layer(nv, H, xb.shape[0])
    codes, scales, ts = gl.quantize_act(xb.to(DEV))
    oc, os_, ot = OQ.quantize_tensor(xb.float().numpy())
    assert np.float32(ts.item()) == ot == np.float32(1.0)
    np.testing.assert_array_equal(scales.cpu().numpy(), os_)
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)


# ------------------------------------------------------------- whole layer

def _check_layer(cfg, gpu, orc, check_perm=True, tight=Hp.TIGHT_FP32):
    assert np.float32(gpu["xq_tensor_scale"][0]) == orc["s_x"]
    np.testing.assert_array_equal(gpu["xq_codes"], orc["xq_codes"])
    np.testing.assert_array_equal(gpu["xq_scales"], orc["xq_scales"])
    near_ties = Hp.compare_routing(cfg, gpu, orc)
    n_pos = int(gpu["offsets"][-1])      # pairs computed (fewer than T * k under a route-tail skip)
    gpu = dict(gpu, perm=gpu["perm"][:n_pos], hq=gpu["hq"][:n_pos], hs=gpu["hs"][:n_pos])
    if check_perm and near_ties == 0:
        for k in ("counts", "offsets", "perm", "inv"):
            np.testing.assert_array_equal(gpu[k], orc[k])
    elif check_perm:
        counts, offsets, perm, inv = OP.permute(gpu["idx"], cfg.experts)  # validity only
        np.testing.assert_array_equal(gpu["perm"], perm)
    flips = Hp.compare_h(cfg, gpu["hq"], gpu["hs"], orc, Hp.perm_pairs(gpu["perm"], cfg.top_k))
    Hp.assert_flip_ceiling(cfg, flips, orc, Hp.perm_pairs(gpu["perm"], cfg.top_k))
    err = Hp.rel_l2(gpu["y"], orc["y"])
    assert err <= Hp.Y_REL_L2, f"y rel-L2 {err}"
    if flips == 0 and near_ties == 0:
        assert err <= tight, f"y rel-L2 {err} with identical codes"
    return err, flips, near_ties


@pytest.mark.parametrize("name", ["tiny", "mid_ragged", "mid_zipf"])
def test_layer_parity_small(nv, name):
    cfg = synth.get_config(name)
    w = Hp.layer_weights(cfg)
    gl = Hp.GpuLayer(cfg, w, cfg.tokens)
    x = synth.make_x(cfg.tokens, cfg.hidden, cfg.seed)
    gpu = gl.forward(x.to(DEV))
    orc = Hp.run_oracle(cfg, x, w)
    np.testing.assert_array_equal(gpu["idx"].shape, orc["idx"].shape)
    _check_layer(cfg, gpu, orc)


@pytest.mark.parametrize("tokens,flags", [(1, 0), (8, 0), (300, 0), (300, 1)],
                         ids=["fused-decode-1", "fused-decode-8", "tensor-core-300", "per-step-300"])
def test_dense_w4a4_ffn(nv, tokens, flags):
    """E = 1, k = 1: a dense W4A4 NVFP4 SwiGLU FFN (every token to expert 0,
    weight exactly 1) on each path, against the oracle."""
    cfg = synth.get_config("dense_w4a4").with_(tokens=tokens)
    w = Hp.layer_weights(cfg)
    gl = Hp.GpuLayer(cfg, w, 300, flags=flags)
    x = synth.make_x(tokens, cfg.hidden, cfg.seed)
    gpu = gl.forward(x.to(DEV))
    orc = Hp.run_oracle(cfg, x, w)
    assert np.all(gpu["idx"] == 0) and np.all(gpu["weights"] == np.float32(1.0))
    tensor_core = tokens > 8 and flags == 0
    err, flips, _ = _check_layer(cfg, gpu, orc,
                                 tight=Hp.TIGHT_FP16_PARTIALS if tensor_core else Hp.TIGHT_FP32)
    print(f"dense W4A4 FFN, {tokens} tokens, flags {flags}: rel-L2 {err:.2e}, h flips {flips}")


@pytest.mark.parametrize("name", ["tiny", "mid_ragged"])
def test_layer_given_xq_matches_internal(nv, name):
    """Same per-step kernels with and without a caller-supplied xq: bit-identical."""
    cfg = synth.get_config(name)
    w = Hp.layer_weights(cfg)
    gl = Hp.GpuLayer(cfg, w, cfg.tokens, flags=nv.MOE_FLAG_MULTI_KERNEL)
    x = synth.make_x(cfg.tokens, cfg.hidden, cfg.seed).to(DEV)
    a = gl.forward(x)
    b = gl.forward(x, xq=gl.quantize_act(x))
    np.testing.assert_array_equal(a["y"], b["y"])


def test_residual_and_determinism(nv):
    cfg = synth.get_config("mid_ragged")
    w = Hp.layer_weights(cfg)
    gl = Hp.GpuLayer(cfg, w, cfg.tokens)
    x = synth.make_x(cfg.tokens, cfg.hidden, cfg.seed)
    a = gl.forward(x.to(DEV), residual=True)
    b = gl.forward(x.to(DEV), residual=True)
    np.testing.assert_array_equal(a["y"], b["y"])
    np.testing.assert_array_equal(a["x_next_bits"], b["x_next_bits"])
    ref = (x.float() + torch.from_numpy(a["y"])).to(torch.bfloat16)
    np.testing.assert_array_equal(a["x_next_bits"], ref.view(torch.int16).numpy().view(np.uint16))
    orc = Hp.run_oracle(cfg, x, w, residual=True)
    Hp.check_x_next(a["x_next_bits"], orc["x_next_bits"], a["y"], orc["y"])


def test_empty_call_and_errors(nv):
    cfg = synth.get_config("tiny")
    gl = Hp.GpuLayer(cfg, Hp.layer_weights(cfg), 4)
    x = torch.zeros(0, cfg.hidden, dtype=torch.bfloat16, device=DEV)
    y = torch.full((1, cfg.hidden), 7.0, device=DEV)
    nv.moe_forward(gl.layer, x, y, gl.ws, tokens=0)      # no-op
    assert torch.all(y == 7.0)
    xx = torch.zeros(5, cfg.hidden, dtype=torch.bfloat16, device=DEV)
    yy = torch.empty(5, cfg.hidden, device=DEV)
    with pytest.raises(nv.MoeError) as ei:
        nv.moe_forward(gl.layer, xx, yy, gl.ws)          # T > max_tokens
    assert ei.value.status == nv.MOE_ERR_INVALID_ARGUMENT
    bad = nv.make_desc(100, 16, 2, 128, 4)
    assert nv.moe_workspace_bytes(bad) == 0


def test_graph_capture_replay(nv):
    cfg = synth.get_config("mid_zipf")
    w = Hp.layer_weights(cfg)
    gl = Hp.GpuLayer(cfg, w, cfg.tokens)
    x = synth.make_x(cfg.tokens, cfg.hidden, cfg.seed).to(DEV)
    ref = gl.forward(x, debug=False)["y"]
    y = torch.empty(cfg.tokens, cfg.hidden, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        nv.moe_forward(gl.layer, x, y, gl.ws, stream=s)  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        nv.moe_forward(gl.layer, x, y, gl.ws, stream=s)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(y.cpu().numpy(), ref)


# ------------------------------------------------------- full-size layer

@pytest.fixture(scope="module")
def full_layer(nv):
    cfg = synth.get_config("decode_b1")
    w = Hp.layer_weights(cfg, device=DEV)
    gl = Hp.GpuLayer(cfg, w, 65536)
    experts = {m: Hp.oracle_experts(w[m]) for m in ("gate", "up", "down")}
    yield cfg, w, gl, experts
    gl.layer.close()


@pytest.mark.parametrize("name", ["decode_b1", "decode_b8"])
def test_decode_full_size(nv, full_layer, name):
    _, w, gl, experts = full_layer
    cfg = synth.get_config(name)
    gl.cfg = cfg
    for step in range(2):
        x = synth.make_x(cfg.tokens, cfg.hidden, cfg.seed, step=step)
        gpu = gl.forward(x.to(DEV))
        orc = Hp.run_oracle(cfg, x, w, experts=experts)
        err, flips, ties = _check_layer(cfg, gpu, orc)
        print(f"{name} step {step}: rel-L2 {err:.3e}, h flips {flips}, near ties {ties}")


def _sampled_prefill(nv, full_layer, cfg, samples):
    _, w, gl, experts = full_layer
    if cfg.zipf_bias:
        w = dict(w, bias=synth.make_router_bias(cfg.experts, cfg.seed, device=DEV))
        gl = gl.with_bias(w["bias"])
    gl.cfg = cfg
    x = synth.make_x(cfg.tokens, cfg.hidden, cfg.seed)
    gpu = gl.forward(x.to(DEV))
    xf = x.float().numpy()
    # routing over every token, in fp64
    b = w["bias"].cpu().numpy() if w["bias"] is not None else None
    logits = OL.router_logits(xf, w["router_w"].cpu().numpy(), b)
    idx, wt = OL.route(logits, cfg.top_k)
    near = Hp.compare_routing(cfg, gpu, dict(logits=logits, idx=idx, w=wt))
    # permutation: exact when no near tie decided a pick, else valid for the GPU's picks
    ref = OP.permute(gpu["idx"] if near else idx, cfg.experts)
    for k, v in zip(("counts", "offsets", "perm", "inv"), ref):
        np.testing.assert_array_equal(gpu[k], v)
    # sampled tokens, full oracle: the tensor-core GEMMs' edge rows on purpose
    # (every token in the last, ragged 128-row tile of the most loaded expert,
    # the tokens routed to experts with a single row, the first and the last
    # token) plus a random draw
    counts, offsets, perm = gpu["counts"], gpu["offsets"], gpu["perm"]
    big = int(np.argmax(counts))
    last_tile = perm[offsets[big] + (counts[big] - 1) // 128 * 128: offsets[big + 1]] // cfg.top_k
    singles = np.concatenate([perm[offsets[e]:offsets[e] + 1] for e in np.nonzero(counts == 1)[0]] +
                             [np.zeros(0, np.int32)]) // cfg.top_k
    rng = np.random.default_rng(cfg.tokens)
    chosen = np.concatenate([last_tile[:64], singles[:16], [0, cfg.tokens - 1],
                             rng.choice(cfg.tokens, size=samples, replace=False)])
    rows = np.unique(chosen.astype(np.int64))
    orc = Hp.run_oracle(cfg, x, w, tokens=rows, experts=experts)
    # the experts' NVFP4 activations: one tensor scale over all tokens
    assert np.float32(gpu["xq_tensor_scale"][0]) == orc["s_x"]
    np.testing.assert_array_equal(gpu["xq_codes"][rows], orc["xq_codes"])
    np.testing.assert_array_equal(gpu["xq_scales"][rows], orc["xq_scales"])
    err = Hp.rel_l2(gpu["y"][rows], orc["y"])
    assert err <= Hp.Y_REL_L2, f"sampled y rel-L2 {err}"
    # sampled h rows: position of pair (t, j) is inv[t*k + j]
    pos = gpu["inv"].reshape(cfg.tokens, cfg.top_k)[rows].reshape(-1)
    pairs = np.array([(ri, j) for ri in range(len(rows)) for j in range(cfg.top_k)])
    flips = Hp.compare_h(cfg, gpu["hq"][pos], gpu["hs"][pos], orc, pairs)
    Hp.assert_flip_ceiling(cfg, flips, orc, pairs)
    print(f"{cfg.name}: {len(rows)} sampled tokens ({len(last_tile)} in the largest expert's last "
          f"tile, {len(singles)} on single-row experts), rel-L2 {err:.3e}, h flips {flips}, "
          f"near ties {near}")


@pytest.mark.parametrize("tokens", [9, 16])
def test_small_batch_verify_full_size(nv, full_layer, tokens):
    """9 and 16 tokens (speculative-verify batches just past the fused kernel's
    8) through the full-size layer on the tensor-core path, every token against
    the oracle."""
    cfg0, w, gl, experts = full_layer
    cfg = cfg0.with_(tokens=tokens)
    gl.cfg = cfg
    x = synth.make_x(tokens, cfg.hidden, cfg.seed, step=500 + tokens)
    n0 = nv.moe_kernel_launches()
    gpu = gl.forward(x.to(DEV), residual=True)
    assert nv.moe_kernel_launches() - n0 > 1      # not the fused decode kernel
    orc = Hp.run_oracle(cfg, x, w, experts=experts, residual=True)
    err, flips, ties = _check_layer(cfg, gpu, orc, tight=Hp.TIGHT_FP16_PARTIALS)
    Hp.check_x_next(gpu["x_next_bits"], orc["x_next_bits"], gpu["y"], orc["y"])
    print(f"verify batch T={tokens}: rel-L2 {err:.2e}, h flips {flips}, near ties {ties}")


def test_prefill_4k_zipf_full_size(nv, full_layer):
    _sampled_prefill(nv, full_layer, synth.get_config("prefill_4k_zipf"), samples=48)


def test_prefill_64k_full_size(nv, full_layer):
    _sampled_prefill(nv, full_layer, synth.get_config("prefill_64k"), samples=24)


def test_stacked_decode_four_layers(nv):
    """Four stacked full-size layers with the bf16 residual; the oracle runs its
    own chain from the same x_0."""
    cfg = synth.get_config("decode_b1_stack48")
    layers, orc_layers = [], []
    for l in range(4):
        w = Hp.layer_weights(cfg, layer=l, device=DEV)
        layers.append(Hp.GpuLayer(cfg, w, 1))
        orc_layers.append(dict(router_w=w["router_w"].cpu().numpy(), bias=None,
                               **{m: Hp.oracle_experts(w[m]) for m in ("gate", "up", "down")}))
    x0 = synth.make_x(1, cfg.hidden, cfg.seed)
    cur = x0.to(DEV)
    gpu_y = []
    for gl in layers:
        out = gl.forward(cur, residual=True, debug=False)
        gpu_y.append(out["y"])
        cur = torch.from_numpy(out["x_next_bits"].view(np.int16)).view(torch.bfloat16).to(DEV)
    res = OL.moe_stack(x0.float().numpy(), orc_layers, cfg.top_k, cfg.h_tensor_scale)
    for l, r in enumerate(res):
        err = Hp.rel_l2(gpu_y[l], r["y"])
        print(f"stack layer {l}: rel-L2 {err:.3e}")
        assert err <= Hp.Y_REL_L2
    for gl in layers:
        gl.layer.close()


def test_stack_48_layers_teacher_forced(nv):
    """The bench's decode workload: one token through 48 stacked full-size
    layers in one moe_stack_forward launch, every layer's y recorded.  Each
    layer l is checked against the oracle run on the GPU's own input x_l
    (teacher forcing: x_(l+1) = bf16(x_l + y_l) rebuilt on the host from the
    recorded y, exactly as the kernel forms it), within rel-L2 2e-3; the
    oracle's own 48-layer chain is also run and its end-to-end drift reported."""
    cfg = synth.get_config("decode_b1_stack48")
    L = cfg.layers
    gls, orc_layers = [], []
    def regen(layer, m):
        # the oracle's copy of one expert, redrawn on the device from its own seed
        # (the same draw as the layer's), so 48 layers of fp32 weights never sit in memory
        rows, cols = (cfg.hidden, cfg.inter) if m == "down" else (cfg.inter, cfg.hidden)
        src = lambda e: synth.make_expert_weight(layer, m, e, rows, cols, cfg.seed, device=DEV).cpu().numpy()
        return OL.LazyExperts(src, cfg.experts, rows)

    for l in range(L):
        w = Hp.layer_weights(cfg, layer=l, device=DEV)
        gls.append(Hp.GpuLayer(cfg, w, 1))
        orc_layers.append(dict(router_w=w["router_w"].cpu().numpy(), bias=None,
                               **{m: regen(l, m) for m in ("gate", "up", "down")}))
        del w
        torch.cuda.empty_cache()
    x0 = synth.make_x(1, cfg.hidden, cfg.seed, step=48)
    ys = [torch.empty(1, cfg.hidden, device=DEV) for _ in range(L)]
    x_out = torch.empty(1, cfg.hidden, dtype=torch.bfloat16, device=DEV)
    nv.moe_stack_forward([g.layer for g in gls], x0.to(DEV), x_out, gls[0].ws, ys=ys)
    torch.cuda.synchronize()
    assert nv.moe_layer_status(gls[0].layer) == nv.MOE_OK
    cur = x0.float()
    worst = 0.0
    for l in range(L):
        y = ys[l].cpu()
        p = orc_layers[l]
        r = OL.moe_layer(cur.numpy(), p["router_w"], None, p["gate"], p["up"], p["down"], cfg.top_k,
                         cfg.h_tensor_scale)
        err = Hp.rel_l2(y.numpy(), r["y"])
        worst = max(worst, err)
        assert err <= Hp.Y_REL_L2, f"layer {l}: rel-L2 {err}"
        cur = (cur + y).to(torch.bfloat16).float()       # the kernel's x_(l+1) = bf16(x_l + y_l)
    np.testing.assert_array_equal(cur.to(torch.bfloat16).view(torch.int16).numpy(),
                                  x_out.view(torch.int16).cpu().numpy())
    res = OL.moe_stack(x0.float().numpy(), orc_layers, cfg.top_k, cfg.h_tensor_scale)
    from oracle.formats import f32_from_bf16_bits
    drift = Hp.rel_l2(x_out.float().cpu().numpy(), f32_from_bf16_bits(res[-1]["x_next_bits"]))
    print(f"48 stacked layers, teacher forced: worst per-layer rel-L2 {worst:.2e}; "
          f"end-to-end drift of x_48 against the oracle's own chain {drift:.2e}")
    for g in gls:
        g.layer.close()


# --------------------------------------------------- fused decode kernel

def _compare_paths(cfg, a, b, tight=Hp.TIGHT_FP32):
    """Fused decode vs per-step kernels: identical routing, permutation and
    activation codes; h codes may differ only where rounding order can move
    them, y within fp32 round-off when they do not."""
    for key in ("idx", "counts", "offsets", "perm", "inv", "xq_codes", "xq_scales",
                "xq_tensor_scale"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    np.testing.assert_allclose(a["logits"], b["logits"], rtol=0, atol=Hp.LOGIT_TOL)
    dl = float(np.max(np.abs(a["logits"].astype(np.float64) - b["logits"]), initial=0.0))
    dw = np.abs(a["weights"].astype(np.float64) - b["weights"])
    assert np.all(dw <= Hp.weight_tol(b["weights"], dl)), np.max(dw)
    diff = int(np.count_nonzero(a["hq"] != b["hq"]) + np.count_nonzero(a["hs"] != b["hs"]))
    err = Hp.rel_l2(a["y"], b["y"])
    assert err <= (tight if diff == 0 else Hp.Y_REL_L2), (err, diff)
    return err, diff


def test_fused_decode_tiny_matches_oracle_and_multikernel(nv):
    cfg = synth.get_config("tiny")
    w = Hp.layer_weights(cfg)
    fused = Hp.GpuLayer(cfg, w, cfg.tokens)
    multi = fused.with_flags(nv.MOE_FLAG_MULTI_KERNEL)
    x = synth.make_x(cfg.tokens, cfg.hidden, cfg.seed)
    a = fused.forward(x.to(DEV), residual=True)
    b = multi.forward(x.to(DEV), residual=True)
    _compare_paths(cfg, a, b)
    orc = Hp.run_oracle(cfg, x, w, residual=True)
    _check_layer(cfg, a, orc)


# every shared-memory plan of the fused kernel at this shape: one token (gate/up
# slots in the ring), 2-6 tokens (slots over the x staging and router rows,
# five or four of them), 8 tokens (four slots, down units streaming through)
@pytest.mark.parametrize("tokens", [1, 2, 3, 5, 6, 8])
def test_fused_decode_full_size_matches_multikernel(nv, full_layer, tokens):
    cfg0, w, gl, experts = full_layer
    cfg = cfg0.with_(tokens=tokens)
    gl.cfg = cfg
    multi = gl.with_flags(nv.MOE_FLAG_MULTI_KERNEL)
    multi.cfg = cfg
    x = synth.make_x(tokens, cfg.hidden, cfg.seed, step=100 + tokens)
    a = gl.forward(x.to(DEV), residual=True)
    b = multi.forward(x.to(DEV), residual=True)
    err, diff = _compare_paths(cfg, a, b)
    orc = Hp.run_oracle(cfg, x, w, experts=experts, residual=True)
    e2, flips, ties = _check_layer(cfg, a, orc)
    print(f"fused T={tokens}: vs per-step rel-L2 {err:.2e} ({diff} h bytes differ); "
          f"vs oracle {e2:.2e}, flips {flips}, near ties {ties}")
    multi.layer.close()


def _stack(nv, layers_n=4):
    cfg = synth.get_config("decode_b1_stack48")
    gls, orc_layers = [], []
    for l in range(layers_n):
        w = Hp.layer_weights(cfg, layer=l, device=DEV)
        gls.append(Hp.GpuLayer(cfg, w, 8))
        orc_layers.append(dict(router_w=w["router_w"].cpu().numpy(), bias=None,
                               **{m: Hp.oracle_experts(w[m]) for m in ("gate", "up", "down")}))
    return cfg, gls, orc_layers


@pytest.fixture(scope="module")
def stack4(nv):
    cfg, gls, orc_layers = _stack(nv, 4)
    yield cfg, gls, orc_layers
    for g in gls:
        g.layer.close()


@pytest.mark.parametrize("tokens", [1, 5])
def test_stack_forward_matches_oracle_chain_and_per_layer_calls(nv, stack4, tokens):
    cfg, gls, orc_layers = stack4
    L = len(gls)
    x0 = synth.make_x(tokens, cfg.hidden, cfg.seed, step=7)
    xd = x0.to(DEV)
    ys = [torch.empty(tokens, cfg.hidden, device=DEV) for _ in range(L)]
    x_out = torch.empty(tokens, cfg.hidden, dtype=torch.bfloat16, device=DEV)
    nv.moe_stack_forward([g.layer for g in gls], xd, x_out, gls[0].ws, ys=ys)
    torch.cuda.synchronize()
    assert nv.moe_layer_status(gls[0].layer) == nv.MOE_OK
    # the same chain as separate per-layer calls: the same kernel, bit for bit
    cur = xd
    for l, g in enumerate(gls):
        g.cfg = cfg.with_(tokens=tokens)
        out = g.forward(cur, residual=True, debug=False)
        np.testing.assert_array_equal(ys[l].cpu().numpy(), out["y"])
        cur = torch.from_numpy(out["x_next_bits"].view(np.int16)).view(torch.bfloat16).to(DEV)
    np.testing.assert_array_equal(x_out.view(torch.int16).cpu().numpy(),
                                  cur.view(torch.int16).cpu().numpy())
    # and the oracle's own chain from the same x0
    res = OL.moe_stack(x0.float().numpy(), orc_layers, cfg.top_k, cfg.h_tensor_scale)
    for l, r in enumerate(res):
        err = Hp.rel_l2(ys[l].cpu().numpy(), r["y"])
        print(f"stack T={tokens} layer {l}: rel-L2 {err:.3e}")
        assert err <= Hp.Y_REL_L2


def test_stack_forward_graph_capture(nv, stack4):
    cfg, gls, _ = stack4
    x = synth.make_x(2, cfg.hidden, cfg.seed, step=9).to(DEV)
    ref = torch.empty(2, cfg.hidden, dtype=torch.bfloat16, device=DEV)
    nv.moe_stack_forward([g.layer for g in gls], x, ref, gls[0].ws)
    torch.cuda.synchronize()
    out = torch.zeros_like(ref)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        nv.moe_stack_forward([gl.layer for gl in gls], x, out, gls[0].ws, stream=s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.view(torch.int16).cpu().numpy(),
                                      ref.view(torch.int16).cpu().numpy())
    assert nv.moe_layer_status(gls[0].layer) == nv.MOE_OK


def test_stack_forward_rejects_large_batches(nv, stack4):
    cfg, gls, _ = stack4
    x = torch.zeros(9, cfg.hidden, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(nv.MoeError) as ei:
        nv.moe_stack_forward([g.layer for g in gls], x, x.clone(), gls[0].ws)
    assert ei.value.status in (nv.MOE_ERR_INVALID_ARGUMENT, nv.MOE_ERR_UNSUPPORTED_SHAPE)


# ------------------------------------------------ tensor-core prefill GEMMs

@pytest.mark.parametrize("name", ["mid_tc", "mid_tc_zipf"])
def test_tensor_core_prefill_matches_oracle_and_cuda_cores(nv, name):
    cfg = synth.get_config(name)
    w = Hp.layer_weights(cfg)
    tc = Hp.GpuLayer(cfg, w, cfg.tokens)
    cc = tc.with_flags(nv.MOE_FLAG_MULTI_KERNEL)
    x = synth.make_x(cfg.tokens, cfg.hidden, cfg.seed)
    a = tc.forward(x.to(DEV), residual=True)
    b = cc.forward(x.to(DEV), residual=True)
    orc = Hp.run_oracle(cfg, x, w, residual=True)
    err, flips, ties = _check_layer(cfg, a, orc, tight=Hp.TIGHT_FP16_PARTIALS)
    counts = np.sort(orc["counts"])[::-1]
    print(f"{name}: tensor-core vs oracle rel-L2 {err:.2e}, flips {flips}, near ties {ties}, "
          f"largest expert {counts[0]} rows")
    assert counts[0] > 128                     # several M-tiles for one expert
    _compare_paths(cfg, a, b, tight=Hp.TIGHT_FP16_PARTIALS)
    Hp.check_x_next(a["x_next_bits"], orc["x_next_bits"], a["y"], orc["y"])


def test_tensor_core_prefill_deterministic_and_capturable(nv):
    cfg = synth.get_config("mid_tc")
    gl = Hp.GpuLayer(cfg, Hp.layer_weights(cfg), cfg.tokens)
    x = synth.make_x(cfg.tokens, cfg.hidden, cfg.seed).to(DEV)
    ref = gl.forward(x, debug=False)["y"]
    again = gl.forward(x, debug=False)["y"]
    np.testing.assert_array_equal(ref, again)
    y = torch.empty(cfg.tokens, cfg.hidden, device=DEV)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        nv.moe_forward(gl.layer, x, y, gl.ws, stream=s)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(y.cpu().numpy(), ref)
    assert nv.moe_layer_status(gl.layer) == nv.MOE_OK


# ------------------------------------------------------- route-tail skip

@pytest.mark.parametrize("path,name,tokens,keep", [("fused", "mid_tc", 1, 1), ("fused", "mid_tc", 8, 2),
                                                  ("per-step", "mid_zipf", 37, 2),
                                                  ("tensor-core", "mid_tc", 300, 2)])
def test_route_tail_skip(nv, path, name, tokens, keep):
    """Route-tail skip (keep ranks < r and the resident experts, renormalise
    over the kept picks) on every path against the oracle: dropped picks read
    -1 with weight 0, the permutation holds only the kept pairs, y is the
    weighted sum over the kept picks."""
    cfg = synth.get_config(name).with_(tokens=tokens)
    w = Hp.layer_weights(cfg)
    resident = np.zeros(cfg.experts, dtype=np.uint8)
    resident[::3] = 1                                    # every third expert is "cached"
    flags = nv.MOE_FLAG_MULTI_KERNEL if path == "per-step" else 0
    gl = Hp.GpuLayer(cfg, w, tokens, flags=flags, route_keep=keep, resident=resident)
    x = synth.make_x(tokens, cfg.hidden, cfg.seed, step=keep)
    n0 = nv.moe_kernel_launches()
    gpu = gl.forward(x.to(DEV), residual=True)
    launches = nv.moe_kernel_launches() - n0
    assert (launches == 1) == (path == "fused"), launches   # the path under test really ran
    orc = Hp.run_oracle(cfg, x, w, residual=True, keep=keep, resident=resident)
    dropped = int((orc["idx"] < 0).sum())
    assert 0 < dropped < tokens * cfg.top_k              # the skip did something, not everything
    err, flips, ties = _check_layer(cfg, gpu, orc,
                                    tight=Hp.TIGHT_FP16_PARTIALS if path == "tensor-core" else Hp.TIGHT_FP32)
    if ties == 0:
        np.testing.assert_array_equal(gpu["idx"], orc["idx"])
    Hp.check_x_next(gpu["x_next_bits"], orc["x_next_bits"], gpu["y"], orc["y"])
    # without a residency mask the whole tail is dropped: every token keeps exactly r picks
    nv.moe_layer_set_resident(gl.layer, None)
    gl.resident = None
    gpu2 = gl.forward(x.to(DEV))
    orc2 = Hp.run_oracle(cfg, x, w, keep=keep)
    assert int(gpu2["offsets"][-1]) == tokens * keep
    _check_layer(cfg, gpu2, orc2, tight=Hp.TIGHT_FP16_PARTIALS if path == "tensor-core" else Hp.TIGHT_FP32)
    print(f"route-tail skip {path} T={tokens} keep={keep}: {dropped} picks dropped, rel-L2 {err:.2e}, "
          f"flips {flips}, near ties {ties}")


# ------------------------------------------------- fp16 partial range check

def test_fp16_partial_overflow_is_reported(nv):
    """The tensor-core path stores each pair's w * o as an fp16 partial: down
    weights scaled up until |w o| passes 65520 make the forward report
    MOE_ERR_PARTIAL_OVERFLOW (read and cleared by moe_layer_status) instead of
    an output with infinities in it.  The CUDA-core paths keep fp32 partials and
    report nothing; ordinary weights report nothing on the tensor-core path."""
    cfg = synth.get_config("mid_tc").with_(tokens=300)
    w = Hp.layer_weights(cfg)
    big = dict(w, down=w["down"] * 1e8)
    x = synth.make_x(cfg.tokens, cfg.hidden, cfg.seed).to(DEV)
    y = torch.empty(cfg.tokens, cfg.hidden, dtype=torch.float32, device=DEV)
    for weights, flags, expect in ((big, 0, nv.MOE_ERR_PARTIAL_OVERFLOW),
                                   (big, nv.MOE_FLAG_MULTI_KERNEL, nv.MOE_OK),
                                   (w, 0, nv.MOE_OK)):
        gl = Hp.GpuLayer(cfg, weights, cfg.tokens, flags=flags)
        nv.moe_forward(gl.layer, x, y, gl.ws)
        torch.cuda.synchronize()
        st = nv.moe_layer_status(gl.layer)
        assert st == expect, (flags, nv.status_string(st))
        assert nv.moe_layer_status(gl.layer) == nv.MOE_OK     # the status word was cleared
        if expect == nv.MOE_OK:
            assert torch.isfinite(y).all()
