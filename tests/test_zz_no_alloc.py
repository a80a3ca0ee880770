"""moe_forward_noalloc, the forward for callers that cannot allocate device
memory (a host framework that owns all device allocations, a plugin handed only
buffers and a stream, a loop where cudaMalloc's synchronisation is not
allowed).  It must give what moe_forward gives, call after call, although its
scratch is one device array shared by every call.

This file is collected last on purpose: it also runs after every other GPU
test in the same process, where earlier calls have left the library's state
behind."""
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


def _forward_pair(nv, gl, x):
    """(y, x_next) from moe_forward with a workspace and from moe_forward_noalloc."""
    cfg = gl.cfg
    T = x.shape[0]
    ref_y = torch.empty(T, cfg.hidden, device=DEV)
    ref_xn = torch.empty(T, cfg.hidden, dtype=torch.bfloat16, device=DEV)
    nv.moe_forward(gl.layer, x, ref_y, gl.ws, residual=x, x_next=ref_xn)
    y = torch.full((T, cfg.hidden), float("nan"), device=DEV)
    xn = torch.zeros(T, cfg.hidden, dtype=torch.bfloat16, device=DEV)
    nv.moe_forward_noalloc(gl.layer, x, y, residual=x, x_next=xn)
    torch.cuda.synchronize()
    assert nv.moe_layer_status(gl.layer) == nv.MOE_OK
    return ref_y.cpu().numpy(), ref_xn, y.cpu().numpy(), xn


@pytest.mark.parametrize("name", ["tiny", "mid_zipf"])
def test_noalloc_matches_forward_two_calls_in_a_row(nv, name):
    cfg = synth.get_config(name)
    gl = Hp.GpuLayer(cfg, Hp.layer_weights(cfg), cfg.tokens)
    for step in range(2):  # two calls in a row, different inputs: stale scratch must not leak
        x = synth.make_x(cfg.tokens, cfg.hidden, cfg.seed, step=step).to(DEV)
        ref_y, ref_xn, y, xn = _forward_pair(nv, gl, x)
        assert np.all(np.isfinite(y))
        assert Hp.rel_l2(y, ref_y) <= Hp.Y_REL_L2
        Hp.check_x_next(xn.view(torch.int16).cpu().numpy().view(np.uint16),
                        ref_xn.view(torch.int16).cpu().numpy().view(np.uint16), y, ref_y)
    gl.layer.close()


def test_noalloc_fewer_tokens_than_max_and_capacity_limit(nv):
    cfg = synth.get_config("mid_ragged")
    big_t = 16384
    gl = Hp.GpuLayer(cfg, Hp.layer_weights(cfg), big_t)
    x = synth.make_x(5, cfg.hidden, cfg.seed).to(DEV)
    ref_y, _, y, _ = _forward_pair(nv, gl, x)
    assert Hp.rel_l2(y, ref_y) <= Hp.Y_REL_L2
    # past the scratch capacity the call is refused and writes nothing
    big = nv.make_desc(cfg.hidden, cfg.experts, cfg.top_k, cfg.inter, big_t)
    assert nv.moe_workspace_bytes(big) > nv.MOE_NOALLOC_SCRATCH_BYTES
    xb = torch.zeros(big_t, cfg.hidden, dtype=torch.bfloat16, device=DEV)
    yb = torch.full((big_t, cfg.hidden), 3.0, device=DEV)
    with pytest.raises(nv.MoeError) as ei:
        nv.moe_forward_noalloc(gl.layer, xb, yb)
    assert ei.value.status == nv.MOE_ERR_UNSUPPORTED_SHAPE
    torch.cuda.synchronize()
    assert torch.all(yb == 3.0)
    gl.layer.close()


def test_documented_capacity_for_the_decode_shape(nv):
    """The documented capacity (658 tokens at hidden 2048, 512 experts, top-10,
    intermediate 512): 658 tokens run, 659 are refused."""
    cfg = synth.get_config("decode_b1").with_(tokens=659)
    gl = Hp.GpuLayer(cfg, Hp.layer_weights(cfg, device=DEV), 659)
    x = synth.make_x(659, cfg.hidden, cfg.seed).to(DEV)
    y = torch.empty(659, cfg.hidden, device=DEV)
    nv.moe_forward_noalloc(gl.layer, x, y, tokens=658)
    torch.cuda.synchronize()
    assert nv.moe_layer_status(gl.layer) == nv.MOE_OK
    assert torch.isfinite(y[:658]).all()
    with pytest.raises(nv.MoeError) as ei:
        nv.moe_forward_noalloc(gl.layer, x, y, tokens=659)
    assert ei.value.status == nv.MOE_ERR_UNSUPPORTED_SHAPE
    gl.layer.close()
