"""Failure detection on the GPU without a fault: the bounded waits of the
persistent kernels run out on targets that nothing completes (tagged words
nobody writes, an mbarrier nobody arrives on), report the device timeout in
their status words, and leave the context usable for the next forward."""
import time

import numpy as np
import pytest
import torch

import synth
import nvfp4_routed_expert_gb300 as nv
from tests import helpers as Hp

DEV = "cuda"


@pytest.mark.gpu
def test_bounded_waits_run_out_and_report():
    scratch = torch.empty(nv.MOE_SELFTEST_SCRATCH_BYTES, dtype=torch.uint8, device=DEV)
    t0 = time.monotonic()
    words = nv.moe_selftest_bounded_waits(scratch)
    dt = time.monotonic() - t0
    assert words == (1, 1), words          # kDevErrTimeout in both status words
    assert dt < 60.0, dt                   # each wait gives up after about a second
    # the context is still usable: a fused decode call matches the oracle
    cfg = synth.get_config("tiny")
    w = Hp.layer_weights(cfg)
    gl = Hp.GpuLayer(cfg, w, cfg.tokens)
    x = synth.make_x(cfg.tokens, cfg.hidden, cfg.seed)
    gpu = gl.forward(x.to(DEV), residual=True)
    orc = Hp.run_oracle(cfg, x, w, residual=True)
    Hp.compare_routing(cfg, gpu, orc)
    assert Hp.rel_l2(gpu["y"], orc["y"]) <= Hp.Y_REL_L2
    assert nv.moe_layer_status(gl.layer) == nv.MOE_OK


@pytest.mark.gpu
def test_selftest_rejects_unaligned_scratch():
    scratch = torch.empty(nv.MOE_SELFTEST_SCRATCH_BYTES + 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(nv.MoeError) as ei:
        nv.moe_selftest_bounded_waits(scratch[1:])
    assert ei.value.status == nv.MOE_ERR_INVALID_ARGUMENT
