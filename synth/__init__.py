"""Seeded synthetic inputs for the routed-expert MoE layer.

This package is shared by the CUDA path's tests/bench and by the CPU oracle.
It draws random numbers and nothing else: no quantisation, routing or expert
arithmetic lives here (the method's steps are implemented separately on each
side).
"""
from .configs import CONFIGS, LayerConfig, get_config  # noqa: F401
from .inputs import (  # noqa: F401
    mix_seed,
    make_x,
    make_router,
    make_router_bias,
    make_expert_weight,
    make_expert_weights,
    MATRIX_IDS,
)
