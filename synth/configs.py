"""Workload shapes for the routed-expert MoE layer.

The page "capy-flash v0.7.1: a 125B MoE on 64 GB of RAM ..." ("What shipped")
gives the model as 48 layers x 512 routed experts; the pages print no hidden or
expert-intermediate width, so the layer widths below (hidden 2048, expert
intermediate 512, top-10) are synthetic stand-ins of that structure.  The
capy-flash status post (feedman.me repost, "Where it stands") measures decode
at one request and a 64k-token prefill, which the decode-b1 / stacked-decode and
65,536-token-prefill workloads stand in for.

Every config is seeded (seed 0) and synthetic.
"""
from dataclasses import dataclass, replace


@dataclass(frozen=True)
class LayerConfig:
    name: str
    tokens: int          # T
    hidden: int          # H
    experts: int         # E
    top_k: int           # k
    inter: int           # I (expert intermediate width)
    layers: int = 1      # stacked layers with a residual add between them
    zipf_bias: bool = False  # per-expert router bias with Zipf(1.1) ranks
    seed: int = 0
    h_tensor_scale: float = 2.0 ** -6  # static tensor scale of the SwiGLU output

    @property
    def pairs(self) -> int:
        return self.tokens * self.top_k

    def with_(self, **kw) -> "LayerConfig":
        return replace(self, **kw)


CONFIGS = {
    # tiny layer: 4 tokens, hidden 256, 16 experts, top-2, intermediate 128
    "tiny": LayerConfig("tiny", tokens=4, hidden=256, experts=16, top_k=2, inter=128),
    # one decode token through one full-size layer
    "decode_b1": LayerConfig("decode_b1", tokens=1, hidden=2048, experts=512, top_k=10, inter=512),
    # 8 independent decode tokens (8 concurrent requests)
    "decode_b8": LayerConfig("decode_b8", tokens=8, hidden=2048, experts=512, top_k=10, inter=512),
    # 4096-token prefill with Zipf-skewed expert loads
    "prefill_4k_zipf": LayerConfig("prefill_4k_zipf", tokens=4096, hidden=2048, experts=512,
                                   top_k=10, inter=512, zipf_bias=True),
    # 48 stacked layers at batch-1 decode (about 43.5 GB of NVFP4 experts)
    "decode_b1_stack48": LayerConfig("decode_b1_stack48", tokens=1, hidden=2048, experts=512,
                                     top_k=10, inter=512, layers=48),
    # one layer at 65,536-token prefill
    "prefill_64k": LayerConfig("prefill_64k", tokens=65536, hidden=2048, experts=512,
                               top_k=10, inter=512),
    # mid-size parity shapes: several tiles per expert, ragged tails, odd token counts
    "mid_ragged": LayerConfig("mid_ragged", tokens=37, hidden=512, experts=32, top_k=4, inter=192),
    "mid_zipf": LayerConfig("mid_zipf", tokens=300, hidden=1024, experts=64, top_k=6, inter=320,
                            zipf_bias=True),
    # tensor-core prefill shapes: several 128-row tiles per expert with ragged tails
    "mid_tc": LayerConfig("mid_tc", tokens=333, hidden=512, experts=8, top_k=3, inter=256),
    "mid_tc_zipf": LayerConfig("mid_tc_zipf", tokens=517, hidden=768, experts=24, top_k=4,
                               inter=512, zipf_bias=True),
    # one expert, top-1: the layer reduces to a dense W4A4 NVFP4 SwiGLU FFN
    # (router weight exactly 1), the form of the pages' dense model's layers
    "dense_w4a4": LayerConfig("dense_w4a4", tokens=300, hidden=1024, experts=1, top_k=1, inter=1024),
}


def get_config(name: str) -> LayerConfig:
    return CONFIGS[name]
