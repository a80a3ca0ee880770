"""Seeded random inputs of the routed-expert MoE layer (random draws only).

Distributions (the layer's synthetic workload):
  * activations x ~ N(0, 1), rounded to bf16;
  * router weights Wr ~ N(0, 0.02), fp32, shape [E][H];
  * expert gate/up/down weights ~ N(0, 0.02), fp32, shapes [I][H], [I][H], [H][I]
    per expert (each side quantises them to NVFP4 with its own quantiser);
  * skewed routing: a per-expert router bias b[e] = -s * ln(rank(e) + 1), where
    rank is a seeded random permutation of 0..E-1 and s = 1.1, i.e. the log of a
    Zipf(s) probability over the experts (the normalising constant cancels in the
    softmax and does not move the top-k).

Every tensor has its own torch.Generator seeded by ``mix_seed(seed, tensor id,
layer, expert)``; the same call on the same device always returns the same
values.  Draws on a CUDA device and on the CPU differ (different generators),
so a test that compares two implementations draws once and hands both the same
tensor.
"""
import math

import torch

MASK64 = (1 << 64) - 1

# tensor ids used in the seed mix
TENSOR_X = 1
TENSOR_ROUTER = 2
TENSOR_BIAS = 3
MATRIX_IDS = {"gate": 10, "up": 11, "down": 12}

WEIGHT_STD = 0.02
ZIPF_S = 1.1


def _splitmix64(z: int) -> int:
    z = (z + 0x9E3779B97F4A7C15) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def mix_seed(*parts: int) -> int:
    """Hash a tuple of small integers into a 63-bit generator seed."""
    h = 0x243F6A8885A308D3
    for p in parts:
        h = _splitmix64(h ^ (int(p) & MASK64))
    return h & ((1 << 63) - 1)


def _gen(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(mix_seed(*parts))
    return g


def make_x(tokens: int, hidden: int, seed: int = 0, layer: int = 0, step: int = 0,
           device="cpu") -> torch.Tensor:
    """Activations [T][H] bf16, N(0,1) rounded to nearest bf16."""
    g = _gen(device, seed, TENSOR_X, layer, step)
    x = torch.randn(tokens, hidden, generator=g, device=device, dtype=torch.float32)
    return x.to(torch.bfloat16)


def make_router(experts: int, hidden: int, seed: int = 0, layer: int = 0,
                device="cpu") -> torch.Tensor:
    """Router weights Wr [E][H] fp32 ~ N(0, 0.02)."""
    g = _gen(device, seed, TENSOR_ROUTER, layer)
    w = torch.empty(experts, hidden, device=device, dtype=torch.float32)
    return w.normal_(0.0, WEIGHT_STD, generator=g)


def make_router_bias(experts: int, seed: int = 0, layer: int = 0, s: float = ZIPF_S,
                     device="cpu") -> torch.Tensor:
    """Per-expert router bias [E] fp32 from a seeded Zipf(s) rank assignment."""
    g = _gen("cpu", seed, TENSOR_BIAS, layer)
    rank = torch.randperm(experts, generator=g)
    b = torch.tensor([-s * math.log(int(r) + 1) for r in rank], dtype=torch.float32)
    return b.to(device)


def make_expert_weight(layer: int, matrix: str, expert: int, rows: int, cols: int,
                       seed: int = 0, device="cpu", out=None) -> torch.Tensor:
    """One expert's fp32 weight matrix [rows][cols] ~ N(0, 0.02).

    gate and up have rows = I, cols = H; down has rows = H, cols = I.
    """
    g = _gen(device, seed, MATRIX_IDS[matrix], layer, expert)
    if out is None:
        out = torch.empty(rows, cols, device=device, dtype=torch.float32)
    return out.normal_(0.0, WEIGHT_STD, generator=g)


def make_expert_weights(layer: int, matrix: str, experts: int, rows: int, cols: int,
                        seed: int = 0, device="cpu") -> torch.Tensor:
    """All experts' fp32 weights [E][rows][cols]: expert e equals make_expert_weight(e)."""
    w = torch.empty(experts, rows, cols, device=device, dtype=torch.float32)
    for e in range(experts):
        make_expert_weight(layer, matrix, e, rows, cols, seed=seed, device=device, out=w[e])
    return w
