"""CPU oracle of the routed-expert NVFP4 MoE layer -- TEST INFRASTRUCTURE ONLY.

This package is the slow, plain reference that the CUDA library is checked
against.  Only the test-suite, the package smoke check and the benchmark's CPU
baseline leg may import it; the library and its Python binding never do.  It
shares no code with the CUDA path: inputs come from ``synth`` (random draws
only), everything else is written here from the layer's definition.

What it computes, and where each step comes from
------------------------------------------------
The pages describe the capy-flash engine, not its kernels:
  * "capy-flash v0.7.1: a 125B MoE on 64 GB of RAM ..." ("What shipped"):
    48 layers x 512 routed experts; ("Why it matters"): the GPU expert path is
    W4A4 (4-bit weights and 4-bit activations) inside a captured CUDA graph,
    and decode is bound by memory bandwidth;
  * capy-flash status post (feedman.me repost, "What it's for"): the engine
    was built for NVIDIA's NVFP4 format; ("Where it stands"): every expert the
    router picks is computed (no route-tail skip).
The arithmetic of each step is therefore the plainest reading of a top-k
routed SwiGLU expert layer over NVFP4 operands:

  formats.py  E2M1 / E4M3 decode tables and round-to-nearest-even encoders
  quant.py    Q: NVFP4 block quantiser (16-element blocks, E4M3 block scale,
              fp32 tensor scale), every step one correctly rounded fp32 op
  router.py   S1 logits in fp64, S2 full-sort top-k (ties -> lower index) and
              the softmax renormalised over the k picks
  permute.py  S4 counting sort of (token, slot) pairs by expert, token order
  expert.py   S5 gate/up products, SwiGLU, requantisation of h;
              S6 down products and the weighted combine in slot order
  layer.py    the whole layer (and a stack of layers with a bf16 residual)

Pins (tests/test_oracle_*.py, run with -m "not gpu"): exhaustive format
tables against bit-field formulas and torch's float8 conversion; exhaustive
round-trips and midpoint/tie cases of Q; exact-rational checks of E4M3 scale
rounding; brute-force top-k; permutation invariants; identical-experts and
single-expert closed forms; a torch.float64 restatement of a whole tiny layer.
"""
