#!/usr/bin/env python
"""Benchmark of the NVFP4 routed-expert MoE layer on GB300.

Workloads (seeded synthetic inputs; random-init weights; no datasets):
  decode  (default) batch-1 decode through 48 stacked MoE layers of hidden
          2048, 512 experts, top-10, expert intermediate 512 (about 43.5 GB
          of NVFP4 experts resident in HBM), bf16 residual between layers.
          One step = 128 consecutive decode tokens, each through all 48 layers
          in one launch of the fused decode kernel (moe_stack_forward),
          replayed from a CUDA graph together with the token's input copy.
  prefill one layer of the same shape at 65,536 tokens; one step = one call.

Metric: MoE-layer tokens/s = (tokens x layers) processed per second.

The printed JSON line also carries
  roofline      the dominant kernel against HBM bandwidth: for decode the
                fused kernel (all of S1-S6 for 48 layers in one launch), its
                algorithmic bytes per launch / its CUDA-event duration measured
                inside the timed region (the last token of the last step)
  e2e           the same metric through the C ABI with host buffers: each
                token's x is copied from pinned host memory and the layer
                stack's output read back, inside the timed region
  cpu_baseline  the CPU oracle timed on this host on a bounded sample
  clocks        SM clocks sampled during the timed region
  prefill_64k   (decode workload) a short measurement of the prefill workload
                with its own roofline: the gate/up grouped GEMM against the
                dense NVFP4 tensor peak (--no-prefill skips it)

--impl reference times the CPU oracle alone (the slow reference) on the
same metric, one bounded sample per step.
"""
import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
DECODE_TOKENS_PER_STEP = 128


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=("decode", "prefill"), default="decode")
    ap.add_argument("--layers", type=int, default=48)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="decode workload only: skip the prefill 64k measurement in the line")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock/throttle sampling every 200 ms in a child process."""

    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append(dict(sm=float(parts[2]), smax=float(parts[3]), active=parts[5],
                                 hw=parts[6], hwt=parts[7], swt=parts[8], pcap=parts[9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median([r["sm"] for r in rows])),
                "sm_max_mhz": max(r["smax"] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            for key in ("hbm_gbs", "hbm_GBs", "hbm"):
                if key in d and d[key]:
                    return float(d[key]), "measured"
        except (ValueError, OSError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


def fp4_tensor_peak():
    """Dense NVFP4 tensor peak (TFLOP/s): the measured bf16 cuBLAS burst x 6, the
    nominal fp4:bf16 ratio (13.5 : 2.25 PFLOP/s); fallback 1900 x 6."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            if d.get("bf16_tflops"):
                return 6.0 * float(d["bf16_tflops"]), "measured bf16 burst x 6 (nominal fp4:bf16)"
        except (ValueError, OSError):
            pass
    return 6.0 * FALLBACK_BF16_TFLOPS, "fallback bf16 x 6 (nominal fp4:bf16)"


# ------------------------------------------------------- measured traffic

# DRAM bytes (read + write) per unit from one ncu capture of each dominant
# kernel (profiles/decode_fused_b1.md, profiles/prefill_64k_gemm.md), valid
# only for the kernel source they were taken on: a changed source reports null.
NCU_TRAFFIC = {
    "decode": ("nvfp4_routed_expert_gb300/csrc/decode.cu",
               "62145f383d1620923cdb6d87f437b0143c8ac92c7c19d0a7655b1efe99dd71dc",
               89_690_624 / 4),          # per layer (4-layer launch, caches flushed)
    "prefill_gateup": ("nvfp4_routed_expert_gb300/csrc/prefill.cu",
                       "6f131f00194ba66b8e654761781300387f6d3015b5ec3b41e8f82ee4df1f10bf",
                       1_258_753_000),   # per launch at 65,536 tokens
}


def ncu_traffic(kind, units=1):
    import hashlib
    path, sha, per_unit = NCU_TRAFFIC[kind]
    try:
        with open(os.path.join(ROOT, path), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != sha:
                return None
    except OSError:
        return None
    return per_unit * units


# ------------------------------------------------------- algorithmic bytes

def nvfp4_bytes(rows, cols):
    return rows * cols // 2 + rows * cols // 16


def gateup_bytes(cfg, active_experts, pairs, tokens):
    """Algorithmic bytes of one S5 launch: every routed expert's gate and up
    matrices once (codes + block scales + tensor scales), the activation
    codes of the tokens, and the requantised h written per pair."""
    w = active_experts * (2 * nvfp4_bytes(cfg.inter, cfg.hidden) + 8)
    x = tokens * (nvfp4_bytes(1, cfg.hidden))
    h = pairs * nvfp4_bytes(1, cfg.inter)
    return w + x + h


def layer_bytes(cfg, active_experts, tokens):
    """Algorithmic bytes of one whole layer call (router weights, x, routed
    experts' three matrices, y and the bf16 residual in/out)."""
    router = cfg.experts * cfg.hidden * 4
    experts = active_experts * (3 * nvfp4_bytes(cfg.inter, cfg.hidden) + 12)
    io = tokens * cfg.hidden * (2 + 4 + 2)
    return router + experts + io


# ----------------------------------------------------------- CPU oracle

def oracle_decode_sample(cfg, layers, seed_step=0):
    """Prepare a bounded oracle sample: one decode token through `layers`
    stacked layers, weights drawn on the CPU for the routed experts only.
    Returns a callable that runs the (already quantised) chain."""
    import synth
    from oracle import layer as OL

    def src(layer, m):
        rows, cols = (cfg.inter, cfg.hidden) if m != "down" else (cfg.hidden, cfg.inter)
        return lambda e: synth.make_expert_weight(layer, m, e, rows, cols, cfg.seed).numpy()

    stack = []
    for l in range(layers):
        stack.append(dict(
            router_w=synth.make_router(cfg.experts, cfg.hidden, cfg.seed, l).numpy(), bias=None,
            **{m: OL.LazyExperts(src(l, m), cfg.experts, cfg.inter if m != "down" else cfg.hidden)
               for m in ("gate", "up", "down")}))
    x0 = synth.make_x(1, cfg.hidden, cfg.seed, step=seed_step).float().numpy()
    run = lambda: OL.moe_stack(x0, stack, cfg.top_k, cfg.h_tensor_scale)
    run()  # draws and quantises the routed experts; later runs reuse them
    return run


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count() or 1


def cpu_baseline_decode(cfg, layers=4, reps=2):
    run = oracle_decode_sample(cfg, layers)
    t0 = time.perf_counter()
    for _ in range(reps):
        run()
    dt = (time.perf_counter() - t0) / reps
    return {"value": layers / dt, "unit": "layer-tokens/s", "cores": blas_threads(),
            "kind": "oracle",
            "sample": f"1 decode token through {layers} full-size stacked layers, x{reps} "
                      f"(experts pre-quantised; numpy fp64, BLAS threads for the contractions)"}


# ------------------------------------------------------------------ ours

def build_stack(nv, torch, cfg, layers, max_tokens, dev):
    import synth
    stack = []
    for l in range(layers):
        router = synth.make_router(cfg.experts, cfg.hidden, cfg.seed, l, device=dev)
        bias = synth.make_router_bias(cfg.experts, cfg.seed, l, device=dev) if cfg.zipf_bias else None
        mats = []
        for m, (r, c) in (("gate", (cfg.inter, cfg.hidden)), ("up", (cfg.inter, cfg.hidden)),
                          ("down", (cfg.hidden, cfg.inter))):
            w = synth.make_expert_weights(l, m, cfg.experts, r, c, cfg.seed, device=dev)
            mats.append(nv.quantize_weights(w))
            del w
        desc = nv.make_desc(cfg.hidden, cfg.experts, cfg.top_k, cfg.inter, max_tokens,
                            cfg.h_tensor_scale)
        stack.append(nv.Layer(desc, router, bias, *mats))
    torch.cuda.synchronize()
    return stack


def run_decode(args, rank, world, local):
    import torch
    import nvfp4_routed_expert_gb300 as nv
    import synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = synth.get_config("decode_b1_stack48").with_(layers=args.layers)
    L = cfg.layers
    stack = build_stack(nv, torch, cfg, L, 1, dev)
    ws = stack[0].workspace(dev)
    x_in = torch.empty(1, cfg.hidden, dtype=torch.bfloat16, device=dev)
    x_out = torch.empty(1, cfg.hidden, dtype=torch.bfloat16, device=dev)
    n_tok = DECODE_TOKENS_PER_STEP
    pool = torch.stack([synth.make_x(1, cfg.hidden, cfg.seed, step=i, device=dev)[0]
                        for i in range(n_tok)])
    ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    stream = torch.cuda.Stream(device=dev)
    for e in ev:
        e.record(stream)
    torch.cuda.synchronize()
    # the fused stack kernel is the dominant (only) kernel: trace brackets it
    nv.moe_layer_set_trace(stack[0], nv.MOE_STEP_GATEUP, ev[0], ev[1])
    handles = [l for l in stack]

    with torch.cuda.stream(stream):
        x_in.copy_(pool[0:1])
        nv.moe_stack_forward(handles, x_in, x_out, ws, stream=stream)  # eager warm-up
    stream.synchronize()
    st = nv.moe_layer_status(stack[0], stream)
    assert st == 0, nv.status_string(st)
    n0 = nv.moe_kernel_launches()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        nv.moe_stack_forward(handles, x_in, x_out, ws, stream=stream)
    launches_per_token = nv.moe_kernel_launches() - n0

    def step():
        for i in range(n_tok):
            x_in.copy_(pool[i:i + 1], non_blocking=True)
            graph.replay()

    clocks = ClockSampler(local)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for _ in range(args.steps):
            step()
        t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    kernel_ms = ev[0].elapsed_time(ev[1])          # the last token of the last timed step
    st = nv.moe_layer_status(stack[0], stream)
    assert st == 0, nv.status_string(st)
    if world > 1:
        t = torch.tensor([elapsed_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    ms_per_step = elapsed_ms / args.steps
    layer_tokens = n_tok * L
    value = world * layer_tokens / (ms_per_step / 1e3)

    e2e = None
    if not args.no_e2e:
        host_in = pool.cpu().pin_memory()
        host_out = torch.empty(1, cfg.hidden, dtype=torch.bfloat16).pin_memory()
        with torch.cuda.stream(stream):
            for i in range(8):
                x_in.copy_(host_in[i:i + 1], non_blocking=True)
                graph.replay()
                host_out.copy_(x_out, non_blocking=True)
            stream.synchronize()
            t0 = time.perf_counter()
            for _ in range(args.steps):
                for i in range(n_tok):
                    x_in.copy_(host_in[i:i + 1], non_blocking=True)
                    graph.replay()
                    host_out.copy_(x_out, non_blocking=True)
                    stream.synchronize()
            dt = (time.perf_counter() - t0) / args.steps
        e2e = {"value": world * layer_tokens / dt, "unit": "layer-tokens/s",
               "h2d_bytes_per_step": n_tok * cfg.hidden * 2,
               "d2h_bytes_per_step": n_tok * cfg.hidden * 2}

    peak, peak_kind = measured_peaks()
    lb = layer_bytes(cfg, cfg.top_k, 1)
    launch_bytes = lb * L                             # one launch = one token through L layers
    achieved = launch_bytes / (kernel_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": f"k_decode (fused S1-S6, {L} layers per launch)",
                "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": peak_kind, "traffic": ncu_traffic("decode", L),
                "bytes_per_launch": launch_bytes, "launch_ms": kernel_ms,
                "per_layer_us": kernel_ms * 1e3 / L,
                "step_GBs": launch_bytes * n_tok / (ms_per_step / 1e3) / 1e9}
    return {
        "metric": "MoE-layer tokens/s (decode b=1)", "value": value, "unit": "layer-tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4",
        "data": "synthetic: seeded N(0,1) bf16 activations, N(0,0.02) weights quantised to NVFP4",
        "config": {"workload": f"decode b=1 through {L} stacked MoE layers (hidden {cfg.hidden}, "
                               f"{cfg.experts} experts, top-{cfg.top_k}, intermediate {cfg.inter})",
                   "tokens_per_step": n_tok, "layers": L,
                   "stack_tokens_per_s": world * n_tok / (ms_per_step / 1e3),
                   "l2": f"inputs larger than L2: {L} layers x {lb / 1e6:.1f} MB touched per token",
                   "parallelism": f"replicas x{world}"},
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": int(launches_per_token * n_tok * args.steps),
        "clocks": clk,
    }


def run_prefill(args, rank, world, local, steps=None, warmup=None):
    """One MoE layer at 65,536 tokens through moe_forward (tensor-core path)."""
    import torch
    import nvfp4_routed_expert_gb300 as nv
    import synth

    steps = args.steps if steps is None else steps
    warmup = args.warmup if warmup is None else warmup
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = synth.get_config("prefill_64k")
    layer = build_stack(nv, torch, cfg, 1, cfg.tokens, dev)[0]
    ws = layer.workspace(dev)
    x = synth.make_x(cfg.tokens, cfg.hidden, cfg.seed, device=dev)
    y = torch.empty(cfg.tokens, cfg.hidden, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    n0 = nv.moe_kernel_launches()
    with torch.cuda.stream(stream):
        nv.moe_forward(layer, x, y, ws, stream=stream)
    per_call = nv.moe_kernel_launches() - n0
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            nv.moe_forward(layer, x, y, ws, stream=stream)
    stream.synchronize()
    # the gate/up grouped GEMM (S5) is the dominant kernel: trace events bracket
    # it (with the tiny M-tile list kernel before it) in every timed call
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for pair in gev:              # torch creates the CUDA event at its first record
        for e in pair:
            e.record(stream)
    stream.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for i in range(steps):
            nv.moe_layer_set_trace(layer, nv.MOE_STEP_GATEUP, gev[i][0], gev[i][1])
            nv.moe_forward(layer, x, y, ws, stream=stream)
        t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    nv.moe_layer_set_trace(layer, nv.MOE_STEP_NONE, None, None)
    ms = t0.elapsed_time(t1) / steps
    gate_ms = float(np.mean([a.elapsed_time(b) for a, b in gev]))
    pairs = cfg.tokens * cfg.top_k
    flops_gateup = 4 * cfg.hidden * cfg.inter * pairs
    flops = 6 * cfg.hidden * cfg.inter * pairs
    peak, peak_src = fp4_tensor_peak()
    achieved = flops_gateup / (gate_ms / 1e3) / 1e12
    roofline = {"bound": "tensor", "kernel": "k_grouped_gemm<kGateUp> (S5: gate/up FP4 grouped GEMM "
                "+ SwiGLU + requantisation)", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": peak_src,
                "traffic": ncu_traffic("prefill_gateup"), "traffic_unit": "bytes",
                "flops_per_launch": flops_gateup, "launch_ms": gate_ms}
    # end to end: x from pinned host memory, y back to pinned host memory
    x_h = x.cpu().pin_memory()
    y_h = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    e_steps = max(1, min(steps, 3))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e_steps):
            x.copy_(x_h, non_blocking=True)
            nv.moe_forward(layer, x, y, ws, stream=stream)
            y_h.copy_(y, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e_ms = e0.elapsed_time(e1) / e_steps
    e2e = {"value": world * cfg.tokens / (e_ms / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": x.numel() * 2, "d2h_bytes_per_step": y.numel() * 4}
    return {
        "metric": "MoE-layer tokens/s (prefill 64k)", "value": world * cfg.tokens / (ms / 1e3),
        "unit": "tokens/s", "n_gpus": world, "steps": steps, "warmup": warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "nvfp4", "data": "synthetic: seeded N(0,1) bf16 activations, N(0,0.02) weights "
                                  "quantised to NVFP4",
        "config": {"workload": "one MoE layer at 65,536-token prefill (hidden 2048, 512 experts, "
                               "top-10, intermediate 512)", "tokens": cfg.tokens,
                   "l2": "inputs larger than L2 (x 268 MB, experts 0.9 GB)",
                   "parallelism": f"replicas x{world}"},
        "expert_tflops": flops / (ms / 1e3) / 1e12,
        "roofline": roofline, "e2e": e2e,
        "gpu_launches": int(per_call * steps), "clocks": clk,
    }


def cpu_baseline_prefill(n=4, reps=2):
    import synth
    from oracle import layer as OL
    cfg = synth.get_config("prefill_64k")
    x = synth.make_x(cfg.tokens, cfg.hidden, cfg.seed).float().numpy()
    Wr = synth.make_router(cfg.experts, cfg.hidden, cfg.seed).numpy()

    def src(m):
        rows, cols = (cfg.inter, cfg.hidden) if m != "down" else (cfg.hidden, cfg.inter)
        return lambda e: synth.make_expert_weight(0, m, e, rows, cols, cfg.seed).numpy()
    ex = {m: OL.LazyExperts(src(m), cfg.experts, cfg.inter if m != "down" else cfg.hidden)
          for m in ("gate", "up", "down")}
    rows = list(range(n))
    run = lambda: OL.moe_layer(x, Wr, None, ex["gate"], ex["up"], ex["down"], cfg.top_k,
                               cfg.h_tensor_scale, tokens=rows)
    run()
    t0 = time.perf_counter()
    for _ in range(reps):
        run()
    dt = (time.perf_counter() - t0) / reps
    return {"value": n / dt, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"{n} of the 65,536 prefill tokens, x{reps} (experts pre-quantised; numpy "
                      f"fp64, BLAS threads for the contractions)"}


# ------------------------------------------------------------- reference

def run_reference(args):
    """The CPU oracle as the reference arm: each step one bounded sample."""
    import synth
    if args.workload == "decode":
        cfg = synth.get_config("decode_b1_stack48")
        run = oracle_decode_sample(cfg, layers=1)
        unit, per_step, metric = "layer-tokens/s", 1, "MoE-layer tokens/s (decode b=1)"
        sample = "1 decode token through 1 full-size layer per step (experts pre-quantised)"
        workload = (f"decode b=1 through 48 stacked MoE layers (hidden {cfg.hidden}, "
                    f"{cfg.experts} experts, top-{cfg.top_k}, intermediate {cfg.inter})")
    else:
        from oracle import layer as OL
        cfg = synth.get_config("prefill_64k")
        n = 4
        x = synth.make_x(cfg.tokens, cfg.hidden, cfg.seed).float().numpy()
        Wr = synth.make_router(cfg.experts, cfg.hidden, cfg.seed).numpy()

        def src(m):
            rows, cols = (cfg.inter, cfg.hidden) if m != "down" else (cfg.hidden, cfg.inter)
            return lambda e: synth.make_expert_weight(0, m, e, rows, cols, cfg.seed).numpy()
        ex = {m: OL.LazyExperts(src(m), cfg.experts, cfg.inter if m != "down" else cfg.hidden)
              for m in ("gate", "up", "down")}
        rows = list(range(n))
        run = lambda: OL.moe_layer(x, Wr, None, ex["gate"], ex["up"], ex["down"], cfg.top_k,
                                   cfg.h_tensor_scale, tokens=rows)
        run()
        unit, per_step, metric = "tokens/s", n, "MoE-layer tokens/s (prefill 64k)"
        sample = f"{n} of the 65,536 prefill tokens per step (experts pre-quantised)"
        workload = "one MoE layer at 65,536-token prefill"
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t0) / args.steps
    value = per_step / dt
    return {"impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload},
            "cpu_baseline": {"value": value, "unit": unit, "kind": "oracle",
                             "cores": blas_threads(), "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    from nvfp4_routed_expert_gb300 import build as B
    B.build()
    out = run_decode(args, rank, world, local) if args.workload == "decode" else \
        run_prefill(args, rank, world, local)
    if args.workload == "decode" and world == 1 and not args.no_prefill:
        # the headline metric names both decode b=1 and prefill 64k: a short
        # prefill measurement rides along with the decode line
        pf = run_prefill(args, rank, world, local, steps=5, warmup=2)
        out["prefill_64k"] = {k: pf[k] for k in ("metric", "value", "unit", "ms_per_step",
                                                 "expert_tflops", "roofline", "e2e",
                                                 "gpu_launches", "clocks")}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import synth
        out["cpu_baseline"] = cpu_baseline_decode(synth.get_config("decode_b1_stack48")) \
            if args.workload == "decode" else cpu_baseline_prefill()
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
