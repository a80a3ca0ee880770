#!/usr/bin/env python
"""Benchmark of the NVFP4 routed-expert MoE layer on GB300.

Workloads (seeded synthetic inputs; random-init weights; no datasets):
  decode     (default) batch-1 decode through 48 stacked MoE layers of hidden
             2048, 512 experts, top-10, expert intermediate 512 (about 43.5 GB
             of NVFP4 experts resident in HBM), bf16 residual between layers.
             One step = 128 consecutive decode tokens, each through all 48
             layers in one launch of the fused decode kernel
             (moe_stack_forward), replayed from a CUDA graph together with the
             token's input copy.
  decode_b8  the same stack at 8 tokens per launch (16 launches per step)
  prefill    one layer of the same shape at 65,536 tokens; one step = one call
  prefill_4k one layer at 4,096 tokens with a per-expert Zipf(1.1) router bias

Metric: MoE-layer tokens/s = (tokens x layers) processed per second.

The printed JSON line also carries
  roofline      the dominant kernel against its roof: for decode the fused
                kernel (all of S1-S6 for 48 layers in one launch), its
                algorithmic bytes per launch / its CUDA-event duration measured
                inside the timed region (the last launch of the timed region);
                for prefill the gate/up grouped GEMM against the dense NVFP4
                tensor peak (and, as hbm_roofline, against HBM)
  e2e           the same metric through the C ABI with host buffers: each
                input copied from pinned host memory and the output read back,
                inside the timed region
  cpu_baseline  the CPU oracle timed on this host on a bounded sample, with
                all threads and with one
  clocks        SM clocks sampled during the timed region (at least ten samples)
  decode_b8, decode_b1_tail_skip_r5, prefill_4k_zipf, prefill_64k
                (decode workload) the other configurations, each with its own
                roofline, e2e and clocks (--no-extras skips them)

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
    ap.add_argument("--workload", choices=("decode", "decode_b8", "prefill", "prefill_4k"),
                    default="decode")
    ap.add_argument("--layers", type=int, default=48)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="decode workload only: skip the other configurations in the line")
    # internal: time the oracle in a child process (see cpu_baseline)
    ap.add_argument("--oracle-sample", choices=("decode", "prefill"), default=None,
                    help=argparse.SUPPRESS)
    ap.add_argument("--sample-layers", type=int, default=4, help=argparse.SUPPRESS)
    ap.add_argument("--min-seconds", type=float, default=8.0, help=argparse.SUPPRESS)
    ap.add_argument("--min-region", type=float, default=2.4,
                    help="shortest timed region in seconds (more steps are run to reach it; "
                         "0 times exactly --steps steps, e.g. under a profiler)")
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
# kernel, valid only for the kernel sources it was taken on (SHA-256 over the
# files in order): a changed source reports null.
_CSRC = "nvfp4_routed_expert_gb300/csrc/"
NCU_TRAFFIC = {
    "decode": ([_CSRC + "decode.cu", _CSRC + "decode.h", _CSRC + "common.cuh", _CSRC + "sync.cuh"],
               "5f109217ce53bdc056edb6b4afe685a7bf494bdae45565ea211720f8e8101858",
               (87_744_768 + 1_379_584) / 4),   # per layer (4-layer launch, caches flushed)
    "prefill_gateup": ([_CSRC + "prefill.cu", _CSRC + "prefill.h", _CSRC + "common.cuh", _CSRC + "sync.cuh"],
                       "64306a624d7ffd513978d02ab189ecb99c81b72e45ff89d26c5314bdb2e66483",
                       1_058_817_280 + 197_969_664),   # per launch at 65,536 tokens
}


def ncu_traffic(kind, units=1):
    import hashlib
    paths, sha, per_unit = NCU_TRAFFIC[kind]
    m = hashlib.sha256()
    try:
        for path in paths:
            with open(os.path.join(ROOT, path), "rb") as f:
                m.update(f.read())
    except OSError:
        return None
    if m.hexdigest() != sha:
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


# ------------------------------------------------------ multi-rank timing

def max_over_ranks(value_ms, world, device=None):
    """The slowest rank's time: every rank's measurement, MAX-reduced over the
    process group (world 1: the value itself)."""
    if world <= 1:
        return float(value_ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, max_ms):
    """Units per second of the whole job: every rank processes units_per_rank
    in the slowest rank's time."""
    return world * units_per_rank / (max_ms / 1e3)


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
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count() or 1


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample_child(args):
    """--oracle-sample: time the oracle in this (child) process and print one
    JSON line; the parent chooses the thread count through the environment."""
    import synth
    if args.oracle_sample == "decode":
        cfg = synth.get_config("decode_b1_stack48")
        run = oracle_decode_sample(cfg, args.sample_layers)
        per_rep, unit = args.sample_layers, "layer-tokens/s"
    else:
        from oracle import layer as OL
        cfg = synth.get_config("prefill_64k")
        x = synth.make_x(cfg.tokens, cfg.hidden, cfg.seed).float().numpy()
        Wr = synth.make_router(cfg.experts, cfg.hidden, cfg.seed).numpy()

        def src(m):
            rows, cols = (cfg.inter, cfg.hidden) if m != "down" else (cfg.hidden, cfg.inter)
            return lambda e: synth.make_expert_weight(0, m, e, rows, cols, cfg.seed).numpy()
        ex = {m: OL.LazyExperts(src(m), cfg.experts, cfg.inter if m != "down" else cfg.hidden)
              for m in ("gate", "up", "down")}
        rows = list(range(args.sample_layers))
        run = lambda: OL.moe_layer(x, Wr, None, ex["gate"], ex["up"], ex["down"], cfg.top_k,
                                   cfg.h_tensor_scale, tokens=rows)
        run()
        per_rep, unit = len(rows), "tokens/s"
    reps, t0 = 0, time.perf_counter()
    while True:
        run()
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= args.min_seconds or reps >= 1000:
            break
    print(json.dumps({"value": per_rep * reps / dt, "unit": unit, "reps": reps, "seconds": dt,
                      "blas_threads": blas_threads()}), flush=True)


def time_oracle(kind, units, min_seconds, single_thread):
    """Run the oracle sample in a fresh process (all threads, or pinned to one
    BLAS / OpenMP thread) and return its JSON result, or None."""
    env = dict(os.environ)
    env.pop("CUDA_VISIBLE_DEVICES", None)
    if single_thread:
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            env[var] = "1"
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--oracle-sample", kind,
           "--sample-layers", str(units), "--min-seconds", str(min_seconds)]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError, OSError):
        return None


def cpu_baseline(kind="decode"):
    """The oracle as it stands on this host: all threads, then one thread."""
    units = 4 if kind == "decode" else 4
    multi = time_oracle(kind, units, 8.0, single_thread=False)
    single = time_oracle(kind, units, 8.0, single_thread=True)
    if multi is None:
        return None
    what = (f"1 decode token through {units} full-size stacked layers per repetition"
            if kind == "decode" else f"{units} of the 65,536 prefill tokens per repetition")
    out = {"value": multi["value"], "unit": multi["unit"], "cores": multi["blas_threads"],
           "host_cores": host_cores(), "kind": "oracle",
           "sample": f"{what}, {multi['reps']} repetitions in {multi['seconds']:.1f} s (experts "
                     f"pre-quantised; numpy fp64 contractions on {multi['blas_threads']} BLAS threads)"}
    if single is not None:
        out["single_thread"] = {"value": single["value"], "unit": single["unit"], "cores": 1,
                                "reps": single["reps"], "seconds": single["seconds"]}
    return out


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


def sibling(nv, layer, max_tokens, bias=False, route_keep=0, cfg=None, dev=None):
    """Another handle on a layer's weights (no copy) with another desc."""
    import synth
    router, b, g, u, d = layer._keep
    if bias:
        b = synth.make_router_bias(cfg.experts, cfg.seed, 0, device=dev)
    de = layer.desc
    desc = nv.make_desc(de.hidden, de.num_experts, de.top_k, de.inter, max_tokens, de.h_tensor_scale,
                        route_keep=route_keep)
    return nv.Layer(desc, router, b, g, u, d)


def timed_region(torch, stream, step, steps, warmup, min_seconds, clock_index):
    """Warm up, then time `steps` steps (more if needed so that the region lasts
    min_seconds, which gives the clock sampler at least ten samples) with CUDA
    events on `stream`; returns (ms per step, steps, clocks)."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
    stream.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    one = max(time.perf_counter() - t0, 1e-6)
    steps = max(steps, int(min_seconds / one) + 1)
    clocks = ClockSampler(clock_index)
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    return e0.elapsed_time(e1) / steps, steps, clk


def distinct_experts_per_layer(nv, torch, stack, x, ws):
    """Routed experts of each layer for input x [T][H] through the stack (the
    chain of single-layer calls gives the stack's own routing, bit for bit)."""
    cur, out = x, []
    T = x.shape[0]
    for layer in stack:
        d = layer.desc
        idx = torch.empty(T, d.top_k, dtype=torch.int32, device=x.device)
        y = torch.empty(T, d.hidden, device=x.device)
        nxt = torch.empty_like(cur)
        nv.moe_forward(layer, cur, y, ws, residual=cur, x_next=nxt, debug={"idx": idx})
        e = idx.cpu().numpy()
        out.append(int(np.unique(e[e >= 0]).size))
        cur = nxt
    return out


def measure_decode(nv, torch, stack, cfg, T, dev, args, world, local, label):
    """T tokens per launch through the whole stack (one fused-kernel launch per
    batch); one step = 128 / T launches from a CUDA graph, fresh tokens each."""
    import synth
    L = len(stack)
    ws = stack[0].workspace(dev)
    n_batch = DECODE_TOKENS_PER_STEP // T
    x_in = torch.empty(T, cfg.hidden, dtype=torch.bfloat16, device=dev)
    x_out = torch.empty(T, cfg.hidden, dtype=torch.bfloat16, device=dev)
    pool = torch.stack([synth.make_x(T, cfg.hidden, cfg.seed, step=1000 * T + i, device=dev)
                        for i in range(n_batch)])
    ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    stream = torch.cuda.Stream(device=dev)
    for e in ev:
        e.record(stream)
    torch.cuda.synchronize()
    # the fused stack kernel is the only kernel of a step: trace events bracket it
    nv.moe_layer_set_trace(stack[0], nv.MOE_STEP_GATEUP, ev[0], ev[1])
    with torch.cuda.stream(stream):
        x_in.copy_(pool[0])
        nv.moe_stack_forward(stack, x_in, x_out, ws, stream=stream)
    stream.synchronize()
    st = nv.moe_layer_status(stack[0], stream)
    assert st == 0, nv.status_string(st)
    n0 = nv.moe_kernel_launches()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        nv.moe_stack_forward(stack, x_in, x_out, ws, stream=stream)
    launches_per_batch = nv.moe_kernel_launches() - n0

    def step():
        for i in range(n_batch):
            x_in.copy_(pool[i], non_blocking=True)
            graph.replay()

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ms, steps, clk = timed_region(torch, stream, step, args.steps, args.warmup, args.min_region, local)
    if world > 1:
        torch.distributed.barrier()
    kernel_ms = ev[0].elapsed_time(ev[1])          # the last launch of the timed region
    nv.moe_layer_set_trace(stack[0], nv.MOE_STEP_NONE, None, None)
    st = nv.moe_layer_status(stack[0], stream)
    assert st == 0, nv.status_string(st)
    ms = max_over_ranks(ms, world, dev)
    layer_tokens = n_batch * T * L
    value = whole_job_rate(layer_tokens, world, ms)

    e2e = None
    if not args.no_e2e:
        host_in = pool.cpu().pin_memory()
        host_out = torch.empty(T, cfg.hidden, dtype=torch.bfloat16).pin_memory()
        with torch.cuda.stream(stream):
            for i in range(min(8, n_batch)):
                x_in.copy_(host_in[i], non_blocking=True)
                graph.replay()
                host_out.copy_(x_out, non_blocking=True)
            stream.synchronize()
            e_steps = max(1, min(steps, 20))
            t0 = time.perf_counter()
            for _ in range(e_steps):
                for i in range(n_batch):
                    x_in.copy_(host_in[i], non_blocking=True)
                    graph.replay()
                    host_out.copy_(x_out, non_blocking=True)
                    stream.synchronize()
            dt = (time.perf_counter() - t0) / e_steps
        dt = max_over_ranks(dt * 1e3, world, dev) / 1e3
        e2e = {"value": world * layer_tokens / dt, "unit": "layer-tokens/s",
               "h2d_bytes_per_step": n_batch * T * cfg.hidden * 2,
               "d2h_bytes_per_step": n_batch * T * cfg.hidden * 2}

    # algorithmic bytes of the last launch: the router and each layer's routed
    # experts (counted from that launch's own routing) plus x in and out
    keep = stack[0].desc.route_keep
    if T == 1 and keep == 0:
        experts = [cfg.top_k] * L
    elif T == 1:
        experts = [keep] * L
    else:
        experts = distinct_experts_per_layer(nv, torch, stack, pool[n_batch - 1], ws)
    launch_bytes = sum(layer_bytes(cfg, n, T) for n in experts)
    peak, peak_kind = measured_peaks()
    achieved = launch_bytes / (kernel_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": f"k_decode<{T}> (fused S1-S6, {L} layers per launch)",
                "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": peak_kind,
                "traffic": ncu_traffic("decode", L) if T == 1 and keep == 0 else None,
                "bytes_per_launch": launch_bytes, "launch_ms": kernel_ms,
                "per_layer_us": kernel_ms * 1e3 / L,
                "routed_experts_per_layer": float(np.mean(experts)),
                "step_GBs": launch_bytes * n_batch / (ms / 1e3) / 1e9}
    return {
        "metric": f"MoE-layer tokens/s ({label})", "value": value, "unit": "layer-tokens/s",
        "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4",
        "data": "synthetic: seeded N(0,1) bf16 activations, N(0,0.02) weights quantised to NVFP4",
        "config": {"workload": f"decode b={T} through {L} stacked MoE layers (hidden {cfg.hidden}, "
                               f"{cfg.experts} experts, top-{cfg.top_k}, intermediate {cfg.inter})"
                               + (f", route-tail skip keeping the top {keep} picks" if keep else ""),
                   "tokens_per_step": n_batch * T, "layers": L,
                   "stack_tokens_per_s": whole_job_rate(n_batch * T, world, ms),
                   "l2": f"inputs larger than L2: {L} layers x "
                         f"{layer_bytes(cfg, experts[0], T) / 1e6:.1f} MB touched per launch",
                   "parallelism": f"replicas x{world}"},
        "roofline": roofline, "e2e": e2e,
        "gpu_launches": int(launches_per_batch * n_batch * steps), "clocks": clk,
    }


def run_decode(args, rank, world, local):
    import torch
    import nvfp4_routed_expert_gb300 as nv
    import synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = synth.get_config("decode_b1_stack48").with_(layers=args.layers)
    stack = build_stack(nv, torch, cfg, cfg.layers, 8, dev)
    out = measure_decode(nv, torch, stack, cfg, 1, dev, args, world, local, "decode b=1")
    if world == 1 and not args.no_extras:
        # the other configurations of the layer, each with its own roofline, e2e and clocks
        out["decode_b8"] = measure_decode(nv, torch, stack, cfg, 8, dev, args, world, local,
                                          "decode b=8")
        skip = [sibling(nv, layer, 8, route_keep=5) for layer in stack]
        out["decode_b1_tail_skip_r5"] = measure_decode(nv, torch, skip, cfg, 1, dev, args, world,
                                                       local, "decode b=1, route-tail skip r=5")
        del skip
        pf4 = sibling(nv, stack[0], 4096, bias=True, cfg=cfg, dev=dev)
        out["prefill_4k_zipf"] = measure_prefill(nv, torch, pf4, synth.get_config("prefill_4k_zipf"),
                                                 dev, args, world, local)
        del pf4
        pf64 = sibling(nv, stack[0], 65536)
        out["prefill_64k"] = measure_prefill(nv, torch, pf64, synth.get_config("prefill_64k"),
                                             dev, args, world, local)
    return out


def measure_prefill(nv, torch, layer, cfg, dev, args, world, local):
    """One layer at cfg.tokens tokens through moe_forward (tensor-core path)."""
    import synth
    ws = layer.workspace(dev)
    x = synth.make_x(cfg.tokens, cfg.hidden, cfg.seed, device=dev)
    y = torch.empty(cfg.tokens, cfg.hidden, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    n0 = nv.moe_kernel_launches()
    with torch.cuda.stream(stream):
        nv.moe_forward(layer, x, y, ws, stream=stream)
    per_call = nv.moe_kernel_launches() - n0
    stream.synchronize()
    # routing of this input: the touched experts (for the HBM roofline)
    counts = torch.empty(cfg.experts, dtype=torch.int32, device=dev)
    nv.moe_forward(layer, x, y, ws, debug={"counts": counts}, stream=stream)
    stream.synchronize()
    active = int((counts > 0).sum().item())
    # The timed calls are replays of a CUDA graph of R calls, the way a serving
    # loop runs the layer.  The gate/up grouped GEMM (S5) is the dominant
    # kernel: trace events bracket it in each captured call, and their times in
    # the last replay of the timed region are averaged.
    R = 4
    gev = []
    for _ in range(R):
        pair = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        for e in pair:            # torch creates the CUDA event at its first record
            e.record(stream)
        gev.append(pair)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for a, b in gev:
            nv.moe_layer_set_trace(layer, nv.MOE_STEP_GATEUP, a, b)
            nv.moe_forward(layer, x, y, ws, stream=stream)
    nv.moe_layer_set_trace(layer, nv.MOE_STEP_NONE, None, None)
    ms, replays, clk = timed_region(torch, stream, graph.replay, max(1, args.steps // R),
                                    args.warmup, args.min_region, local)
    gate_ms = float(np.mean([a.elapsed_time(b) for a, b in gev]))
    ms = max_over_ranks(ms / R, world, dev)     # per call
    steps = replays * R
    pairs = cfg.tokens * cfg.top_k
    flops_gateup = 4 * cfg.hidden * cfg.inter * pairs
    flops = 6 * cfg.hidden * cfg.inter * pairs
    peak, peak_src = fp4_tensor_peak()
    achieved = flops_gateup / (gate_ms / 1e3) / 1e12
    roofline = {"bound": "tensor", "kernel": "k_grouped_gemm<kGateUp> (S5: gate/up FP4 grouped GEMM "
                "+ SwiGLU + requantisation)", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": peak_src,
                "traffic": ncu_traffic("prefill_gateup") if cfg.tokens == 65536 else None,
                "traffic_unit": "bytes", "flops_per_launch": flops_gateup, "launch_ms": gate_ms}
    # the same kernel against HBM: its algorithmic bytes (every touched expert's
    # gate and up matrices once, the activations' NVFP4 codes, h written)
    hbm, hbm_src = measured_peaks()
    gb = gateup_bytes(cfg, active, pairs, cfg.tokens)
    hbm_roofline = {"bound": "hbm", "achieved": gb / (gate_ms / 1e3) / 1e9, "peak": hbm,
                    "unit": "GB/s", "frac": gb / (gate_ms / 1e3) / 1e9 / hbm, "peak_source": hbm_src,
                    "bytes_per_launch": gb, "touched_experts": active}
    e2e = None
    if not args.no_e2e:
        # Every step copies its x in from pinned host memory, runs moe_forward
        # and copies its y out to pinned host memory, the way a serving loop
        # streams prompts: the copy-in of step i + 1 and the copy-out of step
        # i - 1 run on their own streams while step i computes (two device
        # buffers each for x and y; events order every reuse).  The region
        # runs from before the first copy-in to after the last copy-out.
        x_h = x.cpu().pin_memory()
        y_h = torch.empty(y.shape, dtype=y.dtype).pin_memory()
        xb, yb = [x, torch.empty_like(x)], [y, torch.empty_like(y)]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        e_steps = max(3, min(steps, 20))
        ev_in = [torch.cuda.Event() for _ in range(e_steps)]
        ev_comp = [torch.cuda.Event() for _ in range(e_steps)]
        ev_out = [torch.cuda.Event() for _ in range(e_steps)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(s_in)
        for i in range(e_steps):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[i - 2])     # step i - 2 has read xb[b]
                xb[b].copy_(x_h, non_blocking=True)
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])        # yb[b] has been copied out
            nv.moe_forward(layer, xb[b], yb[b], ws, stream=stream)
            ev_comp[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[i])
                y_h.copy_(yb[b], non_blocking=True)
                ev_out[i].record(s_out)
        s_out.wait_event(ev_in[e_steps - 1])
        e1.record(s_out)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps, world, dev)
        e2e = {"value": whole_job_rate(cfg.tokens, world, e_ms), "unit": "tokens/s",
               "h2d_bytes_per_step": x.numel() * 2, "d2h_bytes_per_step": y.numel() * 4,
               "copies": "each step's copy-in and copy-out on two copy streams, overlapping "
                         "the neighbouring steps' compute"}
    name = "prefill 64k" if cfg.tokens == 65536 else f"prefill {cfg.tokens}" + (", Zipf-skewed routing"
                                                                               if cfg.zipf_bias else "")
    return {
        "metric": f"MoE-layer tokens/s ({name})", "value": whole_job_rate(cfg.tokens, world, ms),
        "unit": "tokens/s", "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "nvfp4", "data": "synthetic: seeded N(0,1) bf16 activations, N(0,0.02) weights "
                                  "quantised to NVFP4",
        "config": {"workload": f"one MoE layer at {cfg.tokens}-token prefill (hidden {cfg.hidden}, "
                               f"{cfg.experts} experts, top-{cfg.top_k}, intermediate {cfg.inter})"
                               + (", per-expert Zipf(1.1) router bias" if cfg.zipf_bias else ""),
                   "tokens": cfg.tokens, "touched_experts": active,
                   "l2": f"inputs larger than L2: the touched experts' weights alone are "
                         f"{active * 3 * nvfp4_bytes(cfg.inter, cfg.hidden) / 1e6:.0f} MB",
                   "parallelism": f"replicas x{world}"},
        "expert_tflops": flops / (ms / 1e3) / 1e12,
        "roofline": roofline, "hbm_roofline": hbm_roofline, "e2e": e2e,
        "gpu_launches": int(per_call * steps), "clocks": clk,
    }


def run_prefill(args, rank, world, local):
    import torch
    import nvfp4_routed_expert_gb300 as nv
    import synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = synth.get_config("prefill_4k_zipf" if args.workload == "prefill_4k" else "prefill_64k")
    layer = build_stack(nv, torch, cfg, 1, cfg.tokens, dev)[0]
    return measure_prefill(nv, torch, layer, cfg, dev, args, world, local)


def run_decode_b8(args, rank, world, local):
    import torch
    import nvfp4_routed_expert_gb300 as nv
    import synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = synth.get_config("decode_b1_stack48").with_(layers=args.layers)
    stack = build_stack(nv, torch, cfg, cfg.layers, 8, dev)
    return measure_decode(nv, torch, stack, cfg, 8, dev, args, world, local, "decode b=8")


# ------------------------------------------------------------- reference

def run_reference(args):
    """The CPU oracle as the reference arm: each step one bounded sample."""
    import synth
    if args.workload in ("decode", "decode_b8"):
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
                             "cores": blas_threads(), "host_cores": host_cores(), "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    if args.oracle_sample:
        oracle_sample_child(args)
        return
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
    if args.workload == "decode":
        out = run_decode(args, rank, world, local)
    elif args.workload == "decode_b8":
        out = run_decode_b8(args, rank, world, local)
    else:
        out = run_prefill(args, rank, world, local)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline("decode" if args.workload.startswith("decode") else "prefill")
        if cb is not None:
            out["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
