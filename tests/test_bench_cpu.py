"""The measurement arithmetic of bench.py, without a GPU: the algorithmic
bytes and FLOPs behind roofline.achieved, pinned to figures derived by hand
from the NVFP4 format (per N x K matrix: N K / 2 code bytes, N K / 16 scale
bytes, one fp32 tensor scale) rather than re-derived from bench.py's own
helpers; the source-hash gate of the ncu traffic table; the peaks and the
timing defaults."""
import hashlib
import os

import pytest

import bench
import synth


def test_decode_b1_layer_bytes():
    cfg = synth.get_config("decode_b1")
    # one 512 x 2048 NVFP4 matrix: 524,288 code bytes + 65,536 scale bytes + 4
    assert bench.nvfp4_bytes(512, 2048) == 589_824
    # router 512 x 2048 fp32 (4 MiB) + 10 experts x (3 matrices of 589,828 B)
    # + x bf16 (4 KiB) + y fp32 (8 KiB) + x_next bf16 (4 KiB)
    assert bench.layer_bytes(cfg, 10, 1) == 4_194_304 + 10 * 1_769_484 + 16_384 == 21_905_528
    # the stacked workload touches 48 such layers per decode token (~1.05 GB)
    assert 48 * bench.layer_bytes(cfg, 10, 1) == 1_051_465_344


def test_gateup_bytes_counts_each_routed_expert_once():
    cfg = synth.get_config("decode_b1")
    one = bench.gateup_bytes(cfg, 1, 1, 1)
    # gate + up (2 x 589,824 + 2 tensor scales) + x codes/scales 1,152 + h codes/scales 288
    assert one == 2 * 589_824 + 8 + 1_152 + 288
    # a second pair of the same expert adds only its h row
    assert bench.gateup_bytes(cfg, 1, 2, 2) - one == 1_152 + 288


def test_prefill_64k_flops():
    cfg = synth.get_config("prefill_64k")
    pairs = cfg.tokens * cfg.top_k
    assert pairs == 655_360
    # gate/up: two 2048 x 512 GEMVs per pair, 2 FLOP per multiply-add
    gateup = 2 * 2 * cfg.hidden * cfg.inter * pairs
    assert gateup == 2_748_779_069_440
    # with down (one more 512 x 2048 product per pair) the layer's expert work is
    # 6 H I per pair = 4.12 TFLOP
    assert gateup * 3 // 2 == 4_123_168_604_160


def test_ncu_traffic_is_gated_by_the_source_hash(tmp_path, monkeypatch):
    src, hdr = tmp_path / "kernel.cu", tmp_path / "shared.cuh"
    src.write_bytes(b"// one kernel\n")
    hdr.write_bytes(b"// a header it includes\n")
    sha = hashlib.sha256(src.read_bytes() + hdr.read_bytes()).hexdigest()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setitem(bench.NCU_TRAFFIC, "probe", (["kernel.cu", "shared.cuh"], sha, 1000.0))
    assert bench.ncu_traffic("probe", 3) == 3000.0
    hdr.write_bytes(b"// a header it includes, changed\n")   # a changed header counts too
    assert bench.ncu_traffic("probe", 3) is None
    hdr.write_bytes(b"// a header it includes\n")
    assert bench.ncu_traffic("probe", 3) == 3000.0
    src.write_bytes(b"// one kernel, changed\n")
    assert bench.ncu_traffic("probe", 3) is None
    os.remove(src)
    assert bench.ncu_traffic("probe", 3) is None


def test_peaks_and_defaults(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    gbs, src = bench.measured_peaks()
    assert src == "fallback" and gbs == bench.FALLBACK_HBM_GBS
    tf, src = bench.fp4_tensor_peak()
    assert src.startswith("fallback") and tf == pytest.approx(6 * bench.FALLBACK_BF16_TFLOPS)
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 6000.5, "bf16_tflops": 2000.0}')
    assert bench.measured_peaks() == (6000.5, "measured")
    tf, src = bench.fp4_tensor_peak()
    assert tf == 12000.0 and src.startswith("measured")
    monkeypatch.setattr("sys.argv", ["bench.py"])
    args = bench.parse_args()
    assert args.gpus == 1 and args.warmup >= 3 and args.steps >= 1 and args.impl == "ours"


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    ms = 10.0 + 5.0 * rank                       # rank 1 is the slower one
    dist.barrier()
    slowest = bench.max_over_ranks(ms, world)
    out[rank] = (slowest, bench.whole_job_rate(128, world, slowest))
    dist.destroy_process_group()


def test_replica_timing_over_two_gloo_ranks():
    """The multi-rank timing of bench.py (barrier, MAX over the ranks, whole-job
    rate = ranks x units / slowest time) with two gloo ranks on the CPU."""
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
    for rank in range(2):
        slowest, rate = out[rank]
        assert slowest == 15.0
        assert rate == pytest.approx(2 * 128 / 0.015)
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.whole_job_rate(128, 1, 64.0) == pytest.approx(2000.0)
