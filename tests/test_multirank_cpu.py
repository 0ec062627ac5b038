"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2): the timing
reductions over ranks, the per-rank independent batches, and the reference arm's
rank-0-only rule. No GPU is involved."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    from mixture_experts_layer_102_b300 import configs, inputs
    bench.init_dist(world, "gloo")
    mx = bench.reduce_max(1.5 + rank, world)
    sm = bench.reduce_sum(100 * (rank + 1), world)
    cfg = configs.TINY_F32
    inp = inputs.make_inputs(cfg, rank=rank)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "1"])
    q.put((rank, mx, sm, inp.x.sum(), inp.w1.sum(), buf.getvalue()))
    if dist.is_initialized():   # bench.main tears the group down itself
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted([q.get(timeout=300) for _ in procs])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (_, mx0, sm0, x0, w0, out0), (_, mx1, sm1, x1, w1, out1) = res
    assert mx0 == mx1 == 2.5
    assert sm0 == sm1 == 300.0
    assert x0 != x1          # independent batches per rank
    assert w0 == w1          # the same experts on every rank
    line = json.loads(out0.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert out1.strip() == ""  # only rank 0 prints


def test_algorithmic_units_match_hand_counts():
    sys.path.insert(0, ROOT)
    import bench
    from mixture_experts_layer_102_b300 import configs
    c = configs.BF16_T4096
    u = bench.algorithmic_units(c, kept_slots=8192, touched_experts=16)
    assert u["gemm1_swiglu"][0] == 4.0 * 1024 * 2816 * 8192
    assert u["gemm2"][0] == 2.0 * 1024 * 2816 * 8192
    # 6*H*F per kept slot in total: 141.7 GFLOP for 8192 kept slots
    assert abs(u["gemm1_swiglu"][0] + u["gemm2"][0] - 141.7e9) < 0.1e9
    # GEMM1 reads W1 and W3 of all 16 experts (184.5 MB) plus xp, and writes h
    assert u["gemm1_swiglu"][1] == 16 * 2 * 2816 * 1024 * 2 + 8192 * 1024 * 2 + 8192 * 2816 * 2
    assert u["combine"] == (0.0, 8192 * 1024 * 2 + 4096 * 1024 * 2)
    peaks = {"bf16_tflops": 1797.5, "hbm_gbs": 6484.3}
    assert bench.bound_of(*u["gemm1_swiglu"], peaks) == "tensor"
    assert bench.bound_of(*u["combine"], peaks) == "hbm"
    d = configs.DECODE_T64  # 128 slots over 75 experts: weight streaming, ~1 FLOP/B
    ud = bench.algorithmic_units(d, kept_slots=128, touched_experts=75)
    assert bench.bound_of(*ud["gemm1_swiglu"], peaks) == "hbm"


def test_stage_names_and_launch_counts():
    sys.path.insert(0, ROOT)
    import bench
    from mixture_experts_layer_102_b300 import build, configs
    build.build(quiet=True)  # the stages come from the library's plan (host only)
    bf = configs.BF16_T4096
    f32 = configs.TINY_F32
    assert bench.stage_names(bf) == ["route", "dispatch", "gemm1_swiglu", "gemm2", "combine"]
    assert bench.stage_names(f32) == bench.STAGES
    assert bench.stage_names(configs.DECODE_T64) == bench.STAGES     # 1 tile: split router
    assert bench.launches_per_forward(bf) == 5 and bench.launches_per_forward(f32) == 6
    u = bench.algorithmic_units(bf, kept_slots=8192, touched_experts=16)
    assert u["route"][0] == u["router_logits"][0]
    assert u["route"][1] == u["router_logits"][1] + u["route_select"][1]


def test_reference_arm_line_has_every_contract_key():
    # one process (no torchrun environment): rank 0 of 1 prints one JSON line
    sys.path.insert(0, ROOT)
    import bench
    for var in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(var, None)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "1"])
    lines = [l for l in buf.getvalue().strip().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["value"] > 0
    assert (d["steps"], d["warmup"]) == (2, 1) and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny_f32_t64_h128_n8_k2_f256"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["unit"] == d["unit"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_clock_samples_summary():
    sys.path.insert(0, ROOT)
    import bench
    lines = [
        "0, 2032, 2032, 812.50, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n",
        "0, 1980, 2032, 1099.10, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n",
        "0, 2010, 2032, 1002.00, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n",
        "0, [N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A]\n",
        "\n",
    ]
    d = bench.ClockSampler.summarise(lines)
    assert d == {"sm_mhz": 2010.0, "sm_max_mhz": 2032.0, "reasons": ["sw_power_cap"],
                 "samples": 4}
    hot = bench.ClockSampler.summarise(
        ["0, 1500, 2032, 1100, 0x48, Active, Active, Not Active, Active\n"])
    assert hot["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap"]
    assert bench.ClockSampler.summarise([]) is None


def test_traffic_record_follows_the_captured_sources(tmp_path, monkeypatch):
    # a record counts only for its workload and while its sources hash as captured
    import hashlib
    sys.path.insert(0, ROOT)
    import bench
    (tmp_path / "profiles").mkdir()
    src = tmp_path / "kernel.cu"
    src.write_text("__global__ void k() {}\n")
    rec = {"gemm1_swiglu": {"config": "wl", "bytes_per_launch": 123.0,
                            "sources": ["kernel.cu"],
                            "sha256": hashlib.sha256(src.read_bytes()).hexdigest()}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("gemm1_swiglu", "wl") == 123.0
    assert bench.traffic_record("gemm1_swiglu", "other") is None
    assert bench.traffic_record("gemm2", "wl") is None
    src.write_text("__global__ void k() { /* changed */ }\n")
    assert bench.traffic_record("gemm1_swiglu", "wl") is None
    src.unlink()
    assert bench.traffic_record("gemm1_swiglu", "wl") is None


def test_tensor_peak_follows_the_power_regime_of_the_timed_region():
    # a tensor-bound kernel timed inside a power-capped loop is measured against the
    # sustained bf16 figure, one that ran at full clock against the burst figure
    sys.path.insert(0, ROOT)
    import bench
    peaks = {"hbm_gbs": 6486.1, "bf16_tflops": 1768.2, "bf16_tflops_sustained": 1385.5}
    assert bench.tensor_peak(peaks, {"reasons": ["sw_power_cap"]})[0] == 1385.5
    assert bench.tensor_peak(peaks, {"reasons": []})[0] == 1768.2
    assert bench.tensor_peak(peaks, None)[0] == 1768.2
    assert bench.tensor_peak({"hbm_gbs": 1.0, "bf16_tflops": 2.0},
                             {"reasons": ["sw_power_cap"]})[0] == 2.0


def test_routing_stats_from_the_layer_outputs():
    # utilisation figures the bench prints, computed from routing outputs alone
    import types

    import torch
    sys.path.insert(0, ROOT)
    import bench
    from mixture_experts_layer_102_b300 import configs
    cfg = configs.TINY_F32.with_(N=4, k=2)
    r = types.SimpleNamespace(expert_counts=torch.tensor([60, 30, 20, 18], dtype=torch.int32),
                              kept_counts=torch.tensor([40, 30, 20, 18], dtype=torch.int32),
                              aux_loss=torch.tensor([1.25]))
    d = bench.routing_stats(cfg, r)
    assert d["dropped_slots"] == 20 and d["routed_rows_max"] == 60 and d["routed_rows_min"] == 18
    assert d["kept_rows_max"] == 40 and d["active_fraction"] == 0.5 and d["aux_loss"] == 1.25
    c = torch.tensor([60., 30., 20., 18.])
    assert abs(d["load_cv"] - float(c.std(unbiased=False) / c.mean())) < 1e-4
