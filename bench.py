#!/usr/bin/env python
"""Benchmark of the sparse MoE SwiGLU layer forward on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl {moe,reference}]

One step = one full layer forward (router, dispatch, gate/up GEMM + SwiGLU,
down GEMM, combine, aux statistics) over one batch of synthetic tokens of the
workload, inputs resident in HBM.  The default workload is the largest one,
the Mixtral-shaped layer (d=4096, F=14336, E=8, top-2) at T=16384 tokens.
L2 is flushed (a 256 MiB write) between timed steps; each step is timed with
CUDA events on the launching stream.  Prints one JSON line; on one GPU the
line also carries the other workloads (top-2 d=1024, the fine-grained E=64
layer, expert choice, and the large layer at T=16/256/4096) under
"workloads".  Under torchrun every rank runs its own replica of the workload
(tokens are independent, no collective on the data path); the time is the max
over ranks and the value counts the tokens of all ranks.

--impl reference times the fp64 CPU oracle on bounded samples of the same
workload on the host cores (rank 0 only).
"""

from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_mixture_experts_67_b300 import synth  # noqa: E402

METRIC = "MoE-layer fwd tokens/s and active TFLOP/s (% of B300 BF16 peak), 1 GPU"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
KERNEL_SOURCES = {"gateup": "sparse_mixture_experts_67_b300/csrc/grouped_tc.cuh"}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="large_d4096")
    ap.add_argument("--tokens", type=int, default=0, help="override T (large_d4096 sweep)")
    ap.add_argument("--impl", default="moe", choices=["moe", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-sweep", action="store_true", help="skip the other workloads")
    return ap.parse_args(argv)


def workload_config(args) -> synth.LayerConfig:
    cfg = synth.CONFIGS[args.workload]
    if args.tokens:
        cfg = cfg.with_tokens(args.tokens)
    return cfg


def describe(cfg: synth.LayerConfig) -> str:
    if cfg.routing == "expert_choice":
        return (f"{cfg.name}: expert-choice T={cfg.T} d={cfg.d} F={cfg.F} E={cfg.E} "
                f"cf={cfg.capacity_factor} C={cfg.C} {cfg.dtype}")
    return f"{cfg.name}: top-{cfg.k} T={cfg.T} d={cfg.d} F={cfg.F} E={cfg.E} {cfg.dtype}"


def workload_keys(cfg: synth.LayerConfig, ws: int) -> dict:
    """The workload part of the JSON line's config (the same in both arms)."""
    return {"workload": describe(cfg), "T_per_gpu": cfg.T, "d_model": cfg.d, "d_ff": cfg.F,
            "experts": cfg.E, "k": cfg.k, "routing": cfg.routing,
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None if the kernel changed
    since or the capture was of another workload."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)[kernel]
        if rec.get("workload") != workload:
            return None
        with open(os.path.join(ROOT, rec["source"]), "rb") as fh:
            sha = hashlib.sha256(fh.read()).hexdigest()
        return rec if sha == rec["source_sha256"] else None
    except (OSError, ValueError, KeyError):
        return None


# ---------------------------------------------------------------- distributed


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return ws, int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def aggregate(local_seconds: float, local_units: float, world_size: int, dist=None, device=None):
    """Whole-job throughput: units of all ranks / max over ranks of the timed seconds."""
    if world_size == 1 or dist is None:
        return local_units / local_seconds, local_seconds, local_units
    import torch

    t = torch.tensor([local_seconds], dtype=torch.float64, device=device)
    u = torch.tensor([local_units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(u.item()) / float(t.item()), float(t.item()), float(u.item())


# ---------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark(self, which: str):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 9]
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for i, n in enumerate(names):
                if r[5 + i].strip().lower() == "active":
                    reasons.add(n)
        loaded = [v for v in sm if mx and v > 0.3 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(rows)}


# ---------------------------------------------------------------- GPU arm


def _upload(torch, dev, a):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def _device_weights(torch, dev, inp):
    return {"w_g": _upload(torch, dev, inp.w_g),
            "bias": None if inp.bias is None else _upload(torch, dev, inp.bias),
            "w_gate": _upload(torch, dev, inp.w_gate), "w_up": _upload(torch, dev, inp.w_up),
            "w_down": _upload(torch, dev, inp.w_down)}


def _capture(torch, layer, x, y, warmup):
    """Warm-up launches, then the layer captured once into a CUDA graph."""
    for _ in range(max(3, warmup)):
        layer(x, y=y)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        layer(x, y=y)
    torch.cuda.current_stream().wait_stream(side)
    with torch.cuda.graph(graph, capture_error_mode="relaxed"):
        layer(x, y=y)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    return graph


def _timed_replays(torch, graph, flush, stream, steps):
    """Device ms of each graph replay, L2 flushed before each."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        graph.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def _weight_bytes(cfg, experts_used: int) -> float:
    """Expert weight bytes a forward reads when `experts_used` experts hold rows."""
    return 3.0 * experts_used * cfg.F * cfg.d * (2 if cfg.dtype == "bf16" else 4)


def dominant_kernel(cfg, stages, peaks, peak_src, experts_used=None):
    """Roofline entry of the stage that takes the most time: the gate/up GEMM against the
    bf16 tensor peak when the expert segments are compute-bound, against HBM on its
    weight bytes when they are not (fewer rows per expert than the ridge point).  The
    fp32 workload (FFMA kernels, microseconds per launch) is launch-latency-bound and
    has no roofline entry."""
    gu_ms = stages["gateup_ms"]
    if cfg.dtype != "bf16":
        return {"kernel": "grouped gate/up (fp32 FFMA)", "bound": "latency", "frac": None,
                "note": "a few microseconds per launch; parity workload, not a throughput target"}
    flops = 4.0 * cfg.R * cfg.d * cfg.F
    used = cfg.E if experts_used is None else experts_used
    rows_per_expert = cfg.R / max(used, 1)
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)  # flop per byte
    b = 2 if cfg.dtype == "bf16" else 4
    if rows_per_expert * 2 / b >= ridge / 2:  # ~rows flop per weight byte
        achieved = flops / (gu_ms / 1e3) / 1e12
        return {"kernel": "grouped gate/up GEMM + SwiGLU", "bound": "tensor",
                "achieved": achieved, "peak": peaks["bf16_tflops"],
                "peak_kind": f"bf16 dense burst ({peak_src})", "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"],
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                "algorithmic_flops_per_launch": flops}
    byts = 2.0 * used * cfg.F * cfg.d * b + cfg.R * cfg.d * b + cfg.R * cfg.F * b
    achieved = byts / (gu_ms / 1e3) / 1e9
    return {"kernel": "grouped gate/up GEMM + SwiGLU (weight-bandwidth-bound)", "bound": "hbm",
            "achieved": achieved, "peak": peaks["hbm_gbs"], "peak_kind": f"HBM copy ({peak_src})",
            "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
            "algorithmic_bytes_per_launch": byts}


def run_gpu(args, cfg):
    import torch

    import sparse_mixture_experts_67_b300 as moe

    ws, rank, local_rank = dist_env()
    dist = None
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    inp = synth.make_inputs(cfg)
    w = _device_weights(torch, dev, inp)
    x = _upload(torch, dev, inp.x)
    ec = cfg.routing == "expert_choice"
    layer = moe.MoELayer(w, k=cfg.k, routing=1 if ec else 0, capacity_factor=cfg.capacity_factor)
    y = torch.empty((cfg.T, cfg.d), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    # the step is replayed from a CUDA graph: one launch per step, no host work
    graph = _capture(torch, layer, x, y, args.warmup)

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    K = args.steps
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    step_ms = _timed_replays(torch, graph, flush, stream, K)
    if dist:
        dist.barrier()
    local_s = sum(step_ms) / 1e3
    # the same step launched eagerly through the API, for comparison
    eager = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(min(K, 20))]
    for i, (a, b) in enumerate(eager):
        flush.fill_(i & 0xFF)
        a.record(stream)
        layer(x, y=y)
        b.record(stream)
    torch.cuda.synchronize()
    eager_ms = sum(a.elapsed_time(b) for a, b in eager) / len(eager)
    del graph

    # per-stage breakdown through the individual entry points (same kernels)
    stages = (stage_breakdown_ec if ec else stage_breakdown)(moe, torch, cfg, x, w, flush, stream,
                                                             min(K, 50))
    # end to end through the public API with host buffers
    e2e = run_e2e(moe, torch, layer, inp.x, cfg, dev, min(K, 50))
    clk = clocks.stop()

    value, max_s, units = aggregate(local_s, float(cfg.T * K), ws, dist, dev)
    if dist:
        dist.destroy_process_group()
    if rank != 0:
        return None
    ms = max_s * 1e3 / K
    flops = cfg.active_flops()
    peaks, peak_src = load_peaks()
    tflops = flops / (ms / 1e3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if cfg.dtype == "bf16" else "f32",
        "data": "synthetic (seeded normal x and weights of the workload's shape; no dataset)",
        "config": dict(workload_keys(cfg, ws),
                       l2="flushed between timed steps (256 MiB write)",
                       launch="CUDA graph replay of moe_layer_forward (one graph launch per step)"),
        "ms_per_step_median": float(np.median(step_ms)),
        "ms_per_step_eager_launch": eager_ms,
        "active_tflops": tflops,
        "frac_of_bf16_peak": {"burst": tflops / peaks["bf16_tflops"],
                              "sustained": tflops / peaks["bf16_tflops_sustained"],
                              "source": peak_src},
        "stages_ms": {k_: v for k_, v in stages.items() if k_ != "experts_used"},
        "gpu_launches": launches_per_step(cfg) * K,
        "clocks": clk,
        "e2e": e2e,
    }
    if stages:
        # the GEMM is timed alone (events around its launch): the burst figure is its
        # denominator; the sustained one is reported beside it
        roof = dominant_kernel(cfg, stages, peaks, peak_src, stages.get("experts_used"))
        traffic = recorded_traffic("gateup", cfg.name)
        roof["traffic"] = None if traffic is None else traffic["bytes_per_launch"]
        line["roofline"] = roof
    if ws == 1 and not args.no_sweep:
        del layer, y, x
        torch.cuda.empty_cache()
        line["workloads"] = sweep(moe, torch, dev, cfg, inp, w, flush, stream, peaks, peak_src,
                                  min(K, 30), args.warmup)
    if not args.no_cpu_baseline and ws == 1:
        del w
        torch.cuda.empty_cache()
        line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_seconds, inp)
    return line


# the other workloads reported beside the headline: (name, T override)
SWEEP = (("tiny_fp32", 0), ("top2_d1024", 0), ("fine_e64", 0), ("ec_e16", 0), ("large_d4096", 16),
         ("large_d4096", 256), ("large_d4096", 4096))


def sweep(moe, torch, dev, main_cfg, main_inp, main_w, flush, stream, peaks, peak_src, steps,
          warmup):
    """ms per step (CUDA-graph replay, L2 flushed), tokens/s, active TFLOP/s and the
    dominant kernel's roofline fraction of each workload in SWEEP; the large layer at
    smaller T reuses the headline's weights and the leading rows of its x."""
    out = []
    for name, T in SWEEP:
        base = synth.CONFIGS[name]
        cfg = base.with_tokens(T) if T else base
        if cfg == main_cfg:
            continue
        same_weights = name == main_cfg.name.split("@")[0] and T <= main_cfg.T
        if same_weights:
            inp, w = None, main_w
            x = _upload(torch, dev, main_inp.x[:cfg.T])
        else:
            inp = synth.make_inputs(cfg)
            w = _device_weights(torch, dev, inp)
            x = _upload(torch, dev, inp.x)
        ec = cfg.routing == "expert_choice"
        layer = moe.MoELayer(w, k=cfg.k, routing=1 if ec else 0,
                             capacity_factor=cfg.capacity_factor)
        y = torch.empty((cfg.T, cfg.d), dtype=torch.float32, device=dev)
        graph = _capture(torch, layer, x, y, warmup)
        ms_list = _timed_replays(torch, graph, flush, stream, steps)
        del graph
        ms = float(np.mean(ms_list))
        stages = (stage_breakdown_ec if ec else stage_breakdown)(moe, torch, cfg, x, w, flush,
                                                                 stream, min(steps, 10))
        used = stages.get("experts_used")
        rec = {"workload": describe(cfg), "ms_per_step": ms,
               "ms_per_step_median": float(np.median(ms_list)), "steps": steps,
               "tokens_per_s": cfg.T / (ms / 1e3),
               "active_tflops": cfg.active_flops() / (ms / 1e3) / 1e12,
               "stages_ms": {k_: v for k_, v in stages.items() if k_ != "experts_used"},
               "dominant_kernel": dominant_kernel(cfg, stages, peaks, peak_src, used)}
        rec["frac_of_bf16_burst"] = (rec["active_tflops"] / peaks["bf16_tflops"]
                                     if cfg.dtype == "bf16" else None)
        if used is not None and rec["dominant_kernel"]["bound"] == "hbm":
            wb = _weight_bytes(cfg, used)
            rec["step_weight_bytes"] = wb
            rec["step_hbm_frac"] = wb / (ms / 1e3) / 1e9 / peaks["hbm_gbs"]
        out.append(rec)
        del layer, y, x
        if not same_weights:
            del w, inp
        torch.cuda.empty_cache()
    return out


def launches_per_step(cfg) -> int:
    if cfg.routing == "expert_choice":
        return 7  # logits, EC select, offsets, gather, gate/up, down, EC combine
    # the scatter reduces the per-tile count matrix itself unless tiles^2 * E exceeds
    # 4 Mi reads; then a one-CTA scan and the aux finalisation run as two more launches
    tile_tokens = 32 if cfg.E <= 16 else 64
    tiles = -(-cfg.T // tile_tokens)
    extra = 2 if tiles * tiles * cfg.E > 4 * 1024 * 1024 else 0
    if cfg.dtype == "bf16" and cfg.k <= 2:
        return 4 + extra  # router (+ dispatch counts), scatter (+ scan, aux, y = 0), gate/up, down + combine
    return 5 + extra  # router (+ dispatch counts), scatter (+ scan, aux), gate/up, down, combine


def stage_breakdown(moe, torch, cfg, x, w, flush, stream, steps):
    """Average device ms per stage, timed with events between the entry points.

    A spin kernel at the head of each iteration holds the stream while the host
    queues every stage, so the events bracket device work only, not the
    Python-side launch gaps between entry points."""
    names = ["route_ms", "permute_ms", "gateup_ms", "down_ms", "combine_ms", "aux_ms"]
    acc = {n: 0.0 for n in names}
    for i in range(steps + 3):
        flush.fill_(i & 0xFF)
        torch.cuda._sleep(5_000_000)  # ~2.5-4 ms of device time, longer than the host's queueing
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
        evs[0].record(stream)
        r = moe.moe_route(x, w["w_g"], w["bias"], cfg.k)
        evs[1].record(stream)
        p = moe.moe_permute(x, r["topk_idx"], cfg.E)
        evs[2].record(stream)
        h = moe.moe_grouped_gateup_swiglu(p["x_perm"], p["offsets"], w["w_gate"], w["w_up"])
        evs[3].record(stream)
        yp = moe.moe_grouped_down(h, p["offsets"], w["w_down"])
        evs[4].record(stream)
        moe.moe_combine(yp, p["inv_perm"], r["topk_w"])
        evs[5].record(stream)
        moe.moe_aux_loss(p["counts"], cfg.T, cfg.k, aux_partials=r["aux_partials"])
        evs[6].record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            for j, n in enumerate(names):
                acc[n] += evs[j].elapsed_time(evs[j + 1])
    res = {n: v / steps for n, v in acc.items()}
    res["experts_used"] = int((p["counts"] > 0).sum().item())
    return res


def stage_breakdown_ec(moe, torch, cfg, x, w, flush, stream, steps):
    """Expert-choice stages, timed as in stage_breakdown."""
    names = ["route_ms", "gather_ms", "gateup_ms", "down_ms", "combine_ms"]
    acc = {n: 0.0 for n in names}
    for i in range(steps + 3):
        flush.fill_(i & 0xFF)
        torch.cuda._sleep(5_000_000)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
        evs[0].record(stream)
        r = moe.moe_expert_choice_route(x, w["w_g"], w["bias"], cfg.capacity_factor)
        evs[1].record(stream)
        C = r["C"]
        offsets = torch.arange(cfg.E + 1, device=x.device, dtype=torch.int32) * C
        xp = moe.moe_gather_rows(x, r["ec_idx"].view(-1), 1)
        evs[2].record(stream)
        h = moe.moe_grouped_gateup_swiglu(xp, offsets, w["w_gate"], w["w_up"])
        evs[3].record(stream)
        yp = moe.moe_grouped_down(h, offsets, w["w_down"])
        evs[4].record(stream)
        moe.moe_ec_combine(yp, r["pos"], r["ec_score"])
        evs[5].record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            for j, n in enumerate(names):
                acc[n] += evs[j].elapsed_time(evs[j + 1])
    return {n: v / steps for n, v in acc.items()}


def run_e2e(moe, torch, layer, x_host_np, cfg, dev, steps):
    """Same metric with host buffers, through the public HostPipeline: every step copies
    its x from pinned host memory to the device and its y back, inside the timed region.
    The pipeline overlaps batch i's forward with the copies of batches i+1 and i-1; the
    strictly serial form (copy in, forward, copy out, one step at a time) is reported
    beside it."""
    if x_host_np.dtype == np.uint16:
        xh = torch.from_numpy(x_host_np.view(np.int16)).view(torch.bfloat16).pin_memory()
    else:
        xh = torch.from_numpy(x_host_np).pin_memory()
    yhs = [torch.empty((cfg.T, cfg.d), dtype=torch.float32).pin_memory() for _ in range(2)]
    stream = torch.cuda.current_stream()
    pipe = moe.HostPipeline(layer, cfg.T, cfg.d, xh.dtype, dev)
    pipe.run([xh] * 3, [yhs[i % 2] for i in range(3)])
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    pipe.run([xh] * steps, [yhs[i % 2] for i in range(steps)])
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    # serial reference: one batch at a time on one stream
    xd = torch.empty_like(xh, device=dev)
    yd = torch.empty((cfg.T, cfg.d), dtype=torch.float32, device=dev)
    serial = 0.0
    n_serial = min(steps, 20)
    for i in range(n_serial + 3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        xd.copy_(xh, non_blocking=True)
        layer(xd, y=yd)
        yhs[0].copy_(yd, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            serial += a.elapsed_time(b)
    return {"value": cfg.T / (ms / 1e3), "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": int(xh.numel() * xh.element_size()),
            "d2h_bytes_per_step": int(yhs[0].numel() * yhs[0].element_size()),
            "api": "HostPipeline.run (copies of neighbouring batches overlap the forward)",
            "serial_ms_per_step": serial / n_serial}


# ---------------------------------------------------------------- CPU oracle


def _oracle_threads():
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:  # noqa: BLE001
        return os.cpu_count() or 1


def _oracle_step(oracle, cfg, x64, wg64, experts, tokens):
    xs = x64[tokens]
    if cfg.routing == "expert_choice":
        # expert choice needs every token's logits; the experts run on this sample's picks
        s = oracle.router_logits(x64, wg64, cfg_bias(cfg))
        C, idx, sc, pos = oracle.expert_choice_route(s, cfg.capacity_factor)
        keep = np.isin(idx, tokens)
        for e in range(cfg.E):
            rows = idx[e][keep[e]]
            if rows.size:
                oracle.swiglu_expert(x64[rows], *experts[e])
        return
    s = oracle.router_logits(xs, wg64, cfg_bias(cfg))
    idx, w, g = oracle.topk_route(s, cfg.k)
    oracle.aux_stats(g, idx, cfg.E)
    oracle.dispatch(idx, cfg.E)
    oracle.moe_forward(xs, idx, w, experts)


def cfg_bias(cfg):
    return synth.router_bias(cfg)


class _Pre:
    """fp64 copies of the stored weights (input preparation, outside the timing)."""

    def __init__(self, inp):
        self.items = [tuple(synth.to_f64(w[e]) for w in (inp.w_gate, inp.w_up, inp.w_down))
                      for e in range(inp.cfg.E)]

    def __len__(self):
        return len(self.items)

    def __getitem__(self, e):
        return self.items[e]


def cpu_baseline(cfg, seconds: float, inp=None, sample_tokens: int = 256):
    import oracle

    inp = inp if inp is not None else synth.make_inputs(cfg)
    x64, wg64 = synth.to_f64(inp.x), synth.to_f64(inp.w_g)
    experts = _Pre(inp)
    rng = np.random.default_rng(7)
    done = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        tokens = np.sort(rng.choice(cfg.T, size=min(sample_tokens, cfg.T), replace=False))
        _oracle_step(oracle, cfg, x64, wg64, experts, tokens)
        done += tokens.size
    dt = time.perf_counter() - t0
    return {"value": done / dt, "unit": UNIT, "cores": _oracle_threads(), "kind": "oracle",
            "sample": f"{done} tokens of {cfg.name} in chunks of {sample_tokens} (routing, aux, "
                      f"dispatch and fp64 SwiGLU experts per chunk), {dt:.1f} s"}


def run_reference(args, cfg):
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle

    inp = synth.make_inputs(cfg)
    x64, wg64 = synth.to_f64(inp.x), synth.to_f64(inp.w_g)
    experts = _Pre(inp)
    rng = np.random.default_rng(11)
    per_step = min(128, cfg.T)
    for _ in range(args.warmup):
        _oracle_step(oracle, cfg, x64, wg64, experts, np.sort(rng.choice(cfg.T, per_step, replace=False)))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(oracle, cfg, x64, wg64, experts, np.sort(rng.choice(cfg.T, per_step, replace=False)))
    dt = time.perf_counter() - t0
    value = per_step * args.steps / dt
    cores = _oracle_threads()
    sample = f"{per_step} random tokens of {cfg.name} per step"
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload_keys(cfg, ws), l2="not applicable (host CPU)",
                           launch="fp64 oracle on the host cores, one sample per step"),
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    args = parse_args(argv)
    cfg = workload_config(args)
    line = run_reference(args, cfg) if args.impl == "reference" else run_gpu(args, cfg)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
