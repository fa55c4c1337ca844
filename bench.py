#!/usr/bin/env python3
"""Benchmark of the ternary FWHT-128 linear-layer hot path on GB300.

Headline (the `value` of the JSON line): decode GEMV throughput on packed
weight bytes (codes + fp16 scales), GB/s, for one decode step = one token
(M = 1) through the linear layers of a 64-layer stack of 27B-class shapes
(per layer 5120x5120 x2, 27648x5120 x2, 5120x27648; 2-bit codes; gate and up
read the same x, so their rows are stored as one 55296x5120 matrix and run as
one GEMV): 256 GEMV launches and 8.1 GB of packed weights per step, far larger
than L2, so every
step streams its weights from HBM.  The activation FWHT-128 runs inside every
GEMV launch.  Extra keys report the other hot-path rows: skinny M = 2..16
(2-bit and base-3), the tensor-core prefill GEMM (M = 2048), and the offline
quantise + pack sweep.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

`--impl reference` times the CPU oracle (single core) on a bounded sample of
the same workload and prints the same JSON line with "impl": "reference".
Multi-GPU runs are independent replicas (the path has no exchange step).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HIDDEN, FFN, LAYERS = 5120, 27648, 64
# (name, N, K) per layer: two 5120x5120, gate and up (two 27648x5120 that read
# the same x, stored as one matrix of 2 x 27648 rows), one 5120x27648
LAYER_SHAPES = [("h2h_a", HIDDEN, HIDDEN), ("h2h_b", HIDDEN, HIDDEN), ("gate_up", 2 * FFN, HIDDEN),
                ("down", HIDDEN, FFN)]
METRIC = "ternary GEMV packed-weight HBM GB/s (% of peak); prefill GEMM TFLOP/s"
# DRAM bytes per algorithmic byte of k_gemv_tc, from an ncu capture of one
# 27648x5120 launch of the current kernel: dram__bytes_read.sum +
# dram__bytes_write.sum = 37,666,560 + 0 for 37,601,280 packed bytes
# (every weight byte read once).
GEMV_TC_TRAFFIC_RATIO = 37666560 / 37601280
WORKLOAD = ("decode GEMV M=1, 2-bit codes, 64-layer stack of 27B-class shapes "
            "{5120x5120 x2, 27648x5120 x2, 5120x27648} per layer; gate and up (the two 27648x5120, same x) "
            "stored as one 55296x5120 matrix and run as one GEMV (256 launches, FWHT-128 fused)")


def packed_bytes(N: int, K: int, fmt: str = "2bit") -> int:
    """Algorithmic bytes a GEMV must read: packed codes + fp16 scales."""
    codes = N * (K // 4) if fmt == "2bit" else N * (((K + 4) // 5 + 15) // 16 * 16)
    return codes + N * (K // 128) * 2


def step_bytes() -> int:
    return LAYERS * sum(packed_bytes(N, K) for _, N, K in LAYER_SHAPES)


def peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------- ranks

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over all ranks (x itself when running alone)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None) -> None:
    if world > 1:
        import torch.distributed as dist
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons while active."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=2)

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- GPU arm

def synth_weight(torch, gen, dev, N: int, K: int):
    """W [N][K] bf16 ~N(0, 0.02) with 0.1% of the entries (chosen without
    replacement) x20, drawn on the device from a seeded generator."""
    W = torch.randn(N, K, device=dev, generator=gen, dtype=torch.float32).mul_(0.02)
    n_out = max(1, (N * K) // 1000)
    idx = torch.randperm(N * K, device=dev, generator=gen)[:n_out]
    W.view(-1)[idx] *= 20.0
    del idx
    return W.to(torch.bfloat16)


def build_stack(tq, torch, dev, seed: int, keep_weights: bool = False):
    """64 layers of packed weights, quantised on the GPU from seeded synthetic
    bf16 weights ~N(0, 0.02) with 0.1% of entries x20.  keep_weights: also
    return the bf16 weights (the offline sweep re-quantises them)."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    stack, weights = [], []
    for layer in range(LAYERS):
        mats, wl = [], []
        for name, N, K in LAYER_SHAPES:
            Wb = synth_weight(torch, gen, dev, N, K)
            # base-3 codes as well for the shapes the skinny comparison uses
            fmt = tq.TQ_PACK_BOTH if name in ("gate_up", "down") else tq.TQ_PACK_2BIT
            c2, c3, s = tq.quantize_pack(Wb, fmt)
            mats.append((name, N, K, c2, s, c3))
            if keep_weights:
                wl.append(Wb)
            del Wb
        stack.append(mats)
        weights.append(wl)
    return stack, weights


def activations(torch, dev, K: int, M: int, seed: int):
    """x [M][K] bf16 ~N(0, 1) with 4 channels x30 (seeded)."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    x = torch.randn(M, K, device=dev, generator=gen)
    ch = torch.randperm(K, device=dev, generator=gen)[:4]
    x[:, ch] *= 30.0
    return x.to(torch.bfloat16)


def capture(torch, fn):
    """fn's launches captured once into a CUDA graph (replayed per step)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def timing_event(torch):
    """A timing event that, inside a graph capture, becomes an event-record
    node of its own (needs torch's `external` events; None without them)."""
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return None


def launch_times(args, tq, torch, launches, path_of) -> dict:
    """Per-kernel launch durations in the step: a copy of the step graph with
    a timing event before and after every launch, replayed `steps` times (the
    events cut the programmatic overlap between neighbours, so each duration
    is one launch on its own in the stream).  Without graph-capturable events
    the same launches run eagerly between events."""
    ev = [(timing_event(torch), timing_event(torch)) for _ in launches]
    graphed = all(a is not None for a, _ in ev)
    if not graphed:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in launches]

    def body():
        for (e0, e1), fn in zip(ev, launches):
            e0.record()
            fn()
            e1.record()

    g = capture(torch, body) if graphed else None
    reps = max(3, min(args.steps, 10))
    sums: dict[int, list[float]] = {}
    for _ in range(reps):
        if graphed:
            g.replay()
        else:
            body()
        torch.cuda.synchronize()
        for i, (e0, e1) in enumerate(ev):
            sums.setdefault(path_of[i], []).append(e0.elapsed_time(e1))
    return {"graphed": graphed, "reps": reps, "ms": sums}


def gpu_arm(args, world, rank, local):
    import torch
    import ternary_weight_fwht128_gb300 as tq

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    pk = peaks()
    stream = torch.cuda.current_stream()

    stack, sweep_w = build_stack(tq, torch, dev, seed=1000 + rank, keep_weights=not args.quick)
    xs = {K: activations(torch, dev, K, 1, seed=K) for K in (HIDDEN, FFN)}
    ys = {N: torch.empty(1, N, device=dev) for N in sorted({N for _, N, _ in LAYER_SHAPES})}
    launches_per_step = LAYERS * len(LAYER_SHAPES)

    # the weights are written once, before any timing: every GEMV may start
    # streaming them while the one before it finishes (TQ_GEMV_WEIGHTS_READY)
    def gemv_calls(xsrc):
        return [(lambda c2=c2, s=s, N=N, K=K: tq.gemv(c2, s, xsrc[K], K, tq.TQ_PACK_2BIT, out=ys[N],
                                                      weights_ready=True))
                for mats in stack for _, N, K, c2, s, _ in mats]

    calls = gemv_calls(xs)

    def step():
        for fn in calls:
            fn()

    # eager steps first: one-time set-up (attributes, occupancy queries) runs
    # before the capture; then the step's 256 launches become one CUDA graph
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    graph = capture(torch, step)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world, dev)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world, dev)
    ms_local = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(ms_local, world, dev)
    bytes_step = step_bytes()
    gbs = world * bytes_step / (ms * 1e-3) / 1e9

    # ---- per-kernel launch durations (roofline of the dominant kernel)
    shapes = [(N, K) for mats in stack for _, N, K, _, _, _ in mats]
    path_of = [tq.gemv_path(N, K, 1, tq.TQ_PACK_2BIT) for N, K in shapes]
    lt = launch_times(args, tq, torch, calls, path_of)
    names = {tq.TQ_GEMV_TENSOR_MEMORY: "k_gemv_tc (tcgen05, weights in tensor memory)",
             tq.TQ_GEMV_MMA_SYNC: "k_gemv<1> (mma.sync)"}
    kernels = []
    for pth, times in lt["ms"].items():
        idx = [i for i, q in enumerate(path_of) if q == pth]
        nbytes = sum(packed_bytes(*shapes[i]) for i in idx)
        per_launch_ms = sum(times) / len(times)
        step_ms = per_launch_ms * len(idx)
        kernels.append({"kernel": names[pth], "launches_per_step": len(idx),
                        "us_per_launch": round(per_launch_ms * 1e3, 3),
                        "bytes_per_launch": nbytes // len(idx),
                        "GB/s": round(nbytes / len(idx) / (per_launch_ms * 1e-3) / 1e9, 1),
                        "ms_per_step_alone": round(step_ms, 4)})
    kernels.sort(key=lambda k: -k["ms_per_step_alone"])
    total_alone = sum(k["ms_per_step_alone"] for k in kernels)
    for k in kernels:
        k["share"] = round(k["ms_per_step_alone"] / total_alone, 4)
    dom = kernels[0]
    dom_is_tc = dom["kernel"].startswith("k_gemv_tc")

    # ---- end to end through the public API with host buffers: every step
    # copies its activations in from pinned host memory (one token row per
    # input width), replays the step's 256 GEMVs, and reads its outputs back.
    hx = {K: xs[K].cpu().pin_memory() for K in xs}
    hy = {N: torch.empty(1, N, dtype=torch.float32).pin_memory() for N in ys}
    dx = {K: torch.empty_like(xs[K]) for K in xs}
    h2d = sum(t.numel() * t.element_size() for t in hx.values())
    d2h = sum(t.numel() * t.element_size() for t in hy.values())
    e2e_calls = gemv_calls(dx)

    def e2e_compute():
        for fn in e2e_calls:
            fn()

    e2e_graph = capture(torch, e2e_compute)

    def e2e_step():
        for K in dx:
            dx[K].copy_(hx[K], non_blocking=True)
        e2e_graph.replay()
        for N in hy:
            hy[N].copy_(ys[N], non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(args.warmup):
        e2e_step()
    barrier(world, dev)
    # each step timed on the host clock (the copies and the host's wait are
    # part of it); the value uses the median step, which a host hiccup (a
    # freshly booted machine still starting services) does not move -- the
    # mean is reported beside it
    step_s = []
    t_all = time.perf_counter()
    for _ in range(args.steps):
        t0 = time.perf_counter()
        e2e_step()
        step_s.append(time.perf_counter() - t0)
    e2e_mean_s = max_over_ranks((time.perf_counter() - t_all) / args.steps, world, dev)
    e2e_s = max_over_ranks(statistics.median(step_s), world, dev)
    e2e_gbs = world * bytes_step / e2e_s / 1e9
    e2e_mean_gbs = world * bytes_step / e2e_mean_s / 1e9

    extras = {}
    if not args.quick:
        extras = gpu_extras(args, tq, torch, dev, stack, pk)
        extras["sweep"] = sweep_bench(tq, torch, sweep_w, pk, world)
    del sweep_w

    if rank != 0:
        return
    # achieved rate of the dominant kernel: when it makes every launch of the
    # step, its average launch duration in the timed region is the step time
    # over the launch count (CUDA events around the graph replays); otherwise
    # the isolated per-launch durations above are the best available figure.
    if dom["launches_per_step"] == launches_per_step:
        dom_gbs = round(bytes_step / launches_per_step / (ms_local / launches_per_step * 1e-3) / 1e9, 1)
        dom_timing = "CUDA events around the timed graph replays; step time / launches per step"
    else:
        dom_gbs = dom["GB/s"]
        dom_timing = ("timing-event nodes around each launch in a replay of the step graph"
                      if lt["graphed"] else "CUDA events around each eager launch of the step")
    line = {
        "metric": METRIC,
        "value": round(gbs, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u8 codes; e4m3 x e4m3 (tcgen05) and f16 x f16 (mma.sync) MMAs; f32 accumulate",
        "data": "synthetic (seeded; weights N(0,0.02)+0.1% x20 outliers, x N(0,1)+4 channels x30)",
        "config": {"workload": WORKLOAD, "M": 1, "layers": LAYERS, "packed_bytes_per_step": bytes_step,
                   "launches_per_step": launches_per_step,
                   "launch": "one CUDA graph per step (256 launches, programmatic dependent launch edges; "
                             "tq_gemv_ex with TQ_GEMV_WEIGHTS_READY: weights stream while the previous GEMV ends)",
                   "l2": "inputs larger than L2 (8.1 GB of packed weights streamed per step)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "frac_of_peak": round(gbs / world / pk["hbm_gbs"], 4),
        "roofline": {"bound": "hbm", "achieved": dom_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(dom_gbs / pk["hbm_gbs"], 4),
                     "traffic": (int(GEMV_TC_TRAFFIC_RATIO * dom["bytes_per_launch"])
                                 if dom_is_tc and GEMV_TC_TRAFFIC_RATIO else None),
                     "traffic_note": "DRAM bytes per launch of the dominant kernel, ncu capture of one "
                                     "27648x5120 launch (same algorithmic bytes as every launch of it here)",
                     "kernel": dom["kernel"],
                     "us_per_launch": round(ms_local / launches_per_step * 1e3, 3)
                     if dom["launches_per_step"] == launches_per_step else dom["us_per_launch"],
                     "kernel_timing": dom_timing,
                     "peak_source": pk["source"] + " (MEASURED_PEAKS.json hbm_gbs)"},
        "kernels_isolated": {"note": "each launch timed alone (event nodes between launches cut the "
                                     "programmatic overlap of neighbours)", "kernels": kernels},
        "e2e": {"value": round(e2e_gbs, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "timing": "host clock around each step (pinned-host copies in, the step's graph, copies out, "
                          "stream synchronise); value from the median step",
                "mean_GB/s": round(e2e_mean_gbs, 1)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    line.update(extras)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_budget)
    print(json.dumps(line), flush=True)


def time_events(fn, reps: int, torch) -> float:
    """Average ms of fn() over reps, CUDA events on the current stream."""
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fn()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def gpu_extras(args, tq, torch, dev, stack, pk) -> dict:
    """Skinny decode (2-bit vs base-3), prefill GEMM and the quantise sweep."""
    out = {}
    # --- skinny M in {2,4,8,16} on 27648x5120 and 5120x27648: cycle over the
    # stack's layers so that every launch streams from HBM
    skinny = []
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    def rows_of(m, n):
        # (name, N, K, c2, s, c3) restricted to the first n rows (gate of gate_up)
        nm, _, K, c2, s, c3 = m
        return (nm, n, K, c2[:n], s[:n], c3[:n] if c3 is not None else None)

    for (name, N, K) in (("gate_up", FFN, HIDDEN), ("down", HIDDEN, FFN)):
        mats = [rows_of([m for m in layer if m[0] == name][0], N) for layer in stack]
        for fmt_name, fmt in (("2bit", tq.TQ_PACK_2BIT), ("base3", tq.TQ_PACK_BASE3)):
            for M in (1, 2, 4, 8, 16):
                x = activations(torch, dev, K, M, seed=K + M)
                y = torch.empty(M, N, device=dev)
                it = [0]

                def run():
                    _, _, _, c2, s, c3 = mats[it[0] % len(mats)]
                    it[0] += 1
                    tq.gemv(c2 if fmt == tq.TQ_PACK_2BIT else c3, s, x, K, fmt, out=y)

                ms = time_events(run, 3 * len(mats), torch)
                gb = packed_bytes(N, K, fmt_name) / (ms * 1e-3) / 1e9
                path = tq.gemv_path(N, K, M, fmt)
                skinny.append({"shape": f"{N}x{K}", "M": M, "fmt": fmt_name,
                               "kernel": "k_gemv_tc" if path == tq.TQ_GEMV_TENSOR_MEMORY else "k_gemv (mma.sync)",
                               "us": round(ms * 1e3, 2),
                               "GB/s": round(gb, 1), "frac_of_peak": round(gb / pk["hbm_gbs"], 4),
                               "TFLOP/s": round(2 * M * N * K / (ms * 1e-3) / 1e12, 2)})
    out["skinny"] = skinny
    # --- prefill GEMM, M = 2048 on the three shapes
    prefill = []
    for name, N, K in (("h2h_a", HIDDEN, HIDDEN), ("gate_up", FFN, HIDDEN), ("down", HIDDEN, FFN)):
        _, _, _, c2, s, _ = rows_of([m for m in stack[0] if m[0] == name][0], N)
        M = 2048
        x = activations(torch, dev, K, M, seed=11 + K)
        ws = torch.empty(tq.gemm_workspace_bytes(M, K), dtype=torch.uint8, device=dev)
        y = torch.empty(M, N, device=dev)
        try:
            ms = time_events(lambda: tq.gemm(c2, s, x, K, tq.TQ_PACK_2BIT, workspace=ws, out=y), 10, torch)
        except tq.TQError as e:
            prefill.append({"shape": f"{N}x{K}", "M": M, "unavailable": str(e)})
            continue
        tf = 2 * M * N * K / (ms * 1e-3) / 1e12
        prefill.append({"shape": f"{N}x{K}", "M": M, "us": round(ms * 1e3, 1), "TFLOP/s": round(tf, 1),
                        "frac_of_bf16_peak": round(tf / pk["bf16_tflops"], 4),
                        "l2": "one layer's weights, repeated: its codes (6.6-35 MB) stay in L2; the GEMM is "
                              "tensor-bound, x' (21-113 MB) and y stream"})
    # gate and up of one layer read the same x: the second call reuses the
    # rotated x' in the workspace (TQ_GEMM_REUSE_ROTATED), one pre-pass per pair
    mats = {m[0]: m for m in stack[0]}
    N, K, M = FFN, HIDDEN, 2048
    x = activations(torch, dev, K, M, seed=11 + K)
    ws = torch.empty(tq.gemm_workspace_bytes(M, K), dtype=torch.uint8, device=dev)
    yg, yu = torch.empty(M, N, device=dev), torch.empty(M, N, device=dev)

    def pair():
        gu = mats["gate_up"]
        tq.gemm(gu[3][:FFN], gu[4][:FFN], x, K, tq.TQ_PACK_2BIT, workspace=ws, out=yg)
        tq.gemm(gu[3][FFN:], gu[4][FFN:], x, K, tq.TQ_PACK_2BIT, workspace=ws, out=yu, reuse_rotated=True)

    try:
        ms = time_events(pair, 10, torch)
        tf = 2 * 2 * M * N * K / (ms * 1e-3) / 1e12
        prefill.append({"shape": f"2x{N}x{K} (gate, up: one x' pre-pass)", "M": M, "us": round(ms * 1e3, 1),
                        "TFLOP/s": round(tf, 1), "frac_of_bf16_peak": round(tf / pk["bf16_tflops"], 4)})
    except tq.TQError as e:
        prefill.append({"shape": f"2x{N}x{K} (gate, up: one x' pre-pass)", "M": M, "unavailable": str(e)})
    # a layer whose input is the previous layer's output: the first GEMM writes
    # the second's x' in its epilogue (tq_gemm_rotate_next) and the second
    # skips its pre-pass; against two plain calls, each with its pre-pass
    N = K = HIDDEN
    M = 2048
    x = activations(torch, dev, K, M, seed=13 + K)
    ws1 = torch.empty(tq.gemm_workspace_bytes(M, K), dtype=torch.uint8, device=dev)
    ws2 = torch.empty(tq.gemm_workspace_bytes(M, N), dtype=torch.uint8, device=dev)
    ya, yb = torch.empty(M, N, device=dev), torch.empty(M, N, device=dev)
    xz = torch.zeros(M, N, dtype=torch.bfloat16, device=dev)

    def chained():
        tq.gemm_rotate_next(mats["h2h_a"][3], mats["h2h_a"][4], x, K, ws2, workspace=ws1, out=ya)
        tq.gemm(mats["h2h_b"][3], mats["h2h_b"][4], xz, N, tq.TQ_PACK_2BIT, workspace=ws2, out=yb,
                reuse_rotated=True)

    def two_plain():
        tq.gemm(mats["h2h_a"][3], mats["h2h_a"][4], x, K, tq.TQ_PACK_2BIT, workspace=ws1, out=ya)
        tq.gemm(mats["h2h_b"][3], mats["h2h_b"][4], x, N, tq.TQ_PACK_2BIT, workspace=ws2, out=yb)

    try:
        ms_c = time_events(chained, 10, torch)
        ms_p = time_events(two_plain, 10, torch)
        for label, ms in (("chained: x' of the second written by the first's epilogue", ms_c),
                          ("two plain calls, each with its pre-pass", ms_p)):
            tf = 2 * 2 * M * N * K / (ms * 1e-3) / 1e12
            prefill.append({"shape": f"2x{N}x{K} ({label})", "M": M, "us": round(ms * 1e3, 1),
                            "TFLOP/s": round(tf, 1), "frac_of_bf16_peak": round(tf / pk["bf16_tflops"], 4)})
    except tq.TQError as e:
        prefill.append({"shape": f"2x{N}x{K} chained", "M": M, "unavailable": str(e)})
    out["prefill"] = prefill
    # --- offline quantise + pack of one layer group, weights resident (bf16)
    sweep = []
    for name, N, K in (("h2h_a", HIDDEN, HIDDEN), ("gate", FFN, HIDDEN), ("down", HIDDEN, FFN)):
        W = (torch.randn(N, K, device=dev, generator=gen) * 0.02).to(torch.bfloat16)
        ms = time_events(lambda: tq.quantize_pack(W, tq.TQ_PACK_BOTH), 5, torch)
        nbytes = N * K * 2 + N * (K // 4) + N * tq.packed_ld(K, tq.TQ_PACK_BASE3) + N * (K // 128) * 2
        sweep.append({"shape": f"{N}x{K}", "fmt": "2bit+base3", "us": round(ms * 1e3, 1),
                      "Gparams/s": round(N * K / (ms * 1e-3) / 1e9, 1),
                      "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1)})
        del W
    out["quantize_pack"] = sweep
    out["layouts"] = layout_bench(tq, torch, dev, pk, gen)
    out["sparse24"] = sparse24_bench(tq, torch, dev, pk, gen)
    return out


def layout_bench(tq, torch, dev, pk, gen) -> list:
    """The layout variants (FWHT block 64/256, a scale per 256 weights, the
    residual two-pass form) on the benchmark's shapes: the decode GEMV (M = 1,
    27648x5120, cycling over 8 copies of the codes so each launch streams from
    HBM), the prefill GEMM (M = 2048, 5120x5120) and quantise + pack
    (5120x5120, bf16).  Work is counted over both passes of a residual layout."""
    rows = []
    W = (torch.randn(FFN, HIDDEN, device=dev, generator=gen) * 0.02).to(torch.bfloat16)
    Wh = (torch.randn(HIDDEN, HIDDEN, device=dev, generator=gen) * 0.02).to(torch.bfloat16)
    for (b, g, res) in ((64, 128, False), (256, 128, False), (128, 256, False), (128, 128, True)):
        lay = tq.layout(b, g, res)
        name = f"block {b}, group {g}" + (", residual" if res else "")
        r = {"layout": name}
        try:
            c2, _, s = tq.quantize_pack_layout(W, lay, tq.TQ_PACK_2BIT)
            copies = [(c2.clone(), s.clone()) for _ in range(8)]
            del c2, s
            N, K = FFN, HIDDEN
            x = activations(torch, dev, K, 1, seed=K + 1)
            y = torch.empty(1, N, device=dev)
            it = [0]

            def run():
                c, sc = copies[it[0] % len(copies)]
                it[0] += 1
                tq.gemv_layout(c, sc, x, K, lay, out=y)

            ms = time_events(run, 3 * len(copies), torch)
            nbytes = copies[0][0].numel() + copies[0][1].numel() * 2
            gb = nbytes / (ms * 1e-3) / 1e9
            r["gemv_M1_27648x5120"] = {"us": round(ms * 1e3, 2), "GB/s": round(gb, 1),
                                       "frac_of_peak": round(gb / pk["hbm_gbs"], 4), "bytes": nbytes}
            del copies
            N = K = HIDDEN
            c2, c3, s = tq.quantize_pack_layout(Wh, lay, tq.TQ_PACK_BOTH)
            Keff = K * (2 if res else 1)
            ms = time_events(lambda: tq.quantize_pack_layout(Wh, lay, tq.TQ_PACK_BOTH), 5, torch)
            qbytes = N * K * 2 + c2.numel() + c3.numel() + s.numel() * 2
            r["quantize_pack_5120x5120"] = {"us": round(ms * 1e3, 1), "Gparams/s": round(N * K / (ms * 1e-3) / 1e9, 1),
                                            "GB/s": round(qbytes / (ms * 1e-3) / 1e9, 1),
                                            "frac_of_peak": round(qbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4)}
            M = 2048
            xg = activations(torch, dev, K, M, seed=11 + K)
            ws = torch.empty(tq.gemm_workspace_bytes_layout(M, K, lay), dtype=torch.uint8, device=dev)
            yg = torch.empty(M, N, device=dev)
            ms = time_events(lambda: tq.gemm_layout(c2, s, xg, K, lay, workspace=ws, out=yg), 10, torch)
            tf = 2 * M * N * Keff / (ms * 1e-3) / 1e12
            r["gemm_M2048_5120x5120"] = {"us": round(ms * 1e3, 1), "TFLOP/s": round(tf, 1),
                                         "frac_of_bf16_peak": round(tf / pk["bf16_tflops"], 4),
                                         "flops": "2 M N Keff (both passes)"}
            del c2, c3, s, ws, yg
        except tq.TQError as e:
            r["unavailable"] = str(e)
        rows.append(r)
    return rows


def sparse24_bench(tq, torch, dev, pk, gen) -> dict:
    """The 2:4-sparse ternary format: quantise + pack (bf16 in), and the
    GEMV on the decode shapes (M = 1 and 16; the tensor-memory kernel, the
    codes expanded through a table), cycling over 8 copies of the codes so
    each launch streams from HBM.  GB/s counts the sparse codes and scales
    (26 bytes per 128 weights) of one launch."""
    out = {"bits_per_weight": 1.625}
    try:
        W = (torch.randn(HIDDEN, HIDDEN, device=dev, generator=gen) * 0.02).to(torch.bfloat16)
        ms = time_events(lambda: tq.quantize_pack_sparse24(W), 5, torch)
        N = K = HIDDEN
        qbytes = N * K * 2 + N * tq.sparse24_ld(K) + N * (K // 128) * 2
        out["quantize_pack_5120x5120"] = {"us": round(ms * 1e3, 1), "Gparams/s": round(N * K / (ms * 1e-3) / 1e9, 1),
                                          "GB/s": round(qbytes / (ms * 1e-3) / 1e9, 1),
                                          "frac_of_peak": round(qbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4)}
        del W
        for (N, K) in ((FFN, HIDDEN), (HIDDEN, FFN)):
            W = (torch.randn(N, K, device=dev, generator=gen) * 0.02).to(torch.bfloat16)
            c, sc = tq.quantize_pack_sparse24(W)
            del W
            copies = [(c.clone(), sc.clone()) for _ in range(8)]
            del c, sc
            nbytes = copies[0][0].numel() + copies[0][1].numel() * 2
            for M in (1, 16):
                x = activations(torch, dev, K, M, seed=K + M)
                y = torch.empty(M, N, device=dev)
                ws = torch.empty(tq.gemv_sparse24_workspace_bytes(N, K, M), dtype=torch.uint8, device=dev)
                it = [0]

                def run():
                    cc, ss = copies[it[0] % len(copies)]
                    it[0] += 1
                    tq.gemv_sparse24(cc, ss, x, K, out=y, workspace=ws)

                for _ in range(len(copies)):
                    run()
                ms = time_events(run, 3 * len(copies), torch)
                gb = nbytes / (ms * 1e-3) / 1e9
                path = tq.gemv_sparse24_path(N, K, M)
                out[f"gemv_M{M}_{N}x{K}"] = {"us": round(ms * 1e3, 2), "GB/s": round(gb, 1),
                                             "frac_of_peak": round(gb / pk["hbm_gbs"], 4), "bytes": nbytes,
                                             "kernel": "k_gemv_tc (2:4 codes)" if path == tq.TQ_GEMV_TENSOR_MEMORY
                                             else "k_gemv_sparse24 (CUDA cores)"}
            del copies
        # prefill M = 2048: dense fp16 MMAs on the expanded tiles (2 M N K flops)
        M = 2048
        for (N, K) in ((HIDDEN, HIDDEN), (FFN, HIDDEN)):
            W = (torch.randn(N, K, device=dev, generator=gen) * 0.02).to(torch.bfloat16)
            c, sc = tq.quantize_pack_sparse24(W)
            del W
            xg = activations(torch, dev, K, M, seed=K + 7)
            ws = torch.empty(tq.gemm_workspace_bytes(M, K), dtype=torch.uint8, device=dev)
            yg = torch.empty(M, N, device=dev)
            ms = time_events(lambda: tq.gemm_sparse24(c, sc, xg, K, workspace=ws, out=yg), 10, torch)
            tf = 2 * M * N * K / (ms * 1e-3) / 1e12
            out[f"gemm_M{M}_{N}x{K}"] = {"us": round(ms * 1e3, 1), "TFLOP/s": round(tf, 1),
                                         "frac_of_bf16_peak": round(tf / pk["bf16_tflops"], 4)}
            del c, sc, ws, yg
    except tq.TQError as e:
        out["unavailable"] = str(e)
    return out


def sweep_bench(tq, torch, weights, pk, world: int) -> dict:
    """The offline quantise + pack sweep: all 64 layers x {5120x5120 x2,
    27648x5120 x2, 5120x27648} of resident bf16 weights (30.5 G parameters,
    61 GB, far larger than L2), 2-bit and base-3 codes plus scales in one pass
    per matrix, into per-matrix outputs; CUDA events around whole sweeps."""
    outs = []
    params, nbytes = 0, 0
    for wl in weights:
        for Wb in wl:
            N, K = Wb.shape
            ld3 = tq.packed_ld(K, tq.TQ_PACK_BASE3)
            o = (torch.empty(N, K // 4, dtype=torch.uint8, device=Wb.device),
                 torch.empty(N, ld3, dtype=torch.uint8, device=Wb.device),
                 torch.empty(N, K // 128, dtype=torch.int16, device=Wb.device))
            outs.append((Wb, o))
            params += N * K
            nbytes += N * K * 2 + N * (K // 4) + N * ld3 + N * (K // 128) * 2

    def sweep():
        for Wb, o in outs:
            tq.quantize_pack(Wb, tq.TQ_PACK_BOTH, out=o)

    reps = 3
    ms = time_events(sweep, reps, torch)
    line = {"workload": "64 layers x {5120x5120 x2, 27648x5120 x2, 5120x27648}, bf16 N(0,0.02)+0.1% x20, "
                        "2-bit + base-3 + fp16 scales in one pass per matrix",
            "matrices": len(outs), "params": params, "bytes": nbytes, "ms": round(ms, 3),
            "Gparams/s": round(world * params / (ms * 1e-3) / 1e9, 1),
            "GB/s": round(world * nbytes / (ms * 1e-3) / 1e9, 1),
            "frac_of_peak": round(nbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
            "timing": f"CUDA events around {reps} whole sweeps after one warm-up sweep; inputs larger than L2",
            "launches": len(outs) * (reps + 1)}
    del outs
    return line


# ---------------------------------------------------------------- CPU oracle

def host_cpu() -> dict:
    """Host core count and CPU model (the oracle runs on one of the cores)."""
    import platform
    model = platform.processor() or platform.machine()
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu part", "hardware"):
                    model = line.split(":", 1)[1].strip()
                    if key == "cpu part":
                        model = f"{platform.machine()} (CPU part {model})"
                    break
    except OSError:
        pass
    return {"nproc": os.cpu_count(), "cpu_model": model}


class OracleGemv:
    """The oracle's fp64 GEMV (M = 1) over oracle-quantised synthetic layers
    of the decode shapes (5120x5120, 1024 rows of 27648 inputs, 3456 rows of
    5120 inputs), prepared once; run() times it on one core for a budget."""

    def __init__(self, orc):
        from ternary_weight_fwht128_gb300 import synth
        self.orc = orc
        self.prepared = []
        for (N, K) in [(HIDDEN, HIDDEN), (1024, FFN), (FFN // 8, HIDDEN)]:
            W = synth.weights(N, K, N + K, dtype="bf16")
            T, S = orc.quantize(W)
            x = synth.bf16_bits_to_f32(synth.activations(1, K, K))
            self.prepared.append((N, K, T, S, x))

    def run(self, budget_s: float) -> dict:
        done_bytes, spent, calls = 0, 0.0, 0
        while spent < budget_s:
            for (N, K, T, S, x) in self.prepared:
                t0 = time.perf_counter()
                self.orc.gemv(T, S, x)
                spent += time.perf_counter() - t0
                done_bytes += packed_bytes(N, K)
                calls += 1
        return {"value": round(done_bytes / spent / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": f"{calls} oracle fp64 GEMVs (M=1) over 5120x5120, 1024x27648, 3456x5120 rows of "
                          f"oracle-quantised synthetic weights, {spent:.1f} s of one host core"}


def cpu_baseline(budget_s: float = 12.0) -> dict:
    """The CPU oracle, as it stands, on a bounded sample of the decode
    workload: fp64 GEMV of oracle-quantised 5120x5120 and 27648x5120 layers
    (single core), repeated until the time budget is spent.  Reported in the
    same unit: packed weight bytes consumed per second.  Beside it: the small
    end-to-end case (256x256: quantise, pack, GEMV) in ms, and the offline
    sweep's quantise + pack rate on sampled rows, extrapolated to the 64-layer
    sweep."""
    import numpy as np

    import oracle
    from ternary_weight_fwht128_gb300 import synth

    orc = oracle.load()
    # small end-to-end case, whole
    W, xb = synth.tiny_config()
    xt = synth.bf16_bits_to_f32(xb)
    t0 = time.perf_counter()
    reps = 0
    while reps < 5 or time.perf_counter() - t0 < 0.5:
        T, S = orc.quantize(W)
        orc.pack2(T)
        orc.gemv(T, S, xt)
        reps += 1
    tiny_ms = (time.perf_counter() - t0) / reps * 1e3
    # offline sweep: 1% of the rows of each of the five shapes of a layer
    sweep_rows, sweep_s, sweep_params = 0, 0.0, 0
    sample = []
    for i, (_, N, K) in enumerate(LAYER_SHAPES):
        sample.append(synth.weights(max(1, N // 100), K, 700 + i, dtype="bf16"))
    while sweep_s < min(3.0, budget_s / 4):
        for Ws in sample:
            t0 = time.perf_counter()
            T, S = orc.quantize(Ws)
            orc.pack2(T)
            orc.pack3(T)
            sweep_s += time.perf_counter() - t0
            sweep_params += Ws.size
            sweep_rows += Ws.shape[0]
    sweep_pps = sweep_params / sweep_s
    total_params = LAYERS * sum(N * K for _, N, K in LAYER_SHAPES)
    # decode GEMV, the unit of the headline metric
    gemv = OracleGemv(orc)
    out = gemv.run(budget_s)
    out.update({"tiny_ms": round(tiny_ms, 3),
                "tiny_sample": "256x256 layer: oracle quantise + 2-bit pack + fp64 GEMV (M=1), whole, one core",
                "sweep_params_per_s": round(sweep_pps, 1),
                "sweep_s_extrapolated": round(total_params / sweep_pps, 1),
                "sweep_sample": f"oracle quantise + 2-bit + base-3 pack of 1% of the rows of each layer shape "
                                f"({sweep_rows} rows, {sweep_s:.1f} s, one core), extrapolated to the 64-layer "
                                f"sweep ({total_params / 1e9:.2f} G params)"})
    out.update(host_cpu())
    return out


def reference_arm(args, world, rank):
    """The oracle as the reference implementation (single host core): each
    step is a bounded sample of the decode workload (fp64 GEMVs of the
    decode shapes), sized so the whole run takes about two minutes."""
    if rank != 0:
        return
    import oracle
    orc = oracle.load()
    gemv = OracleGemv(orc)
    per_step = max(0.3, min(args.ref_budget, 120.0 / (args.warmup + args.steps)))
    for _ in range(args.warmup):
        gemv.run(per_step)
    vals, samples = [], []
    for _ in range(args.steps):
        r = gemv.run(per_step)
        vals.append(r["value"])
        samples.append(r["sample"])
    value = round(statistics.median(vals), 4)
    base = {"kind": "oracle", "cores": 1, "value": value, "unit": "GB/s",
            "sample": f"median of {args.steps} steps, each: {samples[-1]}"}
    base.update(host_cpu())
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": WORKLOAD, "M": 1, "sample": "bounded oracle sample per step"},
            "cpu_baseline": base,
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def only_arm(args):
    """One operation on one shape, `warmup` + `steps` launches, timed with
    CUDA events: the small, self-contained command the ncu captures use."""
    import torch
    import ternary_weight_fwht128_gb300 as tq

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    N, K = (int(v) for v in args.shape.lower().split("x"))
    M = args.M
    gen = torch.Generator(device=dev)
    gen.manual_seed(5)
    W = (torch.randn(N, K, device=dev, generator=gen) * 0.02).to(torch.bfloat16)
    fmt = tq.TQ_PACK_BASE3 if args.fmt == "base3" else tq.TQ_PACK_2BIT
    x = activations(torch, dev, K, M, seed=K + M)
    lay = None
    if args.layout:
        b, g, r = (int(v) for v in args.layout.split(","))
        lay = tq.layout(b, g, bool(r))
    if args.only == "quantize" and lay is not None:
        c2, c3, s = tq.quantize_pack_layout(W, lay, tq.TQ_PACK_BOTH)
        run = lambda: tq.quantize_pack_layout(W, lay, tq.TQ_PACK_BOTH)
        work, unit = N * K * 2 + c2.numel() + c3.numel() + s.numel() * 2, "GB/s"
    elif args.only == "quantize":
        run = lambda: tq.quantize_pack(W, tq.TQ_PACK_BOTH)
        work, unit = N * K * 2 + N * (K // 4) + N * tq.packed_ld(K, tq.TQ_PACK_BASE3) + N * (K // 128) * 2, "GB/s"
    elif args.only == "sparse24_quantize":
        run = lambda: tq.quantize_pack_sparse24(W)
        work, unit = N * K * 2 + N * tq.sparse24_ld(K) + N * (K // 128) * 2, "GB/s"
    elif args.only == "sparse24_gemv":
        c24, s24 = tq.quantize_pack_sparse24(W)
        del W
        y = torch.empty(M, N, device=dev)
        ws = torch.empty(tq.gemv_sparse24_workspace_bytes(N, K, M), dtype=torch.uint8, device=dev)
        run = lambda: tq.gemv_sparse24(c24, s24, x, K, out=y, workspace=ws)
        work, unit = c24.numel() + s24.numel() * 2, "GB/s"
    elif args.only == "sparse24_gemm":
        c24, s24 = tq.quantize_pack_sparse24(W)
        del W
        y = torch.empty(M, N, device=dev)
        ws = torch.empty(tq.gemm_workspace_bytes(M, K), dtype=torch.uint8, device=dev)
        run = lambda: tq.gemm_sparse24(c24, s24, x, K, workspace=ws, out=y)
        work, unit = 2 * M * N * K, "TFLOP/s"
    elif args.only == "fwht":
        out = torch.empty(M, K, device=dev, dtype=torch.float16)
        run = lambda: tq.fwht128(x, out=out)
        work, unit = M * K * 4, "GB/s"
    else:
        c2, c3, s = tq.quantize_pack(W, fmt | tq.TQ_PACK_2BIT)
        codes = c3 if fmt == tq.TQ_PACK_BASE3 else c2
        del W
        if args.only == "gemv":
            y = torch.empty(M, N, device=dev)
            run = lambda: tq.gemv(codes, s, x, K, fmt, out=y)
            work, unit = packed_bytes(N, K, "base3" if fmt == tq.TQ_PACK_BASE3 else "2bit"), "GB/s"
        elif args.only in ("gemv_chain", "gemv_pair"):
            # layer a (N x K) then layer b (K x N), as up and down: chained, a
            # writes b's rotated x; as a pair, b takes a bf16 x of its own
            Wb = (torch.randn(K, N, device=dev, generator=gen) * 0.02).to(torch.bfloat16)
            cb, cb3, sb = tq.quantize_pack(Wb, fmt | tq.TQ_PACK_2BIT)
            cb = cb3 if fmt == tq.TQ_PACK_BASE3 else cb
            del Wb
            ya, yb = torch.empty(M, N, device=dev), torch.empty(M, K, device=dev)
            xn = torch.empty(M, N, device=dev)
            xb = activations(torch, dev, N, M, seed=N + M)
            if args.only == "gemv_chain":
                def run():
                    tq.gemv_rotate_next(codes, s, x, K, fmt, xnext=xn, out=ya, weights_ready=True)
                    tq.gemv(cb, sb, xn, N, fmt, out=yb, weights_ready=True, x_rotated=True)
            else:
                def run():
                    tq.gemv(codes, s, x, K, fmt, out=ya, weights_ready=True)
                    tq.gemv(cb, sb, xb, N, fmt, out=yb, weights_ready=True)
            fk = "base3" if fmt == tq.TQ_PACK_BASE3 else "2bit"
            work, unit = packed_bytes(N, K, fk) + packed_bytes(K, N, fk), "GB/s"
        elif args.only == "gemm_chain":
            # layer a (N x K) writes layer b's x' in its epilogue; b (N x N) skips its pre-pass
            Wb = (torch.randn(N, N, device=dev, generator=gen) * 0.02).to(torch.bfloat16)
            cb, _, sb = tq.quantize_pack(Wb, tq.TQ_PACK_2BIT)
            del Wb
            ws1 = torch.empty(tq.gemm_workspace_bytes(M, K), dtype=torch.uint8, device=dev)
            ws2 = torch.empty(tq.gemm_workspace_bytes(M, N), dtype=torch.uint8, device=dev)
            ya, yb = torch.empty(M, N, device=dev), torch.empty(M, N, device=dev)
            xz = torch.zeros(M, N, dtype=torch.bfloat16, device=dev)

            def run():
                tq.gemm_rotate_next(codes, s, x, K, ws2, workspace=ws1, out=ya)
                tq.gemm(cb, sb, xz, N, workspace=ws2, out=yb, reuse_rotated=True)

            work, unit = 2 * M * N * (K + N), "TFLOP/s"
        else:
            ws = torch.empty(tq.gemm_workspace_bytes(M, K), dtype=torch.uint8, device=dev)
            y = torch.empty(M, N, device=dev)
            run = lambda: tq.gemm(codes, s, x, K, fmt, workspace=ws, out=y)
            work, unit = 2 * M * N * K, "TFLOP/s"
    for _ in range(args.warmup):
        run()
    ms = time_events(run, args.steps, torch)
    rate = work / (ms * 1e-3) / (1e12 if unit == "TFLOP/s" else 1e9)
    print(json.dumps({"only": args.only, "shape": f"{N}x{K}", "M": M, "fmt": args.fmt, "us": round(ms * 1e3, 2),
                      unit: round(rate, 1)}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--quick", action="store_true", help="headline decode step only (no extra sections)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--ref-budget", type=float, default=4.0)
    ap.add_argument("--layout", default="", help="block,group,residual for --only quantize (layout variants)")
    ap.add_argument("--only", choices=["gemv", "gemm", "gemm_chain", "quantize", "fwht", "sparse24_gemv",
                                       "sparse24_quantize", "sparse24_gemm", "gemv_chain", "gemv_pair"],
                    help="time one operation on one shape (for profiler captures)")
    ap.add_argument("--shape", default="27648x5120", help="NxK for --only")
    ap.add_argument("--M", type=int, default=1, help="activation rows for --only")
    ap.add_argument("--fmt", choices=["2bit", "base3"], default="2bit")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    if args.only:
        only_arm(args)
        return
    if args.impl == "reference":
        reference_arm(args, world, rank)
        return
    gpu_arm(args, world, rank, local)


if __name__ == "__main__":
    main()
