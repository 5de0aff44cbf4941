#!/usr/bin/env python
"""Benchmark of the W8A8 / W4A8 online-activation-quantized linear on GB300.

One step = one whole layer call through the public API (per-token activation
quantization + integer GEMM with fused dequant) on one batch of seeded
synthetic inputs already resident in HBM.  The default workload is the W8A8
per-channel linear at M=4096, N=10240, K=2560, on which the metric is quoted.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints ONE JSON line on stdout (rank 0).  Under torchrun every rank runs the
same workload on its own GPU (replicas: the layer has no exchange step), and
the value is the sum of all ranks' work over the slowest rank's time.

Timing: CUDA events on the launching stream around exactly K steps, bracketed
by a barrier and a device synchronize; inputs, weights and outputs rotate
through enough sets to exceed twice the L2 size, so every step reads HBM.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "W8A8 linear TOPS @M=4096 N=10240 K=2560; % of INT8/HBM roofline"
UNIT = "TOPS"
# The pages' own number for this workload: 4.41 ms on an Apple M5 Pro
# (per-channel W8A8, N=10240, K=2560, M=4096) = 48.7 TOPS.  Context only.
PAGES_TOPS = 2 * 4096 * 10240 * 2560 / 4.41e-3 / 1e12
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--M", type=int, default=4096)
    ap.add_argument("--N", type=int, default=10240)
    ap.add_argument("--K", type=int, default=2560)
    ap.add_argument("--gs", type=int, default=0, help="0 = per channel, else 64 / 128")
    ap.add_argument("--bits", type=int, default=8, choices=[8, 4])
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", choices=["on", "off"], default="on",
                    help="replay the timed steps from a CUDA graph (off: direct launches from "
                         "Python, whose host-side path is longer than one call below M ~ 2048)")
    a = ap.parse_args()
    a.warmup = max(a.warmup, 3)
    return a


def workload_name(a):
    gran = f"per-group gs={a.gs}" if a.gs else "per-channel"
    return f"W{a.bits}A8 {gran} linear M={a.M} N={a.N} K={a.K}"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, device=None) -> float:
    """The largest of one float across all ranks (a no-op on one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tops(ops_per_rank_step: float, steps: int, world: int, elapsed_ms: float) -> float:
    """Whole-job throughput: the work of all ranks over the slowest rank's time."""
    return ops_per_rank_step * steps * world / (elapsed_ms * 1e-3) / 1e12


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={CLOCK_QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            f = [s.strip() for s in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((ts, float(f[1]), float(f[2]), f))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if self.t0 <= r[0] <= self.t1 + 0.2]
        use = inside or sorted(rows, key=lambda r: abs(r[0] - self.t0))[:2]
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = set()
        for r in use:
            for nm, v in zip(names[1:], r[3][5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(r[1] for r in use),
                "sm_max_mhz": max(r[2] for r in use),
                "reasons": sorted(reasons), "samples": len(use),
                "in_timed_region": bool(inside)}


# ----------------------------------------------------------------------------- helpers
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


def kernel_source_sha(names=("gemm_pair.cu", "gemm_pg.cu", "gemm_tc.cu", "gemv.cu",
                             "cider_device.cuh")) -> str:
    """Hash of the kernels' CUDA sources with comments and blank lines removed,
    so that counters taken on a kernel stay attached to it until its code
    changes."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "w4a8_quantized_linear_gb300", "csrc")
    for name in names:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            for line in f:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def library_path(M: int, N: int, K: int, gs: int, bits: int = 8, num_sms: int = 152):
    """(dominant kernel, kernel launches per step) of the library's dispatch for
    one linear call: the same limits as gemv_fits() and launch_gemm_tc() in the
    CUDA sources (small-M GEMV up to M=16 when its activation block and a ring
    of at least four 4 KiB weight tiles fit in shared memory; it quantizes the
    rows itself for one token or M * K <= 8192 unless it cuts K into slices,
    which adds the quantization kernel and a combine kernel; otherwise the
    quantization kernel followed by one tensor-core GEMM)."""
    if 1 <= M <= 16:
        mb = 1
        while mb < M:
            mb *= 2
        if mb * K <= 200 * 1024 and (227 * 1024 - 4096 - mb * K) // 4096 >= 4:
            from w4a8_quantized_linear_gb300 import cider_debug_small_m_slices
            slices = cider_debug_small_m_slices(M, N, K, bits, gs, num_sms)
            form = "tensor-core form" if M >= 4 else "dp4a form"
            if slices > 1:
                return (f"gemv_kernel (small-M weight-streaming GEMV, {form}, K in {slices} "
                        "slices + combine kernel)"), 3
            if M == 1 or M * K <= 8192:   # gemv_quantizes_itself()
                return "gemv_kernel (small-M weight-streaming GEMV, fused quantization)", 1
            return f"gemv_kernel (small-M weight-streaming GEMV, {form})", 2
    if gs:
        return ("gemm_pg_kernel (tcgen05 cta_group::2 on CTA pairs, 256x256 tiles, per-group drain "
                "into fp32 running sums)"), 2
    return "gemm_pair_kernel (tcgen05 cta_group::2 on CTA pairs, 256x256 tiles)", 2


def ncu_traffic(workload: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel source and workload."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_source_sha") != kernel_source_sha(tuple(e.get("sources", ()))):
        return None
    return e.get("dram_bytes_per_launch")


def make_host_inputs(a, rank: int, n_sets: int):
    from w4a8_quantized_linear_gb300 import inputs
    xs, ws = [], []
    for s in range(n_sets):
        x, w = inputs.layer(a.M, a.N, a.K, base_seed=1000 * rank, index=s)
        xs.append(x)
        ws.append(w)
    return xs, ws


# ----------------------------------------------------------------------------- reference arm
def run_reference(a):
    """The oracle (plain single-threaded C) on the host cores, on a bounded
    sample of rows per step of the same workload."""
    import oracle
    from w4a8_quantized_linear_gb300 import inputs

    ws, rank, _ = dist_env()
    if rank != 0:
        return
    oracle.build()
    x, W = inputs.layer(a.M, a.N, a.K)
    if a.bits == 8:
        qv, sw = oracle.quantize_weight_int8(W, a.gs)
    else:
        qv, sw = oracle.quantize_weight_int4(W, a.gs)
    # calibrate: one row
    t = time.perf_counter()
    oracle.linear(x, qv, sw, a.gs, rows=[0])
    row_s = time.perf_counter() - t
    budget = 120.0
    rows_per_step = int(max(1, min(16, budget / max(row_s, 1e-6) / (a.steps + a.warmup))))
    rng = np.random.default_rng(0)
    for _ in range(a.warmup):
        oracle.linear(x, qv, sw, a.gs, rows=rng.integers(0, a.M, rows_per_step))
    t = time.perf_counter()
    for _ in range(a.steps):
        oracle.linear(x, qv, sw, a.gs, rows=rng.integers(0, a.M, rows_per_step))
    el = time.perf_counter() - t
    ops = 2.0 * rows_per_step * a.N * a.K * a.steps
    val = ops / el / 1e12
    sample = (f"{rows_per_step} random rows of {a.M} per step (all N={a.N}, K={a.K}), "
              f"single-threaded C oracle, {el:.1f} s timed")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT,
            "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": el / a.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8", "data": "synthetic",
            "config": {"workload": workload_name(a), "M": a.M, "N": a.N, "K": a.K,
                       "group_size": a.gs, "bits": a.bits,
                       "note": "CPU oracle; each step computes a row sample of the workload"},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "host": host_cpu(), "sample": sample},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def host_cpu() -> dict:
    """The host's logical CPU count and model name (for the CPU baseline)."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu model", "processor name") and ":" in line:
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if model is None:
        # Arm hosts list no model name in /proc/cpuinfo; lscpu decodes the part number
        try:
            import subprocess
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.lower().startswith("model name:"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    if model is None:
        import platform
        model = platform.processor() or platform.machine()
    return {"nproc": os.cpu_count(), "cpu_model": model}


def cpu_baseline(a, x, qv, sw, budget_s=12.0):
    """The oracle as it stands, timed on this host on a bounded row sample."""
    import oracle
    oracle.build()
    rows, el = 0, 0.0
    chunk = 4
    t = time.perf_counter()
    while el < budget_s and rows < a.M:
        oracle.linear(x, qv, sw, a.gs, rows=np.arange(rows, min(rows + chunk, a.M)))
        rows = min(rows + chunk, a.M)
        el = time.perf_counter() - t
    val = 2.0 * rows * a.N * a.K / el / 1e12
    return {"value": val, "unit": UNIT, "cores": 1, "kind": "oracle", "host": host_cpu(),
            "sample": f"rows 0..{rows - 1} of the {workload_name(a)} workload "
                      f"({rows} x {a.N} x {a.K}), single-threaded C oracle, {el:.1f} s"}


# ----------------------------------------------------------------------------- our arm
def run_ours(a):
    import torch

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    from w4a8_quantized_linear_gb300 import _build
    _build.build()
    import w4a8_quantized_linear_gb300 as cider
    if not cider.cider_is_available():
        raise SystemExit("libcider: current device is not a supported sm_103 GPU")

    set_bytes = 2 * a.M * a.K + (a.N * a.K if a.bits == 8 else a.N * a.K // 2) + 2 * a.M * a.N
    n_sets = max(2, -(-2 * L2_BYTES // set_bytes) + 1)
    log(f"[bench] {workload_name(a)}: {n_sets} rotating sets of {set_bytes / 1e6:.1f} MB")
    xs_h, ws_h = make_host_inputs(a, rank, n_sets)
    xs, qws, sws, ys = [], [], [], []
    for x, w in zip(xs_h, ws_h):
        xs.append(torch.from_numpy(x).to(dev))
        wd = torch.from_numpy(w).to(dev)
        if a.bits == 8:
            q, s = cider.cider_quantize_weight_int8(wd, a.gs)
        else:
            q, s = cider.cider_quantize_weight_int4(wd, a.gs)
        del wd
        qws.append(q)
        sws.append(s)
        ys.append(torch.empty((a.M, a.N), dtype=torch.float16, device=dev))
    lin = cider.cider_w8a8_linear if a.bits == 8 else cider.cider_w4a8_linear
    torch.cuda.synchronize()

    def step(i):
        s = i % n_sets
        lin(xs[s], qws[s], sws[s], a.gs, out=ys[s])

    for i in range(a.warmup):
        step(i)
    torch.cuda.synchronize()

    use_graph = a.graph == "on"
    graph = graph_timed = None
    per_graph = 1
    if use_graph:
        # one graph holds `per_graph` consecutive steps (a divisor of K), replayed K / per_graph
        # times in the timed region.  A second graph of the same steps with the library's kernel
        # timing events as nodes is replayed as often right after it, for the kernel durations:
        # the event nodes add gaps between the launches, so they stay out of the timed steps.
        per_graph = max(d for d in range(1, min(a.steps, 64) + 1) if a.steps % d == 0)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(per_graph):
                step(i)
        cider.cider_timing_begin(per_graph)    # the kernel-timing events become graph nodes
        graph_timed = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_timed):
            for i in range(per_graph):
                step(i)
        torch.cuda.synchronize()
        for _ in range(3):
            graph.replay()
            graph_timed.replay()
        torch.cuda.synchronize()
    else:
        cider.cider_timing_begin(a.steps)   # events are created here, outside the timed region
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.5)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.mark(True)
    start.record()
    if graph is not None:
        for _ in range(a.steps // per_graph):
            graph.replay()
    else:
        for i in range(a.steps):
            step(i)
    stop.record()
    torch.cuda.synchronize()
    if graph_timed is not None:
        # kernel durations: the same steps, replayed with the timing events
        for _ in range(a.steps // per_graph):
            graph_timed.replay()
        torch.cuda.synchronize()
    if clocks:
        clocks.mark(False)
    n_timed, gemm_total_ms = cider.cider_timing_end()
    del graph_timed
    if ws > 1:
        torch.distributed.barrier()
    clk = clocks.stop() if clocks else None
    el_ms = start.elapsed_time(stop)
    # with a graph, the events hold the last replay's `per_graph` launches
    assert n_timed == (per_graph if graph is not None else a.steps), (n_timed, a.steps)
    if cider.cider_check_device_error() != 0:
        raise SystemExit("libcider reported a timed-out wait inside a kernel")
    el_ms = max_over_ranks(el_ms, dev)

    ops_step = 2.0 * a.M * a.N * a.K
    value = job_tops(ops_step, a.steps, ws, el_ms)
    gemm_avg_s = gemm_total_ms / n_timed * 1e-3

    # end to end through the public API with host buffers (copies inside the timed region):
    # every step copies its input from pinned host memory, runs the layer and copies its
    # output back; the copies and the layer run on three streams with two buffer sets, as a
    # serving loop would run them (step i + 1's input copy and step i - 1's output copy
    # overlap step i's layer call)
    e2e = None
    n_e2e = max(3, min(a.e2e_steps, a.steps))
    xh = [torch.from_numpy(x).pin_memory() for x in xs_h[:2]]
    yh = [torch.empty((a.M, a.N), dtype=torch.float16).pin_memory() for _ in range(2)]
    s_in, s_c, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]    # x[b] copied in
    ev_c = [torch.cuda.Event() for _ in range(2)]     # y[b] computed, x[b] no longer read
    ev_out = [torch.cuda.Event() for _ in range(2)]   # y[b] copied out

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_c[b])
            xs[b].copy_(xh[b], non_blocking=True)
            ev_in[b].record(s_in)
        with torch.cuda.stream(s_c):
            s_c.wait_event(ev_in[b])
            if i >= 2:
                s_c.wait_event(ev_out[b])
            lin(xs[b], qws[b], sws[b], a.gs, out=ys[b])
            ev_c[b].record(s_c)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_c[b])
            yh[b].copy_(ys[b], non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    main = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for st_ in (s_in, s_c, s_out):
        st_.wait_event(e0)
    for i in range(n_e2e):
        e2e_step(i)
    main.wait_event(ev_out[0])
    main.wait_event(ev_out[1])
    e1.record(main)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, dev)
    e2e = {"value": job_tops(ops_step, n_e2e, ws, e2e_ms), "unit": UNIT,
           "h2d_bytes_per_step": 2 * a.M * a.K, "d2h_bytes_per_step": 2 * a.M * a.N,
           "steps": n_e2e,
           "pipeline": "input copy, layer and output copy on three streams, two buffer sets"}

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return

    peaks, peak_src = measured_peaks()
    kernel_name, launches_per_step = library_path(
        a.M, a.N, a.K, a.gs, a.bits, torch.cuda.get_device_properties(dev).multi_processor_count)
    small_m = kernel_name.startswith("gemv")
    wl = workload_name(a)
    if small_m:
        wbytes = a.N * a.K if a.bits == 8 else a.N * a.K // 2
        G = a.K // a.gs if a.gs else 1
        # algorithmic bytes of the step: weight codes and scales, x (fp16), y.  The step is
        # timed as CUDA-graph replays; its duration bounds the kernels' from above, so
        # achieved = bytes / step time is a lower bound.  (Timing events placed as graph
        # nodes around a ~10 us kernel add several us of gaps to what they measure.)
        alg_bytes = wbytes + 4 * a.N * G + 2 * a.M * a.K + 2 * a.M * a.N
        achieved = alg_bytes / (el_ms / a.steps * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": ncu_traffic(wl),
                "kernel": kernel_name + ("" if launches_per_step == 1 else
                                         " with the quantization kernel (whole step)"),
                "timing": "whole step per CUDA-graph replay (upper bound of the kernel time)",
                "peak_source": f"{peak_src} hbm_gbs",
                "algorithmic_bytes_per_launch": alg_bytes}
    else:
        long_region = el_ms > 1000.0
        pk = peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]
        achieved = ops_step / gemm_avg_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk, "unit": "TFLOP/s",
                "frac": achieved / pk, "traffic": ncu_traffic(wl),
                "kernel": kernel_name,
                "peak_source": (f"{peak_src} bf16_tflops"
                                f"{'_sustained' if long_region else ''}"
                                " x 1.0 (fp16 and bf16 dense tensor rates are equal)"),
                "algorithmic_ops_per_launch": ops_step}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": el_ms / a.steps, "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": (value / PAGES_TOPS) if (a.M, a.N, a.K, a.gs, a.bits) == (4096, 10240, 2560, 0, 8) else None,
        "dtype": "int8", "data": "synthetic",
        "config": {"workload": wl, "M": a.M, "N": a.N, "K": a.K, "group_size": a.gs,
                   "bits": a.bits, "parallelism": f"replicas x{ws}",
                   "l2": f"inputs larger than L2: {n_sets} rotating x/qw/y sets "
                         f"({n_sets * set_bytes / 1e6:.0f} MB)",
                   "gemm_ms_avg": gemm_avg_s * 1e3,
                   "launch": (f"CUDA graph of {per_graph} steps, replayed {a.steps // per_graph} times; "
                              "kernel durations from a second replay pass with timing events"
                              if graph is not None else "direct launches from Python")},
        "roofline": roof,
        "gpu_launches": launches_per_step * a.steps,
        "e2e": e2e,
        "clocks": clk,
    }
    if ws == 1 and not a.no_cpu_baseline:
        import oracle
        x0 = xs_h[0]
        if a.bits == 8:
            qv, sw = oracle.quantize_weight_int8(ws_h[0], a.gs)
        else:
            qv, sw = oracle.quantize_weight_int4(ws_h[0], a.gs)
        line["cpu_baseline"] = cpu_baseline(a, x0, qv, sw)
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def main():
    a = parse_args()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)


if __name__ == "__main__":
    main()
