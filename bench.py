"""Benchmark of the block-quantized GEMV hot path on GB300.

Workload (default): Q4_0 GEMV, W 4096 rows x 14336 cols (the FFN down
projection shape), fp32 activations, batch 1.  One step = one GEMV over one
activation vector (block decode, unpack + scale, dot product, row reduction).

Metric: effective GB/s = algorithmic bytes (W + x + y) per step / time, also
reported as a fraction of the HBM peak.  Inputs are synthetic and seeded
(qsynth); the weights rotate over enough distinct device copies that the
working set exceeds L2 between reuses.

Timed region: K steps replayed from CUDA graphs (each step one kernel launch
of the library, consecutive launches linked by programmatic dependent launch,
the weights declared static with qgemv_set_option) between a barrier +
synchronize on both sides; the kernel's average launch duration for the
roofline is the timed region's CUDA-event time / K.  A separate short graph
with an event pair around every launch gives the duration of one launch that
does not overlap its neighbours (reported as kernel_ms_isolated).  Before the
start event, a spin kernel (torch.cuda._sleep, outside the timed region)
keeps the stream busy while the host queues the timed launches, so the
host's launch latency is not counted as device time.  `e2e` repeats the metric through the public
Python API with host buffers: each step copies x from pinned host memory,
runs the GEMV and copies y back.

--impl reference runs the CPU oracle (the plain C definition) on the host
cores instead, on a bounded sample of rows per step.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--profile-call OP FMT DIMS... runs a few calls of one library entry point on
seeded synthetic inputs and exits (for ncu captures of a single kernel; no
timing):
    gemv FMT NROWS NCOLS BATCH   six qgemv calls over four copies of W (so the
                                 captured launch does not find W in L2)
    mmvq FMT NROWS NCOLS BATCH   six quantized-activation GEMV calls (quantizer +
                                 GEMV each); mmvq_xq: the GEMV alone
    id FMT NROWS NCOLS N_EXPERT BATCH X_GROUP
                                 six expert-selected GEMV calls, column b of
                                 call i on expert (i*BATCH + b) % N_EXPERT
    dequant FMT NROWS NCOLS      four to-fp16 calls
    gemm FMT NROWS NCOLS M       four prefill calls
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import qsynth  # noqa: E402

WORKLOAD = {"name": "q4_0_gemv_4096x14336_b1", "fmt": "q4_0", "nrows": 4096, "ncols": 14336, "batch": 1}
METRIC = "Q4_0 GEMV 4096x14336 batch-1: effective GB/s and % of GB300 HBM peak"
HBM_NOMINAL_GBS = 8000.0
# dram__bytes_read.sum + dram__bytes_write.sum of one launch of the headline
# GEMV kernel, from the ncu capture summarized in profiles/ (set to None when
# the kernel changes until it is captured again)
NCU_TRAFFIC_BYTES = 33156096
BLOCK_BYTES = {"q4_0": 18, "q4_1": 20, "q8_0": 34}


def gemv_bytes(fmt, nrows, ncols, batch):
    return nrows * (ncols // 32) * BLOCK_BYTES[fmt] + 4 * batch * ncols + 4 * batch * nrows


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="qgemv_clocks_%d_" % self.gpu, suffix=".csv")
            self.f = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        try:
            os.unlink(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------- graph timing helpers
_cudart = None


def cudart():
    """libcudart (the instance torch and libqgemv already share in this process)."""
    global _cudart
    if _cudart is None:
        for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
            try:
                _cudart = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if _cudart is None:
            raise RuntimeError("libcudart not found")
        vp, u = ctypes.c_void_p, ctypes.c_uint
        _cudart.cudaEventCreateWithFlags.argtypes = [ctypes.POINTER(vp), u]
        _cudart.cudaEventRecordWithFlags.argtypes = [vp, vp, u]
        _cudart.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), vp, vp]
        _cudart.cudaEventDestroy.argtypes = [vp]
        for f in ("cudaEventCreateWithFlags", "cudaEventRecordWithFlags", "cudaEventElapsedTime",
                  "cudaEventDestroy"):
            getattr(_cudart, f).restype = ctypes.c_int
    return _cudart


class RawEvent:
    """A timing CUDA event recorded with cudaEventRecordExternal, so that it
    becomes an event-record node when captured into a graph."""

    def __init__(self):
        self.h = ctypes.c_void_p()
        rc = cudart().cudaEventCreateWithFlags(ctypes.byref(self.h), 0)
        if rc != 0:
            raise RuntimeError("cudaEventCreateWithFlags failed: %d" % rc)

    def record(self, stream):
        rc = cudart().cudaEventRecordWithFlags(self.h, ctypes.c_void_p(stream.cuda_stream), 1)
        if rc != 0:
            raise RuntimeError("cudaEventRecordWithFlags failed: %d" % rc)

    def elapsed_time(self, other):
        ms = ctypes.c_float()
        rc = cudart().cudaEventElapsedTime(ctypes.byref(ms), self.h, other.h)
        if rc != 0:
            raise RuntimeError("cudaEventElapsedTime failed: %d" % rc)
        return float(ms.value)

    def __del__(self):
        try:
            cudart().cudaEventDestroy(self.h)
        except Exception:
            pass


_KEEP_ALIVE = []


def build_graphs(torch, launch, n_launch, chunk, timed_events):
    """CUDA graphs that replay exactly n_launch calls of launch(i) in total.

    Returns (list of (graph, count)), events[(start, end)] of the last chunk
    graph when timed_events is set (launch i of that graph is bracketed)."""
    graphs = []
    ev_pairs = []
    done = 0
    sizes = []
    while done < n_launch:
        c = min(chunk, n_launch - done)
        sizes.append(c)
        done += c
    cache = {}
    for c in sizes:
        if c in cache:
            graphs.append((cache[c], c))
            continue
        g = torch.cuda.CUDAGraph()
        pairs = []
        s = torch.cuda.Stream()
        with torch.cuda.graph(g, stream=s):
            cs = torch.cuda.current_stream()
            for i in range(c):
                if timed_events:
                    e0, e1 = RawEvent(), RawEvent()
                    e0.record(cs)
                    launch(i)
                    e1.record(cs)
                    pairs.append((e0, e1))
                else:
                    launch(i)
        cache[c] = g
        graphs.append((g, c))
        _KEEP_ALIVE.append(pairs)         # events referenced by graph nodes must outlive the graph
        if pairs:
            ev_pairs = pairs
    return graphs, ev_pairs


# ------------------------------------------------------------ distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier(torch, world):
    if world > 1:
        torch.distributed.barrier()


def replica_value(step_bytes, steps, world, elapsed_s):
    """Whole-job GB/s of `world` replicas that each ran `steps` steps of
    `step_bytes` algorithmic bytes, the slowest in `elapsed_s` seconds."""
    return step_bytes * steps * world / elapsed_s / 1e9


def max_over_ranks(torch, world, value, device):
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------- CPU oracle
def oracle_rate(oracle, fmt, Wn, xn, nrows, ncols, batch, seconds, threads):
    """Oracle GEMV on row samples for about `seconds`; returns (GB/s, rows done, elapsed)."""
    oracle.set_threads(threads)
    per_row = ncols // 32 * BLOCK_BYTES[fmt] + 4 * batch
    rows_done, t0 = 0, time.perf_counter()
    g = qsynth.rng(123)
    n = min(nrows, max(threads * 8, 64))
    while True:
        rows = g.integers(0, nrows, n)
        oracle.gemv_rows(fmt, Wn, xn, nrows, ncols, batch, rows)
        rows_done += n
        el = time.perf_counter() - t0
        if el >= seconds:
            break
        n = min(nrows, n * 2) if el < seconds / 4 else n
    gbs = (rows_done * per_row + 4 * batch * ncols) / el / 1e9
    return gbs, rows_done, el


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args):
    world, rank, local = dist_setup()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    wl = WORKLOAD
    fmt, nrows, ncols, batch = wl["fmt"], wl["nrows"], wl["ncols"], wl["batch"]
    Wn = qsynth.make_weights(fmt, nrows, ncols, seed=2024)
    xn = qsynth.make_x(batch, ncols, seed=2025)
    cores = host_cores()
    oracle.set_threads(cores)
    # calibrate: rows per step so that warmup + steps take about 60 s
    t0 = time.perf_counter()
    oracle.gemv_rows(fmt, Wn, xn, nrows, ncols, batch, np.arange(min(nrows, 256)))
    per_row = (time.perf_counter() - t0) / min(nrows, 256)
    total = max(1, args.steps + args.warmup)
    rows_per_step = int(max(1, min(nrows, 60.0 / total / max(per_row, 1e-9))))
    g = qsynth.rng(7)
    for _ in range(args.warmup):
        oracle.gemv_rows(fmt, Wn, xn, nrows, ncols, batch, g.integers(0, nrows, rows_per_step))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gemv_rows(fmt, Wn, xn, nrows, ncols, batch, g.integers(0, nrows, rows_per_step))
    el = time.perf_counter() - t0
    step_bytes = rows_per_step * (ncols // 32 * BLOCK_BYTES[fmt] + 4 * batch) + 4 * batch * ncols
    value = step_bytes * args.steps / el / 1e9
    sample = "%d random rows of %dx%d per step (full row = %d blocks), x batch %d" % (
        rows_per_step, nrows, ncols, ncols // 32, batch)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl["name"], "fmt": fmt, "nrows": nrows, "ncols": ncols, "batch": batch},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------ main
def run_ours(args):
    import torch

    world, rank, local = dist_setup()
    if world > 1:
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from block_quantized_weight_qgemv_gb300 import build as qbuild
    qbuild.build()
    import block_quantized_weight_qgemv_gb300 as q

    hbm_peak, bf16_peak, bf16_sus, peak_src = measured_peaks()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))

    wl = WORKLOAD
    fmt, nrows, ncols, batch = wl["fmt"], wl["nrows"], wl["ncols"], wl["batch"]
    wbytes = nrows * (ncols // 32) * BLOCK_BYTES[fmt]
    step_bytes = gemv_bytes(fmt, nrows, ncols, batch)
    ncopy = max(2, math.ceil(2.5 * l2 / wbytes))
    Wn = qsynth.make_weights(fmt, nrows, ncols, seed=2024 + rank)
    xn = qsynth.make_x(batch, ncols, seed=2025 + rank)
    W0 = torch.from_numpy(Wn).to(dev)
    Ws = [W0] + [W0.clone() for _ in range(ncopy - 1)]
    x = torch.from_numpy(xn).to(dev)
    y = torch.empty(batch, nrows, dtype=torch.float32, device=dev)
    fn = getattr(q, "qgemv_" + fmt)
    # a stream of GEMVs over fixed weights: W is never written by the kernel
    # before a GEMV, so its copies may start before that kernel has finished
    q.qgemv_set_option(q.OPT_WEIGHTS_STATIC, 1)

    def launch(i):
        fn(Ws[i % ncopy], x, y, nrows, ncols, batch)

    # warmup (eager, also initializes the library's per-device state)
    for i in range(max(args.warmup, 3)):
        launch(i)
    torch.cuda.synchronize()
    q.qgemv_sync_check()

    chunk = min(args.steps, 2000)
    graphs, _ = build_graphs(torch, launch, args.steps, chunk, timed_events=False)
    # one launch at a time (event pairs between launches break the overlap)
    iso_graphs, pairs = build_graphs(torch, launch, min(args.steps, 200), 200, timed_events=True)
    iso_graphs[0][0].replay()
    torch.cuda.synchronize()
    # warm the graphs (untimed)
    for g, _ in graphs[:2]:
        g.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    barrier(torch, world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    hold_stream(torch)
    s0.record()
    for g, _ in graphs:
        g.replay()
    s1.record()
    torch.cuda.synchronize()
    barrier(torch, world)
    clk = clocks.stop()
    elapsed_ms = s0.elapsed_time(s1)
    elapsed_ms = max_over_ranks(torch, world, elapsed_ms, dev)
    q.qgemv_sync_check()

    durs = [a.elapsed_time(b) for a, b in pairs] if pairs else []
    iso_ms = statistics.mean(durs) if durs else None
    kern_ms = elapsed_ms / args.steps
    value = replica_value(step_bytes, args.steps, world, elapsed_ms * 1e-3)
    achieved = step_bytes / (kern_ms * 1e-3) / 1e9

    # ---- e2e through the public API with host buffers
    e2e_steps = min(args.steps, 2000)
    x_host = [torch.from_numpy(qsynth.make_x(batch, ncols, seed=3000 + i)).pin_memory() for i in range(8)]
    y_host = torch.empty(batch, nrows, dtype=torch.float32).pin_memory()
    for i in range(5):
        x.copy_(x_host[i % 8], non_blocking=True)
        launch(i)
        y_host.copy_(y, non_blocking=True)
    torch.cuda.synchronize()
    barrier(torch, world)
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        x.copy_(x_host[i % 8], non_blocking=True)
        launch(i)
        y_host.copy_(y, non_blocking=True)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(torch, world, time.perf_counter() - t0, dev)
    e2e_value = replica_value(step_bytes, e2e_steps, world, e2e_s)

    # ---- CPU baseline: the oracle on the host cores (rank 0 only)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        cores = host_cores()
        gbs, rows_done, el = oracle_rate(oracle, fmt, Wn, xn, nrows, ncols, batch, args.cpu_seconds, cores)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": "%d random rows of the %dx%d workload in %.1f s (C oracle, fp64, OpenMP %d threads)" % (
                   rows_done, nrows, ncols, el, cores)}

    extras = {}
    if rank == 0 and not args.no_extras:
        extras = run_extras(torch, q, dev, l2, hbm_peak, bf16_peak)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16*f16->f32",
        "dtype_note": "tensor-core MMA on fp16 operands (the weights' exact integer codes; x scaled per "
                      "128 values by a power of two) with fp32 accumulation; fp32 x and y",
        "data": "synthetic",
        "config": {"workload": wl["name"], "fmt": fmt, "nrows": nrows, "ncols": ncols, "batch": batch,
                   "bytes_per_step": step_bytes,
                   "l2": "inputs larger than L2: %d rotating weight copies (%.0f MB > %.0f MB L2)" % (
                       ncopy, ncopy * wbytes / 1e6, l2 / 1e6),
                   "launch": "CUDA graphs of up to %d library calls, programmatic dependent launch, "
                             "weights declared static" % chunk,
                   "parallelism": "replicas" if world > 1 else "single-gpu"},
        "pct_of_hbm_nominal": round(value / HBM_NOMINAL_GBS, 4),
        "pct_of_hbm_measured": round(value / hbm_peak, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4),
                     "traffic": args.traffic if args.traffic is not None else NCU_TRAFFIC_BYTES,
                     "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs, copy burst)",
                     "kernel_ms": round(kern_ms, 6),
                     "kernel_ms_isolated": round(iso_ms, 6) if iso_ms is not None else None},
        "e2e": {"value": round(e2e_value, 3), "unit": "GB/s", "h2d_bytes_per_step": 4 * batch * ncols,
                "d2h_bytes_per_step": 4 * batch * nrows,
                "note": "public Python API, eager launches, W resident, x/y via pinned host buffers"},
        "gpu_launches": args.steps * world,
        "clocks": clk,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if extras:
        line["other_configs"] = extras
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def hold_stream(torch):
    """Queue a ~1.5 ms spin kernel on the current stream: the start event and
    the launches queued after it then run back to back on the device instead
    of waiting for the host to submit them."""
    torch.cuda._sleep(3_000_000)


def time_graph(torch, launch, n, reps):
    """(ms per launch in a graph of n back-to-back launches, ms of one launch
    bracketed by events on its own)."""
    # eager first call: lazily created per-device state (e.g. the prefill
    # workspace) must exist before stream capture
    launch(0)
    torch.cuda.synchronize()
    graphs, _ = build_graphs(torch, launch, n, n, timed_events=False)
    iso, pairs = build_graphs(torch, launch, n, n, timed_events=True)
    g = graphs[0][0]
    g.replay()
    iso[0][0].replay()
    torch.cuda.synchronize()
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    hold_stream(torch)
    s0.record()
    for _ in range(reps):
        g.replay()
    s1.record()
    torch.cuda.synchronize()
    per_step = s0.elapsed_time(s1) / (n * reps)
    iso_ms = statistics.mean(a.elapsed_time(b) for a, b in pairs)
    return per_step, iso_ms


def run_extras(torch, q, dev, l2, hbm_peak, bf16_peak):
    """The other configurations, timed briefly (graph replays, events)."""
    out = {}
    # GEMV: both FFN shapes, all formats, batch 1/2/4/8, plus the 4096x4096 projection
    shapes = [("q4_0", 4096, 4096)] + [(f, r, c) for f in ("q4_0", "q4_1", "q8_0")
                                       for (r, c) in ((14336, 4096), (4096, 14336))]
    for fmt, nrows, ncols in shapes:
        Wn = qsynth.make_weights(fmt, nrows, ncols, seed=7)
        wbytes = Wn.size
        ncopy = max(2, math.ceil(2.5 * l2 / wbytes))
        W0 = torch.from_numpy(Wn).to(dev)
        Ws = [W0] + [W0.clone() for _ in range(ncopy - 1)]
        fn = getattr(q, "qgemv_" + fmt)
        for batch in ((1,) if ncols == nrows else (1, 2, 4, 8)):
            x = torch.randn(batch, ncols, device=dev)
            y = torch.empty(batch, nrows, device=dev)
            per, iso = time_graph(torch, lambda i: fn(Ws[i % ncopy], x, y, nrows, ncols, batch), 200, 5)
            b = gemv_bytes(fmt, nrows, ncols, batch)
            out["gemv_%s_%dx%d_b%d" % (fmt, nrows, ncols, batch)] = {
                "GBps": round(b / (per * 1e-3) / 1e9, 1),
                "frac_hbm_measured": round(b / (per * 1e-3) / 1e9 / hbm_peak, 4),
                "us_per_call": round(per * 1e3, 3), "us_isolated": round(iso * 1e3, 3),
                "rows_per_s": round(nrows * batch / (per * 1e-3), 1),
                "TFLOPs": round(2 * nrows * ncols * batch / (per * 1e-3) / 1e12, 3)}
        del Ws, W0
        torch.cuda.empty_cache()
    # quantized-activation GEMV (int8 activations, integer dot products): the
    # one-call form (quantizer + GEMV) and the GEMV alone on quantized x
    for fmt, nrows, ncols in [(f, r, c) for f in ("q4_0", "q4_1", "q8_0") for (r, c) in ((4096, 14336), (14336, 4096))]:
        Wn = qsynth.make_weights(fmt, nrows, ncols, seed=7)
        wbytes = Wn.size
        ncopy = max(2, math.ceil(2.5 * l2 / wbytes))
        W0 = torch.from_numpy(Wn).to(dev)
        Ws = [W0] + [W0.clone() for _ in range(ncopy - 1)]
        fn = getattr(q, "qgemv_mmvq_" + fmt)
        fxq = getattr(q, "qgemv_mmvq_xq_" + fmt)
        for batch in (1, 8):
            x = torch.randn(batch, ncols, device=dev)
            y = torch.empty(batch, nrows, device=dev)
            xq = torch.empty(q.q8_1_size(ncols, batch), dtype=torch.uint8, device=dev)
            q.qquantize_q8_1(x, xq, ncols, batch)
            per, iso = time_graph(torch, lambda i: fn(Ws[i % ncopy], x, y, nrows, ncols, batch), 200, 5)
            per_g, iso_g = time_graph(torch, lambda i: fxq(Ws[i % ncopy], xq, y, nrows, ncols, batch), 200, 5)
            b = gemv_bytes(fmt, nrows, ncols, batch)
            bg = wbytes + q.q8_1_size(ncols, batch) + 4 * batch * nrows
            out["mmvq_%s_%dx%d_b%d" % (fmt, nrows, ncols, batch)] = {
                "GBps": round(b / (per * 1e-3) / 1e9, 1),
                "frac_hbm_measured": round(b / (per * 1e-3) / 1e9 / hbm_peak, 4),
                "us_per_call": round(per * 1e3, 3), "us_isolated": round(iso * 1e3, 3),
                "gemv_only_GBps": round(bg / (per_g * 1e-3) / 1e9, 1),
                "gemv_only_frac_hbm_measured": round(bg / (per_g * 1e-3) / 1e9 / hbm_peak, 4),
                "gemv_only_us_per_call": round(per_g * 1e3, 3), "gemv_only_us_isolated": round(iso_g * 1e3, 3)}
        del Ws, W0
        torch.cuda.empty_cache()
    # expert-selected GEMV: a stack of 8 experts (Mixtral-style FFN), one
    # token's top-2 experts for the up projection (2 columns sharing x) and the
    # down projection (one x row per column), and 8 tokens x top-2 (16 columns
    # grouped by expert on the device); and 256 experts (DeepSeek-style, hidden
    # 7168, expert width 2048), one token's top-8.  Calls rotate over disjoint
    # expert sets (1 token) or two id sets (8 tokens) so that each reads W from
    # HBM.  Bytes: the distinct experts' matrices + x + y.
    # (format, rows, cols, tokens, experts, top-k, up/gate projection)
    for fmt, nrows, ncols, ntok, n_expert, top_k, up in [
            ("q4_0", 14336, 4096, 1, 8, 2, True), ("q4_0", 4096, 14336, 1, 8, 2, False),
            ("q4_1", 14336, 4096, 1, 8, 2, True), ("q8_0", 14336, 4096, 1, 8, 2, True),
            ("q4_0", 14336, 4096, 8, 8, 2, True),
            ("q4_0", 2048, 7168, 1, 256, 8, True), ("q4_0", 7168, 2048, 1, 256, 8, False)]:
        ebytes = nrows * (ncols // 32) * {"q4_0": 18, "q4_1": 20, "q8_0": 34}[fmt]
        W = torch.from_numpy(qsynth.make_weights(fmt, n_expert * nrows, ncols, seed=17)).to(dev)
        batch = ntok * top_k
        x_group = top_k if up else 1           # up/gate: a token's experts share its x; down: one row per column
        g = np.random.default_rng(19)
        if ntok == 1:
            # disjoint expert sets, rotated so that each call reads its experts from HBM
            sets = [np.arange(top_k * i, top_k * (i + 1), dtype=np.int32) % n_expert for i in range(max(4, min(32, n_expert // top_k)))]
        else:
            sets = [np.concatenate([g.choice(n_expert, top_k, replace=False) for _ in range(ntok)]).astype(np.int32)
                    for _ in range(2)]
        ids = [torch.from_numpy(v).to(dev) for v in sets]
        x = torch.randn(batch // x_group, ncols, device=dev)
        y = torch.empty(batch, nrows, device=dev)
        fn = getattr(q, "qgemv_id_" + fmt)
        per, iso = time_graph(torch, lambda i: fn(W, n_expert, ids[i % len(ids)], x, y, nrows, ncols, batch,
                                                  x_group=x_group), 200, 5)
        distinct = statistics.mean(len(set(v.tolist())) for v in sets)
        b = distinct * ebytes + 4 * x.numel() + 4 * y.numel()
        out["gemv_id_%s_%dx%d_E%d_tok%d_top%d" % (fmt, nrows, ncols, n_expert, ntok, top_k)] = {
            "GBps": round(b / (per * 1e-3) / 1e9, 1),
            "frac_hbm_measured": round(b / (per * 1e-3) / 1e9 / hbm_peak, 4),
            "us_per_call": round(per * 1e3, 3), "us_isolated": round(iso * 1e3, 3),
            "experts_read_per_call": distinct, "columns": batch}
        del W
        torch.cuda.empty_cache()
    # standalone dequant of 2^27 elements (4096 x 32768), Q4_0 and Q8_0, to fp16 and fp32
    nrows, ncols = 4096, 32768
    for fmt in ("q4_0", "q8_0"):
        W = torch.from_numpy(qsynth.make_weights(fmt, nrows, ncols, seed=11)).to(dev)
        fn = getattr(q, "qdequant_" + fmt)
        for dt, esz in ((torch.float16, 2), (torch.float32, 4)):
            o = torch.empty(nrows, ncols, dtype=dt, device=dev)
            per, iso = time_graph(torch, lambda i: fn(W, o, nrows, ncols), 20, 3)
            b = W.numel() + nrows * ncols * esz
            out["dequant_%s_%s_2p27" % (fmt, "f16" if esz == 2 else "f32")] = {
                "GBps": round(b / (per * 1e-3) / 1e9, 1), "frac_hbm_measured": round(b / (per * 1e-3) / 1e9 / hbm_peak, 4),
                "us_per_call": round(per * 1e3, 2), "us_isolated": round(iso * 1e3, 2)}
            del o
        del W
        torch.cuda.empty_cache()
    # prefill: 14336 x 4096 weights, 512 tokens, each format
    nrows, ncols, m = 14336, 4096, 512
    X = torch.randn(m, ncols, device=dev).to(torch.bfloat16)
    Y = torch.empty(m, nrows, device=dev)
    flops = 2.0 * nrows * ncols * m
    for fmt in ("q4_0", "q4_1", "q8_0"):
        W = torch.from_numpy(qsynth.make_weights(fmt, nrows, ncols, seed=13)).to(dev)
        fn = getattr(q, "qgemm_" + fmt)
        per, iso = time_graph(torch, lambda i: fn(W, X, Y, nrows, ncols, m), 10, 3)
        out["prefill_%s_14336x4096_m512" % fmt] = {
            "TFLOPs": round(flops / (per * 1e-3) / 1e12, 2),
            "frac_bf16_measured": round(flops / (per * 1e-3) / 1e12 / bf16_peak, 4),
            "us_per_call": round(per * 1e3, 2), "us_isolated": round(iso * 1e3, 2)}
        del W
    return out


def profile_call(argv):
    """Entry-point calls for a profiler capture (see the module docstring)."""
    import torch

    from block_quantized_weight_qgemv_gb300 import build as qbuild
    qbuild.build()
    import block_quantized_weight_qgemv_gb300 as q

    what, fmt = argv[0], argv[1]
    dims = [int(v) for v in argv[2:]]
    if what == "gemv":
        nrows, ncols, batch = dims
        Wn = qsynth.make_weights(fmt, nrows, ncols, 1)
        copies = [torch.from_numpy(Wn).cuda() for _ in range(4)]
        x = torch.from_numpy(qsynth.make_x(batch, ncols, 2)).cuda()
        y = torch.empty(batch, nrows, device="cuda")
        for i in range(6):
            getattr(q, "qgemv_" + fmt)(copies[i % 4], x, y, nrows, ncols, batch)
    elif what in ("mmvq", "mmvq_xq"):
        nrows, ncols, batch = dims
        Wn = qsynth.make_weights(fmt, nrows, ncols, 1)
        copies = [torch.from_numpy(Wn).cuda() for _ in range(4)]
        x = torch.from_numpy(qsynth.make_x(batch, ncols, 2)).cuda()
        y = torch.empty(batch, nrows, device="cuda")
        xq = torch.empty(q.q8_1_size(ncols, batch), dtype=torch.uint8, device="cuda")
        q.qquantize_q8_1(x, xq, ncols, batch)
        for i in range(6):
            if what == "mmvq":
                getattr(q, "qgemv_mmvq_" + fmt)(copies[i % 4], x, y, nrows, ncols, batch)
            else:
                getattr(q, "qgemv_mmvq_xq_" + fmt)(copies[i % 4], xq, y, nrows, ncols, batch)
    elif what == "id":
        nrows, ncols, n_expert, batch, x_group = dims
        W = torch.from_numpy(qsynth.make_weights(fmt, n_expert * nrows, ncols, 1)).cuda()
        x = torch.from_numpy(qsynth.make_x(batch // x_group, ncols, 2)).cuda()
        y = torch.empty(batch, nrows, device="cuda")
        for i in range(6):
            ids = torch.tensor([(i * batch + b) % n_expert for b in range(batch)], dtype=torch.int32, device="cuda")
            getattr(q, "qgemv_id_" + fmt)(W, n_expert, ids, x, y, nrows, ncols, batch, x_group=x_group)
    elif what == "dequant":
        nrows, ncols = dims
        W = torch.from_numpy(qsynth.make_weights(fmt, nrows, ncols, 1)).cuda()
        out = torch.empty(nrows, ncols, dtype=torch.float16, device="cuda")
        for _ in range(4):
            getattr(q, "qdequant_" + fmt)(W, out, nrows, ncols)
    elif what == "gemm":
        nrows, ncols, m = dims
        W = torch.from_numpy(qsynth.make_weights(fmt, nrows, ncols, 1)).cuda()
        X = torch.from_numpy(qsynth.make_X_bf16(m, ncols, 2).view(np.int16)).cuda()
        Y = torch.empty(m, nrows, device="cuda")
        for _ in range(4):
            getattr(q, "qgemm_" + fmt)(W, X.view(torch.bfloat16), Y, nrows, ncols, m)
    else:
        raise SystemExit("unknown operation %r" % what)
    torch.cuda.synchronize()
    q.qgemv_sync_check()
    print("ok")
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes (read+write) per launch of the GEMV kernel, if captured")
    ap.add_argument("--profile-call", nargs="+", metavar="ARG",
                    help="OP FMT DIMS...: a few calls of one entry point for a profiler capture, then exit")
    args = ap.parse_args()
    if args.profile_call:
        return profile_call(args.profile_call)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
