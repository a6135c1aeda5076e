#!/usr/bin/env python3
"""Benchmark of the GB300 GEMV c = B @ a (one JSON line on stdout).

Workload: n=7168, k=16384, fp16 B (row-major) and fp16 a, fp32 accumulate,
fp16 output; B normal(0, 0.02), a normal(0, 1), seed 0 -- about 235 MB of B
per call.  A step is one call of the whole path (one GEMV).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
    python bench.py --sweep OUT.jsonl     # every workload shape, one line each

Timing: W untimed calls, then K plain gemv() calls (the public entry point,
as a caller makes it) bracketed by a barrier and torch.cuda.synchronize() on
both sides, with CUDA events on the launching stream at both ends.  Consecutive calls alternate between two copies of B,
each larger than the 129 MB L2, so no call finds its B in L2.  value = bytes
of all ranks / the slowest rank's elapsed time; bytes per call are the
algorithmic n*k*2 + k*2 + n*out_bytes (B read once, a once, c written once),
the count TileLang Case Studies Case C uses (66 us <-> 3.55 TB/s at this
shape).  Under torchrun each rank runs an independent replica (the GEMV is
one device's work; nothing is exchanged).

--impl reference times the oracle (a single-threaded C fp64 loop) on the host
cores on a bounded sample of rows of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMV achieved HBM GB/s and % of GB300 peak (µs/call) at n×k fp16/bf16"
WORKLOAD = dict(n=7168, k=16384, dtype="f16", out_fp32=False, dist="normal", seed=0)
WORKLOAD_DESC = ("gemv n=7168 k=16384: fp16 B row-major and fp16 a, fp32 accumulate, fp16 output; "
                 "B normal(0,0.02), a normal(0,1), seed 0")
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1000 * 1000
# Best figure the pages give for this exact workload (fp16, 7168x16384):
# TileLang Case Studies, Case B.2 table, O1+O2 on an H200: 3.67 TB/s.
PAGES_BEST_GBS = 3670.0
# Queue prefill before a timed batch: a sleep kernel of this many SM clock
# cycles (~1.5 ms at 2 GHz) ahead of the first event, long enough for the
# host to enqueue hundreds of calls before the GPU reaches the first.
PREFILL_CYCLES = 3_000_000
# Calls of the benchmark workload (~0.45 s) run right after the timed region,
# inside the clock sampler's window.
CLOCK_WINDOW_CALLS = 13_500
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

SWEEP_SHAPES = (
    [(256, 512, "f16", False, "uniform")]
    + [(7168, 16384, "f16", False, "normal"), (18432, 7168, "bf16", False, "normal"),
       (18432, 7168, "bf16", True, "normal")]
    + [(n, k, "bf16", False, "normal") for n, k in ((4096, 4096), (14336, 4096), (4096, 14336), (28672, 8192))]
    + [(n, k, dt, False, "uniform") for dt in ("f16", "bf16") for n in (1024, 4099, 18433, 65536)
       for k in (1000, 4096, 7169, 16384)]
    + [(57344, 7168, dt, False, "normal") for dt in ("f16", "bf16")]
)


# ------------------------------------------------------------ arithmetic --

def algorithmic_bytes(n: int, k: int, in_bytes: int = 2, out_bytes: int = 2) -> int:
    """B read once, a read once, c written once."""
    return n * k * in_bytes + k * in_bytes + n * out_bytes


def frac_of_peak(achieved: float, peak: float) -> float:
    return achieved / peak


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# Sources that make up the device code of the tiles kernel (the kernel the
# benchmark times and whose ncu capture gives `roofline.traffic`): its
# translation units and every header they include.
KERNEL_SOURCES = ("gemv_internal.h", "gemv_kernels.cuh", "gemv_tiles.cuh", "gemv_kernels_f16.cu",
                  "gemv_kernels_bf16.cu")
# ... and of the bulk kernel, which shares them.
BULK_SOURCES = KERNEL_SOURCES + ("gemv_bulk.cuh", "gemv_bulk_f16.cu", "gemv_bulk_bf16.cu")


def kernel_source_digest(names=KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "memory_bound_gemv_02_gb300", "csrc")
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def launch_signature(cfg: dict) -> str:
    """The launch configuration a profile was taken with."""
    return " ".join(f"{kk}={cfg[kk]}" for kk in ("variant", "rows_per_warp", "unroll", "warps_per_cta",
                                                 "warp_split", "grid_split", "ctas", "stages"))


def profiled_traffic(workload_tag: str, cfg: dict):
    """DRAM bytes per launch from the committed ncu summary of this workload,
    if it was taken on the current kernel sources and the launch
    configuration ``cfg`` (else None)."""
    path = os.path.join(ROOT, "profiles", f"gemv_{workload_tag}.md")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    vals = {}
    for line in lines:
        if line.startswith("- ") and ":" in line:
            key, _, v = line[2:].partition(":")
            vals[key.strip()] = v.strip().strip("`")
    if vals.get("source_digest") != kernel_source_digest() or vals.get("launch") != launch_signature(cfg):
        return None
    try:
        return int(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def parse_clock_rows(header_line: str, row_lines) -> dict:
    """Summarise nvidia-smi clock samples: a CSV header and data lines."""
    header = [h.strip() for h in next(csv.reader([header_line]))] if header_line else []
    data = [[c.strip() for c in r] for r in csv.reader(list(row_lines)) if len(r) == len(header)]

    def col(*prefixes):
        for prefix in prefixes:
            for i, h in enumerate(header):
                if h.startswith(prefix):
                    return i
        return None

    def num(s):
        try:
            return float(s.split()[0])
        except (ValueError, IndexError):
            return None

    i_sm, i_max = col("clocks.current.sm", "clocks.sm"), col("clocks.max.sm")
    sms = [v for v in (num(r[i_sm]) for r in data) if v is not None] if i_sm is not None else []
    maxs = [v for v in (num(r[i_max]) for r in data) if v is not None] if i_max is not None else []
    reasons = set()
    for name in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"):
        i = col(f"clocks_event_reasons.{name}")
        if i is not None and any(r[i].lower().startswith("active") for r in data):
            reasons.add(name)
    return {"sm_mhz": statistics.median(sms) if sms else None,
            "sm_max_mhz": max(maxs) if maxs else None,
            "reasons": sorted(reasons), "samples": len(sms)}


class ClockSampler:
    """nvidia-smi clock samples every 200 ms, stamped with host time."""

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.lines = []
        self.stamps = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={CLOCK_QUERY}", "--format=csv",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
        except OSError:
            self.proc = None
            return self
        import threading

        def reader():
            for line in self.proc.stdout:
                self.lines.append(line.rstrip("\n"))
                self.stamps.append(time.time())
        self.th = threading.Thread(target=reader, daemon=True)
        self.th.start()
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.th.join(timeout=2)

    def summary(self, t0, t1, label="timed region"):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        header = self.lines[0]
        rows = [(ln, t) for ln, t in zip(self.lines[1:], self.stamps[1:]) if ln != header]
        inside = [ln for ln, t in rows if t0 <= t <= t1]
        out = parse_clock_rows(header, inside if inside else [ln for ln, _ in rows])
        out["window"] = label if inside else f"whole run (no sample fell inside the {label})"
        return out


# --------------------------------------------------------------- ranks --

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------- CPU oracle leg --

def oracle_rows_rate(B_bits, a_bits, fmt, budget_s: float, rows_cap=None):
    """Run the oracle over rows of B until ~budget_s of CPU time; return
    (rows done, seconds).  Single thread."""
    import numpy as np

    import oracle
    n = B_bits.shape[0]
    t0 = time.perf_counter()
    oracle.gemv_ref(np.ascontiguousarray(B_bits[:8]), a_bits, fmt)
    per_row = max((time.perf_counter() - t0) / 8, 1e-7)
    done, spent, start = 0, 0.0, 0
    while spent < budget_s and (rows_cap is None or done < rows_cap):
        m = int(min(max(1, (budget_s - spent) / per_row), n - start, 4096))
        if rows_cap is not None:
            m = min(m, rows_cap - done)
        t1 = time.perf_counter()
        oracle.gemv_ref(np.ascontiguousarray(B_bits[start:start + m]), a_bits, fmt)
        spent += time.perf_counter() - t1
        done += m
        start = (start + m) % n
    return done, spent


def cpu_baseline(B_bits, a_bits, fmt, n, k, out_bytes, budget_s=12.0):
    rows, secs = oracle_rows_rate(B_bits, a_bits, fmt, budget_s)
    bytes_done = rows * k * 2 + k * 2 + rows * out_bytes
    return {"value": round(bytes_done / secs / 1e9, 4), "unit": "GB/s", "cores": 1,
            "host_cores": os.cpu_count(), "kind": "oracle",
            "us_per_call": round(secs / (rows / n) * 1e6, 1),
            "sample": f"{rows} rows of the {n}x{k} matrix ({rows / n:.2f} passes), "
                      f"{secs:.1f} s single-threaded fp64 C loop on 1 of {os.cpu_count()} host cores"}


# ---------------------------------------------------------- reference arm --

def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import numpy as np
    import torch

    from memory_bound_gemv_02_gb300 import inputs
    import oracle
    w = WORKLOAD
    n, k = w["n"], w["k"]
    B, a = inputs.make_inputs(n, k, w["dtype"], w["dist"], w["seed"], "cpu")
    B_bits, a_bits = inputs.to_bits(B), inputs.to_bits(a)
    del B
    oracle.build()
    total = args.steps + args.warmup
    t0 = time.perf_counter()
    oracle.gemv_ref(np.ascontiguousarray(B_bits[:8]), a_bits, w["dtype"])
    per_row = max((time.perf_counter() - t0) / 8, 1e-7)
    budget = float(os.environ.get("GEMV_REFERENCE_BUDGET_S", "120"))
    m = int(max(1, min(n, budget / total / per_row)))
    start = 0
    for _ in range(args.warmup):
        oracle.gemv_ref(np.ascontiguousarray(B_bits[start:start + m]), a_bits, w["dtype"])
        start = (start + m) % max(1, n - m + 1)
    t1 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gemv_ref(np.ascontiguousarray(B_bits[start:start + m]), a_bits, w["dtype"])
        start = (start + m) % max(1, n - m + 1)
    secs = time.perf_counter() - t1
    bytes_step = m * k * 2 + k * 2 + m * 2
    value = bytes_step * args.steps / secs / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC, "sample_rows_per_step": m},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "host_cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"{m} rows of {n} per step, single-threaded fp64 C loop on 1 of "
                                   f"{os.cpu_count()} host cores"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------- our arm --

def time_calls(L, calls, stream, steps, warmup):
    """Run `calls` round-robin; return (elapsed_s, per-launch durations in ms)."""
    import torch
    for i in range(warmup):
        fn, args = calls[i % len(calls)]
        st = fn(*args)
        if st != 0:
            raise RuntimeError(f"gemv failed with status {st}")
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s = torch.cuda.current_stream()
    torch.cuda._sleep(PREFILL_CYCLES)  # keep the GPU busy while the launches queue up
    e0.record(s)
    for i in range(steps):
        fn, args = calls[i % len(calls)]
        starts[i].record(s)
        fn(*args)
        ends[i].record(s)
    e1.record(s)
    torch.cuda.synchronize()
    per = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    return e0.elapsed_time(e1) / 1e3, per


def time_batch(calls, steps, warmup, prefill=True):
    """Run `calls` round-robin back to back with CUDA events only at both
    ends of the batch; return the elapsed seconds.  ``prefill``: a sleep
    kernel ahead of the first event keeps the GPU busy while the launches
    queue up."""
    import torch
    for i in range(warmup):
        fn, args = calls[i % len(calls)]
        if fn(*args) != 0:
            raise RuntimeError("gemv failed")
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s = torch.cuda.current_stream()
    if prefill:
        torch.cuda._sleep(PREFILL_CYCLES)
    e0.record(s)
    for i in range(steps):
        fn, args = calls[i % len(calls)]
        fn(*args)
    e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3


def host_overhead_us(L, n, k, dt, dev, stream):
    """Host time of one cached-key gemv() call (enqueue only), in bursts of
    200 calls so the launch queue never fills; median over bursts."""
    import torch
    B = torch.zeros((n, k), dtype=torch.float16, device=dev)
    a = torch.zeros(k, dtype=torch.float16, device=dev)
    c = torch.empty(n, dtype=torch.float16, device=dev)
    args = (B.data_ptr(), a.data_ptr(), c.data_ptr(), n, k, dt, stream)
    L.gemv(*args)
    torch.cuda.synchronize()
    per = []
    for _ in range(30):
        t0 = time.perf_counter()
        for _ in range(200):
            L.gemv(*args)
        per.append((time.perf_counter() - t0) / 200)
        torch.cuda.synchronize()
    return statistics.median(per) * 1e6


def native_measurements(b_bytes: int):
    """The library's native measurement tool (C++): host microseconds per
    cached gemv() call and per empty-kernel launch (steady_clock, 10^4
    calls), and the read-only streaming bandwidth back to back over two 1
    GiB buffers and over two buffers of ``b_bytes`` (plain launches, and
    programmatic launches that overlap completely); None if the tool is not
    built."""
    from memory_bound_gemv_02_gb300 import _build
    if not os.path.exists(_build.HOST_TOOL):
        return None
    r = subprocess.run([_build.HOST_TOOL, str(b_bytes)], capture_output=True, text=True, timeout=300)
    if r.returncode != 0:
        raise RuntimeError(f"native measurement tool failed: {r.stdout} {r.stderr}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def bench_shape(g, L, n, k, dtype, out_fp32, dist, seed, steps, warmup, dev, variant=0):
    """One shape: µs per call four ways -- isolated (CUDA events around each
    launch), back to back, back to back as gemv() launches (programmatic
    dependent launch, first tile prefetched into L2 before the wait), and
    back to back with the first tile read before the wait (B promised
    unwritten) -- and the launch configuration.  ``variant``: a
    GEMV_VARIANT_* forced on every call (0: the planner's choice)."""
    import torch

    from memory_bound_gemv_02_gb300 import inputs
    out_bytes = 4 if out_fp32 else 2
    nbytes = algorithmic_bytes(n, k, 2, out_bytes)
    B, a = inputs.make_inputs(n, k, dtype, dist, seed, dev)
    copies = max(2, min(16, -(-3 * L2_BYTES // max(1, n * k * 2))))
    Bs = [B] + [B.clone() for _ in range(copies - 1)]
    c = torch.empty(n, dtype=torch.float32 if out_fp32 else B.dtype, device=dev)
    dt = g.dtype_code(B.dtype, out_fp32)
    s = torch.cuda.current_stream().cuda_stream
    fc = g.GemvConfig()  # overlap 0: plain launches
    fc.variant = variant
    g.gemv_ex(B, a, c=c, out_fp32=out_fp32, config=fc)
    cfg = g.gemv_last_config()
    plain = [(L.gemv_ex, (Bx.data_ptr(), a.data_ptr(), c.data_ptr(), n, k, dt, ctypes.byref(fc), s))
             for Bx in Bs]
    ov = g.GemvConfig()
    ov.variant = variant
    ov.overlap = g.GEMV_OVERLAP_PDL_PREFETCH_B
    pdl = [(L.gemv_ex, (Bx.data_ptr(), a.data_ptr(), c.data_ptr(), n, k, dt, ctypes.byref(ov), s)) for Bx in Bs]
    dc = g.GemvConfig()
    dc.variant = variant
    dc.overlap = g.GEMV_OVERLAP_PDL
    dflt = [(L.gemv_ex, (Bx.data_ptr(), a.data_ptr(), c.data_ptr(), n, k, dt, ctypes.byref(dc), s)) for Bx in Bs]
    _, per = time_calls(L, plain, s, steps, warmup)
    el_plain = time_batch(plain, steps, warmup)
    el_pdl = time_batch(pdl, steps, warmup)
    el_dflt = time_batch(dflt, steps, warmup)
    iso = statistics.median(per) * 1e3
    b2b = el_plain / steps * 1e6
    b2b_pdl = el_pdl / steps * 1e6
    return {"n": n, "k": k, "dtype": dtype, "out": "f32" if out_fp32 else dtype, "dist": dist,
            "bytes": nbytes, "b_copies": copies,
            "us_isolated_median": round(iso, 3), "us_isolated_min": round(min(per) * 1e3, 3),
            "us_isolated_p90": round(sorted(per)[int(0.9 * (len(per) - 1))] * 1e3, 3),
            "stddev_over_median": round(statistics.pstdev(per) / statistics.median(per), 4),
            "us_back_to_back": round(b2b, 3), "us_back_to_back_pdl": round(b2b_pdl, 3),
            "us_back_to_back_default": round(el_dflt / steps * 1e6, 3),
            "gbs_isolated": round(nbytes / iso / 1e3, 1), "gbs_back_to_back": round(nbytes / b2b / 1e3, 1),
            "gbs_back_to_back_pdl": round(nbytes / b2b_pdl / 1e3, 1),
            "config": {kk: cfg[kk] for kk in ("variant", "rows_per_warp", "unroll", "warps_per_cta",
                                              "warp_split", "grid_split", "ctas", "stages")}}


def torch_mv_us(n, k, dtype, out_fp32, dist, dev, steps):
    """torch.mv on the same shape (back to back over copies of B larger than
    L2; output in the input type), for context."""
    import torch

    from memory_bound_gemv_02_gb300 import inputs
    B, a = inputs.make_inputs(n, k, dtype, dist, 0, dev)
    copies = max(2, min(16, -(-3 * L2_BYTES // max(1, n * k * 2))))
    Bs = [B] + [B.clone() for _ in range(copies - 1)]
    outs = [torch.empty(n, dtype=B.dtype, device=dev) for _ in Bs]
    def mv(Bx, o):
        torch.mv(Bx, a, out=o)
        return 0

    el = time_batch([(mv, (Bx, o)) for Bx, o in zip(Bs, outs)], steps, 10)
    del Bs, outs
    return el / steps * 1e6


def run_sweep(args, dev):
    import torch

    import memory_bound_gemv_02_gb300 as g
    L = g.lib()
    peak, kind = measured_peak()
    out = open(args.sweep, "w")
    for n, k, dtype, out_fp32, dist in SWEEP_SHAPES:
        r = bench_shape(g, L, n, k, dtype, out_fp32, dist, 0, args.sweep_steps, 20, dev)
        r["pct_of_8tbps_pdl"] = round(100 * r["gbs_back_to_back_pdl"] / NOMINAL_HBM_GBS, 1)
        r[f"frac_of_{kind}_peak_pdl"] = round(r["gbs_back_to_back_pdl"] / peak, 4)
        # the same shape with B staged through shared memory (bulk variant)
        rb = bench_shape(g, L, n, k, dtype, out_fp32, dist, 0, args.sweep_steps, 20, dev,
                         variant=g.GEMV_VARIANT_BULK)
        r["bulk"] = {kk: rb[kk] for kk in ("us_isolated_median", "us_back_to_back", "us_back_to_back_pdl",
                                           "us_back_to_back_default", "gbs_back_to_back_pdl", "config")}
        # context only (never a target): torch.mv (cuBLAS) on the same shape and box
        r["torch_mv_us_back_to_back"] = round(torch_mv_us(n, k, dtype, out_fp32, dist, dev, args.sweep_steps), 3)
        out.write(json.dumps(r) + "\n")
        out.flush()
        print(json.dumps(r), file=sys.stderr, flush=True)
        torch.cuda.empty_cache()
    out.close()
    return 0


GLA_WORKLOADS = [(2048, 128, 128, "bf16"), (2048, 128, 128, "f32"), (1024, 256, 256, "bf16"), (4096, 64, 64, "f16"),
                 (8192, 64, 64, "bf16"), (4096, 128, 128, "bf16"), (16384, 16, 64, "f16")]


def run_gla(args, dev):
    """GLA decode step (gla_decode): one JSON line per workload on stderr and
    the list on stdout.  Each call updates one head-state buffer in place;
    calls rotate over copies so that no call finds its state in L2."""
    import torch

    import memory_bound_gemv_02_gb300 as g
    L = g.lib()
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
    code = {"f16": g.GLA_F16, "bf16": g.GLA_BF16, "f32": g.GLA_F32}
    s = torch.cuda.current_stream().cuda_stream
    out = []
    for bh, dk, dv, dt in GLA_WORKLOADS:
        es = 4 if dt == "f32" else 2
        state_bytes = bh * dk * dv * es
        nbytes = 2 * state_bytes + bh * (3 * dk + 2 * dv) * es
        copies = max(2, min(8, -(-3 * L2_BYTES // state_bytes)))
        gen = torch.Generator(device=dev)
        gen.manual_seed(0)
        sets = []
        for _ in range(copies):
            q, k, v = (torch.rand((bh, x), generator=gen, device=dev) * 2 - 1 for x in (dk, dk, dv))
            gk = -3 * torch.rand((bh, dk), generator=gen, device=dev)
            S = torch.randn((bh, dk, dv), generator=gen, device=dev)
            q, k, v, gk, S = (x.to(tdt[dt]) for x in (q, k, v, gk, S))
            o = torch.empty((bh, dv), dtype=tdt[dt], device=dev)
            sets.append((q, k, v, gk, S, o))
        S_outs = [torch.empty_like(x[4]) for x in sets]

        def timed(variant, flags=0, out_of_place=False):
            calls = [(L.gla_decode_ex, (q.data_ptr(), k.data_ptr(), v.data_ptr(), gk.data_ptr(), S.data_ptr(),
                                        (S_out if out_of_place else S).data_ptr(), o.data_ptr(), bh, dk, dv,
                                        ctypes.c_float(dk ** -0.5), code[dt], variant, flags, s))
                     for (q, k, v, gk, S, o), S_out in zip(sets, S_outs)]
            if calls[0][0](*calls[0][1]) != 0:
                return None
            _, per = time_calls(L, calls, s, args.gla_steps, 10)
            el = time_batch(calls, args.gla_steps, 10)
            return statistics.median(per) * 1e3, el / args.gla_steps * 1e6

        iso, b2b = timed(g.GLA_VARIANT_AUTO)
        r = {"workload": f"gla_decode bh={bh} dk={dk} dv={dv} {dt} (in place)", "bytes": nbytes,
             "us_isolated_median": round(iso, 3), "us_back_to_back": round(b2b, 3),
             "gbs_back_to_back": round(nbytes / b2b / 1e3, 1), "gbs_isolated": round(nbytes / iso / 1e3, 1),
             "pct_of_8tbps": round(100 * nbytes / b2b / 1e3 / NOMINAL_HBM_GBS, 1), "state_copies": copies}
        # each kernel layout forced, for comparison; and the state requested
        # before the wait, against the same calls without it.  Those write
        # S_new to a second copy of each state instead of S, so that no call
        # in flight writes a state any call reads (the flag's promise).
        for name, variant in (("cta", g.GLA_VARIANT_CTA), ("warp", g.GLA_VARIANT_WARP), ("pipe", g.GLA_VARIANT_PIPE)):
            t = timed(variant)
            r[f"us_back_to_back_{name}"] = None if t is None else round(t[1], 3)
        for name, flags in (("out_of_place", 0), ("prefetch_state", g.GLA_PREFETCH_STATE)):
            t = timed(g.GLA_VARIANT_AUTO, flags, out_of_place=True)
            r[f"us_back_to_back_{name}"] = None if t is None else round(t[1], 3)
        out.append(r)
        print(json.dumps(r), file=sys.stderr, flush=True)
        del sets, S_outs
        torch.cuda.empty_cache()
    print(json.dumps({"gla_decode": out}), flush=True)
    return 0


def run_case(args, dev):
    """Run one shape a few times and exit (for profiler captures):
    --case N,K,DTYPE[,f32] [--calls C] [--config JSON] [--epilogue ACT]
    [--b-offset E] (ACT: run gemv_fused with alpha 0.5, an fp32 bias and
    that activation; E: B starts E elements past a 512-byte boundary).
    With --range R, R more calls follow back to back between
    cudaProfilerStart and cudaProfilerStop, alternating copies of B that
    together exceed L2 (as the timed calls do).  With --graph as well, the R
    calls are captured in a CUDA graph and the range is one replay of it, so
    that a profiler taking whole graphs as its unit measures consecutive
    launches together, with their programmatic overlap."""
    import torch

    import memory_bound_gemv_02_gb300 as g
    from memory_bound_gemv_02_gb300 import inputs
    parts = args.case.split(",")
    n, k, dtype = int(parts[0]), int(parts[1]), parts[2]
    out_fp32 = len(parts) > 3 and parts[3] == "f32"
    B, a = inputs.make_inputs(n, k, dtype, "normal", 0, dev)
    if args.b_offset:
        # the same matrix at an element offset past a 512-byte boundary
        buf = torch.empty(n * k + args.b_offset, dtype=B.dtype, device=dev)
        Bo = buf[args.b_offset:].view(n, k)
        Bo.copy_(B)
        B = Bo
    c = torch.empty(n, dtype=torch.float32 if out_fp32 else B.dtype, device=dev)
    cfg = json.loads(args.config) if args.config else None
    bias = torch.linspace(-1, 1, n, device=dev) if args.epilogue else None

    def call(Bx):
        if args.epilogue:
            g.gemv_fused(Bx, a, c=c, out_fp32=out_fp32, alpha=0.5, beta=1.0, bias=bias, activation=args.epilogue,
                         config=cfg)
        else:
            g.gemv_ex(Bx, a, c=c, out_fp32=out_fp32, config=cfg)

    for _ in range(args.calls):
        call(B)
    torch.cuda.synchronize()
    graph_us = None
    if args.range:
        copies = max(2, min(16, -(-3 * L2_BYTES // max(1, n * k * 2))))
        Bs = [B]
        for _ in range(copies - 1):  # each copy at B's offset
            buf = torch.empty(n * k + args.b_offset, dtype=B.dtype, device=dev)
            Bs.append(buf[args.b_offset:].view(n, k))
            Bs[-1].copy_(B)
        for i in range(len(Bs)):  # every copy once before the range
            call(Bs[i])
        # raw C-ABI calls (the launch configuration built once), so the
        # host enqueues far faster than the GPU runs them
        L = g.lib()
        fc = g.GemvConfig()
        for key, val in (cfg or {}).items():
            setattr(fc, key, val)
        dt = g.dtype_code(B.dtype, out_fp32)
        st = torch.cuda.current_stream().cuda_stream
        if cfg is None:  # gemv()'s own launch
            fn = L.gemv
            raw = [(Bx.data_ptr(), a.data_ptr(), c.data_ptr(), n, k, dt, st) for Bx in Bs]
        else:
            fn = L.gemv_ex
            raw = [(Bx.data_ptr(), a.data_ptr(), c.data_ptr(), n, k, dt, ctypes.byref(fc), st) for Bx in Bs]
        torch.cuda.synchronize()

        def run_range():
            for i in range(args.range):
                if args.epilogue:
                    call(Bs[i % len(Bs)])
                elif fn(*raw[i % len(raw)]) != 0:
                    raise RuntimeError("gemv failed inside the profiler range")

        if args.graph:
            # the same calls captured once into a CUDA graph (programmatic
            # launches become programmatic edges) and replayed as one unit
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                st = torch.cuda.current_stream().cuda_stream
                raw = [r[:-1] + (st,) for r in raw]
                run_range()
            gr.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            gr.replay()
            e1.record()
            torch.cuda.synchronize()
            graph_us = e0.elapsed_time(e1) * 1e3 / args.range
            torch.cuda.profiler.start()
            gr.replay()
            torch.cuda.synchronize()
            torch.cuda.profiler.stop()
        else:
            torch.cuda.profiler.start()
            run_range()
            torch.cuda.synchronize()
            torch.cuda.profiler.stop()
    print(json.dumps({"case": args.case, "calls": args.calls, "b_offset": args.b_offset, "range": args.range,
                      "graph": bool(args.graph),
                      "graph_us_per_call": graph_us, "epilogue": args.epilogue,
                      "config": g.gemv_last_config()}))
    return 0


def run_gla_case(args, dev):
    """One GLA decode workload a few times, in place (for profiler captures):
    --gla-case BH,DK,DV,DTYPE [--calls C] [--gla-variant V]."""
    import torch

    import memory_bound_gemv_02_gb300 as g
    bh, dk, dv = (int(x) for x in args.gla_case.split(",")[:3])
    dt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[args.gla_case.split(",")[3]]
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    q, k, v = ((torch.rand((bh, x), generator=gen, device=dev) * 2 - 1).to(dt) for x in (dk, dk, dv))
    gk = (-3 * torch.rand((bh, dk), generator=gen, device=dev)).to(dt)
    S = torch.randn((bh, dk, dv), generator=gen, device=dev).to(dt)
    o = torch.empty((bh, dv), dtype=dt, device=dev)
    for _ in range(args.calls):
        g.gla_decode(q, k, v, gk, S, scale=dk ** -0.5, S_new=S, o=o, variant=args.gla_variant)
    torch.cuda.synchronize()
    print(json.dumps({"gla_case": args.gla_case, "calls": args.calls, "variant": args.gla_variant}))
    return 0


def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    import memory_bound_gemv_02_gb300 as g
    from memory_bound_gemv_02_gb300 import _build, inputs
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    _build.ensure_built()
    L = g.lib()
    if args.sweep:
        return run_sweep(args, dev)
    if args.case:
        return run_case(args, dev)
    if args.gla_case:
        return run_gla_case(args, dev)
    if args.gla:
        return run_gla(args, dev)

    w = WORKLOAD
    n, k, fmt = w["n"], w["k"], w["dtype"]
    out_bytes = 4 if w["out_fp32"] else 2
    nbytes = algorithmic_bytes(n, k, 2, out_bytes)
    B, a = inputs.make_inputs(n, k, fmt, w["dist"], w["seed"], dev)
    B2 = B.clone()  # second copy: consecutive calls alternate, each copy > L2
    c = torch.empty(n, dtype=torch.float32 if w["out_fp32"] else B.dtype, device=dev)
    dt = g.dtype_code(B.dtype, w["out_fp32"])
    stream = torch.cuda.current_stream()
    s = stream.cuda_stream
    g.gemv_prepare(n, k, dt, True, s)
    g.gemv(B, a, c=c, out_fp32=w["out_fp32"])
    torch.cuda.synchronize()
    cfg = g.gemv_last_config()
    # The timed calls are plain gemv() calls back to back: the public entry
    # point as a caller makes it (a programmatic dependent launch that reads
    # nothing before the previous call has completed; it only asks L2 for
    # its first B tile).
    calls = [(L.gemv, (Bx.data_ptr(), a.data_ptr(), c.data_ptr(), n, k, dt, s)) for Bx in (B, B2)]

    # timed region: the W warm-up calls run right before it (after the clock
    # sampler has started), then barrier + synchronize, then a queue prefill
    # (a sleep kernel ahead of the first event, outside the region) so that
    # the host has enqueued the calls before the GPU reaches them and the
    # events time the GPU's K calls, not the host's first launch latency.
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    props = torch.cuda.get_device_properties(dev)
    gpu_id = f"GPU-{props.uuid}" if getattr(props, "uuid", None) else str(local)
    with ClockSampler(gpu_id) as clk:
        time.sleep(0.3)  # let the sampler start
        for i in range(args.warmup):
            fn, cargs = calls[i % 2]
            if fn(*cargs) != 0:
                raise RuntimeError("gemv failed in warm-up")
        barrier(world)
        torch.cuda.synchronize()
        torch.cuda._sleep(PREFILL_CYCLES)
        t_host0 = time.time()
        ev0.record(stream)
        for i in range(args.steps):
            fn, cargs = calls[i % 2]
            fn(*cargs)
        ev1.record(stream)
        torch.cuda.synchronize()
        t_host1 = time.time()
        barrier(world)
        # context, in the same sampler window: the same calls 2000 times,
        # and K calls without the prefill (the GPU idle when the first
        # event is recorded)
        us_2000 = time_batch(calls, 2000, 10) / 2000 * 1e6
        # ~0.45 s more of the same calls, so that clock samples (every 200
        # ms) fall inside the loaded window
        us_long = time_batch(calls, CLOCK_WINDOW_CALLS, 0) / CLOCK_WINDOW_CALLS * 1e6
        t_host2 = time.time()
        us_unprefilled = time_batch(calls, args.steps, 10, prefill=False) / args.steps * 1e6
        time.sleep(0.25)
    # clock samples from the timed region through the 2000-call batch (the
    # region alone at K = 20 is shorter than one 200 ms sample period)
    clocks = clk.summary(t_host0, t_host2, "timed region and the 2,000- and 13,500-call batches after it")
    elapsed = ev0.elapsed_time(ev1) / 1e3
    elapsed_max = max_over_ranks(elapsed, world)
    value = world * nbytes * args.steps / elapsed_max / 1e9
    mean_launch_ms = elapsed / args.steps * 1e3  # average launch duration over the timed region
    achieved = nbytes / (mean_launch_ms / 1e3) / 1e9
    peak, peak_kind = measured_peak()

    # Context (untimed for `value`): the same calls without overlap, back to
    # back, and one at a time with CUDA events around each launch; and calls
    # that promise B unwritten by the work in flight (weights), which read
    # their first B tile before the wait.
    none_cfg = g.GemvConfig()  # overlap 0
    plain = [(L.gemv_ex, (Bx.data_ptr(), a.data_ptr(), c.data_ptr(), n, k, dt, ctypes.byref(none_cfg), s))
             for Bx in (B, B2)]
    nplain = 2000
    us_plain = time_batch(plain, nplain, 10) / nplain * 1e6
    pb_cfg = g.GemvConfig()
    pb_cfg.overlap = g.GEMV_OVERLAP_PDL_PREFETCH_B
    prefetch_b = [(L.gemv_ex, (Bx.data_ptr(), a.data_ptr(), c.data_ptr(), n, k, dt, ctypes.byref(pb_cfg), s))
                  for Bx in (B, B2)]
    us_prefetch_b = time_batch(prefetch_b, nplain, 10) / nplain * 1e6
    # Calls that share their input vector (both B and a unwritten by the
    # work in flight, e.g. the projections of one activation) may also stage
    # a before the wait.
    ba_cfg = g.GemvConfig()
    ba_cfg.overlap = g.GEMV_OVERLAP_PDL_PREFETCH_BA
    shared = [(L.gemv_ex, (Bx.data_ptr(), a.data_ptr(), c.data_ptr(), n, k, dt, ctypes.byref(ba_cfg), s))
              for Bx in (B, B2)]
    us_shared = time_batch(shared, nplain, 10) / nplain * 1e6
    _, per_iso = time_calls(L, plain, s, 200, 10)
    us_iso = statistics.median(per_iso) * 1e3

    # e2e through the C-ABI from pinned host buffers (H2D of B and a, D2H of c)
    Bh = B.cpu().pin_memory()
    ah = a.cpu().pin_memory()
    ch = torch.empty(n, dtype=c.dtype).pin_memory()
    B_dev, a_dev, c_dev = torch.empty_like(B), torch.empty_like(a), torch.empty_like(c)
    host_args = (Bh.data_ptr(), ah.data_ptr(), ch.data_ptr(), B_dev.data_ptr(), a_dev.data_ptr(),
                 c_dev.data_ptr(), n, k, dt, s)
    e2e_steps = max(3, min(50, args.steps))
    for _ in range(3):
        L.gemv_host(*host_args)
    torch.cuda.synchronize()
    barrier(world)
    te0 = time.perf_counter()
    for _ in range(e2e_steps):
        if L.gemv_host(*host_args) != 0:
            raise RuntimeError("gemv_host failed")
    torch.cuda.synchronize()
    e2e_elapsed = max_over_ranks(time.perf_counter() - te0, world)
    e2e_value = world * nbytes * e2e_steps / e2e_elapsed / 1e9
    del B_dev, Bh

    host_us = host_overhead_us(L, 256, 512, 0, dev, s)
    native = native_measurements(n * k * 2)
    read_ceiling = None if native is None else native["read_gbs_1gib_overlapped"]

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(elapsed_max / args.steps * 1e3, 5),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": round(value / world / PAGES_BEST_GBS, 3),
        "vs_baseline_ref": "pages' best for this workload: 3.67 TB/s on an H200 (Case B.2, O1+O2); context only",
        "dtype": "f16", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC, "n": n, "k": k, "in_dtype": fmt,
                   "out_dtype": "f32" if w["out_fp32"] else fmt,
                   "l2": "inputs larger than L2: calls alternate two 235 MB copies of B (L2 is 129 MB)",
                   "launch": {**{kk: cfg[kk] for kk in ("variant", "rows_per_warp", "warps_per_cta", "warp_split",
                                                         "grid_split", "ctas", "smem_bytes", "unroll")},
                              "overlap": "gemv() as called: programmatic dependent launch, first B tile "
                                         "prefetched into L2 before the wait"},
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "us_per_call": round(mean_launch_ms * 1e3, 3),
        "us_per_call_no_overlap": round(us_plain, 3),
        "us_per_call_b_read_before_wait": round(us_prefetch_b, 3),
        "us_per_call_shared_input": round(us_shared, 3),
        "us_per_call_isolated_median": round(us_iso, 3),
        "pct_of_nominal_8tbps": round(100 * achieved / NOMINAL_HBM_GBS, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(frac_of_peak(achieved, peak), 4), "peak_kind": f"of {peak_kind}",
                     "traffic": profiled_traffic("7168x16384_f16", cfg)},
        "us_per_call_2000_calls": round(us_2000, 3),
        "us_per_call_13500_calls": round(us_long, 3),
        "us_per_call_unprefilled": round(us_unprefilled, 3),
        "probe_read_gbs": None if read_ceiling is None else round(read_ceiling, 1),
        "frac_of_read_ceiling": None if read_ceiling is None else round(achieved / read_ceiling, 4),
        "read_ceiling": None if native is None else {
            "how": "read-only 32-byte streaming loads, back to back over two buffers, CUDA events after a "
                   "queue prefill; 'overlapped' = programmatic launches that never wait",
            "gbs_1gib_overlapped": native["read_gbs_1gib_overlapped"],
            "gbs_1gib_plain": native["read_gbs_1gib_plain"],
            "gbs_b_bytes_overlapped": native["read_gbs_small_overlapped"],
            "gbs_b_bytes_plain": native["read_gbs_small_plain"]},
        "host_us_per_call": round(host_us, 3),
        "host_us_per_call_native": None if native is None else native["gemv_us"],
        "empty_launch_us_native": None if native is None else native["empty_launch_us"],
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s",
                "h2d_bytes_per_step": n * k * 2 + k * 2, "d2h_bytes_per_step": n * out_bytes},
        "gpu_launches": args.steps * int(cfg["launches"]),
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        B_bits, a_bits = inputs.to_bits(B), inputs.to_bits(a)
        line["cpu_baseline"] = cpu_baseline(B_bits, a_bits, fmt, n, k, out_bytes)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", default=None, help="write one JSON line per workload shape here")
    ap.add_argument("--sweep-steps", type=int, default=300)
    ap.add_argument("--case", default=None, help="N,K,DTYPE[,f32]: run that shape --calls times, no timing")
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--range", type=int, default=0,
                    help="with --case: R more calls back to back inside a cudaProfilerStart/Stop range")
    ap.add_argument("--b-offset", type=int, default=0,
                    help="with --case: B starts this many elements past a 512-byte boundary")
    ap.add_argument("--graph", action="store_true",
                    help="with --range: capture the R calls in a CUDA graph; the range is one replay of it")
    ap.add_argument("--gla", action="store_true", help="time the GLA decode step workloads instead")
    ap.add_argument("--gla-steps", type=int, default=300)
    ap.add_argument("--config", default=None, help="JSON launch configuration forced with --case")
    ap.add_argument("--epilogue", default=None, choices=["none", "relu", "sigmoid", "silu"],
                    help="with --case: run the fused-epilogue entry point with this activation and a bias")
    ap.add_argument("--gla-case", default=None, help="BH,DK,DV,DTYPE: run that GLA decode step --calls times")
    ap.add_argument("--gla-variant", type=int, default=0, help="GLA kernel layout forced with --gla-case")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
