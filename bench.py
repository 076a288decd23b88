#!/usr/bin/env python3
"""Throughput benchmark of the Cholesky forward + adjoint hot path on GB300.

One step = ``chol_fwd`` then ``chol_adj`` over one batch of synthetic input,
inputs resident in HBM when the timed region starts.  The default workload is
the largest single-GPU configuration: one 8192x8192 float64 ``A = E E^T``
(``E`` lower banded, bandwidth 32), tile 128, ``adj_L = tril(N(0, 1))``.  In
the same process the four other workloads (batched 65536 x 16x16 and
8192 x 64x64 float32, one 512x512 bidiagonal and 256 x 512x512 float64) are
timed kernel by kernel and reported under ``workloads``.

Prints ONE JSON line (rank 0).  ``value`` = matrices/s over all ranks,
``e2e`` = the same metric through the public API with pinned host buffers and
the host<->device copies inside the timed region, ``roofline`` = the
dominant call against its measured roof (HBM copy bandwidth for the batched
small matrices, the measured FP64 rate for the blocked path),
``cpu_baseline`` = the CPU oracle on a bounded sample of the same workload.

``--impl reference`` times the CPU oracle itself as the reference arm.
Multi-GPU (torchrun): every rank factors its own batch (weak scaling, no
collective on the data path; a barrier and a max-reduction of the time only).
"""
from __future__ import annotations

import argparse
import json
import math
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

METRIC = "Cholesky fwd+adjoint matrices/s and GFLOP/s (1 GB300), % of HBM/FP64 roofline"
UNIT = "matrices/s"
FALLBACK_BF16_TFLOPS = 1900.0   # the profiling recipe's fallback, if no measured file
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024
DEFAULT_WORKLOAD = "banded_8192"


# ----------------------------------------------------------------------------
# Workload description and algorithmic bytes / flops
# ----------------------------------------------------------------------------

WORKLOADS = {
    # name: (batch, n, numpy dtype, description, tile)
    "batched_16": (65536, 16, np.float32,
                   "65536 x 16x16 fp32, A = G G^T/16 + I (G ~ N(0,1), seed 0), adj_L = tril(N(0,1)) (seed 1)", 0),
    "batched_64": (8192, 64, np.float32,
                   "8192 x 64x64 fp32, A = G G^T/64 + 0.5 I, every 100th matrix non-PD (A[k,k] = -1)", 0),
    "bidiagonal_512": (1, 512, np.float64,
                       "1 x 512x512 fp64, A = E E^T with E lower bidiagonal (diag linspace(1,2), subdiag 0.5), default tile", 0),
    "batched_512": (256, 512, np.float64,
                    "256 x 512x512 fp64, A = G G^T/512 + I, tile 128", 128),
    "banded_8192": (1, 8192, np.float64,
                    "1 x 8192x8192 fp64, A = E E^T with E lower banded (bandwidth 32), tile 128", 128),
}

# Timed steps of the workloads reported beside the main line (each timed
# region spans well over 100 ms, so the clock sampler sees it).
EXTRA_STEPS = {"batched_16": 3000, "batched_64": 1000, "bidiagonal_512": 100,
               "batched_512": 10, "banded_8192": 3}


def lower_sector_bytes(n: int, esize: int) -> int:
    """Bytes of the 32-byte DRAM sectors that hold the lower triangle of one
    row-major n x n matrix (row i needs ceil((i+1) * esize / 32) sectors)."""
    return sum(math.ceil((i + 1) * esize / 32) * 32 for i in range(n))


def algorithmic_bytes(n: int, esize: int):
    low = lower_sector_bytes(n, esize)
    fwd = low + n * n * esize + 4          # tril(A) in, full L out, status out
    adj = 4 * low + 4                      # tril(L), tril(adj_L), tril(adj_A) in and out, status in
    return fwd, adj


def nominal_flops(n: int):
    return n ** 3 / 3.0, float(n ** 3)     # forward n^3/3, adjoint ~n^3 (nominal)


def executed_flops(n: int):
    """Flops the blocked kernels execute: forward n^3/3; the adjoint's blocked
    reverse sweep 2 n^3 / 3 (lower-order terms left out)."""
    return n ** 3 / 3.0, 2.0 * n ** 3 / 3.0


def default_tile(n: int, batch: int, sms: int = 152, float64: bool = False) -> int:
    """The library's default blocked tile (mirrors pick_tile and
    blocked_default_tile) for a device with `sms` multiprocessors."""
    if float64 and n > 128 and batch * 8 <= sms:
        return 128
    if n >= 2048:
        return 128
    per_side = (n + 63) // 64
    return 64 if batch * per_side * per_side >= 4 * sms else 32


def launches_per_step(n: int, tile: int, batch: int = 1, float64: bool = False,
                      sms: int = 152) -> int:
    """Kernels the library launches for one chol_fwd + chol_adj (mirrors the
    dispatch of blocked.cu and ozaki.cu; float64 with 128-wide tiles takes
    the tensor-core path, with lookahead once there are three tile columns)."""
    if n <= 64:
        return 2
    nt = (n + tile - 1) // tile
    tc = float64 and tile == 128
    tc_fwd = tc and n > 128
    look = tc_fwd and nt >= 3
    cluster = batch * 8 <= sms and tile > 32  # the cluster factor also inverts the tile
    fwd = 1 + nt                              # copy, diagonal factors
    for k in range(nt - 1):
        if tc_fwd:
            # inverse (unless the cluster factor made it), one slicing of the
            # panel and the inverse, assign; slicing, update (lookahead: column
            # k + 1, then the rest while there is one)
            fwd += (2 if cluster else 3) + 1 + ((1 + (1 if nt - k - 1 >= 2 else 0)) if look else 1)
        else:
            fwd += 2                          # panel solve, trailing update
    if not tc:
        # copy, per tile column: solve, row update, panel update, diagonal
        # sweep, symmetric update (the first and last columns skip some), add
        adj = 3 if nt == 1 else 5 * nt - 3
        return fwd + adj
    adj = 1 + 4 + 1                           # copy, prepare (4), add
    lit = batch * 4 <= sms

    def splits(k_n, chunks):
        tiles = batch * k_n
        return max(1, min((2 * sms + 2 * tiles - 1) // (2 * tiles), chunks))

    for J in range(nt):
        if J < nt - 1:
            chunks = nt - J - 1
            adj += 2 + 2                      # solve (slicing, assign); row (slicing, products)
            if look and J >= 2:
                # row update of block columns J - 1 .. J, then (side stream) the rest
                adj += 1 if splits(2, chunks) > 1 else 0
                adj += 1 + (1 if splits(J - 1, chunks) > 1 else 0)
            else:
                adj += 1 if splits(J + 1, chunks) > 1 else 0   # ordered reduce
        adj += 3 if lit else 1                # diagonal tile: literal form or sweep
        if J > 0:
            # update: slicing, products (lookahead: block column J - 1, then
            # the rest while there is one)
            adj += 2 + (1 if look and J >= 2 else 0)
    return fwd + adj


# DRAM bytes (read + write) per launch of a dominant kernel, from an ncu
# capture of that kernel (the summaries under profiles/).  Reported only while
# the kernel source still hashes to what was captured; otherwise null.
MEASURED_TRAFFIC = {
    # the tensor-core trailing update of step 0 on the workload's own factor
    # (the launch this bench times; captured at full size with the two DRAM
    # counters alone: 1 pass)
    "banded_8192": {"kernel": "tc_update", "bytes": (279.03 + 3.13) * 1e6,
                    "source": "differentiable_cholesky_gb300/csrc/ozaki.cu",
                    "code_sha256": "1029fc8b26e103612b89a868ef1c1c392add11c7e836d1be0f9269fa1b356a15"},
    "batched_16": {"kernel": "adj", "bytes": (201.624320 + 24.680448) * 1e6,
                   "source": "differentiable_cholesky_gb300/csrc/small_kernels.cuh",
                   "code_sha256": "4cab99b375b376b0c2a57aaea19c8dc55f9e22ad1b35cee7aa66e8af7dac280d"},
}


def code_sha256(text: str) -> str:
    """sha256 of a C/CUDA source with its comments, indentation and blank lines
    removed, so that a comment edit does not retire a measurement but a code
    edit does."""
    import hashlib
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = [re.sub(r"//.*$", "", ln).strip() for ln in text.splitlines()]
    return hashlib.sha256("\n".join(ln for ln in lines if ln).encode()).hexdigest()


def measured_traffic(workload: str, kernel: str):
    rec = MEASURED_TRAFFIC.get(workload)
    if rec is None or rec["kernel"] != kernel:
        return None
    try:
        with open(os.path.join(ROOT, rec["source"])) as f:
            if code_sha256(f.read()) != rec["code_sha256"]:
                return None
    except OSError:
        return None
    return rec["bytes"]


def read_bf16_peak():
    """The measured bf16 dense matmul rate (burst), TFLOP/s, or the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_BF16_TFLOPS, "fallback"


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for key in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
            if key in d:
                return float(d[key]), "measured"
        for k, v in d.items():
            if "hbm" in k.lower() and isinstance(v, (int, float)):
                return float(v), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------------------
# Clock sampling during the timed regions
# ----------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.samples = []  # (t, sm, smmax, reasons)
        self.proc = None
        self.thread = None
        cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._reader, daemon=True)
        self.thread.start()

    def _reader(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.strip().split(",")]
            if len(parts) < 8:
                continue
            try:
                sm, smmax = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            reasons = [name for name, v in zip(self.REASONS, parts[4:8]) if v.lower() == "active"]
            self.samples.append((time.monotonic(), sm, smmax, reasons))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        note = "sampled during the timed region"
        if not inside:
            # timed region shorter than the sampling period: nearest samples
            inside = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            note = "timed region shorter than the 100 ms sampling period; nearest samples"
        reasons = sorted({r for s in inside for r in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in inside),
                "sm_max_mhz": max(s[2] for s in inside), "reasons": reasons,
                "samples": len(inside), "note": note}


def max_over_ranks(value_ms: float, dist, device) -> float:
    """The slowest rank's time (the job's time), or the value itself on one rank."""
    if dist is None:
        return value_ms
    import torch
    t = torch.tensor([value_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, world: int, slowest_ms: float) -> float:
    """Whole-job units per second: every rank's units over the slowest rank's time."""
    return units_per_rank * world / (slowest_ms / 1e3)


def gpu_identifier(torch):
    try:
        u = torch.cuda.get_device_properties(0).uuid
        s = str(u)
        if s and not s.startswith("GPU-"):
            s = "GPU-" + s
        return s
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        first = vis.split(",")[0].strip() if vis else ""
        return first or None


# ----------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# ----------------------------------------------------------------------------

def host_threads() -> int:
    return max(1, os.cpu_count() or 1)


def time_oracle(A, Lbar, threads: int):
    """Oracle fwd + adjoint over the matrices of A; returns seconds."""
    import oracle
    t0 = time.perf_counter()
    L, st = oracle.potrf(A, threads=threads)
    oracle.potrf_adj(L, Lbar, status=st, threads=threads)
    return time.perf_counter() - t0


class OracleSample:
    """A bounded sample of a workload for the CPU oracle, and how one timed
    sample scales to matrices/s of the full workload.

    Batched workloads take their first `count` matrices (the unit is the
    matrix, so the scale is 1).  A single matrix of order n takes its leading
    m x m principal block (itself SPD, from the same construction) and counts
    as (m/n)^3 of a matrix, the share of the n^3 flops it does; the oracle's
    column-strided solves only get slower per flop as m grows, so this
    extrapolation flatters the oracle."""

    def __init__(self, w, budget_s: float, threads: int):
        self.w, self.threads = w, threads
        if w.batch > 1:
            probe = min(w.batch, 64)
            t = max(time_oracle(w.A[:probe], w.adj_L[:probe], threads), 1e-6)
            self.count = int(min(w.batch, max(probe, probe * budget_s / t)))
            self.m = w.n
            self.A, self.Lbar = w.A[:self.count], w.adj_L[:self.count]
            self.units = float(self.count)
            self.desc = f"first {self.count} of {w.batch} matrices"
        else:
            m = min(w.n, 256)
            t = max(time_oracle(*self._block(m), threads), 1e-6)
            # the literal adjoint grows faster than m^3 (its column accesses
            # leave the caches): grow m by halving steps of the cube root
            while m < w.n:
                m2 = min(w.n, int(m * 1.26) // 64 * 64 or m + 64)
                if t * (m2 / m) ** 4 > budget_s:
                    break
                m = m2
                t = max(time_oracle(*self._block(m), threads), 1e-6)
            self.count = 1
            self.m = m
            self.A, self.Lbar = self._block(m)
            self.units = (m / w.n) ** 3
            self.desc = (f"leading {m}x{m} principal block of the {w.n}x{w.n} matrix, "
                         f"counted as (m/n)^3 = {self.units:.3g} of a matrix")

    def _block(self, m):
        # a single (2-D) matrix: the oracle's threaded single-matrix routines
        A = np.ascontiguousarray(self.w.A[0, :m, :m])
        Lb = np.ascontiguousarray(self.w.adj_L[0, :m, :m])
        return A, Lb

    def run(self) -> float:
        return time_oracle(self.A, self.Lbar, self.threads)


def cpu_baseline(w):
    threads = host_threads()
    s = OracleSample(w, budget_s=10.0, threads=threads)
    t = s.run()
    return {"value": s.units / t, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{s.desc}; oracle fwd + literal adjoint, OpenMP on {threads} host "
                      f"threads, {t:.2f} s"}


def run_reference(args, w, desc, tile):
    import oracle
    oracle.build()
    threads = host_threads()
    # a bounded sample per step, sized so the whole run stays within ~2 minutes
    per_step = max(0.05, min(5.0, 120.0 / max(1, args.steps + args.warmup)))
    s = OracleSample(w, budget_s=per_step, threads=threads)
    for _ in range(args.warmup):
        s.run()
    times = [s.run() for _ in range(args.steps)]
    total = sum(times)
    value = args.steps * s.units / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if w.dtype == np.float32 else "f64", "data": "synthetic",
        "config": workload_config(args.workload, desc, w, tile, 1),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{s.desc} per step; oracle fwd + literal adjoint, OpenMP on "
                                   f"{threads} host threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def make_workload(name):
    from differentiable_cholesky_gb300 import workloads as W
    return W.WORKLOADS[name]()


def workload_config(name, desc, w, tile, world):
    esize = np.dtype(w.dtype).itemsize
    return {"workload": f"{name}: {desc}", "batch_per_gpu": w.batch, "n": w.n,
            "tile": (tile or "default") if w.n > 64 else None,
            "parallelism": f"independent batches per GPU x{world}" if world > 1 else "1 GPU",
            "l2": "inputs larger than L2 (two buffer sets alternated)"
            if w.batch * w.n * w.n * esize * 2 > L2_BYTES else
            "working set below L2 size: steps run back to back on two buffer sets"}


class GpuWorkload:
    """Device buffers of one workload (two sets, alternated between steps) and
    its timed step."""

    def __init__(self, name, torch, binding, dev, stream, sets=2):
        self.name = name
        self.batch, self.n, self.np_dtype, self.desc, self.tile = WORKLOADS[name]
        self.torch, self.binding, self.dev, self.stream = torch, binding, dev, stream
        self.w = make_workload(name)
        self.esize = np.dtype(self.np_dtype).itemsize
        self.sets = []
        for _ in range(sets):
            A = torch.from_numpy(self.w.A).to(dev)
            Lb = torch.from_numpy(self.w.adj_L).to(dev)
            self.sets.append((A, Lb, torch.empty_like(A), torch.zeros_like(A),
                              torch.empty(self.batch, dtype=torch.int32, device=dev)))

    def step(self, k, ev=None):
        A, Lb, L, G, st = self.sets[k % len(self.sets)]
        if ev is not None:
            ev[0].record(self.stream)
        self.binding.chol_fwd(A, L=L, status=st, tile=self.tile)
        if ev is not None:
            ev[1].record(self.stream)
        self.binding.chol_adj(L, Lb, adj_A=G, status=st, tile=self.tile)
        if ev is not None:
            ev[2].record(self.stream)

    def timed(self, steps, warmup, dist=None, sampler=None):
        """Times `steps` steps after `warmup`: (total ms, mean fwd ms, mean adj
        ms, clocks during the timed region)."""
        torch = self.torch
        for k in range(warmup):
            self.step(k)
        torch.cuda.synchronize()
        events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.monotonic()
        start.record(self.stream)
        for k in range(steps):
            self.step(k, events[k])
        stop.record(self.stream)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        t1 = time.monotonic()
        total = start.elapsed_time(stop)
        fwd = statistics.mean(e[0].elapsed_time(e[1]) for e in events)
        adj = statistics.mean(e[1].elapsed_time(e[2]) for e in events)
        clocks = sampler.summary(t0, t1) if sampler is not None else None
        return total, fwd, adj, clocks

    def kernel_report(self, fwd_ms, adj_ms, hbm_peak, fp64_peak, fp32_peak):
        """Per-call ms, algorithmic GB/s (small path) or executed TFLOP/s
        (blocked path), and the fraction of the relevant measured roof."""
        n, batch = self.n, self.batch
        fwd_b, adj_b = algorithmic_bytes(n, self.esize)
        rep = {"fwd": {"ms": fwd_ms}, "adj": {"ms": adj_ms}}
        if n <= 64:
            for k, ms, b in (("fwd", fwd_ms, fwd_b), ("adj", adj_ms, adj_b)):
                gbs = b * batch / (ms / 1e3) / 1e9
                rep[k].update({"algorithmic_GBps": gbs, "bytes_per_matrix": b,
                               "bound": "hbm", "frac": gbs / hbm_peak})
        else:
            peak = fp64_peak if self.esize == 8 else fp32_peak
            for k, ms, f in zip(("fwd", "adj"), (fwd_ms, adj_ms), executed_flops(n)):
                tf = f * batch / (ms / 1e3) / 1e12
                rep[k].update({"executed_TFLOPs": tf, "flops_per_matrix": f,
                               "bound": "fp64" if self.esize == 8 else "fp32",
                               "frac": tf / peak})
        rep["matrices_per_s"] = batch / ((fwd_ms + adj_ms) / 1e3)
        return rep

    def free(self):
        self.sets = []
        self.w = None


def measure_fp_peaks(binding, torch):
    """Measured FP64 rates of both pipes (FMA chains and f64 mma.sync) and the
    FP32 FMA rate, TFLOP/s.  The FP64 roof is the faster pipe."""
    p = {"dfma": binding.probe_fma_peak(torch.float64, iters=1 << 15) / 1e12,
         "ffma": binding.probe_fma_peak(torch.float32, iters=1 << 15) / 1e12}
    for s in binding.DMMA_SHAPES:
        p[f"dmma_{s}"] = binding.probe_dmma_peak(s, iters=1 << 14) / 1e12
    fp64 = max(v for k, v in p.items() if k == "dfma" or k.startswith("dmma"))
    return p, fp64, p["ffma"]


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 2000 for n <= 64, 10 for n = 512, else 5)")
    ap.add_argument("--warmup", type=int, default=None, help="warm-up steps (default 3)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="end-to-end steps (default: 20 for n <= 64, else 6)")
    ap.add_argument("--e2e-chunks", type=int, default=2,
                    help="chunks of the batch in the end-to-end step (n <= 64)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip timing the other workloads in the same run")
    args = ap.parse_args()
    batch, n, np_dtype, desc, tile = WORKLOADS[args.workload]
    if args.steps is None:
        args.steps = 2000 if n <= 64 else (10 if n <= 512 else 5)
    if args.warmup is None:
        args.warmup = 20 if n <= 64 else 3
    if args.e2e_steps is None:
        args.e2e_steps = 20 if n <= 64 else 6
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args, make_workload(args.workload), desc, tile)
        return

    import torch
    from differentiable_cholesky_gb300 import binding

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    binding.load_library()
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    sampler = ClockSampler(gpu_identifier(torch)) if rank == 0 else None
    if sampler is not None:
        time.sleep(0.3)

    # ---------------- main workload: the bench line -------------------------
    g = GpuWorkload(args.workload, torch, binding, dev, stream)
    w = g.w
    esize = g.esize
    elapsed_ms, fwd_ms, adj_ms, clocks = g.timed(args.steps, args.warmup, dist, sampler)
    elapsed_ms = max_over_ranks(elapsed_ms, dist, dev)

    # The in-place forms on the same workload: two work sets, each restored
    # from the pristine inputs right after its step.  Events bracket the two
    # in-place calls only.
    ip_steps = min(args.steps, 500 if n <= 64 else 3)
    work = [(g.sets[i][0].clone(), g.sets[i][1].clone(), torch.empty_like(g.sets[i][4]))
            for i in range(2)]

    def ip_step(k, ev=None):
        X, Y, ip_st = work[k & 1]
        if ev is not None:
            ev[0].record(stream)
        binding.chol_fwd_inplace(X, status=ip_st, tile=tile)
        if ev is not None:
            ev[1].record(stream)
        binding.chol_adj_inplace(X, Y, status=ip_st, tile=tile)
        if ev is not None:
            ev[2].record(stream)
        X.copy_(g.sets[k & 1][0])
        Y.copy_(g.sets[k & 1][1])

    for k in range(2 if n > 64 else args.warmup):
        ip_step(k)
    ip_events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(ip_steps)]
    for k in range(ip_steps):
        ip_step(k, ip_events[k])
    torch.cuda.synchronize()
    ip_fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ip_events)
    ip_adj_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ip_events)
    del work

    # end-to-end through the public API: pinned host in, pinned host out
    hA = torch.from_numpy(w.A).pin_memory()
    hLb = torch.from_numpy(w.adj_L).pin_memory()
    hL = torch.empty_like(hA).pin_memory()
    hG = torch.empty_like(hA).pin_memory()
    hst = torch.empty(batch, dtype=torch.int32).pin_memory()

    # The batch goes through in chunks, and consecutive steps use the two
    # device buffer sets in turn: chunk c of a step on set k % 2 runs on its
    # own stream, so one chunk's host-to-device copies, another's kernels and
    # a third's (or the previous step's) device-to-host copies overlap, while
    # each (set, chunk) pair stays ordered on its stream.  Every input is
    # still copied in and every result read back once per step.
    chunks = max(1, min(args.e2e_chunks, batch // 1024)) if n <= 64 else 1
    bounds = [batch * c // chunks for c in range(chunks + 1)]
    streams = [torch.cuda.Stream() for _ in range(2 * chunks)]
    host_out = [(hL, hG, hst), (torch.empty_like(hL).pin_memory(), torch.empty_like(hG).pin_memory(),
                                torch.empty_like(hst).pin_memory())]

    # Copies of one step overlap the compute of another.  For the single-
    # matrix (blocked) workloads the compute of consecutive steps stays in
    # order (an event chain), so the end-to-end rate never counts two
    # matrices' kernels running side by side; batched chunks are parts of
    # one batch and may overlap.
    compute_done = [None]
    chain = n > 64

    def e2e_step(k):
        dA_, dLb_, dL_, dG_, dst_ = g.sets[k & 1]
        hL_, hG_, hst_ = host_out[k & 1]
        for c in range(chunks):
            b0, b1 = bounds[c], bounds[c + 1]
            s = streams[(k & 1) * chunks + c]
            with torch.cuda.stream(s):
                dA_[b0:b1].copy_(hA[b0:b1], non_blocking=True)
                dLb_[b0:b1].copy_(hLb[b0:b1], non_blocking=True)
                dG_[b0:b1].zero_()
                if chain and compute_done[0] is not None:
                    s.wait_event(compute_done[0])
                binding.chol_fwd(dA_[b0:b1], L=dL_[b0:b1], status=dst_[b0:b1], tile=tile, stream=s)
                binding.chol_adj(dL_[b0:b1], dLb_[b0:b1], adj_A=dG_[b0:b1], status=dst_[b0:b1],
                                 tile=tile, stream=s)
                if chain:
                    done = torch.cuda.Event()
                    done.record(s)
                    compute_done[0] = done
                hL_[b0:b1].copy_(dL_[b0:b1], non_blocking=True)
                hst_[b0:b1].copy_(dst_[b0:b1], non_blocking=True)
                hG_[b0:b1].copy_(dG_[b0:b1], non_blocking=True)

    def e2e_run(count):
        go = torch.cuda.Event()
        go.record(stream)
        for s in streams:
            s.wait_event(go)
        for k in range(count):
            e2e_step(k)
        for s in streams:
            ev = torch.cuda.Event()
            ev.record(s)
            stream.wait_event(ev)

    e2e_run(3 if n <= 64 else 1)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    e0.record(stream)
    e2e_run(args.e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    h2d = int(hA.numel() * esize + hLb.numel() * esize)
    d2h = int(hL.numel() * esize + hG.numel() * esize + hst.numel() * 4)
    del hA, hLb, hL, hG, hst, host_out, streams

    peaks, fp64_peak, fp32_peak = measure_fp_peaks(binding, torch)
    hbm_peak, peak_src = read_peaks()
    main_report = g.kernel_report(fwd_ms, adj_ms, hbm_peak, fp64_peak, fp32_peak)
    # the dominant kernel of the float64 tensor-core path timed alone: step 0's
    # trailing update of one matrix, on a scratch copy of its factor
    tc_probe = None
    if np_dtype == np.float64:
        t_eff = tile or default_tile(n, batch, sms, True)
        if n > 128 and t_eff == 128:
            scratch = g.sets[0][2][0].clone()
            ms_l, bf_l, fp_l = binding.probe_tc_update(scratch, k=0, reps=3, stream=stream)
            m = (n + 127) // 128 - 1
            tc_probe = {"ms": ms_l, "bf16_TFLOPs": bf_l / 1e12, "fp64_equiv_TFLOPs": fp_l / 1e12,
                        "tiles": m * (m + 1) // 2, "ctas": 4 * (m * (m + 1) // 2)}
            del scratch
    g.free()
    del g
    torch.cuda.empty_cache()

    # ---------------- the other workloads, same process ---------------------
    others = {}
    if not args.no_workloads:
        for name in WORKLOADS:
            if name == args.workload:
                continue
            o = GpuWorkload(name, torch, binding, dev, stream)
            steps = EXTRA_STEPS[name]
            tot, f_ms, a_ms, ck = o.timed(steps, 5 if o.n <= 64 else 2, None, sampler)
            rep = o.kernel_report(f_ms, a_ms, hbm_peak, fp64_peak, fp32_peak)
            rep.update({"steps": steps, "step_ms": tot / steps, "clocks": ck,
                        "tile": (o.tile or default_tile(o.n, o.batch, sms, o.np_dtype == np.float64))
                        if o.n > 64 else None,
                        "config": f"{name}: {o.desc}"})
            others[name] = rep
            o.free()
            del o
            torch.cuda.empty_cache()
    if sampler is not None:
        sampler.stop()

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    value = job_throughput(args.steps * batch, world, elapsed_ms)
    e2e_value = job_throughput(args.e2e_steps * batch, world, e2e_ms)
    fwd_f, adj_f = nominal_flops(n)
    dominant = "adj" if adj_ms >= fwd_ms else "fwd"
    dk = main_report[dominant]
    if n <= 64:
        roofline = {"bound": "hbm", "kernel": f"{dominant} call", "achieved": dk["algorithmic_GBps"],
                    "peak": hbm_peak, "unit": "GB/s", "frac": dk["frac"],
                    "peak_source": f"{peak_src} HBM copy bandwidth (MEASURED_PEAKS.json)",
                    "traffic": measured_traffic(args.workload, dominant)}
    elif tc_probe is not None:
        bf16_peak, bf16_src = read_bf16_peak()
        roofline = {"bound": "tensor",
                    "kernel": "oz_gemm_kernel: the forward's trailing update of step 0 on the bf16 "
                              f"tensor cores ({tc_probe['tiles']} lower 128x128 tiles, "
                              f"{tc_probe['ctas']} CTAs), timed alone with CUDA events "
                              "(chol_probe_tc_update)",
                    "achieved": tc_probe["bf16_TFLOPs"], "peak": bf16_peak, "unit": "TFLOP/s",
                    "frac": tc_probe["bf16_TFLOPs"] / bf16_peak,
                    "peak_source": f"{bf16_src} bf16 dense matmul, burst (MEASURED_PEAKS.json)",
                    "launch_ms": tc_probe["ms"],
                    "fp64_equivalent_TFLOPs": tc_probe["fp64_equiv_TFLOPs"],
                    "fp64_roof_TFLOPs": fp64_peak, "peaks_TFLOPs": peaks,
                    "traffic": measured_traffic(args.workload, "tc_update")}
    else:
        roofline = {"bound": "alu", "pipe": "fp64" if esize == 8 else "fp32",
                    "kernel": f"{dominant} call (all its launches)",
                    "achieved": dk["executed_TFLOPs"],
                    "peak": fp64_peak if esize == 8 else fp32_peak, "unit": "TFLOP/s",
                    "frac": dk["frac"],
                    "peak_source": "measured in this run: the faster of the FP64 FMA-chain probe and "
                                   "the f64 mma.sync (DMMA) probes, all shapes (peaks_TFLOPs)",
                    "peaks_TFLOPs": peaks, "traffic": None}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if np_dtype == np.float32 else "f64", "data": "synthetic",
        "config": workload_config(args.workload, desc, w, tile, world),
        "gflops": value * (fwd_f + adj_f) / 1e9,
        "kernels": main_report,
        "roofline": roofline,
        "gpu_launches": launches_per_step(
            n, (tile or default_tile(n, batch, sms, np_dtype == np.float64)) if n > 64 else 0,
            batch, np_dtype == np.float64, sms) * args.steps,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": args.e2e_steps, "chunks": chunks,
                "overlap": "chunks on their own streams, consecutive steps on alternate buffer sets: "
                           "copies overlap compute" + ("; compute stays in step order" if n > 64 else "")},
        "clocks": clocks,
        "inplace": {"value": batch * world / ((ip_fwd_ms + ip_adj_ms) / 1e3), "unit": UNIT,
                    "fwd_ms": ip_fwd_ms, "adj_ms": ip_adj_ms, "steps": ip_steps,
                    "timed": "chol_fwd_inplace + chol_adj_inplace (CUDA events around the "
                             "two calls; inputs restored outside them), rank 0"},
        "workloads": others,
    }
    if not args.no_cpu_baseline:
        import oracle
        oracle.build()
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
