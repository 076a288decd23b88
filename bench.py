#!/usr/bin/env python3
"""Throughput benchmark of the Cholesky forward + adjoint hot path on GB300.

One step = ``chol_fwd`` then ``chol_adj`` over one batch of synthetic input
(default workload: 65536 independent 16x16 float32 SPD matrices,
``A = G G^T / 16 + I``, ``adj_L = tril(N(0, 1))``).  Inputs are resident in HBM
when the timed region starts; each step reads 256 MiB of distinct buffers, more
than the 129 MB L2, and steps alternate between two buffer sets.

Prints ONE JSON line (rank 0).  ``value`` = matrices/s over all ranks,
``e2e`` = the same metric through the public API with pinned host buffers and
the host<->device copies inside the timed region, ``roofline`` = the dominant
kernel's algorithmic bandwidth against the measured HBM copy peak,
``cpu_baseline`` = the CPU oracle on the same workload.

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
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


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


def default_tile(n: int, batch: int) -> int:
    """The library's default blocked tile (mirrors blocked_default_tile)."""
    if n >= 2048:
        return 128
    per_side = (n + 63) // 64
    return 64 if batch * per_side * per_side >= 4 * 152 else 32


def launches_per_step(n: int, tile: int) -> int:
    """Kernels the library launches for one chol_fwd + chol_adj."""
    if n <= 64:
        return 2
    nt = (n + tile - 1) // tile
    fwd = 1 + nt + 2 * (nt - 1)              # copy, diagonal factors, panel solves + updates
    # copy, per tile column: solve, row update, panel update, diagonal sweep,
    # symmetric update (the first and last columns skip some), accumulate
    adj = 3 if nt == 1 else 5 * nt - 3
    return fwd + adj


# DRAM bytes (read + write) per launch of the dominant kernel, from the ncu
# capture summarised in profiles/batched_16_kernels.md.  Reported only while
# the kernel source still hashes to what was captured; otherwise null.
MEASURED_TRAFFIC = {
    "batched_16": {"kernel": "adj", "bytes": (201.627904 + 23.920896) * 1e6,
                   "source": "differentiable_cholesky_gb300/csrc/small_kernels.cuh",
                   "code_sha256": "65783f7da4b7300d2208efe580890165b364e544a7082868691a0351e74e3502"},
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
# Clock sampling during the timed region
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

def time_oracle(w, count: int, threads: int = 1):
    """Oracle fwd + adjoint over the first `count` matrices; returns seconds."""
    import oracle
    A = w.A[:count]
    Lbar = w.adj_L[:count]
    t0 = time.perf_counter()
    L, st = oracle.potrf(A, threads=threads)
    oracle.potrf_adj(L, Lbar, status=st, threads=threads)
    return time.perf_counter() - t0


def oracle_sample_size(w, budget_s: float = 2.0, cap: int | None = None):
    """Matrices the oracle handles in about `budget_s` seconds (one thread)."""
    probe = min(w.batch, 256)
    t = max(time_oracle(w, probe), 1e-6)
    count = int(min(w.batch, max(probe, probe * budget_s / t)))
    if cap is not None:
        count = min(count, cap)
    return count


def cpu_baseline(w):
    count = oracle_sample_size(w, budget_s=3.0)
    t = time_oracle(w, count)
    return {"value": count / t, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {count} of {w.batch} matrices of the same workload, fwd + adjoint, "
                      f"one thread, {t:.2f} s"}


def run_reference(args, w, desc):
    import oracle
    oracle.build()
    # a bounded sample per step, sized so the whole run stays within ~2 minutes
    per_step = max(0.02, min(0.5, 120.0 / max(1, args.steps + args.warmup)))
    count = oracle_sample_size(w, budget_s=per_step)
    for _ in range(args.warmup):
        time_oracle(w, count)
    times = [time_oracle(w, count) for _ in range(args.steps)]
    total = sum(times)
    value = args.steps * count / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if w.dtype == np.float32 else "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {desc}", "batch_per_gpu": w.batch, "n": w.n,
                   "tile": (WORKLOADS[args.workload][4] or "default") if w.n > 64 else None,
                   "parallelism": "host, one thread",
                   "step": f"oracle fwd + adjoint over {count} matrices of the batch"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{count} of {w.batch} matrices per step, one thread"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def make_workload(name):
    from differentiable_cholesky_gb300 import workloads as W
    return W.WORKLOADS[name]()


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 2000 for n <= 64, else 3)")
    ap.add_argument("--warmup", type=int, default=None,
                    help="warm-up steps (default: 20 for n <= 64, else 3)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="batched_16")
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="end-to-end steps (default: 20 for n <= 64, else 1)")
    ap.add_argument("--e2e-chunks", type=int, default=2,
                    help="chunks of the batch in the end-to-end step (n <= 64)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    batch, n, np_dtype, desc, tile = WORKLOADS[args.workload]
    if args.steps is None:
        args.steps = 2000 if n <= 64 else 3
    if args.warmup is None:
        args.warmup = 20 if n <= 64 else 3
    if args.e2e_steps is None:
        args.e2e_steps = 20 if n <= 64 else 1
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args, make_workload(args.workload), desc)
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

    w = make_workload(args.workload)
    esize = np.dtype(np_dtype).itemsize
    tdtype = torch.float32 if np_dtype == np.float32 else torch.float64

    # two buffer sets, alternated between steps
    sets = []
    for _ in range(2):
        A = torch.from_numpy(w.A).to(dev)
        Lb = torch.from_numpy(w.adj_L).to(dev)
        L = torch.empty_like(A)
        G = torch.zeros_like(A)
        st = torch.empty(batch, dtype=torch.int32, device=dev)
        sets.append((A, Lb, L, G, st))
    stream = torch.cuda.current_stream()

    def step(k, ev=None):
        A, Lb, L, G, st = sets[k & 1]
        if ev is not None:
            ev[0].record(stream)
        binding.chol_fwd(A, L=L, status=st, tile=tile)
        if ev is not None:
            ev[1].record(stream)
        binding.chol_adj(L, Lb, adj_A=G, status=st, tile=tile)
        if ev is not None:
            ev[2].record(stream)

    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize()

    sampler = ClockSampler(gpu_identifier(torch)) if rank == 0 else None
    if sampler is not None:
        time.sleep(0.3)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.monotonic()
    start.record(stream)
    for k in range(args.steps):
        step(k, events[k])
    stop.record(stream)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall1 = time.monotonic()
    elapsed_ms = start.elapsed_time(stop)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in events)
    adj_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in events)
    elapsed_ms = max_over_ranks(elapsed_ms, dist, dev)
    clocks = sampler.summary(t_wall0, t_wall1) if sampler is not None else None

    # The in-place forms on the same workload: two work sets, each restored
    # from the pristine inputs right after its step, so that the other set's
    # step runs in between and a step's inputs have left L2.  Events bracket
    # the two in-place calls only.
    ip_steps = min(args.steps, 500)
    work = [(sets[i][0].clone(), sets[i][1].clone(), torch.empty_like(sets[i][4])) for i in range(2)]

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
        X.copy_(sets[k & 1][0])
        Y.copy_(sets[k & 1][1])

    for k in range(args.warmup):
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
    n_streams = len(streams)

    def e2e_step(k):
        dA_, dLb_, dL_, dG_, dst_ = sets[k & 1]
        hL_, hG_, hst_ = host_out[k & 1]
        for c in range(chunks):
            b0, b1 = bounds[c], bounds[c + 1]
            s = streams[(k & 1) * chunks + c]
            with torch.cuda.stream(s):
                dA_[b0:b1].copy_(hA[b0:b1], non_blocking=True)
                dLb_[b0:b1].copy_(hLb[b0:b1], non_blocking=True)
                dG_[b0:b1].zero_()
                binding.chol_fwd(dA_[b0:b1], L=dL_[b0:b1], status=dst_[b0:b1], tile=tile, stream=s)
                binding.chol_adj(dL_[b0:b1], dLb_[b0:b1], adj_A=dG_[b0:b1], status=dst_[b0:b1],
                                 tile=tile, stream=s)
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
    if sampler is not None:
        sampler.stop()

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    value = job_throughput(args.steps * batch, world, elapsed_ms)
    e2e_value = job_throughput(args.e2e_steps * batch, world, e2e_ms)
    fwd_b, adj_b = algorithmic_bytes(n, esize)
    fwd_f, adj_f = nominal_flops(n)
    hbm_peak, peak_src = read_peaks()
    fwd_gbs = fwd_b * batch / (fwd_ms / 1e3) / 1e9
    adj_gbs = adj_b * batch / (adj_ms / 1e3) / 1e9
    dominant = "adj" if adj_ms >= fwd_ms else "fwd"
    kernels = {
        "fwd": {"ms": fwd_ms, "algorithmic_GBps": fwd_gbs, "bytes_per_matrix": fwd_b},
        "adj": {"ms": adj_ms, "algorithmic_GBps": adj_gbs, "bytes_per_matrix": adj_b},
    }
    if n <= 64:
        achieved = adj_gbs if dominant == "adj" else fwd_gbs
        roofline = {"bound": "hbm", "kernel": dominant, "achieved": achieved, "peak": hbm_peak,
                    "unit": "GB/s", "frac": achieved / hbm_peak,
                    "peak_source": f"{peak_src} HBM copy bandwidth",
                    "traffic": measured_traffic(args.workload, dominant)}
    else:
        # FP64 FMA-pipe bound: executed flops per call against the FMA peak
        # measured by the library's probe on this GPU.
        ex_f, ex_a = executed_flops(n)
        fp64_peak = binding.probe_fma_peak(tdtype, iters=1 << 15) / 1e12
        tf_f = ex_f * batch / (fwd_ms / 1e3) / 1e12
        tf_a = ex_a * batch / (adj_ms / 1e3) / 1e12
        kernels["fwd"]["executed_TFLOPs"] = tf_f
        kernels["adj"]["executed_TFLOPs"] = tf_a
        achieved = tf_a if dominant == "adj" else tf_f
        roofline = {"bound": "fp64" if np_dtype == np.float64 else "fp32", "kernel": dominant,
                    "achieved": achieved, "peak": fp64_peak, "unit": "TFLOP/s",
                    "frac": achieved / fp64_peak,
                    "peak_source": "measured by chol_probe_fma_peak (independent FMA chains on every SM)",
                    "traffic": None}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if np_dtype == np.float32 else "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {desc}", "batch_per_gpu": batch, "n": n,
                   "tile": (tile or "default") if n > 64 else None,
                   "parallelism": f"independent batches per GPU x{world}" if world > 1 else "1 GPU",
                   "l2": "inputs larger than L2 (256 MiB of distinct buffers per step, two sets alternated)"
                   if batch * n * n * esize * 4 > L2_BYTES else
                   "working set below L2 size: steps run back to back on two buffer sets"},
        "gflops": value * (fwd_f + adj_f) / 1e9,
        "kernels": kernels,
        "roofline": roofline,
        "gpu_launches": launches_per_step(n, (tile or default_tile(n, batch)) if n > 64 else 0) * args.steps,
        "e2e": {"value": e2e_value, "unit": UNIT,
                "h2d_bytes_per_step": int(hA.numel() * esize + hLb.numel() * esize),
                "d2h_bytes_per_step": int(hL.numel() * esize + hG.numel() * esize + hst.numel() * 4),
                "steps": args.e2e_steps, "chunks": chunks, "streams": n_streams,
                "overlap": "chunks on their own streams; consecutive steps on alternate buffer sets"},
        "clocks": clocks,
        "inplace": {"value": batch * world / ((ip_fwd_ms + ip_adj_ms) / 1e3), "unit": UNIT,
                    "fwd_ms": ip_fwd_ms, "adj_ms": ip_adj_ms, "steps": ip_steps,
                    "timed": "chol_fwd_inplace + chol_adj_inplace (CUDA events around the "
                             "two calls; inputs restored outside them), rank 0"},
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
