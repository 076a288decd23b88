"""Run a few forward + adjoint steps of one workload, for profilers.

``python -m differentiable_cholesky_gb300.run_steps --workload banded_8192
--warmup 1 --steps 1`` runs ``chol_fwd`` then ``chol_adj`` on one of the five
synthetic workloads (or ``--n``/``--batch``/``--dtype`` for a Gram matrix of
another size), times each call with CUDA events and prints one line per step.
It is the command the kernel profiles are taken with: a known number of
launches per step, nothing else on the GPU.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--workload", default=None, help="one of the named workloads")
    ap.add_argument("--n", type=int, default=1024)
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--dtype", default="float64",
                    choices=["float32", "float64", "complex64", "complex128"])
    ap.add_argument("--tile", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1)
    ap.add_argument("--fwd-only", action="store_true")
    ap.add_argument("--tc-probe", type=int, default=None, metavar="K",
                    help="instead: time the float64 tensor-core trailing update of step K "
                         "once (chol_probe_tc_update) on the factor of the workload's first "
                         "matrix, or on an n x n Gram matrix")
    args = ap.parse_args()

    import torch
    from differentiable_cholesky_gb300 import binding
    from differentiable_cholesky_gb300 import workloads as W

    if args.tc_probe is not None:
        dev = torch.device("cuda:0")
        if args.workload:
            # as bench.py: on the factor of the workload's first matrix
            w = W.WORKLOADS[args.workload]()
            At, _ = binding.chol_fwd(torch.from_numpy(w.A[:1]).to(dev), tile=128)
            At = At[0].clone()
            n = w.n
        else:
            At = torch.from_numpy(W.gram_spd(1, args.n, 0, 1.0, np.float64)[0]).to(dev)
            n = args.n
        ms, bf, fp = binding.probe_tc_update(At, k=args.tc_probe, reps=1)
        print(f"tc update n={n} k={args.tc_probe}: {ms:.3f} ms, bf16 {bf / 1e12:.1f} TFLOP/s, "
              f"float64-equivalent {fp / 1e12:.2f} TFLOP/s", flush=True)
        return
    if args.workload:
        w = W.WORKLOADS[args.workload]()
        A, Lbar = w.A, w.adj_L
        tile = w.meta.get("tile", 0) if w.n > 64 else 0
        if args.workload == "bidiagonal_512":
            tile = 0
    else:
        dt = np.dtype(args.dtype)
        if np.issubdtype(dt, np.complexfloating):
            A = W.hermitian_spd(args.batch, args.n, 0, 1.0, dt)
            Lbar = W.tril_normal_complex(args.batch, args.n, 1, dt)
        else:
            A = W.gram_spd(args.batch, args.n, 0, 1.0, dt)
            Lbar = W.tril_normal(args.batch, args.n, 1, dt)
        tile = args.tile
    dev = torch.device("cuda:0")
    At = torch.from_numpy(A).to(dev)
    Lbt = torch.from_numpy(Lbar).to(dev)
    L = torch.empty_like(At)
    G = torch.zeros_like(At)
    st = torch.empty(At.shape[0], dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    for k in range(args.warmup + args.steps):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(stream)
        binding.chol_fwd(At, L=L, status=st, tile=tile)
        e[1].record(stream)
        if not args.fwd_only:
            binding.chol_adj(L, Lbt, adj_A=G, status=st, tile=tile)
        e[2].record(stream)
        torch.cuda.synchronize()
        tag = "warmup" if k < args.warmup else "step"
        print(f"{tag} {k}: fwd {e[0].elapsed_time(e[1]):.3f} ms, "
              f"adj {e[1].elapsed_time(e[2]):.3f} ms, status max {int(st.max())}", flush=True)


if __name__ == "__main__":
    main()
