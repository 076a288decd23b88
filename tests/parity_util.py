"""Helpers shared by the GPU parity tests: device round trips and the error
metric (per-matrix relative Frobenius error, maximised over the batch)."""
import numpy as np

# Tolerances (relative Frobenius error against the oracle): fp64 / fp32.
TOL_L = {np.dtype(np.float64): 1e-12, np.dtype(np.float32): 2e-5}
TOL_ADJ = {np.dtype(np.float64): 1e-10, np.dtype(np.float32): 1e-4}


def max_rel_err(x, ref, mask=None, lower=False):
    """max over b of ||x_b - ref_b||_F / ||ref_b||_F (lower triangle if asked)."""
    # complex results keep their imaginary parts (compared in complex128)
    wide = np.complex128 if (np.iscomplexobj(x) or np.iscomplexobj(ref)) else np.float64
    x = np.asarray(x, wide)
    ref = np.asarray(ref, wide)
    if lower:
        tri = np.tril(np.ones(x.shape[-2:], bool))
        x = np.where(tri, x, 0.0)
        ref = np.where(tri, ref, 0.0)
    num = np.linalg.norm((x - ref).reshape(x.shape[0], -1), axis=1)
    den = np.linalg.norm(ref.reshape(ref.shape[0], -1), axis=1)
    err = num / np.where(den > 0, den, 1.0)
    if mask is not None:
        err = err[mask]
    return float(err.max()) if err.size else 0.0


def gpu_fwd_adj(A, Lbar, tile=0, adj_A0=None):
    """Run chol_fwd then chol_adj on cuda:0; returns numpy L, status, adj_A."""
    import torch
    from differentiable_cholesky_gb300 import binding
    dev = torch.device("cuda:0")
    At = torch.from_numpy(np.ascontiguousarray(A)).to(dev)
    Lt, st = binding.chol_fwd(At, tile=tile)
    Gt = None if adj_A0 is None else torch.from_numpy(np.ascontiguousarray(adj_A0)).to(dev)
    Gt = binding.chol_adj(Lt, torch.from_numpy(np.ascontiguousarray(Lbar)).to(dev), adj_A=Gt,
                          status=st, tile=tile)
    torch.cuda.synchronize()
    return Lt.cpu().numpy(), st.cpu().numpy(), Gt.cpu().numpy()
