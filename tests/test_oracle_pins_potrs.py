"""Pins of the oracle's solve with the factor (``oracle.potrs``) and its
reverse mode (``oracle.potrs_adj``) to facts outside itself (CPU only):
LAPACK solves through numpy, closed forms, central finite differences on
every entry of B and of L's lower triangle (real and imaginary parts), and
torch's autograd of ``cholesky_solve``."""
import numpy as np
import pytest

import oracle
from differentiable_cholesky_gb300 import workloads as W


def rel(x, ref):
    den = np.linalg.norm(ref)
    return np.linalg.norm(np.asarray(x) - ref) / (den if den > 0 else 1.0)


def spd(n, seed, dtype):
    if np.issubdtype(dtype, np.complexfloating):
        return W.hermitian_spd(1, n, seed, 1.0, dtype)[0]
    return W.gram_spd(1, n, seed, 1.0, dtype)[0]


def factor(A):
    return (oracle.hpotrf if np.iscomplexobj(A) else oracle.potrf)(A)[0]


def rhs(n, r, seed, dtype):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((2, n, r))
    if np.issubdtype(dtype, np.complexfloating):
        return (x[0] + 1j * x[1]).astype(dtype)
    return x[0].astype(dtype)


@pytest.mark.parametrize("dtype", [np.float64, np.complex128])
@pytest.mark.parametrize("n,r", [(1, 1), (5, 3), (40, 1), (33, 17)])
def test_matches_lapack_solve(n, r, dtype):
    A = spd(n, 100 + n, dtype)
    B = rhs(n, r, 101, dtype)
    X = oracle.potrs(factor(A), B)
    assert rel(X, np.linalg.solve(A, B)) <= 1e-13
    assert rel(A @ X, B) <= 1e-13


def test_closed_forms():
    n = 6
    B = rhs(n, 2, 102, np.float64)
    assert np.array_equal(oracle.potrs(np.eye(n), B), B)
    d = np.array([1.0, 2.0, 4.0, 0.5, 8.0, 0.25])   # powers of two: exact
    X = oracle.potrs(np.diag(d), B)
    assert np.array_equal(X, B / (d * d)[:, None])
    # the pages' bidiagonal E: A = E E^T, solve against the dense A
    E = W.bidiagonal_E(64)
    Bb = rhs(64, 4, 103, np.float64)
    assert rel(oracle.potrs(E, Bb), np.linalg.solve(E @ E.T, Bb)) <= 1e-13


def test_reads_lower_triangle_of_L_only_and_skips_failed():
    n = 8
    A = spd(n, 104, np.float64)
    L = factor(A)
    Lg = L.copy()
    Lg[np.triu_indices(n, 1)] = np.nan
    B = rhs(n, 3, 105, np.float64)
    assert np.array_equal(oracle.potrs(L, B), oracle.potrs(Lg, B))
    Ls = np.stack([L, L])
    Bs = np.stack([B, B])
    X = oracle.potrs(Ls, Bs, status=np.array([0, 4], np.int32))
    assert np.array_equal(X[0], oracle.potrs(L, B)) and np.all(X[1] == 0)


def loss(L, B, Wt):
    return float(np.real(np.sum(np.conj(Wt) * oracle.potrs(L, B))))


@pytest.mark.parametrize("dtype", [np.float64, np.complex128])
@pytest.mark.parametrize("n,r", [(1, 1), (3, 2), (5, 1)])
def test_adjoint_central_differences(n, r, dtype):
    A = spd(n, 106 + n, dtype)
    L = factor(A)
    B = rhs(n, r, 107, dtype)
    Wt = rhs(n, r, 108, dtype)
    X = oracle.potrs(L, B)
    Bb, Lb = oracle.potrs_adj(L, X, Wt)
    cplx = np.iscomplexobj(A)
    parts = (1.0, 1j) if cplx else (1.0,)
    h = 1e-6
    fdB = np.zeros_like(B)
    for i in range(n):
        for c in range(r):
            for p in parts:
                Bp, Bm = B.copy(), B.copy()
                Bp[i, c] += h * p
                Bm[i, c] -= h * p
                fdB[i, c] += (loss(L, Bp, Wt) - loss(L, Bm, Wt)) / (2 * h) * (1 if p == 1.0 else 1j)
    assert rel(Bb, fdB) <= 1e-7
    fdL = np.zeros_like(L)
    for i in range(n):
        for j in range(i + 1):
            for p in (parts if i != j else (1.0,)):   # L's diagonal is real
                Lp, Lm = L.copy(), L.copy()
                Lp[i, j] += h * p
                Lm[i, j] -= h * p
                fdL[i, j] += (loss(Lp, B, Wt) - loss(Lm, B, Wt)) / (2 * h) * (1 if p == 1.0 else 1j)
    assert np.all(np.triu(Lb, 1) == 0)
    Lb_cmp = Lb.copy()
    idx = np.arange(n)
    Lb_cmp[idx, idx] = Lb_cmp[idx, idx].real   # only Re(Lbar_ii) is a derivative
    assert rel(Lb_cmp, fdL) <= 1e-7


@pytest.mark.parametrize("dtype", [np.float64, np.complex128])
def test_adjoint_matches_torch_autograd(dtype):
    import torch
    n, r = 9, 4
    A = spd(n, 109, dtype)
    L = factor(A)
    B = rhs(n, r, 110, dtype)
    Wt = rhs(n, r, 111, dtype)
    Lt = torch.from_numpy(L).requires_grad_(True)
    Bt = torch.from_numpy(B).requires_grad_(True)
    Xt = torch.cholesky_solve(Bt, Lt, upper=False)
    torch.real(torch.sum(torch.conj(torch.from_numpy(Wt)) * Xt)).backward()
    X = oracle.potrs(L, B)
    Bb, Lb = oracle.potrs_adj(L, X, Wt)
    assert rel(Bb, Bt.grad.numpy()) <= 1e-12
    tg = np.tril(Lt.grad.numpy())
    ours = Lb.copy()
    if np.iscomplexobj(A):
        idx = np.arange(n)
        tg[idx, idx] = tg[idx, idx].real
        ours[idx, idx] = ours[idx, idx].real
    assert rel(ours, tg) <= 1e-12


def test_adjoint_accumulates_and_threads_agree():
    n, r = 30, 5
    A = W.gram_spd(3, n, 112, 1.0, np.float64)
    L = oracle.potrf(A)[0]
    B = np.stack([rhs(n, r, 113 + b, np.float64) for b in range(3)])
    Wt = np.stack([rhs(n, r, 120 + b, np.float64) for b in range(3)])
    X = oracle.potrs(L, B)
    B0 = np.full_like(B, 0.5)
    L0 = np.full_like(L, -0.25)
    Bb1, Lb1 = oracle.potrs_adj(L, X, Wt, threads=1)
    Bb2, Lb2 = oracle.potrs_adj(L, X, Wt, Bbar=B0, Lbar=L0, threads=3)
    assert np.allclose(Bb2, Bb1 + 0.5, rtol=0, atol=1e-15)
    tri = np.tril(np.ones((n, n), bool))
    assert np.allclose(np.where(tri, Lb2, 0), np.where(tri, Lb1 - 0.25, 0), rtol=0, atol=1e-14)
    assert np.all(Lb2[:, ~tri] == -0.25)   # upper triangle untouched
