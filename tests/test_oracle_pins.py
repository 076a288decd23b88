"""Pins of the CPU oracle to facts outside itself (CPU only).

Each test checks the oracle against something it does not compute itself: the
pages' worked example, closed forms, exact textbook values, library routines
used as black boxes, exact symbolic differentiation and finite differences.
A dropped term, a wrong sign or index, or a transposed operand anywhere in the
forward or the adjoint fails at least one of them.
"""
import json
import os

import numpy as np
import pytest

import oracle
from differentiable_cholesky_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rel_fro(x, ref):
    den = np.linalg.norm(ref)
    return np.linalg.norm(np.asarray(x, np.float64) - ref) / (den if den > 0 else 1.0)


def phi(X):
    Y = np.tril(X).copy()
    idx = np.arange(X.shape[-1])
    Y[..., idx, idx] *= 0.5
    return Y


def spd(n, seed, shift=1.0):
    return W.gram_spd(1, n, seed, shift, np.float64)[0]


# ----------------------------------------------------------------------------
# Forward
# ----------------------------------------------------------------------------

def test_bidiagonal_worked_example_from_the_pages():
    """jaxmg docs 'Cholesky factorization': A = E E^T, factor must equal E."""
    g = json.load(open(os.path.join(GOLDEN, "bidiagonal_512.json")))
    n = g["N"]
    E = np.diag(np.linspace(g["E_diagonal"]["linspace_start"],
                            g["E_diagonal"]["linspace_stop"], n))
    E += np.diag(np.full(n - 1, g["E_subdiagonal"]), k=-1)
    A = E @ E.T
    L, st = oracle.potrf(A)
    assert int(st) == 0
    assert np.allclose(L, E)                      # the page's own check
    assert rel_fro(L, E) <= 1e-14


def test_textbook_integer_factor_is_exact():
    g = json.load(open(os.path.join(GOLDEN, "textbook_3x3.json")))
    A = np.array(g["A"], np.float64)
    L, st = oracle.potrf(A)
    assert int(st) == 0
    assert np.array_equal(L, np.array(g["L"], np.float64))
    Lf, stf = oracle.potrf(A.astype(np.float32))
    assert np.array_equal(Lf, np.array(g["L"], np.float32)) and int(stf) == 0


@pytest.mark.parametrize("n", [64, 300, 1024])
def test_banded_closed_form(n):
    E = W.banded_E(n, 32, seed=3)
    A = W.banded_gram(E, 32)
    L, st = oracle.potrf(A)
    assert int(st) == 0
    assert rel_fro(L, E) <= 1e-13


def test_small_closed_forms():
    # identity -> identity
    L, st = oracle.potrf(np.eye(7))
    assert int(st) == 0 and np.array_equal(L, np.eye(7))
    # diagonal -> square roots
    d = np.array([4.0, 9.0, 0.25, 2.0, 1e-6])
    L, st = oracle.potrf(np.diag(d))
    assert int(st) == 0 and np.array_equal(L, np.diag(np.sqrt(d)))
    # n = 1
    L, st = oracle.potrf(np.array([[6.25]]))
    assert L[0, 0] == 2.5 and int(st) == 0
    # n = 2: [sqrt a, 0; b / sqrt a, sqrt(c - b^2 / a)]
    a, b, c = 3.0, 1.2, 2.5
    L, st = oracle.potrf(np.array([[a, b], [b, c]]))
    ref = np.array([[np.sqrt(a), 0], [b / np.sqrt(a), np.sqrt(c - b * b / a)]])
    assert int(st) == 0 and rel_fro(L, ref) <= 1e-15


@pytest.mark.parametrize("n", [1, 2, 3, 7, 16, 33, 64, 100])
def test_residual_uniqueness_and_structure(n):
    A = spd(n, seed=n)
    L, st = oracle.potrf(A)
    assert int(st) == 0
    assert rel_fro(L @ L.T, A) <= 10 * n * np.finfo(np.float64).eps
    assert np.all(np.diag(L) > 0)
    assert np.all(np.triu(L, 1) == 0)


@pytest.mark.parametrize("n", [1, 5, 16, 64, 129])
def test_matches_lapack_through_torch(n):
    torch = pytest.importorskip("torch")
    A = spd(n, seed=100 + n)
    L, _ = oracle.potrf(A)
    ref = torch.linalg.cholesky(torch.from_numpy(A)).numpy()
    assert rel_fro(L, ref) <= 1e-13


def test_power_of_two_scaling_is_exact():
    # chol(4 A) = 2 chol(A) with every rounding scaled by the same power of two.
    A = spd(24, seed=5)
    L1, _ = oracle.potrf(A)
    L4, _ = oracle.potrf(4.0 * A)
    assert np.array_equal(L4, 2.0 * L1)


def test_upper_triangle_of_A_is_not_read():
    A = spd(12, seed=6)
    B = A.copy()
    B[np.triu_indices(12, 1)] = np.nan
    L1, s1 = oracle.potrf(A)
    L2, s2 = oracle.potrf(B)
    assert np.array_equal(L1, L2) and int(s1) == int(s2) == 0


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("k", [0, 1, 17, 63])
def test_status_first_bad_pivot(dtype, k):
    A = W.gram_spd(1, 64, 7, 0.5, np.float64)[0]
    A[k, k] = -1.0
    L, st = oracle.potrf(A.astype(dtype))
    assert int(st) == k + 1
    # LAPACK's info agrees (library used as a black box)
    torch = pytest.importorskip("torch")
    _, info = torch.linalg.cholesky_ex(torch.from_numpy(A))
    assert int(info) == k + 1
    # the leading k x k block is still the factor of the leading minor
    if k > 0:
        Lk, sk = oracle.potrf(A[:k, :k].astype(dtype))
        assert int(sk) == 0 and np.array_equal(L[:k, :k], Lk)


def test_status_special_pivots():
    assert int(oracle.potrf(np.zeros((4, 4)))[1]) == 1
    assert int(oracle.potrf(np.diag([1.0, 0.0, 1.0]))[1]) == 2
    A = np.eye(5)
    A[3, 3] = np.nan
    assert int(oracle.potrf(A)[1]) == 4
    assert int(oracle.potrf(-np.eye(3))[1]) == 1
    # singular PSD matrix: rank-1 ones(3) fails at the second pivot
    assert int(oracle.potrf(np.ones((3, 3)))[1]) == 2


def test_float32_tracks_float64():
    for n in (16, 64):
        A = W.gram_spd(4, n, 8, 1.0, np.float32)
        L32, s32 = oracle.potrf(A)
        L64, s64 = oracle.potrf(A.astype(np.float64))
        assert np.all(s32 == 0) and np.all(s64 == 0)
        for b in range(4):
            assert rel_fro(L32[b], L64[b]) <= 1e-6


def test_batched_equals_single():
    A = W.gram_spd(9, 10, 9, 1.0, np.float64)
    A[4, 2, 2] = -3.0
    Lb, sb = oracle.potrf(A, threads=3)
    for b in range(9):
        L, s = oracle.potrf(A[b])
        assert int(s) == int(sb[b])
        if s == 0:
            assert np.array_equal(L, Lb[b])
    assert int(sb[4]) == 3


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_threaded_single_matrix_path_is_bit_identical(dtype):
    """The single-matrix routines share independent rows (forward) and
    columns/rows (adjoint solves) out over threads without changing any sum's
    order: any thread count must give the one-thread result bit for bit."""
    n = 97
    A = spd(n, 21).astype(dtype)
    Lbar = W.tril_normal(1, n, 22, dtype)[0]
    L1, s1 = oracle.potrf(A, threads=1)
    G1 = oracle.potrf_adj(L1, Lbar, threads=1)
    for t in (2, 3, 8):
        Lt, st = oracle.potrf(A, threads=t)
        assert int(st) == int(s1) == 0
        assert np.array_equal(Lt, L1)
        Gt = oracle.potrf_adj(L1, Lbar, threads=t)
        assert np.array_equal(Gt, G1)
    # a failing pivot stops at the same column whatever the threads
    B = A.copy()
    B[40, 40] = -1
    assert int(oracle.potrf(B, threads=4)[1]) == int(oracle.potrf(B, threads=1)[1]) == 41


def test_workload_status_construction():
    w = W.batched_64(batch=500)
    _, st = oracle.potrf(w.A)
    assert np.array_equal(st, w.expected_status)
    assert np.count_nonzero(st) == 5


# ----------------------------------------------------------------------------
# Adjoint
# ----------------------------------------------------------------------------

def loss(A, Lbar):
    L, st = oracle.potrf(A)
    assert int(st) == 0
    return float(np.sum(Lbar * L))


@pytest.mark.parametrize("n", [1, 2, 3, 5, 8])
def test_adjoint_central_differences(n):
    """Brute force: d<tril(Lbar), L(A)>/d a_ij for every lower entry."""
    A = spd(n, seed=20 + n)
    Lbar = W.tril_normal(1, n, 30 + n, np.float64)[0]
    L, _ = oracle.potrf(A)
    G = oracle.potrf_adj(L, Lbar)
    fd = np.zeros_like(A)
    for i in range(n):
        for j in range(i + 1):
            h = 1e-6 * max(1.0, abs(A[i, j]))
            Ap = A.copy(); Ap[i, j] += h
            Am = A.copy(); Am[i, j] -= h
            fd[i, j] = (loss(Ap, Lbar) - loss(Am, Lbar)) / (2 * h)
    assert np.all(np.triu(G, 1) == 0)
    assert rel_fro(np.tril(G), fd) <= 1e-7


def test_adjoint_exact_symbolic_3x3():
    """sympy's own Cholesky, differentiated exactly, at the textbook matrix."""
    sympy = pytest.importorskip("sympy")
    g = json.load(open(os.path.join(GOLDEN, "textbook_3x3.json")))
    A0 = g["A"]
    sym = {}
    M = sympy.zeros(3, 3)
    for i in range(3):
        for j in range(i + 1):
            s = sympy.Symbol(f"a{i}{j}")
            sym[(i, j)] = s
            M[i, j] = s
            M[j, i] = s
    Ls = M.cholesky(hermitian=False)
    Lbar = np.array([[1, 0, 0], [-2, 3, 0], [5, -1, 2]], np.float64)
    f = sum(int(Lbar[i, j]) * Ls[i, j] for i in range(3) for j in range(i + 1))
    subs = {sym[(i, j)]: A0[i][j] for (i, j) in sym}
    exact = np.zeros((3, 3))
    for (i, j), s in sym.items():
        exact[i, j] = float(sympy.nsimplify(sympy.diff(f, s).subs(subs)))
    L, _ = oracle.potrf(np.array(A0, np.float64))
    G = oracle.potrf_adj(L, Lbar)
    assert rel_fro(G, exact) <= 1e-14


def test_adjoint_closed_forms():
    # n = 1: d sqrt(a) / da = 1 / (2 sqrt a)
    G = oracle.potrf_adj(np.array([[3.0]]), np.array([[1.5]]))
    assert abs(G[0, 0] - 1.5 / 6.0) <= 1e-16
    # identity A: Abar = Phi(Lbar)
    Lbar = W.tril_normal(1, 9, 40, np.float64)[0]
    G = oracle.potrf_adj(np.eye(9), Lbar)
    assert np.array_equal(G, phi(Lbar))
    # diagonal A = diag(d^2): Abar_ii = Lbar_ii / (2 d_i), Abar_ij = Lbar_ij / d_j
    d = np.array([1.0, 2.0, 4.0, 0.5, 8.0])
    G = oracle.potrf_adj(np.diag(d), W.tril_normal(1, 5, 41, np.float64)[0])
    Lb = W.tril_normal(1, 5, 41, np.float64)[0]
    ref = np.tril(Lb / d[None, :], -1) + np.diag(np.diag(Lb) / (2 * d))
    assert rel_fro(G, ref) <= 1e-16


@pytest.mark.parametrize("n", [4, 16, 50])
def test_adjoint_matches_torch_autograd(n):
    """torch's symmetric gradient G_t maps to ours as tril(G_t + G_t^T) - diag(G_t)."""
    torch = pytest.importorskip("torch")
    A = spd(n, seed=50 + n)
    Lbar = W.tril_normal(1, n, 60 + n, np.float64)[0]
    At = torch.from_numpy(A).requires_grad_(True)
    Lt = torch.linalg.cholesky(At)
    (Lt * torch.from_numpy(Lbar)).sum().backward()
    Gt = At.grad.numpy()
    ref = np.tril(Gt + Gt.T) - np.diag(np.diag(Gt))
    L, _ = oracle.potrf(A)
    G = oracle.potrf_adj(L, Lbar)
    assert rel_fro(G, ref) <= 1e-12


@pytest.mark.parametrize("n", [64, 200])
def test_adjoint_directional_derivative(n):
    A = spd(n, seed=70 + n)
    Lbar = W.tril_normal(1, n, 80 + n, np.float64)[0]
    D = W.tril_normal(1, n, 90 + n, np.float64)[0]
    L, _ = oracle.potrf(A)
    G = oracle.potrf_adj(L, Lbar)
    h = 1e-6
    fd = (loss(A + h * D, Lbar) - loss(A - h * D, Lbar)) / (2 * h)
    an = float(np.sum(G * D))
    assert abs(an - fd) <= 1e-6 * max(1.0, abs(an))


def test_adjoint_reads_only_lower_triangles_and_accumulates():
    n = 11
    A = spd(n, seed=91)
    L, _ = oracle.potrf(A)
    Lbar = W.tril_normal(1, n, 92, np.float64)[0]
    G = oracle.potrf_adj(L, Lbar)
    # garbage in the upper triangles of L and Lbar is ignored
    Lg, Lbg = L.copy(), Lbar.copy()
    iu = np.triu_indices(n, 1)
    Lg[iu] = 7.0
    Lbg[iu] = -3.0
    assert np.array_equal(oracle.potrf_adj(Lg, Lbg), G)
    # accumulation into Abar; its upper triangle is untouched
    A0 = np.random.default_rng(93).standard_normal((n, n))
    G2 = oracle.potrf_adj(L, Lbar, Abar=A0)
    assert np.array_equal(G2[iu], A0[iu])
    il = np.tril_indices(n)
    assert np.array_equal(G2[il], (A0 + G)[il])


def test_adjoint_skips_failed_matrices():
    A = W.gram_spd(3, 6, 94, 1.0, np.float64)
    L, st = oracle.potrf(A)
    Lbar = W.tril_normal(3, 6, 95, np.float64)
    status = np.array([0, 2, 0], np.int32)
    A0 = np.ones_like(A)
    G = oracle.potrf_adj(L, Lbar, Abar=A0, status=status)
    assert np.array_equal(G[1], A0[1])
    assert not np.array_equal(G[0], A0[0])
    Gb = oracle.potrf_adj(L[2], Lbar[2], Abar=A0[2])
    assert np.array_equal(G[2], Gb)


def test_adjoint_float32_tracks_float64():
    for n in (16, 64):
        A = W.gram_spd(3, n, 96, 1.0, np.float32)
        Lbar = W.tril_normal(3, n, 97, np.float32)
        L32, _ = oracle.potrf(A)
        G32 = oracle.potrf_adj(L32, Lbar)
        L64, _ = oracle.potrf(A.astype(np.float64))
        G64 = oracle.potrf_adj(L64, Lbar.astype(np.float64))
        for b in range(3):
            assert rel_fro(G32[b], G64[b]) <= 1e-5


def test_workload_generators_are_deterministic_and_shaped():
    w = W.batched_16(batch=64)
    w2 = W.batched_16(batch=64)
    assert np.array_equal(w.A, w2.A) and np.array_equal(w.adj_L, w2.adj_L)
    assert w.A.shape == (64, 16, 16) and w.A.dtype == np.float32
    assert np.all(np.triu(w.adj_L, 1) == 0)
    E = W.banded_E(100, 32, 0)
    assert np.abs(W.banded_gram(E, 32) - E @ E.T).max() <= 1e-14
