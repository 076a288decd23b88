"""Pins of the complex Hermitian oracle (``oracle.hpotrf`` / ``hpotrf_adj``)
to facts outside itself (CPU only): closed forms, LAPACK through torch,
central finite differences on the real and imaginary parts of every lower
entry, torch's complex autograd, and the reduction to the (separately pinned)
real case.  A dropped conjugate anywhere fails the finite differences."""
import numpy as np
import pytest

import oracle
from differentiable_cholesky_gb300 import workloads as W


def rel(x, ref):
    den = np.linalg.norm(ref)
    return np.linalg.norm(np.asarray(x) - ref) / (den if den > 0 else 1.0)


def herm(n, seed, shift=1.0):
    return W.hermitian_spd(1, n, seed, shift, np.complex128)[0]


def test_bidiagonal_closed_form():
    """A = E E^H with E lower bidiagonal (real positive diagonal, complex
    sub-diagonal): the factor is E itself."""
    n = 64
    E = np.diag(np.linspace(1.0, 2.0, n)).astype(np.complex128)
    E += np.diag(np.full(n - 1, 0.5 + 0.3j), -1)
    L, s = oracle.hpotrf(E @ E.conj().T)
    assert int(s) == 0
    assert rel(L, E) <= 1e-15


@pytest.mark.parametrize("n", [1, 2, 7, 33])
def test_matches_lapack_through_torch(n):
    import torch
    A = herm(n, 50 + n)
    L, s = oracle.hpotrf(A)
    ref = torch.linalg.cholesky(torch.from_numpy(A)).numpy()
    assert int(s) == 0
    assert rel(L, ref) <= 1e-14
    assert np.all(np.triu(L, 1) == 0)
    assert np.all(L.diagonal().imag == 0) and np.all(L.diagonal().real > 0)
    assert rel(L @ L.conj().T, A) <= 1e-14


def test_reads_lower_triangle_and_real_diagonal_only():
    n = 9
    A = herm(n, 51)
    B = A.copy()
    iu = np.triu_indices(n, 1)
    B[iu] = np.nan
    B[np.arange(n), np.arange(n)] += 1j * np.linspace(-3, 3, n)
    La, _ = oracle.hpotrf(A)
    Lb, _ = oracle.hpotrf(B)
    assert np.array_equal(La, Lb)


def test_real_input_reduces_to_the_real_factor():
    n = 20
    A = W.gram_spd(1, n, 52, 1.0, np.float64)[0]
    Lr, _ = oracle.potrf(A)
    Lc, _ = oracle.hpotrf(A.astype(np.complex128))
    assert np.array_equal(Lc.real, Lr) and np.all(Lc.imag == 0)
    Lbar = W.tril_normal(1, n, 53, np.float64)[0]
    Gr = oracle.potrf_adj(Lr, Lbar)
    Gc = oracle.hpotrf_adj(Lc, Lbar.astype(np.complex128))
    assert rel(Gc.real, Gr) <= 1e-14 and np.abs(Gc.imag).max() <= 1e-14 * np.abs(Gr).max()


@pytest.mark.parametrize("k", [0, 3, 7])
def test_status_first_bad_pivot(k):
    A = herm(8, 54)
    A[k, k] = -1.0
    _, s = oracle.hpotrf(A)
    assert int(s) == k + 1
    A[k, k] = np.nan
    assert int(oracle.hpotrf(A)[1]) == k + 1


def loss(A, G):
    """Real scalar loss Re sum conj(G) * L(A)."""
    L, s = oracle.hpotrf(A)
    assert int(s) == 0
    return float(np.real(np.sum(np.conj(G) * L)))


@pytest.mark.parametrize("n", [1, 2, 3, 5])
def test_adjoint_central_differences(n):
    """dLoss/dRe(a_ij) + i dLoss/dIm(a_ij) for every lower entry, and
    dLoss/dRe(a_ii) on the diagonal (Im(a_ii) is not read)."""
    A = herm(n, 60 + n)
    G = np.tril(W.tril_normal(1, n, 61, np.float64)[0] + 1j * W.tril_normal(1, n, 62, np.float64)[0])
    L, _ = oracle.hpotrf(A)
    Ab = oracle.hpotrf_adj(L, G)
    h = 1e-6
    fd = np.zeros_like(A)
    for i in range(n):
        for j in range(i + 1):
            for part in ((1.0,) if i == j else (1.0, 1j)):
                Ap, Am = A.copy(), A.copy()
                Ap[i, j] += h * part
                Am[i, j] -= h * part
                if i != j:  # keep the matrix Hermitian for numpy's sake (upper not read)
                    Ap[j, i] = np.conj(Ap[i, j])
                    Am[j, i] = np.conj(Am[i, j])
                d = (loss(Ap, G) - loss(Am, G)) / (2 * h)
                fd[i, j] += d * (1.0 if part == 1.0 else 1j)
    assert np.all(np.triu(Ab, 1) == 0)
    assert np.all(Ab.diagonal().imag == 0)
    assert rel(np.tril(Ab), fd) <= 1e-7


def test_adjoint_imaginary_diagonal_of_lbar_is_ignored():
    n = 6
    A = herm(n, 63)
    L, _ = oracle.hpotrf(A)
    G = np.tril(W.tril_normal(1, n, 64, np.float64)[0] + 1j * W.tril_normal(1, n, 65, np.float64)[0])
    G2 = G.copy()
    G2[np.arange(n), np.arange(n)] += 1j * 5.0
    assert rel(oracle.hpotrf_adj(L, G2), oracle.hpotrf_adj(L, G)) <= 1e-14


def test_adjoint_closed_forms():
    # n = 1: d sqrt(a) / da = 1 / (2 sqrt(a)); only Re(Lbar) matters
    a, g = 2.25, 0.8 - 0.4j
    L, _ = oracle.hpotrf(np.array([[a]], np.complex128))
    Ab = oracle.hpotrf_adj(L, np.array([[g]], np.complex128))
    assert abs(Ab[0, 0] - g.real / (2 * np.sqrt(a))) <= 1e-16
    # identity: Abar = Lbar below the diagonal, Re(Lbar_ii) / 2 on it
    n = 5
    G = np.tril(W.tril_normal(1, n, 66, np.float64)[0] + 1j * W.tril_normal(1, n, 67, np.float64)[0])
    I = np.eye(n, dtype=np.complex128)
    Ab = oracle.hpotrf_adj(I, G)
    exp = np.tril(G, -1) + np.diag(G.diagonal().real / 2)
    assert rel(Ab, exp) <= 1e-16


@pytest.mark.parametrize("n", [3, 12])
def test_adjoint_matches_torch_autograd(n):
    """torch's gradient Gt of Re sum conj(G) L(A) with respect to the full
    Hermitian A maps to the lower-entry convention by tril(Gt + Gt^H) - diag(Gt)."""
    import torch
    A = herm(n, 68 + n)
    G = np.tril(W.tril_normal(1, n, 69, np.float64)[0] + 1j * W.tril_normal(1, n, 70, np.float64)[0])
    At = torch.from_numpy(A).requires_grad_(True)
    Lt = torch.linalg.cholesky(At)
    torch.real(torch.sum(torch.conj(torch.from_numpy(G)) * Lt)).backward()
    Gt = At.grad.numpy()
    mapped = np.tril(Gt + Gt.conj().T) - np.diag(np.diag(Gt))
    L, _ = oracle.hpotrf(A)
    Ab = oracle.hpotrf_adj(L, G)
    assert rel(np.tril(Ab, -1), np.tril(mapped, -1)) <= 1e-12
    assert rel(Ab.diagonal().real, mapped.diagonal().real) <= 1e-12


def test_batched_equals_single_and_skips_failed():
    A = W.hermitian_spd(5, 11, 71, 1.0, np.complex128)
    A[2, 4, 4] = -2.0
    G = W.tril_normal(5, 11, 72, np.float64).astype(np.complex128)
    Lb, sb = oracle.hpotrf(A, threads=3)
    assert list(sb) == [0, 0, 5, 0, 0]
    Gb = oracle.hpotrf_adj(Lb, G, status=sb, threads=3)
    assert np.all(Gb[2] == 0)
    for b in (0, 1, 3, 4):
        L, s = oracle.hpotrf(A[b])
        assert np.array_equal(L, Lb[b])
        assert np.array_equal(oracle.hpotrf_adj(L, G[b]), Gb[b])


def test_threaded_single_matrix_is_bit_identical():
    n = 70
    A = herm(n, 73)
    G = np.tril(W.tril_normal(1, n, 74, np.float64)[0] + 1j * W.tril_normal(1, n, 75, np.float64)[0])
    L1, _ = oracle.hpotrf(A, threads=1)
    G1 = oracle.hpotrf_adj(L1, G, threads=1)
    for t in (2, 5):
        assert np.array_equal(oracle.hpotrf(A, threads=t)[0], L1)
        assert np.array_equal(oracle.hpotrf_adj(L1, G, threads=t), G1)


def test_complex64_tracks_complex128():
    A = W.hermitian_spd(4, 16, 76, 1.0, np.complex64)
    L32, s32 = oracle.hpotrf(A)
    L64, s64 = oracle.hpotrf(A.astype(np.complex128))
    assert np.all(s32 == 0) and np.all(s64 == 0)
    G = W.tril_normal(4, 16, 77, np.float32).astype(np.complex64)
    G32 = oracle.hpotrf_adj(L32, G)
    G64 = oracle.hpotrf_adj(L64, G.astype(np.complex128))
    for b in range(4):
        assert rel(L32[b], L64[b]) <= 1e-6
        assert rel(G32[b], G64[b]) <= 1e-5
