"""GPU parity of the solve with the factor (chol_solve) and its reverse mode
(chol_solve_adj) against the oracle, through the C ABI: small and blocked
orders with ragged tiles, one to many right-hand sides, all four element
types, in place, skipped matrices, and the gradient chained through
chol_adj."""
import numpy as np
import pytest

import oracle
from differentiable_cholesky_gb300 import workloads as W
from parity_util import max_rel_err

pytestmark = pytest.mark.gpu

TOL_X = {np.dtype(np.float64): 1e-12, np.dtype(np.float32): 2e-5,
         np.dtype(np.complex128): 1e-12, np.dtype(np.complex64): 2e-5}
TOL_ADJ = {np.dtype(np.float64): 1e-10, np.dtype(np.float32): 1e-4,
           np.dtype(np.complex128): 1e-10, np.dtype(np.complex64): 1e-4}


def is_c(dtype):
    return np.issubdtype(np.dtype(dtype), np.complexfloating)


def make(batch, n, nrhs, seed, dtype):
    if is_c(dtype):
        A = W.hermitian_spd(batch, n, seed, 1.0, np.complex128)
        L = oracle.hpotrf(A)[0]
    else:
        A = W.gram_spd(batch, n, seed, 1.0, np.float64)
        L = oracle.potrf(A)[0]
    rng = np.random.default_rng(seed + 1)
    x = rng.standard_normal((4, batch, n, nrhs))
    B = x[0] + 1j * x[1] if is_c(dtype) else x[0]
    Xb = x[2] + 1j * x[3] if is_c(dtype) else x[2]
    return L.astype(dtype), B.astype(dtype), Xb.astype(dtype)


def dev(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def rel_lower(x, ref):
    return max_rel_err(x, ref, lower=True)


@pytest.mark.parametrize("dtype", [np.float64, np.float32, np.complex128, np.complex64])
@pytest.mark.parametrize("n,nrhs", [(1, 1), (7, 3), (64, 1), (65, 70), (130, 5), (300, 64)])
def test_solve_and_adjoint(n, nrhs, dtype):
    import torch
    from differentiable_cholesky_gb300 import binding
    L, B, Xbar = make(3, n, nrhs, 200 + n, dtype)
    X = binding.chol_solve(dev(L), dev(B))
    Bb, Lb = binding.chol_solve_adj(dev(L), X, dev(Xbar))
    torch.cuda.synchronize()
    X_ref = oracle.potrs(L.astype(np.complex128 if is_c(dtype) else np.float64),
                         B.astype(np.complex128 if is_c(dtype) else np.float64))
    Lh = L.astype(X_ref.dtype)
    Bb_ref, Lb_ref = oracle.potrs_adj(Lh, X_ref, Xbar.astype(X_ref.dtype))
    dt = np.dtype(dtype)
    assert max_rel_err(X.cpu().numpy(), X_ref) <= TOL_X[dt]
    assert max_rel_err(Bb.cpu().numpy(), Bb_ref) <= TOL_ADJ[dt]
    Lbn = Lb.cpu().numpy()
    assert np.all(np.triu(Lbn, 1) == 0)
    assert rel_lower(Lbn, Lb_ref) <= TOL_ADJ[dt]


@pytest.mark.parametrize("n", [20, 200])
def test_in_place_and_skipped_matrices(n):
    import torch
    from differentiable_cholesky_gb300 import binding
    L, B, Xbar = make(4, n, 9, 210, np.float64)
    st = np.array([0, 3, 0, 1], np.int32)
    Bt = dev(B)
    X = binding.chol_solve(dev(L), Bt, X=Bt, status=dev(st))
    assert X.data_ptr() == Bt.data_ptr()
    B0 = np.full_like(B, 0.5)
    L0 = np.full_like(L, -2.0)
    Bb, Lb = binding.chol_solve_adj(dev(L), X, dev(Xbar), adj_B=dev(B0), adj_L=dev(L0),
                                    status=dev(st))
    torch.cuda.synchronize()
    Xn = X.cpu().numpy()
    X_ref = oracle.potrs(L, B, status=st)
    Bb_ref, Lb_ref = oracle.potrs_adj(L, X_ref, Xbar, Bbar=B0, Lbar=L0, status=st)
    assert np.all(Xn[[1, 3]] == 0)
    assert max_rel_err(Xn[[0, 2]], X_ref[[0, 2]]) <= 1e-12
    assert np.all(Bb.cpu().numpy()[[1, 3]] == 0.5)
    assert np.all(Lb.cpu().numpy()[[1, 3]] == -2.0)
    assert max_rel_err(Bb.cpu().numpy(), Bb_ref) <= 1e-10
    assert max_rel_err(Lb.cpu().numpy(), Lb_ref) <= 1e-10   # upper stays -2 on both sides


def test_one_output_at_a_time_and_argument_checks():
    import torch
    from differentiable_cholesky_gb300 import binding
    n, nrhs = 90, 4
    L, B, Xbar = make(2, n, nrhs, 220, np.float64)
    X = binding.chol_solve(dev(L), dev(B))
    Bb, none = binding.chol_solve_adj(dev(L), X, dev(Xbar), want_L=False)
    none2, Lb = binding.chol_solve_adj(dev(L), X, dev(Xbar), want_B=False)
    Bb2, Lb2 = binding.chol_solve_adj(dev(L), X, dev(Xbar))
    torch.cuda.synchronize()
    assert none is None and none2 is None
    assert torch.equal(Bb, Bb2) and torch.equal(Lb, Lb2)
    lib = binding.load_library()
    Lt, Bt = dev(L), dev(B)
    # X overlapping L, a misaligned X, negative nrhs, nrhs = 0 (no-op)
    assert lib.chol_solve(2, n, nrhs, 1, Lt.data_ptr(), Bt.data_ptr(), Lt.data_ptr(), None, None) == -3
    assert lib.chol_solve(2, n, nrhs, 1, Lt.data_ptr(), Bt.data_ptr(), Bt.data_ptr() + 4, None, None) == -1
    assert lib.chol_solve(2, n, -1, 1, Lt.data_ptr(), Bt.data_ptr(), Bt.data_ptr(), None, None) == -1
    assert lib.chol_solve(2, n, 0, 1, None, None, None, None, None) == 0
    # adj_L overlapping X
    Xt = X
    assert lib.chol_solve_adj(2, n, nrhs, 1, Lt.data_ptr(), Xt.data_ptr(), dev(Xbar).data_ptr(),
                              None, Xt.data_ptr(), None, None) == -3


@pytest.mark.parametrize("dtype", [np.float64, np.complex128])
def test_gradient_chained_through_the_factorisation(dtype):
    """loss(X(A, B)) with X = A^-1 B computed as chol_fwd -> chol_solve; the
    reverse pass chol_solve_adj -> chol_adj gives dLoss/dA (lower entries) and
    dLoss/dB; both match the oracle's composition and, for A, the direct
    formula -tril-part of A^-1 Xbar X^H in the lower-entry convention."""
    import torch
    from differentiable_cholesky_gb300 import binding
    n, nrhs = 150, 3
    cx = is_c(dtype)
    A = (W.hermitian_spd(2, n, 230, 1.0, dtype) if cx else W.gram_spd(2, n, 230, 1.0, dtype))
    rng = np.random.default_rng(231)
    x = rng.standard_normal((4, 2, n, nrhs))
    B = (x[0] + 1j * x[1] if cx else x[0]).astype(dtype)
    Xbar = (x[2] + 1j * x[3] if cx else x[2]).astype(dtype)
    Lt, st = binding.chol_fwd(dev(A))
    Xt = binding.chol_solve(Lt, dev(B), status=st)
    Bb, Lb = binding.chol_solve_adj(Lt, Xt, dev(Xbar), status=st)
    Ab = binding.chol_adj(Lt, Lb, status=st)
    torch.cuda.synchronize()
    # direct: G = -A^-1 Xbar X^H (full-matrix gradient), lower-entry form
    X = np.linalg.solve(A, B)
    G = -np.linalg.solve(A, Xbar) @ np.conj(np.swapaxes(X, -1, -2))
    Gh = G + np.conj(np.swapaxes(G, -1, -2))
    idx = np.arange(n)
    exp = np.tril(Gh)
    exp[:, idx, idx] = np.real(G[:, idx, idx])
    assert max_rel_err(Bb.cpu().numpy(), np.linalg.solve(A, Xbar)) <= 1e-10
    assert max_rel_err(Ab.cpu().numpy(), exp, lower=True) <= 1e-9
