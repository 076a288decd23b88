"""GPU parity of the complex Hermitian path (A = L L^H and its adjoint)
against the complex oracle, through the C ABI: the small path (n <= 64, one
block per matrix) and the blocked path (conjugate transposes in the panel
solve and the GEMM-shaped updates), complex64 and complex128."""
import numpy as np
import pytest

import oracle
from differentiable_cholesky_gb300 import workloads as W
from parity_util import max_rel_err

pytestmark = pytest.mark.gpu

TOL_L = {np.dtype(np.complex128): 1e-12, np.dtype(np.complex64): 2e-5}
TOL_ADJ = {np.dtype(np.complex128): 1e-10, np.dtype(np.complex64): 1e-4}


def gpu_run(A, Lbar, tile=0, adj_A0=None, inplace=False):
    import torch
    from differentiable_cholesky_gb300 import binding
    dev = torch.device("cuda:0")
    At = torch.from_numpy(np.ascontiguousarray(A)).to(dev)
    Lbt = torch.from_numpy(np.ascontiguousarray(Lbar)).to(dev)
    if inplace:
        Lt, st = binding.chol_fwd_inplace(At.clone(), tile=tile)
        Gt = binding.chol_adj_inplace(Lt, Lbt.clone(), status=st, tile=tile)
    else:
        Lt, st = binding.chol_fwd(At, tile=tile)
        G0 = None if adj_A0 is None else torch.from_numpy(np.ascontiguousarray(adj_A0)).to(dev)
        Gt = binding.chol_adj(Lt, Lbt, adj_A=G0, status=st, tile=tile)
    torch.cuda.synchronize()
    return Lt.cpu().numpy(), st.cpu().numpy(), Gt.cpu().numpy()


def check(A, Lbar, dtype, tile=0, adj_A0=None, inplace=False):
    dtype = np.dtype(dtype)
    L, st, G = gpu_run(A, Lbar, tile=tile, adj_A0=adj_A0, inplace=inplace)
    _, st_ref = oracle.hpotrf(A, dtype=dtype)
    assert np.array_equal(st.reshape(-1), st_ref.reshape(-1))
    ok = st.reshape(-1) == 0
    L_ref, _ = oracle.hpotrf(A.astype(np.complex128))
    G_ref = oracle.hpotrf_adj(L_ref, Lbar.astype(np.complex128),
                              Abar=None if adj_A0 is None else adj_A0.astype(np.complex128),
                              status=st_ref)
    assert np.all(np.triu(L[ok], 1) == 0)
    assert np.all(L[ok].diagonal(axis1=-2, axis2=-1).imag == 0)
    assert max_rel_err(L, L_ref, mask=ok) <= TOL_L[dtype]
    assert max_rel_err(G, G_ref, mask=ok, lower=True) <= TOL_ADJ[dtype]
    return L, st, G


@pytest.mark.parametrize("dtype", [np.complex128, np.complex64])
@pytest.mark.parametrize("n", [1, 2, 5, 16, 31, 33, 64])
def test_small_sizes(n, dtype):
    A = W.hermitian_spd(37, n, 80 + n, 1.0, dtype)
    Lbar = W.tril_normal_complex(37, n, 81 + n, dtype)
    check(A, Lbar, dtype)


@pytest.mark.parametrize("dtype", [np.complex128, np.complex64])
@pytest.mark.parametrize("n,tile", [(65, 0), (130, 32), (200, 64), (300, 0)])
def test_blocked_sizes(n, tile, dtype):
    A = W.hermitian_spd(3, n, 82 + n, 1.0, dtype)
    Lbar = W.tril_normal_complex(3, n, 83 + n, dtype)
    check(A, Lbar, dtype, tile=tile)


def test_complex64_tile_128():
    A = W.hermitian_spd(2, 260, 84, 1.0, np.complex64)
    Lbar = W.tril_normal_complex(2, 260, 85, np.complex64)
    check(A, Lbar, np.complex64, tile=128)


def test_complex128_rejects_tile_128():
    import torch
    from differentiable_cholesky_gb300 import binding
    A = torch.from_numpy(W.hermitian_spd(1, 130, 86, 1.0, np.complex128)).cuda()
    with pytest.raises(binding.CholError) as e:
        binding.chol_fwd(A, tile=128)
    assert e.value.code == -1


@pytest.mark.parametrize("n", [12, 100])
def test_status_skip_and_accumulate(n):
    A = W.hermitian_spd(4, n, 87, 1.0, np.complex128)
    A[1, n // 2, n // 2] = -1.0
    A[2, 0, 0] = np.nan
    Lbar = W.tril_normal_complex(4, n, 88, np.complex128)
    G0 = np.full_like(A, 1.5 - 0.5j)
    L, st, G = check(A, Lbar, np.complex128, adj_A0=G0)
    assert list(st) == [0, n // 2 + 1, 1, 0]
    assert np.all(G[1:3] == 1.5 - 0.5j)
    # the upper triangle of adj_A is never written
    iu = np.triu_indices(n, 1)
    assert np.all(G[:, iu[0], iu[1]] == 1.5 - 0.5j)


@pytest.mark.parametrize("n", [20, 150])
def test_upper_triangle_and_imaginary_diagonal_ignored(n):
    A = W.hermitian_spd(2, n, 89, 1.0, np.complex128)
    Lbar = W.tril_normal_complex(2, n, 90, np.complex128)
    L1, _, G1 = gpu_run(A, Lbar)
    B = A.copy()
    iu = np.triu_indices(n, 1)
    B[:, iu[0], iu[1]] = np.nan
    B[:, np.arange(n), np.arange(n)] += 1j * 7.0
    Lb2 = Lbar.copy()
    Lb2[:, iu[0], iu[1]] = 1e30
    L2, _, G2 = gpu_run(B, Lb2)
    assert np.array_equal(L1, L2)
    assert np.array_equal(G1, G2)


@pytest.mark.parametrize("n", [16, 130])
def test_inplace_forms(n):
    A = W.hermitian_spd(3, n, 91, 1.0, np.complex128)
    Lbar = W.tril_normal_complex(3, n, 92, np.complex128)
    L1, s1, G1 = gpu_run(A, Lbar)
    L2, s2, G2 = gpu_run(A, Lbar, inplace=True)
    assert np.array_equal(L1, L2) and np.array_equal(s1, s2)
    tri = np.tril(np.ones((n, n), bool))
    assert np.array_equal(np.where(tri, G1, 0), np.where(tri, G2, 0))


def test_autograd_wrapper_complex():
    import torch
    from differentiable_cholesky_gb300 import binding
    n = 24
    A = W.hermitian_spd(2, n, 93, 1.0, np.complex128)
    Lbar = W.tril_normal_complex(2, n, 94, np.complex128)
    At = torch.from_numpy(A).cuda().requires_grad_(True)
    L, st = binding.cholesky(At)
    torch.real(torch.sum(torch.conj(torch.from_numpy(Lbar).cuda()) * L)).backward()
    L_ref, _ = oracle.hpotrf(A)
    G_ref = oracle.hpotrf_adj(L_ref, Lbar)
    assert max_rel_err(At.grad.cpu().numpy(), G_ref) <= 1e-10
