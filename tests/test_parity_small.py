"""GPU parity of the small path (n <= 64) against the oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
from differentiable_cholesky_gb300 import workloads as W
from parity_util import TOL_ADJ, TOL_L, gpu_fwd_adj, max_rel_err

pytestmark = pytest.mark.gpu


def check_against_oracle(A, Lbar, dtype, adj_A0=None, tile=0):
    dtype = np.dtype(dtype)
    L, st, G = gpu_fwd_adj(A, Lbar, tile=tile, adj_A0=adj_A0)
    # status: the same decision in the kernel's precision, bit-exact
    _, st_ref = oracle.potrf(A, dtype=dtype)
    assert np.array_equal(st.reshape(-1), st_ref.reshape(-1))
    ok = st.reshape(-1) == 0
    L_ref, _ = oracle.potrf(A.astype(np.float64))
    G_ref = oracle.potrf_adj(L_ref, Lbar.astype(np.float64),
                             Abar=None if adj_A0 is None else adj_A0.astype(np.float64),
                             status=st_ref)
    assert np.all(np.triu(L[ok], 1) == 0)
    assert max_rel_err(L, L_ref, mask=ok) <= TOL_L[dtype]
    assert max_rel_err(G, G_ref, mask=ok, lower=True) <= TOL_ADJ[dtype]
    return L, st, G


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("n", [1, 2, 3, 5, 7, 8, 9, 12, 15, 16, 17, 24, 31, 32, 33, 48, 63, 64])
def test_sizes(n, dtype):
    batch = 37  # not a multiple of any group count: ragged last block
    A = W.gram_spd(batch, n, 11 + n, 1.0, dtype)
    Lbar = W.tril_normal(batch, n, 12 + n, dtype)
    check_against_oracle(A, Lbar, dtype)


def test_batched_16_full():
    w = W.batched_16()
    check_against_oracle(w.A, w.adj_L, w.dtype)


def test_batched_64_full_with_status():
    w = W.batched_64()
    L, st, G = check_against_oracle(w.A, w.adj_L, w.dtype)
    assert np.array_equal(st, w.expected_status)
    bad = st != 0
    assert np.all(G[bad] == 0)  # skipped matrices keep adj_A untouched (zeros)


@pytest.mark.parametrize("n,dtype", [(16, np.float32), (64, np.float32), (20, np.float64)])
def test_unaligned_pointers_take_the_scalar_path(n, dtype):
    import torch
    from differentiable_cholesky_gb300 import binding
    batch = 9
    A = W.gram_spd(batch, n, 3, 1.0, dtype)
    Lbar = W.tril_normal(batch, n, 4, dtype)
    dev = torch.device("cuda:0")
    total = batch * n * n

    def shifted(x):
        buf = torch.zeros(total + 1, dtype=torch.from_numpy(x).dtype, device=dev)
        v = buf[1:].view(x.shape)
        v.copy_(torch.from_numpy(x))
        return v

    At, Lt, Lbt, Gt = shifted(A), shifted(np.zeros_like(A)), shifted(Lbar), shifted(np.zeros_like(A))
    assert At.data_ptr() % 16 != 0
    _, st = binding.chol_fwd(At, L=Lt)
    binding.chol_adj(Lt, Lbt, adj_A=Gt, status=st)
    torch.cuda.synchronize()
    L_ref, s_ref = oracle.potrf(A.astype(np.float64))
    G_ref = oracle.potrf_adj(L_ref, Lbar.astype(np.float64))
    assert np.array_equal(st.cpu().numpy(), s_ref)
    assert max_rel_err(Lt.cpu().numpy(), L_ref) <= TOL_L[np.dtype(dtype)]
    assert max_rel_err(Gt.cpu().numpy(), G_ref, lower=True) <= TOL_ADJ[np.dtype(dtype)]


@pytest.mark.parametrize("n", [16, 32, 64])
@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_upper_triangles_ignored_and_untouched(dtype, n):
    import torch
    from differentiable_cholesky_gb300 import binding
    batch = 5
    A = W.gram_spd(batch, n, 5, 1.0, dtype)
    Lbar = W.tril_normal(batch, n, 6, dtype)
    iu = np.triu_indices(n, 1)
    Ag = A.copy(); Ag[:, iu[0], iu[1]] = np.nan
    Lbg = Lbar.copy(); Lbg[:, iu[0], iu[1]] = 1e30
    G0 = np.full_like(A, 3.25)
    L1, s1, G1 = gpu_fwd_adj(A, Lbar, adj_A0=G0)
    dev = torch.device("cuda:0")
    Lt, st = binding.chol_fwd(torch.from_numpy(Ag).to(dev))
    Lt2 = Lt.clone()
    Lt2.view(batch, n, n)[:, iu[0], iu[1]] = -7.0  # garbage in L's upper triangle
    Gt = binding.chol_adj(Lt2, torch.from_numpy(Lbg).to(dev), adj_A=torch.from_numpy(G0).to(dev),
                          status=st)
    torch.cuda.synchronize()
    assert np.array_equal(Lt.cpu().numpy(), L1)
    assert np.array_equal(Gt.cpu().numpy(), G1)
    assert np.all(G1[:, iu[0], iu[1]] == 3.25)       # upper never written
    L_ref, _ = oracle.potrf(A.astype(np.float64))
    G_ref = oracle.potrf_adj(L_ref, Lbar.astype(np.float64), Abar=G0.astype(np.float64))
    assert max_rel_err(G1, G_ref, lower=True) <= TOL_ADJ[np.dtype(dtype)]


@pytest.mark.parametrize("n", [8, 16, 33])
def test_non_pd_and_nan_status(n):
    dtype = np.float32
    batch = 12
    A = W.gram_spd(batch, n, 8, 1.0, np.float64)
    A[1, 0, 0] = 0.0
    A[2, n - 1, n - 1] = -5.0
    A[3, n // 2, n // 2] = np.nan
    A[4] = -np.eye(n)
    A[5, :, :] = 1.0             # rank one: fails at the second pivot
    A = A.astype(dtype)
    Lbar = W.tril_normal(batch, n, 9, dtype)
    L, st, G = check_against_oracle(A, Lbar, dtype, adj_A0=np.zeros_like(A))
    assert st[1] == 1 and st[2] == n and st[3] == n // 2 + 1 and st[4] == 1 and st[5] == 2
    assert np.all(G[1:6] == 0)


def test_single_nonzero_seed_reaches_every_entry():
    """One non-zero adj_L entry in one matrix of the batch: the gradient must
    land on all the entries it reaches and on no other matrix."""
    n, batch = 8, 6
    dtype = np.float64
    A = W.gram_spd(batch, n, 13, 1.0, dtype)
    for (i, j) in [(0, 0), (7, 0), (5, 3), (7, 7)]:
        Lbar = np.zeros_like(A)
        Lbar[2, i, j] = 1.0
        L, st, G = check_against_oracle(A, Lbar, dtype)
        assert np.all(G[[0, 1, 3, 4, 5]] == 0)


def test_batch_of_one_and_zero():
    import torch
    from differentiable_cholesky_gb300 import binding
    A = W.gram_spd(1, 10, 14, 1.0, np.float64)
    Lbar = W.tril_normal(1, 10, 15, np.float64)
    check_against_oracle(A, Lbar, np.float64)
    empty = torch.empty((0, 10, 10), dtype=torch.float64, device="cuda:0")
    L, st = binding.chol_fwd(empty)
    G = binding.chol_adj(L, empty)
    assert L.shape == (0, 10, 10) and st.shape == (0,) and G.shape == (0, 10, 10)
