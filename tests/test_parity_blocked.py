"""GPU parity of the blocked path (n > 64) against the oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
from differentiable_cholesky_gb300 import workloads as W
from parity_util import TOL_ADJ, TOL_L, gpu_fwd_adj, max_rel_err

pytestmark = pytest.mark.gpu


def check(A, Lbar, dtype, tile=0, adj_A0=None, expect_L=None):
    dtype = np.dtype(dtype)
    L, st, G = gpu_fwd_adj(A, Lbar, tile=tile, adj_A0=adj_A0)
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
    if expect_L is not None:
        assert max_rel_err(L, expect_L) <= TOL_L[dtype]
    return L, st, G


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("n", [65, 96, 127, 128, 129, 200, 257, 300])
def test_sizes_default_tile(n, dtype):
    A = W.gram_spd(3, n, 21 + n, 1.0, dtype)
    Lbar = W.tril_normal(3, n, 22 + n, dtype)
    check(A, Lbar, dtype)


@pytest.mark.parametrize("tile", [32, 64, 128])
@pytest.mark.parametrize("n", [65, 190, 300])
def test_explicit_tiles(n, tile):
    A = W.gram_spd(2, n, 23, 1.0, np.float64)
    Lbar = W.tril_normal(2, n, 24, np.float64)
    check(A, Lbar, np.float64, tile=tile)


def test_tile_independence():
    n = 300
    A = W.gram_spd(2, n, 25, 1.0, np.float64)
    Lbar = W.tril_normal(2, n, 26, np.float64)
    outs = [gpu_fwd_adj(A, Lbar, tile=t) for t in (32, 64, 128)]
    for L, st, G in outs[1:]:
        assert max_rel_err(L, outs[0][0]) <= 1e-13
        assert max_rel_err(G, outs[0][2], lower=True) <= 1e-12


def test_bidiagonal_512_closed_form():
    """jaxmg docs worked example: the factor of E E^T is E (N = 512, T_A = 128)."""
    w = W.bidiagonal_512()
    check(w.A, w.adj_L, np.float64, tile=128, expect_L=w.expected_L)


def test_batched_512_full_size():
    """All 256 matrices of the 256 x 512x512 float64 workload (tile 128, the
    tensor-core path) against the oracle, batch-parallel on the host cores."""
    w = W.batched_512()
    L, st, G = gpu_fwd_adj(w.A, w.adj_L, tile=128)
    assert np.all(st == 0)
    assert np.all(np.triu(L, 1) == 0)
    th = oracle.max_threads()
    L_ref, s = oracle.potrf(w.A, threads=th)
    assert np.all(s == 0)
    G_ref = oracle.potrf_adj(L_ref, w.adj_L, threads=th)
    assert max_rel_err(L, L_ref) <= 1e-12
    assert max_rel_err(G, G_ref, lower=True) <= 1e-10


def test_banded_8192_full_size():
    """L equals the banded E (closed form); the adjoint satisfies
    L^T Z L = S + S^T with Z = adj_A + adj_A^T, S = Phi(L^T tril(adj_L)),
    checked on 72 columns (the relation determines Z uniquely): the first
    and last, the middle, and 64 drawn at random."""
    w = W.banded_8192()
    L, st, G = gpu_fwd_adj(w.A, w.adj_L, tile=128)
    assert int(st[0]) == 0
    E = w.expected_L[0]
    assert max_rel_err(L, E[None]) <= 1e-12
    Gl = np.tril(G[0])
    Lb = w.adj_L[0]
    n = E.shape[0]
    rng = np.random.default_rng(7)
    J = np.array([0, 1, 2, n // 2, n // 2 + 1, n - 3, n - 2, n - 1]
                 + list(rng.choice(np.arange(3, n - 3), 64, replace=False)))
    EJ = E[:, J]
    lhs = E.T @ (Gl @ EJ + Gl.T @ EJ)             # L^T Z L e_j, column per j
    col_p = E.T @ Lb[:, J]                         # (L^T Lbar)_{:, j}
    row_p = (Lb.T @ EJ)                            # (L^T Lbar)_{j, :} as columns
    rows = np.arange(n)[:, None]
    rhs = np.where(rows > J[None, :], col_p, 0.0)  # S_ij, i > j
    rhs += np.where(rows < J[None, :], row_p, 0.0)  # S_ji, i < j
    rhs += np.where(rows == J[None, :], col_p, 0.0)  # 2 * S_jj = P_jj
    err = np.linalg.norm(lhs - rhs, axis=0) / np.linalg.norm(rhs, axis=0)
    assert err.max() <= 1e-10, (J[err.argmax()], err.max())


@pytest.mark.parametrize("tile", [32, 64, 128])
def test_status_global_column_and_skip(tile):
    n, batch = 200, 4
    A = W.gram_spd(batch, n, 27, 1.0, np.float64)
    A[1, 150, 150] = -1.0
    A[2, 0, 0] = 0.0
    A[3, 199, 199] = np.nan
    Lbar = W.tril_normal(batch, n, 28, np.float64)
    G0 = np.full_like(A, 2.0)
    L, st, G = check(A, Lbar, np.float64, tile=tile, adj_A0=G0)
    assert list(st) == [0, 151, 1, 200]
    assert np.all(G[1:] == 2.0)


@pytest.mark.parametrize("tile", [64, 128])
def test_nonfinite_off_diagonal_sets_the_status_of_its_row(tile):
    """A NaN or Inf below the diagonal reaches the pivot of its row through
    the panel solve and the trailing updates (with 128-wide float64 tiles,
    through the tensor-core update's non-finite rows): the status is that
    row's column + 1, as in the oracle."""
    n, batch = 300, 3
    A = W.gram_spd(batch, n, 41, 1.0, np.float64)
    A[0, 170, 20] = np.nan
    A[1, 250, 140] = np.inf
    Lbar = W.tril_normal(batch, n, 42, np.float64)
    L, st, G = check(A, Lbar, np.float64, tile=tile)
    assert list(st) == [171, 251, 0]


@pytest.mark.parametrize("n", [129, 255, 256, 257, 383, 640])
def test_tensor_core_trailing_update_sizes(n):
    """float64 with 128-wide tiles: the trailing update runs on the tensor
    cores (digit slices, exact fp32 accumulation); ragged last tiles, one and
    several trailing tiles, odd batches."""
    A = W.gram_spd(3, n, 43 + n, 1.0, np.float64)
    Lbar = W.tril_normal(3, n, 44 + n, np.float64)
    check(A, Lbar, np.float64, tile=128)


def test_tensor_core_update_wide_dynamic_range():
    """Rows of very different scales (a diagonal scaling D A D with D spanning
    2^-40 .. 2^40): each row is split with its own power-of-two scale, so the
    factor keeps full relative accuracy, D L, as the FP64 recurrence does."""
    n = 384
    A = W.gram_spd(1, n, 45, 1.0, np.float64)[0]
    d = np.exp2(np.linspace(-40, 40, n))
    As = (d[:, None] * A * d[None, :])[None]
    Lbar = W.tril_normal(1, n, 46, np.float64)
    L, st, G = gpu_fwd_adj(As, Lbar, tile=128)
    assert int(st[0]) == 0
    L_ref, _ = oracle.potrf(As[0])
    # compare row by row, relative to each row's own scale
    Lr = L[0] / d[:, None]
    Rr = L_ref / d[:, None]
    assert np.max(np.abs(Lr - Rr)) <= 1e-12 * np.max(np.abs(Rr))
    # the adjoint scales as D^-1 G D^-1 (G of the unscaled problem with
    # adj_L scaled by D^-1 ... compared entrywise after undoing the scaling)
    G_ref = oracle.potrf_adj(L_ref, Lbar[0])
    Gr = np.tril(G[0]) * d[:, None] * d[None, :]
    Rg = np.tril(G_ref) * d[:, None] * d[None, :]
    assert np.max(np.abs(Gr - Rg)) <= 1e-10 * np.max(np.abs(Rg))


@pytest.mark.parametrize("n", [200, 384])
def test_tensor_core_adjoint_agrees_with_the_fp64_sweep(n):
    """float64 with 128-wide tiles: chol_adj (and chol_adj_inplace) take the
    adjoint's two large updates on the tensor cores (digit slices), while
    chol_adj_noalloc runs the same reverse sweep on the FP64 pipe; both match
    the oracle and each other."""
    import torch
    from differentiable_cholesky_gb300 import binding
    A = W.gram_spd(3, n, 47 + n, 1.0, np.float64)
    Lbar = W.tril_normal(3, n, 48 + n, np.float64)
    dev = torch.device("cuda:0")
    Lt, st = binding.chol_fwd(torch.from_numpy(A).to(dev), tile=128)
    G_tc = binding.chol_adj(Lt, torch.from_numpy(Lbar).to(dev), status=st, tile=128)
    G_ip = torch.zeros_like(Lt)
    Lb = torch.from_numpy(Lbar).to(dev)
    lib = binding.load_library()
    assert lib.chol_adj_noalloc(3, n, 1, Lt.data_ptr(), Lb.data_ptr(), G_ip.data_ptr(),
                                st.data_ptr(), 128,
                                torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    L_ref, _ = oracle.potrf(A)
    G_ref = oracle.potrf_adj(L_ref, Lbar)
    g1, g2 = G_tc.cpu().numpy(), G_ip.cpu().numpy()
    assert max_rel_err(g1, G_ref, lower=True) <= 1e-10
    assert max_rel_err(g2, G_ref, lower=True) <= 1e-10
    assert max_rel_err(g1, g2, lower=True) <= 1e-12


def test_upper_triangles_ignored_and_untouched():
    import torch
    from differentiable_cholesky_gb300 import binding
    n, batch = 150, 2
    A = W.gram_spd(batch, n, 29, 1.0, np.float64)
    Lbar = W.tril_normal(batch, n, 30, np.float64)
    iu = np.triu_indices(n, 1)
    Ag = A.copy(); Ag[:, iu[0], iu[1]] = np.nan
    Lbg = Lbar.copy(); Lbg[:, iu[0], iu[1]] = 1e30
    G0 = np.full_like(A, -1.5)
    L1, s1, G1 = gpu_fwd_adj(A, Lbar, adj_A0=G0, tile=64)
    dev = torch.device("cuda:0")
    Lt, st = binding.chol_fwd(torch.from_numpy(Ag).to(dev), tile=64)
    Lt2 = Lt.clone()
    Lt2[:, iu[0], iu[1]] = 3.0
    Gt = binding.chol_adj(Lt2, torch.from_numpy(Lbg).to(dev), adj_A=torch.from_numpy(G0).to(dev),
                          status=st, tile=64)
    torch.cuda.synchronize()
    assert np.array_equal(Lt.cpu().numpy(), L1)
    assert np.array_equal(Gt.cpu().numpy(), G1)
    assert np.all(G1[:, iu[0], iu[1]] == -1.5)


def test_autograd_wrapper_matches_the_adjoint():
    import torch
    from differentiable_cholesky_gb300 import binding
    dev = torch.device("cuda:0")
    for n in (12, 100):
        A = W.gram_spd(2, n, 31, 1.0, np.float64)
        Lbar = W.tril_normal(2, n, 32, np.float64)
        At = torch.from_numpy(A).to(dev).requires_grad_(True)
        L, st = binding.cholesky(At)
        (L * torch.from_numpy(Lbar).to(dev)).sum().backward()
        L_ref, _ = oracle.potrf(A)
        G_ref = oracle.potrf_adj(L_ref, Lbar)
        assert max_rel_err(At.grad.cpu().numpy(), G_ref) <= 1e-10


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("n,tile", [(128, 128), (200, 128), (300, 64), (383, 128), (97, 64)])
def test_cluster_diagonal_factor_matches_the_single_block_factor(n, tile, dtype):
    """Few matrices factor their diagonal tiles on a cluster of SMs and (float64,
    128-wide tiles) take each diagonal tile's adjoint by its literal formula;
    many matrices use one block per tile and the reverse sweep.  The same
    matrix in a batch of 1 and inside a batch of 40 agrees to rounding, and
    both match the oracle, ragged last tiles included."""
    dtype = np.dtype(dtype)
    A1 = W.gram_spd(1, n, 61 + n, 1.0, dtype)
    Lbar1 = W.tril_normal(1, n, 62 + n, dtype)
    A40 = np.concatenate([W.gram_spd(39, n, 63 + n, 1.0, dtype), A1])
    Lbar40 = np.concatenate([W.tril_normal(39, n, 64 + n, dtype), Lbar1])
    L1, s1, G1 = check(A1, Lbar1, dtype, tile=tile)
    L40, s40, G40 = check(A40, Lbar40, dtype, tile=tile)
    tol = 1e-13 if dtype == np.float64 else 2e-6
    assert max_rel_err(L1, L40[-1:]) <= tol
    assert max_rel_err(G1, G40[-1:], lower=True) <= (1e-11 if dtype == np.float64 else 2e-5)


def test_cluster_of_8_and_cluster_of_16_agree():
    """One or a few matrices take a 16-SM cluster per diagonal tile (where the
    device schedules one), up to SMs / 8 matrices an 8-SM cluster: the same
    matrix factored in a batch of 1 and in a batch of 10 agrees to rounding,
    with and without the tile's inverse (tile 128 float64: the tensor-core
    panel solve uses it; tile 64 does not)."""
    n = 300
    for tile in (128, 64):
        A1 = W.gram_spd(1, n, 93, 1.0, np.float64)
        Lbar1 = W.tril_normal(1, n, 94, np.float64)
        A10 = np.concatenate([W.gram_spd(9, n, 95, 1.0, np.float64), A1])
        Lbar10 = np.concatenate([W.tril_normal(9, n, 96, np.float64), Lbar1])
        L1, _, G1 = check(A1, Lbar1, np.float64, tile=tile)
        L10, _, G10 = check(A10, Lbar10, np.float64, tile=tile)
        assert max_rel_err(L1, L10[-1:]) <= 1e-13
        assert max_rel_err(G1, G10[-1:], lower=True) <= 1e-11


@pytest.mark.parametrize("tile", [64, 128])
def test_cluster_diagonal_factor_status(tile):
    """Failing pivots inside the cluster factor: the first column whose pivot
    is not positive (or is NaN), in the first, a middle and the last panel of
    a tile, and in a later tile; the other matrix of the batch is unaffected."""
    n = 300
    for col in (0, 17, 47, 127, 130, 299):
        A = W.gram_spd(2, n, 71, 1.0, np.float64)
        A[0, col, col] = -2.0 if col % 2 else np.nan
        Lbar = W.tril_normal(2, n, 72, np.float64)
        L, st, G = check(A, Lbar, np.float64, tile=tile)
        assert list(st) == [col + 1, 0]


@pytest.mark.parametrize("n", [300, 520])
def test_tensor_core_path_with_element_aligned_buffers(n):
    """float64 buffers that start 8 bytes past a 32-byte boundary (the header
    allows element-aligned pointers): the tensor-core updates' 32-byte row
    accesses give way to element accesses, with the same results bit for bit."""
    import torch
    from differentiable_cholesky_gb300 import binding
    dev = torch.device("cuda:0")
    batch = 2
    A = W.gram_spd(batch, n, 211 + n, 1.0, np.float64)
    Lbar = W.tril_normal(batch, n, 212 + n, np.float64)
    At, Lbt = torch.from_numpy(A).to(dev), torch.from_numpy(Lbar).to(dev)
    L, st = binding.chol_fwd(At, tile=128)
    G = binding.chol_adj(L, Lbt, status=st, tile=128)

    def shifted(x=None):
        buf = torch.zeros(batch * n * n + 1, dtype=torch.float64, device=dev)
        v = buf[1:].view(batch, n, n)
        assert v.data_ptr() % 32 == 8
        if x is not None:
            v.copy_(x)
        return v
    Au, Lbu, Lu, Gu = shifted(At), shifted(Lbt), shifted(), shifted()
    stu = torch.empty(batch, dtype=torch.int32, device=dev)
    binding.chol_fwd(Au, Lu, stu, tile=128)
    binding.chol_adj(Lu, Lbu, Gu, status=stu, tile=128)
    torch.cuda.synchronize()
    assert torch.equal(st, stu)
    assert torch.equal(L, Lu)
    assert torch.equal(G, Gu)
    L_ref, _ = oracle.potrf(A)
    assert max_rel_err(Lu.cpu().numpy(), L_ref) <= 1e-12
