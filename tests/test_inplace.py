"""GPU parity of the in-place forms (chol_fwd_inplace, chol_adj_inplace)
through the C ABI: bit-identical to the out-of-place calls, which the other
parity tests pin to the oracle, plus the in-place rules of the header."""
import numpy as np
import pytest

import oracle
from differentiable_cholesky_gb300 import workloads as W
from parity_util import TOL_ADJ, TOL_L, max_rel_err

pytestmark = pytest.mark.gpu

# (300 and 520 float64 at tile 128, the default for few such matrices, take
# the tensor-core updates with the lookahead, in place as out of place)
CASES = [(8, np.float32, 0), (16, np.float32, 0), (16, np.float64, 0), (20, np.float32, 0),
         (64, np.float32, 0), (65, np.float64, 0), (130, np.float64, 32), (130, np.float32, 64),
         (300, np.float64, 0), (520, np.float64, 128)]


def _inputs(batch, n, dtype, seed):
    A = W.gram_spd(batch, n, seed, 1.0, dtype)
    A[1, n // 2, n // 2] = -1.0  # one matrix fails: status n//2 + 1
    Lbar = W.tril_normal(batch, n, seed + 1, dtype)
    iu = np.triu_indices(n, 1)
    Lbar[:, iu[0], iu[1]] = 7.5  # upper triangle of the seed: ignored, kept
    return A, Lbar


@pytest.mark.parametrize("n,dtype,tile", CASES)
def test_inplace_matches_out_of_place(n, dtype, tile):
    import torch
    from differentiable_cholesky_gb300 import binding
    dev = torch.device("cuda:0")
    batch = 37 if n <= 64 else 3
    A, Lbar = _inputs(batch, n, dtype, 40 + n)
    At = torch.from_numpy(A).to(dev)
    L_ref, st_ref = binding.chol_fwd(At, tile=tile)
    G_ref = binding.chol_adj(L_ref, torch.from_numpy(Lbar).to(dev), status=st_ref, tile=tile)

    X = At.clone()
    X2, st = binding.chol_fwd_inplace(X, tile=tile)
    assert X2.data_ptr() == X.data_ptr()
    Y = torch.from_numpy(Lbar).to(dev)
    binding.chol_adj_inplace(X, Y, status=st, tile=tile)
    torch.cuda.synchronize()

    assert torch.equal(st, st_ref)
    assert torch.equal(X, L_ref)  # factor, zeros above the diagonal
    il = np.tril_indices(n)
    Yn, Gn = Y.cpu().numpy(), G_ref.cpu().numpy()
    assert np.array_equal(Yn[:, il[0], il[1]], Gn[:, il[0], il[1]])
    iu = np.triu_indices(n, 1)
    assert np.all(Yn[:, iu[0], iu[1]] == 7.5)  # upper triangle never written
    bad = st.cpu().numpy() != 0
    assert bad[1] and not bad[0]
    assert np.all(Yn[bad][:, il[0], il[1]] == 0)  # skipped matrix: zeros

    # and against the oracle directly
    L_o, s_o = oracle.potrf(A, dtype=np.dtype(dtype))
    assert np.array_equal(st.cpu().numpy(), s_o)
    ok = s_o == 0
    L64, _ = oracle.potrf(A.astype(np.float64))
    G_o = oracle.potrf_adj(L64, Lbar.astype(np.float64), status=s_o)
    assert max_rel_err(X.cpu().numpy(), L64, mask=ok) <= TOL_L[np.dtype(dtype)]
    Ylow = np.tril(Yn)
    assert max_rel_err(Ylow, G_o, mask=ok, lower=True) <= TOL_ADJ[np.dtype(dtype)]


def test_inplace_aliasing_rejected():
    import torch
    from differentiable_cholesky_gb300 import binding
    dev = torch.device("cuda:0")
    n, batch = 16, 8
    buf = torch.zeros(batch * n * n + 64, dtype=torch.float32, device=dev)
    X = buf[:batch * n * n].view(batch, n, n)
    st = buf[batch * n * n - 16:batch * n * n - 8].view(torch.int32)  # inside X
    with pytest.raises(binding.CholError) as e:
        binding.chol_fwd_inplace(X, status=st)
    assert e.value.code == -3
    with pytest.raises(binding.CholError) as e:
        binding.chol_adj_inplace(X, X)
    assert e.value.code == -3
