"""chol_adj_noalloc, the adjoint entry point for callers that cannot allocate
device memory while they run, against chol_adj (GPU).

It is called twice in a row on different inputs through the C ABI: the second
call runs on the scratch the first one left behind, and both must match the
allocating entry point within the parity tolerances.  This file is collected
last so that a run stopping at its first failure has run everything else.
"""
import numpy as np
import pytest

from differentiable_cholesky_gb300 import workloads as W
from parity_util import TOL_ADJ, max_rel_err

pytestmark = pytest.mark.gpu

CHOL_OK, CHOL_ENOMEM = 0, -4
SCRATCH_BYTES = 16 << 20


def _inputs(batch, n, dtype, seed):
    import torch
    from differentiable_cholesky_gb300 import binding
    dev = torch.device("cuda:0")
    A = torch.from_numpy(W.gram_spd(batch, n, seed, 1.0, dtype)).to(dev)
    Lb = torch.from_numpy(W.tril_normal(batch, n, seed + 1, dtype)).to(dev)
    L, st = binding.chol_fwd(A)
    return L, Lb, st


def _noalloc(lib, L, Lb, G, st, tile=0):
    import torch
    dt = 0 if L.dtype == torch.float32 else 1
    batch = L.numel() // (L.shape[-1] * L.shape[-1])
    return lib.chol_adj_noalloc(batch, L.shape[-1], dt, L.data_ptr(), Lb.data_ptr(),
                                G.data_ptr(), st.data_ptr(), tile,
                                torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("dtype,n,batch,tile", [(np.float64, 300, 3, 0), (np.float64, 512, 4, 128),
                                                (np.float32, 200, 5, 64), (np.float32, 16, 9, 0)])
def test_two_calls_match_the_allocating_entry_point(dtype, n, batch, tile):
    import torch
    from differentiable_cholesky_gb300 import binding
    lib = binding.load_library()
    for seed in (101, 202):  # two calls in a row, different data
        L, Lb, st = _inputs(batch, n, dtype, seed)
        G0 = torch.full_like(L, 0.25)
        ref = binding.chol_adj(L, Lb, adj_A=G0.clone(), status=st, tile=tile)
        G = G0.clone()
        rc = _noalloc(lib, L, Lb, G, st, tile)
        assert rc == CHOL_OK, lib.chol_strerror(rc).decode()
        torch.cuda.synchronize()
        got, want = G.cpu().numpy(), ref.cpu().numpy()
        assert max_rel_err(got, want, lower=True) <= TOL_ADJ[np.dtype(dtype)]
        iu = np.triu_indices(n, 1)
        assert np.all(got[:, iu[0], iu[1]] == 0.25)


def test_rejects_problems_larger_than_the_scratch():
    import torch
    from differentiable_cholesky_gb300 import binding
    lib = binding.load_library()
    n = 1024                      # 1024^2 * 8 B = 8 MiB per matrix
    batch = SCRATCH_BYTES // (n * n * 8) + 1
    dev = torch.device("cuda:0")
    L = torch.eye(n, dtype=torch.float64, device=dev).repeat(batch, 1, 1)
    Lb = torch.zeros_like(L)
    G = torch.zeros_like(L)
    st = torch.zeros(batch, dtype=torch.int32, device=dev)
    assert _noalloc(lib, L, Lb, G, st) == CHOL_ENOMEM
    torch.cuda.synchronize()
    assert torch.count_nonzero(G).item() == 0
