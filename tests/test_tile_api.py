"""GPU parity of the device-side tile API (include/chol_tile.cuh) against the
oracle: test kernels (tests/tile_api/tile_api_kernels.cu, built here with
nvcc) stage one matrix per block in shared memory and call chol_tile::potrf
and chol_tile::potrf_adj, as a caller's own kernel would."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from differentiable_cholesky_gb300 import workloads as W
from parity_util import TOL_ADJ, TOL_L, max_rel_err

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "tile_api", "tile_api_kernels.cu")
OUT = os.path.join(HERE, "tile_api", "_build", "libtile_demo.so")


@pytest.fixture(scope="module")
def lib():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    subprocess.run([nvcc, "-std=c++17", "-O3", "-Xcompiler", "-fPIC", "-shared",
                    "-I", os.path.join(ROOT, "include"),
                    "-gencode", "arch=compute_103a,code=sm_103a", "-o", OUT, SRC], check=True)
    h = ctypes.CDLL(OUT)
    i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    h.tile_demo_fwd.argtypes = [i64, i32, i32, i32, vp, vp, vp, vp]
    h.tile_demo_adj.argtypes = [i64, i32, i32, i32, i32, vp, vp, vp, vp, vp]
    return h


@pytest.mark.parametrize("threads", [64, 256])
@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("n", [1, 5, 16, 33, 64])
def test_tile_potrf_and_adjoint(lib, n, dtype, threads):
    import torch
    dev = torch.device("cuda:0")
    batch = 6
    A = W.gram_spd(batch, n, 70 + n, 1.0, dtype)
    if n > 1:
        A[2, n // 2, n // 2] = -3.0        # fails at column n//2
    A[4, 0, 0] = np.nan                    # fails at column 0
    Lbar = W.tril_normal(batch, n, 71 + n, dtype)
    At = torch.from_numpy(A).to(dev)
    Lt = torch.empty_like(At)
    st = torch.empty(batch, dtype=torch.int32, device=dev)
    s = torch.cuda.current_stream().cuda_stream
    code = 0 if dtype == np.float32 else 1
    assert lib.tile_demo_fwd(batch, n, code, threads, At.data_ptr(), Lt.data_ptr(),
                             st.data_ptr(), s) == 0
    torch.cuda.synchronize()
    _, s_ref = oracle.potrf(A, dtype=np.dtype(dtype))
    assert np.array_equal(st.cpu().numpy(), s_ref)
    ok = s_ref == 0
    L64, _ = oracle.potrf(A.astype(np.float64))
    assert max_rel_err(Lt.cpu().numpy(), L64, mask=ok) <= TOL_L[np.dtype(dtype)]

    G_ref = oracle.potrf_adj(L64, Lbar.astype(np.float64), status=s_ref)
    for packed in (0, 1):
        Gt = torch.zeros_like(At)
        assert lib.tile_demo_adj(batch, n, code, threads, packed, Lt.data_ptr(),
                                 torch.from_numpy(Lbar).to(dev).data_ptr(), Gt.data_ptr(),
                                 st.data_ptr(), s) == 0
        torch.cuda.synchronize()
        G = Gt.cpu().numpy()
        assert max_rel_err(G, G_ref, mask=ok, lower=True) <= TOL_ADJ[np.dtype(dtype)]
        assert np.all(G[~ok] == 0)
        assert np.all(np.triu(G, 1) == 0)  # nothing above the diagonal written
