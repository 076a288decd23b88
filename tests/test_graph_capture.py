"""The path inside a CUDA graph (GPU): chol_fwd and chol_adj_noalloc are
captured once after an eager warm-up (kernel attributes, occupancy and the
scratch address are looked up on first use) and replayed on new input values
written into the same buffers.  Replays must match eager calls bit for bit.
The adjoint entry is the one that allocates nothing, so the captured work
holds no allocation on either path (n <= 64 and blocked)."""
import numpy as np
import pytest

from differentiable_cholesky_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("batch,n,dtype", [(4096, 16, np.float32), (1000, 64, np.float32),
                                           (37, 20, np.float64), (3, 100, np.float64)])
def test_captured_step_replays_like_eager_calls(batch, n, dtype):
    import torch
    from differentiable_cholesky_gb300 import binding
    lib = binding.load_library()
    dev = torch.device("cuda:0")
    dt = 0 if dtype == np.float32 else 1

    def inputs(seed):
        A = torch.from_numpy(W.gram_spd(batch, n, seed, 1.0, dtype)).to(dev)
        Lb = torch.from_numpy(W.tril_normal(batch, n, seed + 1, dtype)).to(dev)
        return A, Lb

    A, Lb = inputs(200)
    L = torch.empty_like(A)
    G = torch.zeros_like(A)
    st = torch.empty(batch, dtype=torch.int32, device=dev)

    def step():
        s = torch.cuda.current_stream().cuda_stream
        assert lib.chol_fwd_ex(batch, n, dt, A.data_ptr(), L.data_ptr(), st.data_ptr(), 0, s) == 0
        G.zero_()
        assert lib.chol_adj_noalloc(batch, n, dt, L.data_ptr(), Lb.data_ptr(), G.data_ptr(),
                                    st.data_ptr(), 0, s) == 0

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up, eager
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    for seed in (300, 400):
        A2, Lb2 = inputs(seed)
        L_ref, st_ref = binding.chol_fwd(A2)
        G_ref = binding.chol_adj(L_ref, Lb2, status=st_ref)
        A.copy_(A2)
        Lb.copy_(Lb2)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(st, st_ref)
        assert torch.equal(L, L_ref)
        assert torch.equal(G, G_ref)


@pytest.mark.parametrize("batch,n,dtype", [(2048, 16, np.float32), (3, 100, np.float64)])
def test_captured_inplace_step(batch, n, dtype):
    """The in-place pair allocates nothing on either path, so it captures too
    (inputs are copied into the work buffers inside the graph)."""
    import torch
    from differentiable_cholesky_gb300 import binding
    lib = binding.load_library()
    dev = torch.device("cuda:0")
    dt = 0 if dtype == np.float32 else 1
    A = torch.from_numpy(W.gram_spd(batch, n, 500, 1.0, dtype)).to(dev)
    Lb = torch.from_numpy(W.tril_normal(batch, n, 501, dtype)).to(dev)
    X, Y = torch.empty_like(A), torch.empty_like(A)
    st = torch.empty(batch, dtype=torch.int32, device=dev)

    def step():
        s = torch.cuda.current_stream().cuda_stream
        X.copy_(A)
        Y.copy_(Lb)
        assert lib.chol_fwd_inplace(batch, n, dt, X.data_ptr(), st.data_ptr(), 0, s) == 0
        assert lib.chol_adj_inplace(batch, n, dt, X.data_ptr(), Y.data_ptr(), st.data_ptr(), 0, s) == 0

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    A.copy_(torch.from_numpy(W.gram_spd(batch, n, 600, 1.0, dtype)).to(dev))
    Lb.copy_(torch.from_numpy(W.tril_normal(batch, n, 601, dtype)).to(dev))
    L_ref, st_ref = binding.chol_fwd(A)
    G_ref = binding.chol_adj(L_ref, Lb, status=st_ref)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(st, st_ref)
    assert torch.equal(X, L_ref)
    il = torch.tril_indices(n, n, device=dev)
    assert torch.equal(Y[:, il[0], il[1]], G_ref[:, il[0], il[1]])
    iu = torch.triu_indices(n, n, 1, device=dev)
    assert torch.equal(Y[:, iu[0], iu[1]], Lb[:, iu[0], iu[1]])  # upper triangle untouched
