"""Failure detection on the GPU without a GPU fault: a bounded device wait
that cannot complete ends in an error status the host reads, and the CUDA
context stays usable.  The self-test entry point holds back one matrix copy
of every warp's first round in the forward kernel (a lost message), so that
round's arrival barrier cannot complete; every warp must give up after its
poll limit, mark its first round's matrices with status -1, issue the
held-back copy late, wait until every copy it issued has landed and
return."""
import numpy as np
import pytest

import oracle
from differentiable_cholesky_gb300 import workloads as W
from parity_util import TOL_L, max_rel_err

pytestmark = pytest.mark.gpu

SENTINEL = 777


def test_lost_copy_times_out_with_status_and_context_survives():
    import torch
    from differentiable_cholesky_gb300 import binding
    lib = binding.load_library()
    dev = torch.device("cuda:0")
    batch = 40000  # several rounds per warp
    A = torch.from_numpy(W.gram_spd(batch, 16, 90, 1.0, np.float32)).to(dev)
    L = torch.full_like(A, 5.0)
    st = torch.full((batch,), SENTINEL, dtype=torch.int32, device=dev)
    s = torch.cuda.current_stream().cuda_stream
    rc = lib.chol_selftest_wait_timeout(batch, A.data_ptr(), L.data_ptr(), st.data_ptr(),
                                        1 << 16, s)
    assert rc == 0
    torch.cuda.synchronize()  # returns: no hang, no fault
    sv = st.cpu().numpy()
    assert set(np.unique(sv)) <= {-1, SENTINEL}
    timed_out = int((sv == -1).sum())
    assert timed_out > 0
    # only each warp's first round is marked: at most 27 matrices per warp,
    # and rounds are 27 matrices wide
    assert timed_out % 27 == 0 or timed_out == batch
    assert torch.all(L == 5.0)  # nothing of L written

    # the context is still usable: the normal path gives correct results
    L2, st2 = binding.chol_fwd(A)
    torch.cuda.synchronize()
    An = A.cpu().numpy()
    L_ref, s_ref = oracle.potrf(An.astype(np.float64))
    assert np.array_equal(st2.cpu().numpy(), s_ref)
    assert max_rel_err(L2.cpu().numpy(), L_ref) <= TOL_L[np.dtype(np.float32)]


def test_selftest_argument_checks():
    import torch
    from differentiable_cholesky_gb300 import binding
    lib = binding.load_library()
    dev = torch.device("cuda:0")
    A = torch.zeros(4, 16, 16, device=dev)
    L = torch.zeros_like(A)
    st = torch.zeros(4, dtype=torch.int32, device=dev)
    assert lib.chol_selftest_wait_timeout(4, A.data_ptr(), L.data_ptr(), st.data_ptr(), 0, None) == -1
    assert lib.chol_selftest_wait_timeout(4, A.data_ptr(), L.data_ptr(), st.data_ptr(),
                                          (1 << 22) + 1, None) == -1
    assert lib.chol_selftest_wait_timeout(4, A.data_ptr(), A.data_ptr(), st.data_ptr(), 10, None) == -3
