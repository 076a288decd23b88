"""The throughput probes run and report plausible rates (GPU)."""
import pytest

pytestmark = pytest.mark.gpu


def test_probe_reports_positive_rates():
    import torch
    from differentiable_cholesky_gb300 import binding
    f64 = binding.probe_fma_peak(torch.float64, iters=1 << 12)
    f32 = binding.probe_fma_peak(torch.float32, iters=1 << 12)
    assert 1e11 < f64 < 1e15
    assert 1e12 < f32 < 1e15


@pytest.mark.parametrize("shape", ["m8n8k4", "m16n8k4", "m16n8k8", "m16n8k16"])
def test_dmma_probe_reports_positive_rates(shape):
    from differentiable_cholesky_gb300 import binding
    r = binding.probe_dmma_peak(shape, iters=1 << 10)
    assert 1e10 < r < 1e16


def test_dmma_probe_rejects_bad_arguments():
    import ctypes
    import torch
    from differentiable_cholesky_gb300 import binding
    lib = binding.load_library()
    sink = torch.zeros(1, dtype=torch.float64, device="cuda")
    out = ctypes.c_double(0.0)
    assert lib.chol_probe_dmma_peak(7, 16, sink.data_ptr(), ctypes.byref(out), None) == -1
    assert lib.chol_probe_dmma_peak(0, 0, sink.data_ptr(), ctypes.byref(out), None) == -1


def test_tensor_core_update_probe_times_the_real_update():
    """The probe runs the library's own trailing update: one launch on a copy
    of a factored matrix's trailing part equals chol's next step there (the
    update is what the forward does after slicing panel k), and it reports a
    bf16 rate 28 times its float64-equivalent rate."""
    import numpy as np
    import torch
    import oracle
    from differentiable_cholesky_gb300 import binding
    from differentiable_cholesky_gb300 import workloads as W
    n = 512
    A = W.gram_spd(1, n, 91, 1.0, np.float64)[0]
    # panel 0 of the factor, and the trailing part still holding A
    L_ref, _ = oracle.potrf(A)
    M = np.tril(A).copy()
    M[:, :128] = np.tril(L_ref)[:, :128]
    Mt = torch.from_numpy(M).cuda()
    ms, bf16, fp64 = binding.probe_tc_update(Mt, k=0, reps=1)
    torch.cuda.synchronize()
    assert ms > 0 and abs(bf16 / fp64 - 28.0) < 1e-9
    # the Schur complement of the leading block, lower part
    P = np.tril(L_ref)[:, :128]
    S = np.tril(A - P @ P.T)
    got = np.tril(Mt.cpu().numpy())
    assert np.max(np.abs(got[128:, 128:] - S[128:, 128:])) <= 1e-12 * np.max(np.abs(S))
