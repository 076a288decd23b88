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
