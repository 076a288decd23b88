"""The FMA-peak probe runs and reports a plausible rate (GPU)."""
import pytest

pytestmark = pytest.mark.gpu


def test_probe_reports_positive_rates():
    import torch
    from differentiable_cholesky_gb300 import binding
    f64 = binding.probe_fma_peak(torch.float64, iters=1 << 12)
    f32 = binding.probe_fma_peak(torch.float32, iters=1 << 12)
    assert 1e11 < f64 < 1e15
    assert 1e12 < f32 < 1e15
