"""GB300-native differentiable Cholesky: batched/blocked potrf and its adjoint.

The compute path is the C-ABI library ``libchol_gb300.so`` (CUDA for sm_103a,
declared in ``include/chol.h``); :mod:`differentiable_cholesky_gb300.binding`
marshals torch device tensors into it.  The library is loaded on first use, so
importing this package (e.g. for :mod:`.workloads`) needs no GPU.
"""
from __future__ import annotations

__all__ = ["chol_fwd", "chol_adj", "cholesky", "load_library"]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
