"""ctypes binding of ``libchol_gb300.so`` (declared in ``include/chol.h``).

Argument marshalling only: every step of the factorisation and of its adjoint
runs in the library's CUDA kernels.  torch supplies device memory and the
current stream.  There is no fallback: if the library is missing or a call
fails, a ``RuntimeError`` says why.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

CHOL_F32 = 0
CHOL_F64 = 1
CHOL_C64 = 2
CHOL_C128 = 3
_DTYPES = {torch.float32: CHOL_F32, torch.float64: CHOL_F64,
           torch.complex64: CHOL_C64, torch.complex128: CHOL_C128}

_lock = threading.Lock()
_lib = None


class CholError(RuntimeError):
    """A library call returned a negative code."""

    def __init__(self, code: int, msg: str):
        super().__init__(f"{msg} (code {code})")
        self.code = code


def load_library(path: str | None = None):
    """Load (building first if needed) and return the ctypes library handle."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if path is None:
            path = _build.LIB_PATH
            if not _build.up_to_date():
                path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not found at {path}; run the package build first")
        lib = ctypes.CDLL(path)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
        lib.chol_fwd.argtypes = [i64, i32, i32, vp, vp, vp, vp]
        lib.chol_fwd_ex.argtypes = [i64, i32, i32, vp, vp, vp, i32, vp]
        lib.chol_adj.argtypes = [i64, i32, i32, vp, vp, vp, vp, vp]
        lib.chol_adj_ex.argtypes = [i64, i32, i32, vp, vp, vp, vp, i32, vp]
        for f in (lib.chol_fwd, lib.chol_fwd_ex, lib.chol_adj, lib.chol_adj_ex):
            f.restype = ctypes.c_int
        lib.chol_strerror.argtypes = [ctypes.c_int]
        lib.chol_strerror.restype = ctypes.c_char_p
        lib.chol_abi_version.argtypes = []
        lib.chol_abi_version.restype = ctypes.c_int32
        lib.chol_adj_noalloc.argtypes = [i64, i32, i32, vp, vp, vp, vp, i32, vp]
        lib.chol_adj_noalloc.restype = ctypes.c_int
        lib.chol_selftest_wait_timeout.argtypes = [i64, vp, vp, vp, ctypes.c_uint32, vp]
        lib.chol_selftest_wait_timeout.restype = ctypes.c_int
        lib.chol_fwd_inplace.argtypes = [i64, i32, i32, vp, vp, i32, vp]
        lib.chol_fwd_inplace.restype = ctypes.c_int
        lib.chol_adj_inplace.argtypes = [i64, i32, i32, vp, vp, vp, i32, vp]
        lib.chol_adj_inplace.restype = ctypes.c_int
        lib.chol_solve.argtypes = [i64, i32, i32, i32, vp, vp, vp, vp, vp]
        lib.chol_solve.restype = ctypes.c_int
        lib.chol_solve_adj.argtypes = [i64, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
        lib.chol_solve_adj.restype = ctypes.c_int
        lib.chol_probe_fma_peak.argtypes = [i32, i64, vp, ctypes.POINTER(ctypes.c_double), vp]
        lib.chol_probe_fma_peak.restype = ctypes.c_int
        lib.chol_probe_dmma_peak.argtypes = [i32, i64, vp, ctypes.POINTER(ctypes.c_double), vp]
        lib.chol_probe_dmma_peak.restype = ctypes.c_int
        dp = ctypes.POINTER(ctypes.c_double)
        lib.chol_probe_tc_update.argtypes = [i32, vp, i32, i32, dp, dp, dp, vp]
        lib.chol_probe_tc_update.restype = ctypes.c_int
        _lib = lib
        return lib


def _check(rc: int):
    if rc != 0:
        msg = load_library().chol_strerror(rc).decode()
        raise CholError(rc, msg)


def _shape(x: torch.Tensor):
    if x.dim() < 2 or x.shape[-1] != x.shape[-2]:
        raise ValueError(f"expected [..., n, n], got {tuple(x.shape)}")
    n = int(x.shape[-1])
    batch = 1
    for s in x.shape[:-2]:
        batch *= int(s)
    return batch, n


def _require(x: torch.Tensor, name: str, dtype=None):
    if not isinstance(x, torch.Tensor) or not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and x.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}, got {x.dtype}")


def _stream_ptr(stream) -> int | None:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def chol_fwd(A: torch.Tensor, L: torch.Tensor | None = None, status: torch.Tensor | None = None,
             tile: int = 0, stream=None):
    """``L, status = chol_fwd(A)`` for ``A`` of shape ``[..., n, n]`` (float32,
    float64, or complex64/complex128 Hermitian: ``A = L L^H``).

    Only ``tril(A)`` is read (and only the real part of a complex diagonal).  ``status`` is int32 with the batch shape: 0, or
    the 1-based first failing pivot column.  Pre-allocated ``L``/``status`` may
    be passed to avoid allocation (they are fully overwritten).
    """
    _require(A, "A")
    if A.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {A.dtype}")
    batch, n = _shape(A)
    if L is None:
        L = torch.empty_like(A)
    if status is None:
        status = torch.empty(A.shape[:-2], dtype=torch.int32, device=A.device)
    _require(L, "L", A.dtype)
    _require(status, "status", torch.int32)
    if tuple(L.shape) != tuple(A.shape) or status.numel() != batch:
        raise ValueError("L must match A's shape and status must have one entry per matrix")
    lib = load_library()
    rc = lib.chol_fwd_ex(batch, n, _DTYPES[A.dtype], A.data_ptr(), L.data_ptr(),
                         status.data_ptr(), int(tile), _stream_ptr(stream))
    _check(rc)
    return L, status


def chol_adj(L: torch.Tensor, adj_L: torch.Tensor, adj_A: torch.Tensor | None = None,
             status: torch.Tensor | None = None, tile: int = 0, stream=None):
    """Accumulate the Cholesky adjoint into ``adj_A`` (zeros if not given).

    ``adj_A``'s lower triangle gains ``Phi(M + M^T)`` with
    ``M = L^-T Phi(L^T tril(adj_L)) L^-1``; its upper triangle is not written.
    Matrices with non-zero ``status`` are skipped.  Returns ``adj_A``.
    """
    _require(L, "L")
    if L.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {L.dtype}")
    _require(adj_L, "adj_L", L.dtype)
    if tuple(adj_L.shape) != tuple(L.shape):
        raise ValueError("adj_L must match L's shape")
    batch, n = _shape(L)
    if adj_A is None:
        adj_A = torch.zeros_like(L)
    _require(adj_A, "adj_A", L.dtype)
    if tuple(adj_A.shape) != tuple(L.shape):
        raise ValueError("adj_A must match L's shape")
    sp = None
    if status is not None:
        _require(status, "status", torch.int32)
        if status.numel() != batch:
            raise ValueError("status must have one entry per matrix")
        sp = status.data_ptr()
    lib = load_library()
    rc = lib.chol_adj_ex(batch, n, _DTYPES[L.dtype], L.data_ptr(), adj_L.data_ptr(),
                         adj_A.data_ptr(), sp, int(tile), _stream_ptr(stream))
    _check(rc)
    return adj_A


def chol_fwd_inplace(A: torch.Tensor, status: torch.Tensor | None = None, tile: int = 0,
                     stream=None):
    """Factor ``A`` in place: on return ``A`` holds what :func:`chol_fwd`
    returns as ``L`` (zeros above the diagonal).  Returns ``A, status``."""
    _require(A, "A")
    if A.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {A.dtype}")
    batch, n = _shape(A)
    if status is None:
        status = torch.empty(A.shape[:-2], dtype=torch.int32, device=A.device)
    _require(status, "status", torch.int32)
    if status.numel() != batch:
        raise ValueError("status must have one entry per matrix")
    rc = load_library().chol_fwd_inplace(batch, n, _DTYPES[A.dtype], A.data_ptr(),
                                         status.data_ptr(), int(tile), _stream_ptr(stream))
    _check(rc)
    return A, status


def chol_adj_inplace(L: torch.Tensor, adj: torch.Tensor, status: torch.Tensor | None = None,
                     tile: int = 0, stream=None):
    """Replace the lower triangle of ``adj`` (holding ``adj_L``) by the
    gradient :func:`chol_adj` would add to a zero ``adj_A``; matrices with
    non-zero ``status`` get zeros there.  The upper triangle is not written.
    Returns ``adj``."""
    _require(L, "L")
    if L.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {L.dtype}")
    _require(adj, "adj", L.dtype)
    if tuple(adj.shape) != tuple(L.shape):
        raise ValueError("adj must match L's shape")
    batch, n = _shape(L)
    sp = None
    if status is not None:
        _require(status, "status", torch.int32)
        if status.numel() != batch:
            raise ValueError("status must have one entry per matrix")
        sp = status.data_ptr()
    rc = load_library().chol_adj_inplace(batch, n, _DTYPES[L.dtype], L.data_ptr(), adj.data_ptr(),
                                         sp, int(tile), _stream_ptr(stream))
    _check(rc)
    return adj


def _rhs_shape(L: torch.Tensor, B: torch.Tensor):
    batch, n = _shape(L)
    if B.dim() != L.dim() or tuple(B.shape[:-1]) != tuple(L.shape[:-1]):
        raise ValueError(f"expected right-hand sides [..., {n}, nrhs] matching L {tuple(L.shape)}, "
                         f"got {tuple(B.shape)}")
    return batch, n, int(B.shape[-1])


def chol_solve(L: torch.Tensor, B: torch.Tensor, X: torch.Tensor | None = None,
               status: torch.Tensor | None = None, stream=None):
    """``X = A^-1 B`` with ``A = L L^H`` (``L L^T`` for real dtypes): ``L`` is
    ``[..., n, n]`` from :func:`chol_fwd`, ``B`` is ``[..., n, nrhs]``.  ``X``
    may be ``B`` itself (in place).  Matrices with non-zero ``status`` get
    ``X = 0``.  Returns ``X``."""
    _require(L, "L")
    if L.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {L.dtype}")
    _require(B, "B", L.dtype)
    batch, n, nrhs = _rhs_shape(L, B)
    if X is None:
        X = torch.empty_like(B)
    _require(X, "X", L.dtype)
    if tuple(X.shape) != tuple(B.shape):
        raise ValueError("X must match B's shape")
    sp = None
    if status is not None:
        _require(status, "status", torch.int32)
        if status.numel() != batch:
            raise ValueError("status must have one entry per matrix")
        sp = status.data_ptr()
    rc = load_library().chol_solve(batch, n, nrhs, _DTYPES[L.dtype], L.data_ptr(), B.data_ptr(),
                                   X.data_ptr(), sp, _stream_ptr(stream))
    _check(rc)
    return X


def chol_solve_adj(L: torch.Tensor, X: torch.Tensor, adj_X: torch.Tensor,
                   adj_B: torch.Tensor | None = None, adj_L: torch.Tensor | None = None,
                   status: torch.Tensor | None = None, want_B: bool = True, want_L: bool = True,
                   stream=None):
    """Reverse mode of :func:`chol_solve`: accumulates ``A^-1 adj_X`` into
    ``adj_B`` and ``tril(-(Bb X^H + X Bb^H) L)`` into ``adj_L`` (zeros when
    not given; skipped when ``want_B`` / ``want_L`` is false).  Returns
    ``(adj_B, adj_L)``."""
    _require(L, "L")
    if L.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {L.dtype}")
    _require(X, "X", L.dtype)
    _require(adj_X, "adj_X", L.dtype)
    batch, n, nrhs = _rhs_shape(L, X)
    if tuple(adj_X.shape) != tuple(X.shape):
        raise ValueError("adj_X must match X's shape")
    if want_B and adj_B is None:
        adj_B = torch.zeros_like(X)
    if want_L and adj_L is None:
        adj_L = torch.zeros_like(L)
    if adj_B is not None:
        _require(adj_B, "adj_B", L.dtype)
    if adj_L is not None:
        _require(adj_L, "adj_L", L.dtype)
    sp = None
    if status is not None:
        _require(status, "status", torch.int32)
        sp = status.data_ptr()
    rc = load_library().chol_solve_adj(
        batch, n, nrhs, _DTYPES[L.dtype], L.data_ptr(), X.data_ptr(), adj_X.data_ptr(),
        adj_B.data_ptr() if adj_B is not None else None,
        adj_L.data_ptr() if adj_L is not None else None, sp, _stream_ptr(stream))
    _check(rc)
    return adj_B, adj_L


def probe_fma_peak(dtype=torch.float64, iters: int = 1 << 16, stream=None) -> float:
    """Measured FMA throughput of the current device in FLOP/s (2 per FMA)."""
    if dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {dtype}")
    sink = torch.zeros(1, dtype=dtype, device="cuda")
    out = ctypes.c_double(0.0)
    rc = load_library().chol_probe_fma_peak(_DTYPES[dtype], int(iters), sink.data_ptr(),
                                            ctypes.byref(out), _stream_ptr(stream))
    _check(rc)
    return out.value


DMMA_SHAPES = {"m8n8k4": 0, "m16n8k4": 1, "m16n8k8": 2, "m16n8k16": 3}


def probe_dmma_peak(shape: str = "m8n8k4", iters: int = 1 << 14, stream=None) -> float:
    """Measured f64 ``mma.sync`` (DMMA) throughput of the current device in
    FLOP/s for one instruction shape (a key of ``DMMA_SHAPES``)."""
    if shape not in DMMA_SHAPES:
        raise ValueError(f"unknown shape {shape}; expected one of {sorted(DMMA_SHAPES)}")
    sink = torch.zeros(1, dtype=torch.float64, device="cuda")
    out = ctypes.c_double(0.0)
    rc = load_library().chol_probe_dmma_peak(DMMA_SHAPES[shape], int(iters), sink.data_ptr(),
                                             ctypes.byref(out), _stream_ptr(stream))
    _check(rc)
    return out.value


class _Cholesky(torch.autograd.Function):
    """Autograd wrapper: the gradient flows to the lower triangle of A only,
    because the factorisation reads nothing else."""

    @staticmethod
    def forward(ctx, A, tile):
        L, status = chol_fwd(A.contiguous(), tile=tile)
        ctx.save_for_backward(L, status)
        ctx.tile = tile
        ctx.mark_non_differentiable(status)
        return L, status

    @staticmethod
    def backward(ctx, gL, gstatus):
        L, status = ctx.saved_tensors
        if gL is None:
            return None, None
        gA = chol_adj(L, gL.contiguous(), status=status, tile=ctx.tile)
        return gA, None


def cholesky(A: torch.Tensor, tile: int = 0):
    """Differentiable ``(L, status)``; ``A.grad`` gets the lower-triangle adjoint."""
    return _Cholesky.apply(A, tile)


def probe_tc_update(L: torch.Tensor, k: int = 0, reps: int = 3, stream=None):
    """Times the float64 tensor-core trailing update of step ``k`` on the
    square float64 CUDA matrix ``L`` (modified: pass a scratch copy).
    Returns ``(ms_per_launch, bf16_flops_per_s, fp64_equivalent_flops_per_s)``."""
    _require(L, "L", torch.float64)
    if L.dim() != 2 or L.shape[0] != L.shape[1]:
        raise ValueError("L must be a square matrix")
    ms, bf, fp = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    rc = load_library().chol_probe_tc_update(int(L.shape[0]), L.data_ptr(), int(k), int(reps),
                                             ctypes.byref(ms), ctypes.byref(bf), ctypes.byref(fp),
                                             _stream_ptr(stream))
    _check(rc)
    return ms.value, bf.value, fp.value
