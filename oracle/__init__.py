"""CPU oracle for the differentiable Cholesky path -- test infrastructure only.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU library never does: it shares no
code with the oracle, and neither imports the other.

The arithmetic lives in ``chol_oracle.c`` (plain C, no blocking or fusion); this
module compiles it with gcc on first use and marshals numpy arrays through
ctypes.  Each function states the passage it restates:

* :func:`potrf` -- the lower Cholesky factor and the per-matrix status
  (jaxmg docs "Cholesky factorization": intro and the ``factor, status`` result of
  "Advanced: control the outer jax.jit"; status read as LAPACK's info).
* :func:`potrf_adj` -- the symmetric-matrix Cholesky adjoint (Murray 2016) as the
  closing comment of NVIDIA/warp issue #1316 states it: ``S = Phi(L^T tril(Lbar))``,
  solve ``L^T X = S``, solve ``M L = X``, accumulate ``M + M^T`` into the lower
  triangle of ``Abar`` (``M_ii`` on the diagonal).
* :func:`potrs` / :func:`potrs_adj` -- the solve with the factor, ``X = A^-1 B``
  by ``L Y = B`` then ``L^H X = Y`` (the step jaxmg's potrf leaves out, "without
  performing a solve"), and its reverse mode: ``Bbar += A^-1 Xbar`` and
  ``Lbar += tril((G + G^H) L)`` with ``G = -(A^-1 Xbar) X^H``.
* :func:`hpotrf` / :func:`hpotrf_adj` -- the same for complex Hermitian matrices
  (``A = L L^H``, jaxmg docs intro: "symmetric or Hermitian"), with conjugate
  transposes: ``P = L^H tril(Lbar)``, solves against ``L^H`` and ``L``,
  ``Abar_ij += M_ij + conj(M_ji)`` below the diagonal and ``Re(M_ii)`` on it.

Parity pins for every function are in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "chol_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_F64P = ctypes.POINTER(ctypes.c_double)
_F32P = ctypes.POINTER(ctypes.c_float)
_I32P = ctypes.POINTER(ctypes.c_int32)


def build(force: bool = False) -> str:
    """Compile ``chol_oracle.c`` into ``oracle/_build/liboracle.so`` with gcc.

    ``-ffp-contract=off`` keeps the rounding identical on x86-64 and aarch64.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        for sfx, fp in (("d", _F64P), ("s", _F32P)):
            f = getattr(lib, f"orc_potrf_{sfx}")
            f.argtypes = [ctypes.c_int32, fp, fp, ctypes.c_int32]
            f.restype = ctypes.c_int32
            f = getattr(lib, f"orc_potrf_batch_{sfx}")
            f.argtypes = [ctypes.c_int64, ctypes.c_int32, fp, fp, _I32P, ctypes.c_int32]
            f.restype = None
            f = getattr(lib, f"orc_potrf_adj_{sfx}")
            f.argtypes = [ctypes.c_int32, fp, fp, fp, ctypes.c_int32]
            f.restype = ctypes.c_int32
            f = getattr(lib, f"orc_potrf_adj_batch_{sfx}")
            f.argtypes = [ctypes.c_int64, ctypes.c_int32, fp, fp, fp, _I32P, ctypes.c_int32]
            f.restype = ctypes.c_int32
        for sfx in ("z", "c"):
            f = getattr(lib, f"orc_hpotrf_batch_{sfx}")
            f.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                          _I32P, ctypes.c_int32]
            f.restype = None
            f = getattr(lib, f"orc_hpotrf_adj_batch_{sfx}")
            f.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                          ctypes.c_void_p, _I32P, ctypes.c_int32]
            f.restype = ctypes.c_int32
        for sfx in ("d", "s", "z", "c"):
            f = getattr(lib, f"orc_potrs_{sfx}")
            f.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                          ctypes.c_void_p, ctypes.c_void_p, _I32P, ctypes.c_int32]
            f.restype = ctypes.c_int32
            f = getattr(lib, f"orc_potrs_adj_{sfx}")
            f.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                          _I32P, ctypes.c_int32]
            f.restype = ctypes.c_int32
        lib.orc_max_threads.argtypes = []
        lib.orc_max_threads.restype = ctypes.c_int32
        _lib = lib
        return lib


def max_threads() -> int:
    """Threads OpenMP would use by default in this process."""
    return int(_load().orc_max_threads())


def _prep(x, dtype):
    x = np.ascontiguousarray(x, dtype=dtype)
    return x


def _sfx(dtype):
    dtype = np.dtype(dtype)
    if dtype == np.float64:
        return "d", _F64P
    if dtype == np.float32:
        return "s", _F32P
    raise TypeError(f"oracle supports float32/float64, not {dtype}")


def potrf(A, dtype=None, threads: int = 1):
    """Lower Cholesky factor of one matrix or a batch ``[..., n, n]``.

    Arithmetic runs in ``dtype`` (default: ``A``'s dtype).  Returns
    ``(L, status)``: ``L`` has a zero upper triangle; ``status`` is 0 or the
    1-based first column whose pivot is not positive (numpy int32, shaped like
    the batch).  Past a failing pivot ``L`` is whatever was computed so far.
    """
    A = np.asarray(A)
    dtype = np.dtype(dtype or A.dtype)
    sfx, fp = _sfx(dtype)
    A = _prep(A, dtype)
    n = A.shape[-1]
    if A.ndim < 2 or A.shape[-2] != n:
        raise ValueError("A must be [..., n, n]")
    batch_shape = A.shape[:-2]
    nb = int(np.prod(batch_shape)) if batch_shape else 1
    L = np.zeros_like(A)
    status = np.zeros(nb, dtype=np.int32)
    lib = _load()
    if nb == 1:
        status[0] = getattr(lib, f"orc_potrf_{sfx}")(
            n, A.ctypes.data_as(fp), L.ctypes.data_as(fp), int(threads))
    elif nb > 0:
        getattr(lib, f"orc_potrf_batch_{sfx}")(
            nb, n, A.ctypes.data_as(fp), L.ctypes.data_as(fp),
            status.ctypes.data_as(_I32P), int(threads))
    return L, status.reshape(batch_shape)


def potrf_adj(L, Lbar, Abar=None, status=None, dtype=None, threads: int = 1):
    """Literal Murray adjoint; returns ``Abar`` with ``Phi(M + M^T)`` added.

    ``Abar`` (default zeros) is copied, not modified in place.  Matrices whose
    ``status`` is non-zero are skipped (their ``Abar`` is returned unchanged).
    """
    L = np.asarray(L)
    dtype = np.dtype(dtype or L.dtype)
    sfx, fp = _sfx(dtype)
    L = _prep(L, dtype)
    Lbar = _prep(Lbar, dtype)
    if Lbar.shape != L.shape:
        raise ValueError("L and Lbar must have the same shape")
    out = np.zeros_like(L) if Abar is None else np.array(Abar, dtype=dtype, copy=True, order="C")
    n = L.shape[-1]
    batch_shape = L.shape[:-2]
    nb = int(np.prod(batch_shape)) if batch_shape else 1
    lib = _load()
    if nb == 1 and batch_shape == ():
        if status is not None and int(np.asarray(status).reshape(-1)[0]) != 0:
            return out
        rc = getattr(lib, f"orc_potrf_adj_{sfx}")(
            n, L.ctypes.data_as(fp), Lbar.ctypes.data_as(fp), out.ctypes.data_as(fp),
            int(threads))
    else:
        st = None
        if status is not None:
            st = np.ascontiguousarray(np.asarray(status, dtype=np.int32).reshape(-1))
        rc = getattr(lib, f"orc_potrf_adj_batch_{sfx}")(
            nb, n, L.ctypes.data_as(fp), Lbar.ctypes.data_as(fp), out.ctypes.data_as(fp),
            st.ctypes.data_as(_I32P) if st is not None else None, int(threads))
    if rc != 0:
        raise MemoryError("oracle adjoint could not allocate its scratch")
    return out


def _csfx(dtype):
    dtype = np.dtype(dtype)
    if dtype == np.complex128:
        return "z"
    if dtype == np.complex64:
        return "c"
    raise TypeError(f"complex oracle supports complex64/complex128, not {dtype}")


def hpotrf(A, dtype=None, threads: int = 1):
    """Lower Cholesky factor ``A = L L^H`` of a complex Hermitian matrix or a
    batch ``[..., n, n]`` (complex64/complex128).  Only the lower triangle is
    read, and only the real part of the diagonal.  Returns ``(L, status)`` as
    :func:`potrf` does; ``L`` has a real positive diagonal."""
    A = np.asarray(A)
    dtype = np.dtype(dtype or A.dtype)
    sfx = _csfx(dtype)
    A = np.ascontiguousarray(A, dtype=dtype)
    n = A.shape[-1]
    if A.ndim < 2 or A.shape[-2] != n:
        raise ValueError("A must be [..., n, n]")
    batch_shape = A.shape[:-2]
    nb = int(np.prod(batch_shape)) if batch_shape else 1
    L = np.zeros_like(A)
    status = np.zeros(nb, dtype=np.int32)
    if nb > 0:
        getattr(_load(), f"orc_hpotrf_batch_{sfx}")(
            nb, n, A.ctypes.data, L.ctypes.data, status.ctypes.data_as(_I32P), int(threads))
    return L, status.reshape(batch_shape)


def hpotrf_adj(L, Lbar, Abar=None, status=None, dtype=None, threads: int = 1):
    """Literal Hermitian adjoint; returns a copy of ``Abar`` (default zeros)
    with ``M_ij + conj(M_ji)`` added below the diagonal and ``Re(M_ii)`` on
    it, ``M = L^-H Phi(L^H tril(Lbar)) L^-1``.  ``Lbar`` is the gradient of a
    real loss with respect to ``L`` as ``dLoss/dRe + i dLoss/dIm``.  Matrices
    with non-zero ``status`` are skipped."""
    L = np.asarray(L)
    dtype = np.dtype(dtype or L.dtype)
    sfx = _csfx(dtype)
    L = np.ascontiguousarray(L, dtype=dtype)
    Lbar = np.ascontiguousarray(Lbar, dtype=dtype)
    if Lbar.shape != L.shape:
        raise ValueError("L and Lbar must have the same shape")
    out = np.zeros_like(L) if Abar is None else np.array(Abar, dtype=dtype, copy=True, order="C")
    n = L.shape[-1]
    batch_shape = L.shape[:-2]
    nb = int(np.prod(batch_shape)) if batch_shape else 1
    st = None
    if status is not None:
        st = np.ascontiguousarray(np.asarray(status, dtype=np.int32).reshape(-1))
    rc = getattr(_load(), f"orc_hpotrf_adj_batch_{sfx}")(
        nb, n, L.ctypes.data, Lbar.ctypes.data, out.ctypes.data,
        st.ctypes.data_as(_I32P) if st is not None else None, int(threads))
    if rc != 0:
        raise MemoryError("oracle adjoint could not allocate its scratch")
    return out


_ANY_SFX = {np.dtype(np.float64): "d", np.dtype(np.float32): "s",
            np.dtype(np.complex128): "z", np.dtype(np.complex64): "c"}


def _status_arg(status):
    if status is None:
        return None, None
    st = np.ascontiguousarray(np.asarray(status, dtype=np.int32).reshape(-1))
    return st, st.ctypes.data_as(_I32P)


def potrs(L, B, status=None, dtype=None, threads: int = 1):
    """``X = A^-1 B`` with ``A = L L^H`` (``L^T`` for real types): ``L`` is
    ``[..., n, n]`` (lower triangle read), ``B`` is ``[..., n, nrhs]``.
    Matrices with non-zero ``status`` get ``X`` = zeros."""
    L = np.asarray(L)
    dtype = np.dtype(dtype or L.dtype)
    sfx = _ANY_SFX[dtype]
    L = np.ascontiguousarray(L, dtype=dtype)
    B = np.ascontiguousarray(B, dtype=dtype)
    n = L.shape[-1]
    if B.shape[:-1] != L.shape[:-1]:
        raise ValueError("B must be [..., n, nrhs] with L's batch shape and n")
    nrhs = B.shape[-1]
    nb = int(np.prod(L.shape[:-2])) if L.shape[:-2] else 1
    X = np.zeros_like(B)
    st, stp = _status_arg(status)
    if nb > 0 and n > 0 and nrhs > 0:
        rc = getattr(_load(), f"orc_potrs_{sfx}")(nb, n, nrhs, L.ctypes.data, B.ctypes.data,
                                                  X.ctypes.data, stp, int(threads))
        if rc != 0:
            raise MemoryError("oracle solve could not allocate its scratch")
    return X


def potrs_adj(L, X, Xbar, Bbar=None, Lbar=None, status=None, dtype=None, threads: int = 1):
    """Reverse mode of :func:`potrs`.  Returns ``(Bbar + A^-1 Xbar,
    Lbar + tril((G + G^H) L))`` with ``G = -(A^-1 Xbar) X^H`` (copies; the
    defaults are zeros).  Matrices with non-zero ``status`` are skipped."""
    L = np.asarray(L)
    dtype = np.dtype(dtype or L.dtype)
    sfx = _ANY_SFX[dtype]
    L = np.ascontiguousarray(L, dtype=dtype)
    X = np.ascontiguousarray(X, dtype=dtype)
    Xbar = np.ascontiguousarray(Xbar, dtype=dtype)
    n, nrhs = L.shape[-1], X.shape[-1]
    nb = int(np.prod(L.shape[:-2])) if L.shape[:-2] else 1
    Bo = np.zeros_like(X) if Bbar is None else np.array(Bbar, dtype=dtype, copy=True, order="C")
    Lo = np.zeros_like(L) if Lbar is None else np.array(Lbar, dtype=dtype, copy=True, order="C")
    st, stp = _status_arg(status)
    if nb > 0 and n > 0 and nrhs > 0:
        rc = getattr(_load(), f"orc_potrs_adj_{sfx}")(
            nb, n, nrhs, L.ctypes.data, X.ctypes.data, Xbar.ctypes.data, Bo.ctypes.data,
            Lo.ctypes.data, stp, int(threads))
        if rc != 0:
            raise MemoryError("oracle solve adjoint could not allocate its scratch")
    return Bo, Lo
