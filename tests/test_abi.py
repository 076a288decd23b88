"""The C-ABI library loads and exports every symbol include/chol.h declares;
argument checks that need no GPU return the documented codes (CPU only)."""
import ctypes
import os
import re

import numpy as np
import pytest

from differentiable_cholesky_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in sorted(os.listdir(os.path.join(ROOT, "include")))
           if h.endswith(".h")]

CHOL_OK, CHOL_EINVAL, CHOL_EDTYPE = 0, -1, -2


def declared_symbols():
    text = "".join(open(h).read() for h in HEADERS)
    return sorted(set(re.findall(r"CHOL_API\s+[\w\s\*]+?\b(chol_\w+)\s*\(", text)))


def test_header_declares_the_path():
    syms = declared_symbols()
    for s in ("chol_fwd", "chol_adj", "chol_fwd_ex", "chol_adj_ex", "chol_strerror",
              "chol_abi_version", "chol_probe_fma_peak", "chol_fwd_inplace", "chol_adj_inplace"):
        assert s in syms


def test_library_exports_every_declared_symbol():
    lib = binding.load_library()
    for s in declared_symbols():
        assert hasattr(lib, s), f"{s} not exported"
    assert lib.chol_abi_version() == (1 << 16) | 4


def test_strerror_covers_every_code():
    lib = binding.load_library()
    for code in (0, -1, -2, -3, -4, -5):
        txt = lib.chol_strerror(code).decode()
        assert txt and "unknown" not in txt
    assert "unknown" in lib.chol_strerror(-99).decode()


def test_argument_checks_without_gpu():
    lib = binding.load_library()
    buf = (ctypes.c_double * 16)()
    st = (ctypes.c_int32 * 4)()
    p, s = ctypes.addressof(buf), ctypes.addressof(st)
    # bad dtype, bad n, bad batch, bad tile
    assert lib.chol_fwd(1, 4, 7, p, p, s, None) == CHOL_EDTYPE
    assert lib.chol_fwd(1, 0, 1, p, p, s, None) == CHOL_EINVAL
    assert lib.chol_fwd(-1, 4, 1, p, p, s, None) == CHOL_EINVAL
    assert lib.chol_fwd_ex(1, 100, 1, p, p, s, 48, None) == CHOL_EINVAL
    assert lib.chol_adj(1, -3, 0, p, p, p, None, None) == CHOL_EINVAL
    assert lib.chol_adj(1, 4, 5, p, p, p, None, None) == CHOL_EDTYPE
    # complex double takes tiles up to 64
    assert lib.chol_fwd_ex(1, 100, 3, p, p, s, 128, None) == CHOL_EINVAL
    assert lib.chol_adj_ex(1, 100, 3, p, p, p, None, 128, None) == CHOL_EINVAL
    # batch == 0 is a no-op, even with null pointers
    assert lib.chol_fwd(0, 4, 1, None, None, None, None) == CHOL_OK
    assert lib.chol_adj(0, 4, 1, None, None, None, None, None) == CHOL_OK
    # null pointers
    assert lib.chol_fwd(1, 4, 1, None, p, s, None) == CHOL_EINVAL
    assert lib.chol_adj(1, 4, 1, p, None, p, None, None) == CHOL_EINVAL
    # misaligned element pointer
    assert lib.chol_fwd(1, 2, 1, p + 4, p + 64, s, None) == CHOL_EINVAL
    # host memory is rejected (not a device pointer)
    big = (ctypes.c_double * 64)()
    q = ctypes.addressof(big)
    assert lib.chol_fwd(1, 2, 1, q, q + 256, s, None) == CHOL_EINVAL


def test_probe_argument_checks_without_gpu():
    lib = binding.load_library()
    d = ctypes.c_double()
    p = ctypes.byref(d)
    buf = (ctypes.c_double * 16)()
    q = ctypes.addressof(buf)
    lib.chol_probe_tc_update.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
                                         ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p]
    # n <= 128, k out of range, reps <= 0, null pointers: rejected before any GPU call
    assert lib.chol_probe_tc_update(128, q, 0, 1, p, p, p, None) == CHOL_EINVAL
    assert lib.chol_probe_tc_update(512, q, 3, 1, p, p, p, None) == CHOL_EINVAL
    assert lib.chol_probe_tc_update(512, q, -1, 1, p, p, p, None) == CHOL_EINVAL
    assert lib.chol_probe_tc_update(512, q, 0, 0, p, p, p, None) == CHOL_EINVAL
    assert lib.chol_probe_tc_update(512, None, 0, 1, p, p, p, None) == CHOL_EINVAL
    assert lib.chol_probe_tc_update(512, q, 0, 1, None, p, p, None) == CHOL_EINVAL


def test_inplace_argument_checks_without_gpu():
    lib = binding.load_library()
    buf = (ctypes.c_double * 16)()
    st = (ctypes.c_int32 * 4)()
    p, s = ctypes.addressof(buf), ctypes.addressof(st)
    assert lib.chol_fwd_inplace(1, 4, 7, p, s, 0, None) == CHOL_EDTYPE
    assert lib.chol_fwd_inplace(1, 0, 1, p, s, 0, None) == CHOL_EINVAL
    assert lib.chol_fwd_inplace(1, 100, 1, p, s, 48, None) == CHOL_EINVAL
    assert lib.chol_fwd_inplace(0, 4, 1, None, None, 0, None) == CHOL_OK
    assert lib.chol_fwd_inplace(1, 4, 1, None, s, 0, None) == CHOL_EINVAL
    assert lib.chol_fwd_inplace(1, 2, 1, p + 4, s, 0, None) == CHOL_EINVAL
    assert lib.chol_adj_inplace(1, 4, 9, p, p, None, 0, None) == CHOL_EDTYPE
    assert lib.chol_adj_inplace(0, 4, 1, None, None, None, 0, None) == CHOL_OK
    assert lib.chol_adj_inplace(1, 4, 1, p, None, None, 0, None) == CHOL_EINVAL
    assert lib.chol_adj_inplace(1, 4, 1, None, p, None, 0, None) == CHOL_EINVAL
    # host memory is rejected (not a device pointer)
    assert lib.chol_fwd_inplace(1, 2, 1, p, s, 0, None) == CHOL_EINVAL
    assert lib.chol_adj_inplace(1, 2, 1, p, p + 64, None, 0, None) == CHOL_EINVAL


def test_selftest_argument_checks_without_gpu():
    lib = binding.load_library()
    lib.chol_selftest_wait_timeout.argtypes = [ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_uint32, ctypes.c_void_p]
    buf = (ctypes.c_float * 512)()
    st = (ctypes.c_int32 * 2)()
    p, s = ctypes.addressof(buf), ctypes.addressof(st)
    assert lib.chol_selftest_wait_timeout(0, None, None, None, 10, None) == CHOL_OK
    assert lib.chol_selftest_wait_timeout(-1, p, p, s, 10, None) == CHOL_EINVAL
    assert lib.chol_selftest_wait_timeout(1, p, p + 1024, s, 0, None) == CHOL_EINVAL
    assert lib.chol_selftest_wait_timeout(1, None, p, s, 10, None) == CHOL_EINVAL
    # host memory is rejected (not a device pointer)
    assert lib.chol_selftest_wait_timeout(1, p, p + 1024, s, 10, None) == CHOL_EINVAL


def test_tile_header_compiles_in_a_user_kernel():
    """include/chol_tile.cuh is header-only device code: the test kernels that
    use it as a caller would must compile for sm_103a with only include/ on the
    path (the GPU test runs them)."""
    import shutil
    import subprocess
    import tempfile
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    src = os.path.join(ROOT, "tests", "tile_api", "tile_api_kernels.cu")
    with tempfile.TemporaryDirectory() as d:
        subprocess.run([nvcc, "-std=c++17", "-O1", "-I", os.path.join(ROOT, "include"),
                        "-gencode", "arch=compute_103a,code=sm_103a", "-c", src,
                        "-o", os.path.join(d, "t.o")], check=True)


def test_size_overflow_rejected():
    lib = binding.load_library()
    buf = (ctypes.c_double * 4)()
    p = ctypes.addressof(buf)
    assert lib.chol_fwd(1 << 40, 1 << 20, 1, p, p, p, None) == CHOL_EINVAL


def test_binding_rejects_cpu_tensors():
    torch = pytest.importorskip("torch")
    A = torch.eye(4, dtype=torch.float64)
    with pytest.raises(ValueError):
        binding.chol_fwd(A)
    with pytest.raises(ValueError):
        binding.chol_adj(A, A)


def test_noalloc_adjoint_returns_the_same_codes_as_chol_adj_ex():
    """chol_adj_noalloc promises chol_adj_ex's argument checks: both entry
    points must answer every bad argument with the same code."""
    lib = binding.load_library()
    buf = (ctypes.c_double * 64)()
    st = (ctypes.c_int32 * 4)()
    p, s = ctypes.addressof(buf), ctypes.addressof(st)
    cases = [
        (1, 4, 7, p, p, p, None, 0),          # dtype
        (1, 0, 1, p, p, p, None, 0),          # n
        (-2, 4, 1, p, p, p, None, 0),         # batch
        (1, 100, 1, p, p, p, None, 48),       # tile
        (1, 4, 1, None, p, p, None, 0),       # null L
        (1, 4, 1, p, None, p, None, 0),       # null adj_L
        (1, 4, 1, p, p, None, None, 0),       # null adj_A
        (1, 4, 1, p + 4, p, p, None, 0),      # misaligned L
        (1, 4, 1, p, p, p, s + 2, 0),         # misaligned status
        (1, 4, 1, p, p, p, None, 0),          # host pointers
        (0, 4, 1, None, None, None, None, 0), # empty batch: no-op
        (1 << 40, 1 << 20, 1, p, p, p, None, 0),  # size overflow
    ]
    for args in cases:
        a = lib.chol_adj_ex(*args, None)
        b = lib.chol_adj_noalloc(*args, None)
        assert a == b, (args, a, b)
