"""Seeded synthetic inputs shared by the GPU path's tests/bench and the oracle.

This module only draws random numbers and assembles symmetric positive-definite
test matrices; it contains none of the factorisation or adjoint arithmetic and
imports neither the CUDA binding nor the oracle.  All draws use numpy's PCG64
``default_rng(seed)``, which gives the same stream on every platform.

The five workloads (with the pages' own closed-form case first):

* ``bidiagonal_512``: one 512x512 float64 ``A = E E^T`` with ``E`` lower
  bidiagonal, diagonal ``linspace(1, 2, 512)``, sub-diagonal 0.5 -- the worked
  example of the jaxmg docs "Cholesky factorization" (``make_matrix``; tile
  size 128), whose factor must equal ``E``.
* ``batched_16``: 65536 float32 16x16, ``A = G G^T / 16 + I``.
* ``batched_64``: 8192 float32 64x64, ``A = G G^T / 64 + 0.5 I``; every 100th
  matrix gets ``A[k, k] = -1`` (``k`` uniform in [0, 64) from seed 2), so its
  status is exactly ``k + 1``.
* ``batched_512``: 256 float64 512x512, ``A = G G^T / 512 + I``.
* ``banded_8192``: one 8192x8192 float64 ``A = E E^T`` with ``E`` lower banded
  (bandwidth 32), diagonal U[1, 2], band N(0, 0.1); the factor must equal ``E``.

``G`` is drawn with seed 0 (``E`` for the banded case too) and ``adj_L`` is
``tril(N(0, 1))`` with seed 1 (seed 0 for the single bidiagonal matrix).
Products are formed in float64 and rounded once to the workload's dtype.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass
class Workload:
    name: str
    batch: int
    n: int
    dtype: np.dtype
    A: np.ndarray                 # [batch, n, n] (batch kept even when 1)
    adj_L: np.ndarray             # [batch, n, n], lower triangular
    expected_L: np.ndarray | None = None   # closed-form factor, when known
    expected_status: np.ndarray | None = None
    meta: dict = field(default_factory=dict)


def tril_normal(batch: int, n: int, seed: int, dtype) -> np.ndarray:
    """``tril(N(0, 1))`` in ``[batch, n, n]``, drawn in float64, then cast."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((batch, n, n))
    return np.tril(x).astype(dtype)


def gram_spd(batch: int, n: int, seed: int, shift: float, dtype,
             scale: float | None = None) -> np.ndarray:
    """``A_b = G_b G_b^T / scale + shift * I`` (scale defaults to n)."""
    rng = np.random.default_rng(seed)
    G = rng.standard_normal((batch, n, n))
    s = float(n if scale is None else scale)
    A = np.matmul(G, np.swapaxes(G, -1, -2)) / s
    idx = np.arange(n)
    A[:, idx, idx] += shift
    return A.astype(dtype)


def tril_normal_complex(batch: int, n: int, seed: int, dtype) -> np.ndarray:
    """``tril(N(0, 1) + i N(0, 1))`` in ``[batch, n, n]`` (real and imaginary
    parts drawn in that order as one ``[2, batch, n, n]`` array), then cast."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((2, batch, n, n))
    return np.tril(x[0] + 1j * x[1]).astype(dtype)


def hermitian_spd(batch: int, n: int, seed: int, shift: float, dtype,
                  scale: float | None = None) -> np.ndarray:
    """``A_b = G_b G_b^H / scale + shift * I`` with complex Gaussian ``G``
    (real and imaginary parts N(0, 1)); scale defaults to n."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((2, batch, n, n))
    G = x[0] + 1j * x[1]
    s = float(n if scale is None else scale)
    A = np.matmul(G, np.conj(np.swapaxes(G, -1, -2))) / s
    idx = np.arange(n)
    A[:, idx, idx] = A[:, idx, idx].real + shift
    return A.astype(dtype)


def bidiagonal_E(n: int) -> np.ndarray:
    """Lower bidiagonal E: diagonal linspace(1, 2, n), sub-diagonal 0.5."""
    E = np.diag(np.linspace(1.0, 2.0, n))
    if n > 1:
        E += np.diag(np.full(n - 1, 0.5), k=-1)
    return E


def banded_E(n: int, bandwidth: int, seed: int, sigma: float = 0.1) -> np.ndarray:
    """Lower banded E: diagonal U[1, 2], sub-diagonals 1..bandwidth N(0, sigma)."""
    rng = np.random.default_rng(seed)
    diag = rng.uniform(1.0, 2.0, n)
    band = rng.standard_normal((bandwidth, n)) * sigma
    E = np.zeros((n, n))
    idx = np.arange(n)
    E[idx, idx] = diag
    for d in range(1, bandwidth + 1):
        E[idx[d:], idx[:-d]] = band[d - 1, : n - d]
    return E


def banded_gram(E: np.ndarray, bandwidth: int) -> np.ndarray:
    """``E E^T`` for lower-banded E, formed band-wise (O(n * bandwidth^2))."""
    n = E.shape[0]
    A = np.zeros((n, n))
    w = bandwidth
    # (E E^T)_ij = sum_k E_ik E_jk with k in [max(i,j)-w, min(i,j)].
    Eb = np.zeros((n, w + 1))     # Eb[i, t] = E[i, i - t]
    idx = np.arange(n)
    for t in range(w + 1):
        Eb[t:, t] = E[idx[t:], idx[t:] - t]
    for d in range(0, w + 1):      # A[i, i-d]
        i = idx[d:]
        acc = np.zeros(n - d)
        for t in range(0, w + 1 - d):
            # k = i - d - t  =>  E[i, k] = Eb[i, d + t], E[i-d, k] = Eb[i-d, t]
            acc += Eb[i, d + t] * Eb[i - d, t]
        A[i, i - d] = acc
        A[i - d, i] = acc
    return A


def bidiagonal_512(n: int = 512) -> Workload:
    E = bidiagonal_E(n)
    A = (E @ E.T)[None]
    return Workload("bidiagonal_512", 1, n, np.dtype(np.float64), A,
                    tril_normal(1, n, 0, np.float64), expected_L=E[None],
                    expected_status=np.zeros(1, np.int32),
                    meta={"tile": 128})


def batched_16(batch: int = 65536, n: int = 16) -> Workload:
    A = gram_spd(batch, n, 0, 1.0, np.float32)
    return Workload("batched_16", batch, n, np.dtype(np.float32), A,
                    tril_normal(batch, n, 1, np.float32),
                    expected_status=np.zeros(batch, np.int32))


def batched_64(batch: int = 8192, n: int = 64, fail_every: int = 100) -> Workload:
    A = gram_spd(batch, n, 0, 0.5, np.float64)
    rng = np.random.default_rng(2)
    fails = np.arange(0, batch, fail_every)
    ks = rng.integers(0, n, size=fails.size)
    A[fails, ks, ks] = -1.0
    status = np.zeros(batch, np.int32)
    status[fails] = ks + 1
    return Workload("batched_64", batch, n, np.dtype(np.float32), A.astype(np.float32),
                    tril_normal(batch, n, 1, np.float32), expected_status=status,
                    meta={"failing": fails, "k": ks})


def batched_512(batch: int = 256, n: int = 512) -> Workload:
    A = gram_spd(batch, n, 0, 1.0, np.float64)
    return Workload("batched_512", batch, n, np.dtype(np.float64), A,
                    tril_normal(batch, n, 1, np.float64),
                    expected_status=np.zeros(batch, np.int32), meta={"tile": 128})


def banded_8192(n: int = 8192, bandwidth: int = 32) -> Workload:
    E = banded_E(n, bandwidth, 0)
    A = banded_gram(E, bandwidth)[None]
    return Workload("banded_8192", 1, n, np.dtype(np.float64), A,
                    tril_normal(1, n, 1, np.float64), expected_L=E[None],
                    expected_status=np.zeros(1, np.int32),
                    meta={"tile": 128, "bandwidth": bandwidth})


WORKLOADS = {
    "bidiagonal_512": bidiagonal_512,
    "batched_16": batched_16,
    "batched_64": batched_64,
    "batched_512": batched_512,
    "banded_8192": banded_8192,
}
