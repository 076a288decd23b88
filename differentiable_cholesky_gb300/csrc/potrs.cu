// Solve with the Cholesky factor, X = A^-1 B = L^-H L^-1 B, and its reverse
// mode: the step the jaxmg docs "Cholesky factorization" leave out of potrf
// (intro: the lower factor "without performing a solve").  Real types read
// ^H as ^T; complex types are Hermitian.
//
// Solve: forward substitution L Y = B, then back substitution L^H X = Y, on
// the right-hand sides' columns.
//   n <= 64: one block per (matrix, 64 right-hand sides), L packed in shared
//            memory, one thread per right-hand side.
//   n > 64:  64-row tiles: a diagonal-tile solve (as above, on X's rows of
//            the tile) then a tile update of the rows still to solve
//            (X_i -= L_ik X_k going down, X_i -= L_ki^H X_k coming up).
// Reverse mode, for a loss gradient adj_X:
//   Bb = A^-1 adj_X (the same solve), adj_B += Bb, and
//   adj_L += tril(-(Bb X^H + X Bb^H) L) = tril(-(Bb U^H + X V^H))
//   with U = L^H X and V = L^H Bb (n x nrhs each), so that no n x n
//   intermediate is formed: O(n^2 nrhs) instead of O(n^3).
// Matrices whose status is non-zero get X = 0 and are skipped by the adjoint.

#include <cuda_runtime.h>

#include <algorithm>
#include <type_traits>

#include "chol_tile.cuh"
#include "common.cuh"
#include "kernels.h"

namespace chol {
namespace {

using chol_tile::cplx;
using chol_tile::detail::add;
using chol_tile::detail::conj;
using chol_tile::detail::madd;
using chol_tile::detail::msub;
using chol_tile::detail::re;
using chol_tile::detail::scale;
using chol_tile::detail::sub;

constexpr int kTS = 64;      // tile of the blocked solve; right-hand sides per block
constexpr int kThreads = 256;

__device__ __forceinline__ bool skipped(const int32_t* status, int64_t b) {
    return status != nullptr && status[b] != 0;
}

inline unsigned gy(int64_t batch) { return (unsigned)std::min<int64_t>(batch, 65535); }

// ---------------------------------------------------------------------------
// Triangular solves of rows [r0, r0 + m) of X (n x nrhs) against the
// diagonal tile G = L[r0 .. r0+m, r0 .. r0+m] (m <= 64): FWD solves G y = x,
// BWD solves G^H y = x, in place; one thread per right-hand side.
// ---------------------------------------------------------------------------
template <typename T, bool FWD>
__global__ void __launch_bounds__(kTS)
diag_solve_kernel(const T* __restrict__ L, T* X, const int32_t* __restrict__ status,
                  int64_t batch, int n, int nrhs, int r0, int m) {
    using R = typename chol_tile::detail::real_of<T>::type;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* G = reinterpret_cast<T*>(smem_raw);                   // packed lower tile
    T(*Y)[kTS + 1] = reinterpret_cast<T(*)[kTS + 1]>(G + kTS * (kTS + 1) / 2);  // [rhs][row]
    R* ginv = reinterpret_cast<R*>(Y + kTS);
    const int c = threadIdx.x;
    const int col = blockIdx.x * kTS + c;
    for (int64_t b = blockIdx.y; b < batch; b += gridDim.y) {
        if (skipped(status, b)) continue;
        const T* Lb = L + b * (int64_t)n * n;
        T* Xb = X + b * (int64_t)n * nrhs;
        __syncthreads();
        for (int e = threadIdx.x; e < m * m; e += kTS) {
            const int i = e / m, j = e % m;
            if (j <= i) G[i * (i + 1) / 2 + j] = Lb[(int64_t)(r0 + i) * n + r0 + j];
        }
        // rows of X: coalesced over the right-hand sides
        for (int i = 0; i < m; ++i)
            Y[c][i] = col < nrhs ? Xb[(int64_t)(r0 + i) * nrhs + col] : T{};
        __syncthreads();
        for (int i = threadIdx.x; i < m; i += kTS) ginv[i] = R(1) / re(G[i * (i + 1) / 2 + i]);
        __syncthreads();
        T* y = Y[c];
        if (FWD) {
            for (int i = 0; i < m; ++i) {
                T s = y[i];
                const T* g = G + i * (i + 1) / 2;
                for (int k = 0; k < i; ++k) s = msub(g[k], y[k], s);
                y[i] = scale(s, ginv[i]);
            }
        } else {
            for (int i = m - 1; i >= 0; --i) {
                T s = y[i];
                for (int k = i + 1; k < m; ++k) s = msub(conj(G[k * (k + 1) / 2 + i]), y[k], s);
                y[i] = scale(s, ginv[i]);
            }
        }
        __syncthreads();
        if (col < nrhs)
            for (int i = 0; i < m; ++i) Xb[(int64_t)(r0 + i) * nrhs + col] = Y[c][i];
    }
}

// ---------------------------------------------------------------------------
// A 64 x 64 output tile C (+)= sum_k op_a(r, k) op_b(k, c) over a reduction,
// 256 threads with 4 x 4 outputs each; the loaders fetch one element (zero
// outside the operands).
// ---------------------------------------------------------------------------
template <typename T, typename LA, typename LB>
__device__ __forceinline__ void tile_mm(T (&acc)[4][4], int klen, LA load_a, LB load_b) {
    constexpr int BK = 16;
    __shared__ T As[BK][kTS + 1];
    __shared__ T Bs[BK][kTS + 1];
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    for (int k0 = 0; k0 < klen; k0 += BK) {
        __syncthreads();
        for (int e = threadIdx.x; e < BK * kTS; e += kThreads) {
            const int kk = e / kTS, x = e % kTS;
            As[kk][x] = k0 + kk < klen ? load_a(x, k0 + kk) : T{};
            Bs[kk][x] = k0 + kk < klen ? load_b(k0 + kk, x) : T{};
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            T a[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = madd(a[i], bv[j], acc[i][j]);
        }
    }
}

// Rows still to solve, after diagonal tile k (rows k0 .. k0+kb):
// FWD: X_i -= L[i, k-tile] X_k-tile for rows i >= k0 + kb;
// BWD: X_i -= L[k-tile, i]^H X_k-tile for rows i < k0.
template <typename T, bool FWD>
__global__ void __launch_bounds__(kThreads)
solve_update_kernel(const T* __restrict__ L, T* X, const int32_t* __restrict__ status,
                    int64_t batch, int n, int nrhs, int k0, int kb, int row_begin) {
    const int i0 = row_begin + blockIdx.x * kTS;  // first output row
    const int c0 = blockIdx.z * kTS;             // first right-hand side
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    for (int64_t b = blockIdx.y; b < batch; b += gridDim.y) {
        if (skipped(status, b)) continue;
        const T* Lb = L + b * (int64_t)n * n;
        T* Xb = X + b * (int64_t)n * nrhs;
        const int row_end = FWD ? n : k0;
        T acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = T{};
        tile_mm(
            acc, kb,
            [&](int r, int k) -> T {
                const int gi = i0 + r;
                if (gi >= row_end) return T{};
                return FWD ? Lb[(int64_t)gi * n + k0 + k] : conj(Lb[(int64_t)(k0 + k) * n + gi]);
            },
            [&](int k, int c) -> T {
                const int gc = c0 + c;
                return gc < nrhs ? Xb[(int64_t)(k0 + k) * nrhs + gc] : T{};
            });
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int gi = i0 + ty * 4 + i;
            if (gi >= row_end) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int gc = c0 + tx * 4 + j;
                if (gc < nrhs) Xb[(int64_t)gi * nrhs + gc] = sub(Xb[(int64_t)gi * nrhs + gc], acc[i][j]);
            }
        }
    }
}

// Y = L^H Z for n x nrhs Z: Y_j = sum_{i >= j} conj(L_ij) Z_i.
template <typename T>
__global__ void __launch_bounds__(kThreads)
trmm_lh_kernel(const T* __restrict__ L, const T* __restrict__ Z, T* __restrict__ Y,
               const int32_t* __restrict__ status, int64_t batch, int n, int nrhs) {
    const int j0 = blockIdx.x * kTS, c0 = blockIdx.z * kTS;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    for (int64_t b = blockIdx.y; b < batch; b += gridDim.y) {
        if (skipped(status, b)) continue;
        const T* Lb = L + b * (int64_t)n * n;
        const T* Zb = Z + b * (int64_t)n * nrhs;
        T* Yb = Y + b * (int64_t)n * nrhs;
        T acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = T{};
        // reduction over rows i = j0 .. n-1 (the lower part i >= j is tested per element)
        tile_mm(
            acc, n - j0,
            [&](int r, int k) -> T {
                const int j = j0 + r, i = j0 + k;
                return (j < n && i >= j) ? conj(Lb[(int64_t)i * n + j]) : T{};
            },
            [&](int k, int c) -> T {
                const int gc = c0 + c;
                return gc < nrhs ? Zb[(int64_t)(j0 + k) * nrhs + gc] : T{};
            });
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = j0 + ty * 4 + i;
            if (j >= n) continue;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int gc = c0 + tx * 4 + jj;
                if (gc < nrhs) Yb[(int64_t)j * nrhs + gc] = acc[i][jj];
            }
        }
    }
}

// adj_L_ij -= sum_c (P_ic conj(U_jc) + Q_ic conj(V_jc)) on the lower
// triangle (i >= j), one 64 x 64 tile (I >= J) per block.
template <typename T>
__global__ void __launch_bounds__(kThreads)
lower_rank_update_kernel(const T* __restrict__ P, const T* __restrict__ U,
                         const T* __restrict__ Q, const T* __restrict__ V, T* __restrict__ Lbar,
                         const int32_t* __restrict__ status, int64_t batch, int n, int nrhs) {
    // tile (I, J) of a row-major enumeration of the lower tile triangle
    const int t = blockIdx.x;
    int I = (int)((sqrt(8.0 * t + 1.0) - 1.0) * 0.5);
    while ((I + 1) * (I + 2) / 2 <= t) ++I;
    while (I * (I + 1) / 2 > t) --I;
    const int J = t - I * (I + 1) / 2;
    const int i0 = I * kTS, j0 = J * kTS;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    for (int64_t b = blockIdx.y; b < batch; b += gridDim.y) {
        if (skipped(status, b)) continue;
        const int64_t off = b * (int64_t)n * nrhs;
        T acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = T{};
        // reduction of length 2 nrhs: the P U^H half, then the Q V^H half
        tile_mm(
            acc, 2 * nrhs,
            [&](int r, int k) -> T {
                const int i = i0 + r;
                if (i >= n) return T{};
                return k < nrhs ? P[off + (int64_t)i * nrhs + k] : Q[off + (int64_t)i * nrhs + k - nrhs];
            },
            [&](int k, int c) -> T {
                const int j = j0 + c;
                if (j >= n) return T{};
                return conj(k < nrhs ? U[off + (int64_t)j * nrhs + k] : V[off + (int64_t)j * nrhs + k - nrhs]);
            });
        T* Lb = Lbar + b * (int64_t)n * n;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int gi = i0 + ty * 4 + i;
            if (gi >= n) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int gj = j0 + tx * 4 + j;
                if (gj < n && gj <= gi) Lb[(int64_t)gi * n + gj] = sub(Lb[(int64_t)gi * n + gj], acc[i][j]);
            }
        }
    }
}

// X_b = 0 for the matrices with status != 0; dst += src elementwise (skipped
// matrices untouched).
template <typename T>
__global__ void __launch_bounds__(kThreads)
zero_skipped_kernel(T* X, const int32_t* __restrict__ status, int64_t batch, int64_t per) {
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < batch * per;
         e += (int64_t)gridDim.x * blockDim.x)
        if (skipped(status, e / per)) X[e] = T{};
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
add_kernel(const T* __restrict__ src, T* __restrict__ dst, const int32_t* __restrict__ status,
           int64_t batch, int64_t per) {
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < batch * per;
         e += (int64_t)gridDim.x * blockDim.x)
        if (!skipped(status, e / per)) dst[e] = add(dst[e], src[e]);
}

template <typename T>
constexpr size_t diag_solve_smem() {
    return (size_t)kTS * (kTS + 1) / 2 * sizeof(T) + (size_t)kTS * (kTS + 1) * sizeof(T) +
           kTS * sizeof(T);
}

inline unsigned ew_blocks(int64_t total) {
    return (unsigned)std::max<int64_t>(
        1, std::min<int64_t>((total + kThreads - 1) / kThreads, (int64_t)device_sm_count() * 16));
}

#define CHOL_TRY(x)                              \
    do {                                         \
        cudaError_t e_ = (x);                    \
        if (e_ != cudaSuccess) return e_;        \
    } while (0)

// X = A^-1 X in place (X holds B on entry).
template <typename T>
cudaError_t solve_in_place(const T* L, T* X, const int32_t* status, int64_t batch, int n,
                           int nrhs, cudaStream_t stream) {
    const int nt = (n + kTS - 1) / kTS;
    const unsigned rc = (unsigned)((nrhs + kTS - 1) / kTS);
    constexpr size_t dsm = diag_solve_smem<T>();
    static std::atomic<uint64_t> set_fwd{0}, set_bwd{0};
    CHOL_TRY(allow_smem_once(diag_solve_kernel<T, true>, dsm, set_fwd));
    CHOL_TRY(allow_smem_once(diag_solve_kernel<T, false>, dsm, set_bwd));
    for (int k = 0; k < nt; ++k) {
        const int k0 = k * kTS, kb = std::min(kTS, n - k0);
        diag_solve_kernel<T, true><<<dim3(rc, gy(batch)), kTS, dsm, stream>>>(L, X, status, batch,
                                                                             n, nrhs, k0, kb);
        CHOL_TRY(cudaGetLastError());
        const int below = n - k0 - kb;
        if (below > 0) {
            solve_update_kernel<T, true><<<dim3((below + kTS - 1) / kTS, gy(batch), rc), kThreads,
                                           0, stream>>>(L, X, status, batch, n, nrhs, k0, kb,
                                                        k0 + kb);
            CHOL_TRY(cudaGetLastError());
        }
    }
    for (int k = nt - 1; k >= 0; --k) {
        const int k0 = k * kTS, kb = std::min(kTS, n - k0);
        diag_solve_kernel<T, false><<<dim3(rc, gy(batch)), kTS, dsm, stream>>>(L, X, status,
                                                                              batch, n, nrhs, k0,
                                                                              kb);
        CHOL_TRY(cudaGetLastError());
        if (k0 > 0) {
            solve_update_kernel<T, false><<<dim3((k0 + kTS - 1) / kTS, gy(batch), rc), kThreads, 0,
                                            stream>>>(L, X, status, batch, n, nrhs, k0, kb, 0);
            CHOL_TRY(cudaGetLastError());
        }
    }
    return cudaSuccess;
}

}  // namespace

template <typename T>
cudaError_t potrs_solve(const T* L, const T* B, T* X, const int32_t* status, int64_t batch,
                        int n, int nrhs, cudaStream_t stream) {
    const int64_t per = (int64_t)n * nrhs;
    if (X != B)
        CHOL_TRY(cudaMemcpyAsync(X, B, (size_t)(batch * per) * sizeof(T), cudaMemcpyDeviceToDevice,
                                 stream));
    CHOL_TRY(solve_in_place(L, X, status, batch, n, nrhs, stream));
    if (status != nullptr) {
        zero_skipped_kernel<T><<<ew_blocks(batch * per), kThreads, 0, stream>>>(X, status, batch,
                                                                               per);
        CHOL_TRY(cudaGetLastError());
    }
    return cudaSuccess;
}

size_t potrs_adj_workspace_elems(int64_t batch, int n, int nrhs, bool want_L) {
    return (size_t)batch * n * nrhs * (want_L ? 3 : 1);
}

template <typename T>
cudaError_t potrs_adj(const T* L, const T* X, const T* Xbar, T* Bbar, T* Lbar,
                      const int32_t* status, int64_t batch, int n, int nrhs, T* work,
                      cudaStream_t stream) {
    const int64_t per = (int64_t)n * nrhs;
    T* Bb = work;  // A^-1 adj_X
    CHOL_TRY(cudaMemcpyAsync(Bb, Xbar, (size_t)(batch * per) * sizeof(T), cudaMemcpyDeviceToDevice,
                             stream));
    CHOL_TRY(solve_in_place(L, Bb, status, batch, n, nrhs, stream));
    if (Bbar != nullptr) {
        add_kernel<T><<<ew_blocks(batch * per), kThreads, 0, stream>>>(Bb, Bbar, status, batch, per);
        CHOL_TRY(cudaGetLastError());
    }
    if (Lbar == nullptr) return cudaSuccess;
    T* U = work + batch * per;      // L^H X
    T* V = U + batch * per;         // L^H Bb
    const int nt = (n + kTS - 1) / kTS;
    const unsigned rc = (unsigned)((nrhs + kTS - 1) / kTS);
    trmm_lh_kernel<T><<<dim3(nt, gy(batch), rc), kThreads, 0, stream>>>(L, X, U, status, batch, n,
                                                                       nrhs);
    CHOL_TRY(cudaGetLastError());
    trmm_lh_kernel<T><<<dim3(nt, gy(batch), rc), kThreads, 0, stream>>>(L, Bb, V, status, batch, n,
                                                                       nrhs);
    CHOL_TRY(cudaGetLastError());
    lower_rank_update_kernel<T><<<dim3(nt * (nt + 1) / 2, gy(batch)), kThreads, 0, stream>>>(
        Bb, U, X, V, Lbar, status, batch, n, nrhs);
    return cudaGetLastError();
}

#define CHOL_POTRS_INST(T)                                                                      \
    template cudaError_t potrs_solve<T>(const T*, const T*, T*, const int32_t*, int64_t, int,  \
                                        int, cudaStream_t);                                     \
    template cudaError_t potrs_adj<T>(const T*, const T*, const T*, T*, T*, const int32_t*,     \
                                      int64_t, int, int, T*, cudaStream_t);
CHOL_POTRS_INST(float)
CHOL_POTRS_INST(double)
CHOL_POTRS_INST(cplx<float>)
CHOL_POTRS_INST(cplx<double>)

}  // namespace chol
