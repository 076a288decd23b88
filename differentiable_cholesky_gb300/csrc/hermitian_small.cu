// Batched Hermitian Cholesky forward and adjoint for small complex matrices
// (n <= 64): A = L L^H and its reverse mode (jaxmg docs "Cholesky
// factorization", intro: the factorisation of "a symmetric or Hermitian
// positive-definite matrix"; NVIDIA/warp issue #1316: one tile per block,
// the adjoint accumulated into the lower triangle of A's gradient).
//
// One block of 64 threads per matrix, the matrix packed as a lower triangle
// in shared memory, factored and differentiated by the device tile API
// (chol_tile::potrf / potrf_adj on cplx elements: the right-looking column
// recurrence with conjugates, and Murray's reverse sweep).  Global memory is
// read and written row by row, coalesced within a row.

#include <cuda_runtime.h>

#include <algorithm>

#include "chol_tile.cuh"
#include "common.cuh"
#include "kernels.h"

namespace chol {
namespace {

using chol_tile::cplx;
constexpr int kHThreads = 64;

__device__ __forceinline__ int packed(int i, int j) { return i * (i + 1) / 2 + j; }

// A and L may be the same buffer (the in-place forward): the block reads its
// matrix in full before it writes any of it.
template <typename T>
__global__ void __launch_bounds__(kHThreads)
hsmall_potrf_kernel(const T* A, T* L, int32_t* __restrict__ status, int64_t batch, int n) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* S = reinterpret_cast<T*>(smem_raw);
    const int nn = n * n;
    for (int64_t b = blockIdx.x; b < batch; b += gridDim.x) {
        const T* Ab = A + b * nn;
        T* Lb = L + b * nn;
        __syncthreads();
        for (int e = threadIdx.x; e < nn; e += kHThreads) {
            const int i = e / n, j = e % n;
            if (j <= i) S[packed(i, j)] = Ab[e];
        }
        __syncthreads();
        const int st = chol_tile::potrf<kHThreads>(S, n, chol_tile::PackedLower{});
        for (int e = threadIdx.x; e < nn; e += kHThreads) {
            const int i = e / n, j = e % n;
            Lb[e] = j <= i ? S[packed(i, j)] : T{};
        }
        if (threadIdx.x == 0) status[b] = st;
    }
}

// Lbar and Abar may be the same buffer (the in-place adjoint, not
// accumulating): the block reads its matrix in full before it writes.
template <typename T>
__global__ void __launch_bounds__(kHThreads)
hsmall_potrf_adj_kernel(const T* __restrict__ L, const T* Lbar, T* Abar,
                        const int32_t* __restrict__ status, int64_t batch, int n,
                        bool accumulate) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int np = n * (n + 1) / 2;
    T* Ls = reinterpret_cast<T*>(smem_raw);
    T* Ws = Ls + np;
    const int nn = n * n;
    for (int64_t b = blockIdx.x; b < batch; b += gridDim.x) {
        T* Ab = Abar + b * nn;
        if (status != nullptr && status[b] != 0) {
            // skipped: untouched when accumulating, zeros in place
            if (!accumulate)
                for (int e = threadIdx.x; e < nn; e += kHThreads)
                    if (e % n <= e / n) Ab[e] = T{};
            continue;
        }
        const T* Lb = L + b * nn;
        const T* Gb = Lbar + b * nn;
        __syncthreads();
        for (int e = threadIdx.x; e < nn; e += kHThreads) {
            const int i = e / n, j = e % n;
            if (j <= i) {
                Ls[packed(i, j)] = Lb[e];
                Ws[packed(i, j)] = Gb[e];
            }
        }
        __syncthreads();
        chol_tile::potrf_adj<kHThreads>(Ls, Ws, n, chol_tile::PackedLower{});
        for (int e = threadIdx.x; e < nn; e += kHThreads) {
            const int i = e / n, j = e % n;
            if (j > i) continue;
            const T w = Ws[packed(i, j)];
            Ab[e] = accumulate ? chol_tile::detail::add(Ab[e], w) : w;
        }
    }
}

inline unsigned hgrid(int64_t batch) {
    return (unsigned)std::max<int64_t>(
        1, std::min<int64_t>(batch, (int64_t)device_sm_count() * 64));
}

}  // namespace

template <typename T>
cudaError_t hsmall_fwd(const T* A, T* L, int32_t* status, int64_t batch, int n,
                       cudaStream_t stream) {
    const size_t smem = (size_t)n * (n + 1) / 2 * sizeof(T);
    static std::atomic<uint64_t> smem_set{0};
    cudaError_t e = allow_smem_once(hsmall_potrf_kernel<T>, (size_t)64 * 65 / 2 * sizeof(T),
                                    smem_set);
    if (e != cudaSuccess) return e;
    hsmall_potrf_kernel<T><<<hgrid(batch), kHThreads, smem, stream>>>(A, L, status, batch, n);
    return cudaGetLastError();
}

template <typename T>
cudaError_t hsmall_adj(const T* L, const T* Lbar, T* Abar, const int32_t* status, int64_t batch,
                       int n, bool accumulate, cudaStream_t stream) {
    const size_t smem = (size_t)n * (n + 1) * sizeof(T);
    static std::atomic<uint64_t> smem_set{0};
    cudaError_t e =
        allow_smem_once(hsmall_potrf_adj_kernel<T>, (size_t)64 * 65 * sizeof(T), smem_set);
    if (e != cudaSuccess) return e;
    hsmall_potrf_adj_kernel<T><<<hgrid(batch), kHThreads, smem, stream>>>(L, Lbar, Abar, status,
                                                                         batch, n, accumulate);
    return cudaGetLastError();
}

template cudaError_t hsmall_fwd<cplx<float>>(const cplx<float>*, cplx<float>*, int32_t*, int64_t,
                                             int, cudaStream_t);
template cudaError_t hsmall_fwd<cplx<double>>(const cplx<double>*, cplx<double>*, int32_t*,
                                              int64_t, int, cudaStream_t);
template cudaError_t hsmall_adj<cplx<float>>(const cplx<float>*, const cplx<float>*, cplx<float>*,
                                             const int32_t*, int64_t, int, bool, cudaStream_t);
template cudaError_t hsmall_adj<cplx<double>>(const cplx<double>*, const cplx<double>*,
                                              cplx<double>*, const int32_t*, int64_t, int, bool,
                                              cudaStream_t);

}  // namespace chol
