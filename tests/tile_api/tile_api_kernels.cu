// Test kernels for the device-side tile API (include/chol_tile.cuh): one
// block per matrix stages its tile in shared memory and calls
// chol_tile::potrf / chol_tile::potrf_adj, as a caller's own kernel would.
// Built by the test that uses it; not part of the library.
#include <cuda_runtime.h>
#include <stdint.h>

#include "chol_tile.cuh"

namespace {

template <typename T, int THREADS>
__global__ void __launch_bounds__(THREADS)
tile_fwd_kernel(const T* A, T* L, int32_t* status, int n) {
    extern __shared__ __align__(16) unsigned char raw[];
    T* S = reinterpret_cast<T*>(raw);
    const int P = n + 1;
    const int64_t b = blockIdx.x;
    const T* Ab = A + b * (int64_t)n * n;
    for (int e = threadIdx.x; e < n * n; e += THREADS) {
        const int r = e / n, c = e % n;
        if (c <= r) S[r * P + c] = Ab[e];
    }
    __syncthreads();
    const int st = chol_tile::potrf<THREADS>(S, n, chol_tile::RowMajor{P});
    if (threadIdx.x == 0) status[b] = st;
    T* Lb = L + b * (int64_t)n * n;
    for (int e = threadIdx.x; e < n * n; e += THREADS) {
        const int r = e / n, c = e % n;
        Lb[e] = (c <= r) ? S[r * P + c] : T(0);
    }
}

template <typename T, int THREADS, bool PACKED>
__global__ void __launch_bounds__(THREADS)
tile_adj_kernel(const T* L, const T* Lbar, T* Abar, const int32_t* status, int n) {
    extern __shared__ __align__(16) unsigned char raw[];
    const int64_t b = blockIdx.x;
    if (status[b] != 0) return;
    const int tri = n * (n + 1) / 2, P = n + 1;
    T* Ls = reinterpret_cast<T*>(raw);
    T* Ws = Ls + (PACKED ? tri : n * P);
    auto at = [&](int i, int j) { return PACKED ? i * (i + 1) / 2 + j : i * P + j; };
    const T* Lb = L + b * (int64_t)n * n;
    const T* Bb = Lbar + b * (int64_t)n * n;
    for (int e = threadIdx.x; e < n * n; e += THREADS) {
        const int r = e / n, c = e % n;
        if (c <= r) {
            Ls[at(r, c)] = Lb[e];
            Ws[at(r, c)] = Bb[e];
        }
    }
    __syncthreads();
    if constexpr (PACKED)
        chol_tile::potrf_adj<THREADS>(Ls, Ws, n, chol_tile::PackedLower{});
    else
        chol_tile::potrf_adj<THREADS>(Ls, Ws, n, chol_tile::RowMajor{P});
    T* Gb = Abar + b * (int64_t)n * n;
    for (int e = threadIdx.x; e < n * n; e += THREADS) {
        const int r = e / n, c = e % n;
        if (c <= r) Gb[e] = Ws[at(r, c)];
    }
}

template <typename T, int THREADS>
int fwd(int64_t batch, int n, const void* A, void* L, int32_t* status, cudaStream_t s) {
    const size_t smem = (size_t)n * (n + 1) * sizeof(T);
    auto k = tile_fwd_kernel<T, THREADS>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return -1;
    k<<<(unsigned)batch, THREADS, smem, s>>>(static_cast<const T*>(A), static_cast<T*>(L), status, n);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

template <typename T, int THREADS, bool PACKED>
int adj(int64_t batch, int n, const void* L, const void* Lbar, void* Abar, const int32_t* status,
        cudaStream_t s) {
    const size_t smem = (PACKED ? (size_t)n * (n + 1) : 2 * (size_t)n * (n + 1)) * sizeof(T);
    auto k = tile_adj_kernel<T, THREADS, PACKED>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return -1;
    k<<<(unsigned)batch, THREADS, smem, s>>>(static_cast<const T*>(L), static_cast<const T*>(Lbar),
                                             static_cast<T*>(Abar), status, n);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

extern "C" {

// dtype 0 = float, 1 = double; threads 64 or 256.
int tile_demo_fwd(int64_t batch, int n, int dtype, int threads, const void* A, void* L,
                  int32_t* status, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == 0) return threads == 64 ? fwd<float, 64>(batch, n, A, L, status, s)
                                         : fwd<float, 256>(batch, n, A, L, status, s);
    return threads == 64 ? fwd<double, 64>(batch, n, A, L, status, s)
                         : fwd<double, 256>(batch, n, A, L, status, s);
}

int tile_demo_adj(int64_t batch, int n, int dtype, int threads, int packed, const void* L,
                  const void* Lbar, void* Abar, const int32_t* status, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
#define TILE_ADJ(T, TH)                                                                   \
    return packed ? adj<T, TH, true>(batch, n, L, Lbar, Abar, status, s)                  \
                  : adj<T, TH, false>(batch, n, L, Lbar, Abar, status, s);
    if (dtype == 0) {
        if (threads == 64) { TILE_ADJ(float, 64) }
        TILE_ADJ(float, 256)
    }
    if (threads == 64) { TILE_ADJ(double, 64) }
    TILE_ADJ(double, 256)
#undef TILE_ADJ
}

}  // extern "C"
