// Throughput probes: the measured FP64 / FP32 rates that the blocked path's
// roofline is reported against.  Two FP64 pipes exist on sm_103a: the FMA pipe
// (DFMA) and the double-precision tensor path of mma.sync (DMMA); tcgen05 has
// no f64 kind.  Each probe keeps one pipe busy with independent chains per
// thread; a data-dependent store keeps the work alive.

#include <cuda_runtime.h>

#include "chol_probe.h"
#include "kernels.h"

namespace {

constexpr int kChains = 8;
constexpr int kThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kThreads) fma_chain_kernel(int64_t iters, T* sink) {
    T x[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) x[c] = T(threadIdx.x + c) * T(1e-3);
    const T a = T(0.999999), b = T(1e-7);
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int c = 0; c < kChains; ++c) x[c] = fma(x[c], a, b);
    }
    T s = T(0);
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += x[c];
    if (s == T(-1.2345)) *sink = s;  // never true; the compiler cannot tell
}

// One warp-wide f64 MMA of each shape the PTX ISA lists for sm_90 and later:
// D = A B + C with A (M x K, row), B (K x N, col), per-thread fragment sizes
// A: M*K/32, B: K*N/32, C/D: M*N/32 doubles.
template <int SHAPE> struct Dmma;
template <> struct Dmma<0> {  // m8n8k4
    static constexpr int M = 8, N = 8, K = 4;
    __device__ __forceinline__ static void mma(double (&c)[2], const double (&a)[1],
                                               const double (&b)[1]) {
        asm volatile("mma.sync.aligned.m8n8k4.row.col.f64.f64.f64.f64 {%0,%1}, {%2}, {%3}, {%0,%1};"
                     : "+d"(c[0]), "+d"(c[1])
                     : "d"(a[0]), "d"(b[0]));
    }
};
template <> struct Dmma<1> {  // m16n8k4
    static constexpr int M = 16, N = 8, K = 4;
    __device__ __forceinline__ static void mma(double (&c)[4], const double (&a)[2],
                                               const double (&b)[1]) {
        asm volatile(
            "mma.sync.aligned.m16n8k4.row.col.f64.f64.f64.f64 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
            "{%0,%1,%2,%3};"
            : "+d"(c[0]), "+d"(c[1]), "+d"(c[2]), "+d"(c[3])
            : "d"(a[0]), "d"(a[1]), "d"(b[0]));
    }
};
template <> struct Dmma<2> {  // m16n8k8
    static constexpr int M = 16, N = 8, K = 8;
    __device__ __forceinline__ static void mma(double (&c)[4], const double (&a)[4],
                                               const double (&b)[2]) {
        asm volatile(
            "mma.sync.aligned.m16n8k8.row.col.f64.f64.f64.f64 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+d"(c[0]), "+d"(c[1]), "+d"(c[2]), "+d"(c[3])
            : "d"(a[0]), "d"(a[1]), "d"(a[2]), "d"(a[3]), "d"(b[0]), "d"(b[1]));
    }
};
template <> struct Dmma<3> {  // m16n8k16
    static constexpr int M = 16, N = 8, K = 16;
    __device__ __forceinline__ static void mma(double (&c)[4], const double (&a)[8],
                                               const double (&b)[4]) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f64.f64.f64.f64 {%0,%1,%2,%3}, "
            "{%4,%5,%6,%7,%8,%9,%10,%11}, {%12,%13,%14,%15}, {%0,%1,%2,%3};"
            : "+d"(c[0]), "+d"(c[1]), "+d"(c[2]), "+d"(c[3])
            : "d"(a[0]), "d"(a[1]), "d"(a[2]), "d"(a[3]), "d"(a[4]), "d"(a[5]), "d"(a[6]),
              "d"(a[7]), "d"(b[0]), "d"(b[1]), "d"(b[2]), "d"(b[3]));
    }
};

constexpr int kMmaChains = 4;

template <int SHAPE>
__global__ void __launch_bounds__(kThreads) dmma_chain_kernel(int64_t iters, double* sink) {
    using D = Dmma<SHAPE>;
    constexpr int NA = D::M * D::K / 32, NB = D::K * D::N / 32, NC = D::M * D::N / 32;
    double a[NA], b[NB], c[kMmaChains][NC];
#pragma unroll
    for (int i = 0; i < NA; ++i) a[i] = 1e-3 * (threadIdx.x + i);
#pragma unroll
    for (int i = 0; i < NB; ++i) b[i] = 1e-4 * (threadIdx.x + 3 * i);
#pragma unroll
    for (int k = 0; k < kMmaChains; ++k)
#pragma unroll
        for (int i = 0; i < NC; ++i) c[k][i] = 0.0;
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int k = 0; k < kMmaChains; ++k) D::mma(c[k], a, b);
    }
    double s = 0.0;
#pragma unroll
    for (int k = 0; k < kMmaChains; ++k)
#pragma unroll
        for (int i = 0; i < NC; ++i) s += c[k][i];
    if (s == -1.2345) *sink = s;  // never true; the compiler cannot tell
}

// Times `kern` (warm-up launch, then one timed launch on every SM at full
// occupancy) and returns the rate for `flops_per_thread_iter` flops per
// thread and iteration.
template <typename K, typename T>
int time_kernel(K kern, int64_t iters, T* sink, double flops_per_thread_iter, double* flops,
                cudaStream_t stream) {
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CHOL_ECUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return CHOL_ECUDA;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, 0) != cudaSuccess)
        return CHOL_ECUDA;
    const int blocks = sms * (per_sm > 0 ? per_sm : 1);
    cudaEvent_t e0, e1;
    if (cudaEventCreate(&e0) != cudaSuccess) return CHOL_ECUDA;
    if (cudaEventCreate(&e1) != cudaSuccess) {
        cudaEventDestroy(e0);
        return CHOL_ECUDA;
    }
    kern<<<blocks, kThreads, 0, stream>>>(iters / 16 + 1, sink);
    cudaEventRecord(e0, stream);
    kern<<<blocks, kThreads, 0, stream>>>(iters, sink);
    cudaEventRecord(e1, stream);
    cudaError_t err = cudaGetLastError();
    if (err == cudaSuccess) err = cudaEventSynchronize(e1);
    float ms = 0.f;
    if (err == cudaSuccess) err = cudaEventElapsedTime(&ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (err != cudaSuccess || ms <= 0.f) return CHOL_ECUDA;
    *flops = (double)blocks * kThreads * flops_per_thread_iter * (double)iters / (ms * 1e-3);
    return CHOL_OK;
}

template <int SHAPE>
int run_dmma(int64_t iters, void* sink, double* flops, cudaStream_t stream) {
    using D = Dmma<SHAPE>;
    // one warp-wide MMA is 2 M N K flops, i.e. 2 M N K / 32 per thread
    const double per_thread = kMmaChains * 2.0 * D::M * D::N * D::K / 32.0;
    return time_kernel(dmma_chain_kernel<SHAPE>, iters, static_cast<double*>(sink), per_thread,
                       flops, stream);
}

}  // namespace

extern "C" int chol_probe_fma_peak(int32_t dtype, int64_t iters, void* sink, double* flops,
                                   void* stream) {
    if (iters <= 0 || sink == nullptr || flops == nullptr) return CHOL_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == CHOL_F32)
        return time_kernel(fma_chain_kernel<float>, iters, static_cast<float*>(sink),
                           2.0 * kChains, flops, s);
    if (dtype == CHOL_F64)
        return time_kernel(fma_chain_kernel<double>, iters, static_cast<double*>(sink),
                           2.0 * kChains, flops, s);
    return CHOL_EDTYPE;
}

extern "C" int chol_probe_dmma_peak(int32_t shape, int64_t iters, void* sink, double* flops,
                                    void* stream) {
    if (iters <= 0 || sink == nullptr || flops == nullptr) return CHOL_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (shape) {
        case CHOL_DMMA_M8N8K4: return run_dmma<0>(iters, sink, flops, s);
        case CHOL_DMMA_M16N8K4: return run_dmma<1>(iters, sink, flops, s);
        case CHOL_DMMA_M16N8K8: return run_dmma<2>(iters, sink, flops, s);
        case CHOL_DMMA_M16N8K16: return run_dmma<3>(iters, sink, flops, s);
        default: return CHOL_EINVAL;
    }
}

// The dominant kernel of the float64 blocked path, timed alone: step k's
// trailing update on the tensor cores (all lower tiles I >= J > k), with the
// panel's rows sliced once before the timed launches.
extern "C" int chol_probe_tc_update(int32_t n, void* L, int32_t k, int32_t reps, double* ms,
                                    double* bf16_flops, double* fp64_equiv_flops, void* stream) {
    if (n <= 128 || L == nullptr || ms == nullptr || bf16_flops == nullptr ||
        fp64_equiv_flops == nullptr || reps <= 0)
        return CHOL_EINVAL;
    const int nt = (n + 127) / 128;
    if (k < 0 || k >= nt - 1) return CHOL_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    double* Ld = static_cast<double*>(L);
    void* work = nullptr;
    if (cudaMallocAsync(&work, chol::ozaki_workspace_bytes(1, n), s) != cudaSuccess) {
        cudaGetLastError();
        return CHOL_ENOMEM;
    }
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    cudaError_t e = cudaEventCreate(&e0);
    if (e == cudaSuccess) e = cudaEventCreate(&e1);
    if (e == cudaSuccess) e = chol::ozaki_trailing_slice(Ld, work, nullptr, 1, n, k, s);
    if (e == cudaSuccess) e = cudaEventRecord(e0, s);
    for (int r = 0; r < reps && e == cudaSuccess; ++r)
        e = chol::ozaki_trailing_gemm(Ld, work, nullptr, 1, n, k, 0, s);
    if (e == cudaSuccess) e = cudaEventRecord(e1, s);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    float t = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, e0, e1);
    if (e0 != nullptr) cudaEventDestroy(e0);
    if (e1 != nullptr) cudaEventDestroy(e1);
    const cudaError_t ef = cudaFreeAsync(work, s);
    if (e != cudaSuccess || ef != cudaSuccess) return CHOL_ECUDA;
    const double m = nt - k - 1;
    const double tiles = m * (m + 1) / 2;
    const double per_tile = 2.0 * 128.0 * 128.0 * 128.0;
    *ms = (double)t / reps;
    *fp64_equiv_flops = tiles * per_tile / (*ms * 1e-3);
    *bf16_flops = 28.0 * *fp64_equiv_flops;  // 28 digit products per element product
    return CHOL_OK;
}
