// Throughput probes: the measured FP64 / FP32 rates that the blocked path's
// roofline is reported against.  Two FP64 pipes exist on sm_103a: the FMA pipe
// (DFMA) and the double-precision tensor path of mma.sync (DMMA); tcgen05 has
// no f64 kind.  Each probe keeps one pipe busy with independent chains per
// thread; a data-dependent store keeps the work alive.

#include <cuda_runtime.h>

#include "chol_probe.h"

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
