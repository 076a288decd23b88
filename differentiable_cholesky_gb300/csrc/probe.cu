// FMA-throughput probe: the measured FP64 / FP32 peak that the blocked path's
// roofline is reported against.  Independent chains per thread keep every
// FMA pipe busy; a data-dependent store keeps the work alive.

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

template <typename T>
int run(int64_t iters, void* sink, double* flops, cudaStream_t stream) {
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CHOL_ECUDA;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fma_chain_kernel<T>, kThreads, 0) !=
        cudaSuccess)
        return CHOL_ECUDA;
    const int blocks = sms * (per_sm > 0 ? per_sm : 1);
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    fma_chain_kernel<T><<<blocks, kThreads, 0, stream>>>(iters / 16 + 1, static_cast<T*>(sink));
    cudaEventRecord(e0, stream);
    fma_chain_kernel<T><<<blocks, kThreads, 0, stream>>>(iters, static_cast<T*>(sink));
    cudaEventRecord(e1, stream);
    cudaError_t err = cudaEventSynchronize(e1);
    float ms = 0.f;
    if (err == cudaSuccess) err = cudaEventElapsedTime(&ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (err != cudaSuccess || ms <= 0.f) return CHOL_ECUDA;
    const double fmas = (double)blocks * kThreads * kChains * (double)iters;
    *flops = 2.0 * fmas / (ms * 1e-3);
    return CHOL_OK;
}

}  // namespace

extern "C" int chol_probe_fma_peak(int32_t dtype, int64_t iters, void* sink, double* flops,
                                   void* stream) {
    if (iters <= 0 || sink == nullptr || flops == nullptr) return CHOL_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == CHOL_F32) return run<float>(iters, sink, flops, s);
    if (dtype == CHOL_F64) return run<double>(iters, sink, flops, s);
    return CHOL_EDTYPE;
}
