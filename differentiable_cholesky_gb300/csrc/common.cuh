// Shared device helpers for the GB300 Cholesky kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <utility>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <type_traits>

#include "chol.h"

namespace chol {

// ---------------------------------------------------------------------------
// Per-device host-side caches.  Kernel attributes (the raised dynamic
// shared-memory limit) and occupancy figures belong to one device; a process
// that drives several GPUs, from one thread or many, must set and look them
// up per device.  Device ordinals >= kMaxDevices are served uncached.
// ---------------------------------------------------------------------------
constexpr int kMaxDevices = 64;

inline std::mutex& device_cache_mutex() {
    static std::mutex m;
    return m;
}

// Runs `f` (returning cudaError_t) once per device for the current device;
// success is remembered in bit `dev` of `done`, a failure is returned and
// retried on the next call.
template <typename F>
cudaError_t once_per_device(std::atomic<uint64_t>& done, F&& f) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return f();
    const uint64_t bit = 1ull << dev;
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    std::lock_guard<std::mutex> lock(device_cache_mutex());
    if (done.load(std::memory_order_relaxed) & bit) return cudaSuccess;
    e = f();
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// An int computed once per device by `f` (returning a value > 0, or <= 0 on
// failure, which is not cached).
struct PerDeviceInt {
    std::atomic<int> v[kMaxDevices];
    PerDeviceInt() {
        for (auto& x : v) x.store(0, std::memory_order_relaxed);
    }
    template <typename F>
    int get(F&& f) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) {
            cudaGetLastError();
            return f();
        }
        if (dev < 0 || dev >= kMaxDevices) return f();
        int x = v[dev].load(std::memory_order_acquire);
        if (x > 0) return x;
        x = f();
        if (x > 0) v[dev].store(x, std::memory_order_release);
        return x;
    }
};

// Streaming multiprocessors of the current device (152 on a GB300; queried,
// never assumed).
inline int device_sm_count() {
    static PerDeviceInt cache;
    const int n = cache.get([] {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        return sms;
    });
    return n > 0 ? n : 1;
}

// Raise a kernel's dynamic shared-memory limit to `bytes`, once per device
// (the attribute call is host-synchronous, so not once per launch).
template <typename K>
cudaError_t allow_smem_once(K kern, size_t bytes, std::atomic<uint64_t>& done) {
    return once_per_device(done, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    });
}

// Compile-time loop: f(std::integral_constant<int, I>) for I in [B, E).  Used
// where every index must be a constant so that arrays stay in registers,
// whatever the unroller decides about large loop nests.
template <int B, int E, typename F>
__device__ __forceinline__ void static_for(F&& f) {
    if constexpr (B < E) {
        f(std::integral_constant<int, B>{});
        static_for<B + 1, E>(f);
    }
}

// 16-byte vector of the element type: the unit of every vectorised global or
// shared-memory access in these kernels.
template <typename T> struct Vec16;
template <> struct Vec16<float> {
    using type = float4;
    static constexpr int N = 4;
};
template <> struct Vec16<double> {
    using type = double2;
    static constexpr int N = 2;
};

template <typename T>
__device__ __forceinline__ T vget(const typename Vec16<T>::type& v, int e);
template <>
__device__ __forceinline__ float vget<float>(const float4& v, int e) {
    return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}
template <>
__device__ __forceinline__ double vget<double>(const double2& v, int e) {
    return e == 0 ? v.x : v.y;
}

template <typename T>
__device__ __forceinline__ void vset(typename Vec16<T>::type& v, int e, T x);
template <>
__device__ __forceinline__ void vset<float>(float4& v, int e, float x) {
    if (e == 0) v.x = x; else if (e == 1) v.y = x; else if (e == 2) v.z = x; else v.w = x;
}
template <>
__device__ __forceinline__ void vset<double>(double2& v, int e, double x) {
    if (e == 0) v.x = x; else v.y = x;
}

// Reciprocal square root and correctly rounded reciprocal, by element type.
// These call CUDA's own math functions; nothing of their internals is restated.
__device__ __forceinline__ float rsqrt_t(float x) { return rsqrtf(x); }
__device__ __forceinline__ double rsqrt_t(double x) { return rsqrt(x); }
__device__ __forceinline__ float rcp_t(float x) { return __frcp_rn(x); }
__device__ __forceinline__ double rcp_t(double x) { return __drcp_rn(x); }

}  // namespace chol

// ---------------------------------------------------------------------------
// Bulk asynchronous copies (TMA, non-tensor form) and mbarriers, sm_90+ PTX.
// ---------------------------------------------------------------------------
namespace chol {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Programmatic dependent launch: a kernel launched with launch_pdl may be
// scheduled before the previous kernel in its stream has finished; it calls
// pdl_wait() before its first global memory access, which returns once that
// kernel has completed and its writes are visible (at once for a kernel
// launched without the attribute).  Only the launch and scheduling of the
// CTAs overlap the previous kernel's tail.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make an initialised mbarrier visible to the async proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, giving up after
// `max_iter` polls (each poll may itself suspend briefly).  Returns false on
// timeout: callers report it and stop instead of waiting forever.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t max_iter) {
    for (uint32_t it = 0; it < max_iter; ++it)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

constexpr uint32_t kMbarPolls = 1u << 22;

// global -> shared bulk copy; completion counted in bytes on `bar`.
// Addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// shared -> global bulk copy in the calling thread's bulk async-group.
__device__ __forceinline__ void bulk_store(void* gmem_dst, const void* smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
                 "r"(smem_u32(smem_src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// The calling thread's committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// The calling thread's committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// 16-byte global -> shared copy that bypasses L1; the first `src_bytes`
// (0..16) come from `gmem`, the rest of the 16 are zero-filled.  Both
// addresses 16-byte aligned.  Completion: cp_async_wait_all.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem)),
                 "l"(gmem), "r"(src_bytes)
                 : "memory");
}

// The calling thread's cp.async copies have landed in shared memory.
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Bring `bytes` of global memory into L2 without waiting for them (a hint:
// nothing is written and no completion is tracked).  Address 16-byte aligned,
// bytes a multiple of 16.
__device__ __forceinline__ void l2_prefetch(const void* gmem, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gmem), "r"(bytes) : "memory");
}

// Order generic-proxy shared-memory accesses before later async-proxy ones.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace chol
