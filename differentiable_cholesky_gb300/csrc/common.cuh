// Shared device helpers for the GB300 Cholesky kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "chol.h"

namespace chol {

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
__device__ __forceinline__ float sqrt_t(float x) { return __fsqrt_rn(x); }
__device__ __forceinline__ double sqrt_t(double x) { return __dsqrt_rn(x); }

// Read-only, streaming global load of a 16-byte vector (not kept in L1).
template <typename V>
__device__ __forceinline__ V ldg_stream(const V* p) {
    return __ldcs(p);
}

}  // namespace chol
