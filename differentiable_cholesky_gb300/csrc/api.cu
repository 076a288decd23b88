// C ABI of the library (declared in include/chol.h): argument checks, the
// small/blocked dispatch and workspace handling.  No kernel code lives here.

#include <cuda_runtime.h>
#include <stdint.h>

#include <initializer_list>

#include "chol.h"
#include "chol_selftest.h"
#include "kernels.h"

namespace {

constexpr int kSmallMax = 64;

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

bool overlaps(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

Range range_of(const void* p, size_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + bytes};
}

int elem_size(int32_t dtype) { return dtype == CHOL_F32 ? 4 : dtype == CHOL_F64 ? 8 : 0; }

// Device (or managed) memory only: a host pointer handed to a kernel would
// fault or, where the GPU can reach host memory, silently run over the link.
bool is_device_pointer(const void* p) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();  // clear the non-sticky error
        return false;
    }
    return attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Common shape / pointer checks.  On success *bytes is the size of one
// [batch][n][n] array.
int check_shape(int64_t batch, int32_t n, int32_t dtype, size_t* bytes) {
    if (elem_size(dtype) == 0) return CHOL_EDTYPE;
    if (batch < 0 || n <= 0) return CHOL_EINVAL;
    const unsigned __int128 total =
        (unsigned __int128)batch * (unsigned __int128)n * (unsigned __int128)n * elem_size(dtype);
    if (total > ((unsigned __int128)1 << 62)) return CHOL_EINVAL;
    *bytes = (size_t)total;
    return CHOL_OK;
}

int check_tile(int32_t tile) {
    return (tile == 0 || tile == 32 || tile == 64 || tile == 128) ? CHOL_OK : CHOL_EINVAL;
}

int to_code(cudaError_t e) { return e == cudaSuccess ? CHOL_OK : CHOL_ECUDA; }

bool vec_ok(int n, int esize, std::initializer_list<const void*> ptrs) {
    if ((n * esize) % 16 != 0) return false;
    for (const void* p : ptrs)
        if (p != nullptr && !aligned(p, 16)) return false;
    return true;
}

template <typename T>
int fwd_impl(int64_t batch, int32_t n, const void* A, void* L, int32_t* status, int32_t tile,
             cudaStream_t stream) {
    const T* a = static_cast<const T*>(A);
    T* l = static_cast<T*>(L);
    if (n <= kSmallMax) {
        const bool vec = vec_ok(n, sizeof(T), {A, L});
        if constexpr (sizeof(T) == 4) {
            if (vec && chol::tpm_supported(n))
                return to_code(chol::tpm_fwd(a, l, status, batch, n, stream));
        }
        return to_code(chol::small_fwd<T>(a, l, status, batch, n, vec, stream));
    }
    if (tile == 0) tile = chol::blocked_default_tile(n, batch);
    return to_code(chol::blocked_fwd<T>(a, l, status, batch, n, tile, stream));
}

template <typename T>
int adj_impl(int64_t batch, int32_t n, const void* L, const void* Lbar, void* Abar,
             const int32_t* status, int32_t tile, size_t bytes, bool accumulate,
             cudaStream_t stream) {
    const T* l = static_cast<const T*>(L);
    const T* lb = static_cast<const T*>(Lbar);
    T* ab = static_cast<T*>(Abar);
    if (n <= kSmallMax) {
        const bool vec = vec_ok(n, sizeof(T), {L, Lbar, Abar});
        return to_code(chol::small_adj<T>(l, lb, ab, status, batch, n, vec, accumulate, stream));
    }
    if (tile == 0) tile = chol::blocked_default_tile(n, batch);
    if (!accumulate && Lbar == Abar)  // in place: the sweep needs no workspace
        return to_code(chol::blocked_adj<T>(l, lb, ab, status, batch, n, tile, nullptr, false,
                                            stream));
    void* work = nullptr;
    if (cudaMallocAsync(&work, bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return CHOL_ENOMEM;
    }
    const int rc = to_code(chol::blocked_adj<T>(l, lb, ab, status, batch, n, tile,
                                                static_cast<T*>(work), accumulate, stream));
    if (cudaFreeAsync(work, stream) != cudaSuccess) return CHOL_ECUDA;
    return rc;
}

}  // namespace

extern "C" {

int chol_fwd_ex(int64_t batch, int32_t n, int32_t dtype, const void* A, void* L,
                int32_t* status, int32_t tile, void* stream) {
    size_t bytes = 0;
    int rc = check_shape(batch, n, dtype, &bytes);
    if (rc != CHOL_OK) return rc;
    if ((rc = check_tile(tile)) != CHOL_OK) return rc;
    if (batch == 0) return CHOL_OK;
    if (A == nullptr || L == nullptr || status == nullptr) return CHOL_EINVAL;
    const size_t es = (size_t)elem_size(dtype);
    if (!aligned(A, es) || !aligned(L, es) || !aligned(status, 4)) return CHOL_EINVAL;
    if (!is_device_pointer(A) || !is_device_pointer(L) || !is_device_pointer(status))
        return CHOL_EINVAL;
    const Range rA = range_of(A, bytes), rL = range_of(L, bytes),
                rS = range_of(status, (size_t)batch * 4);
    if (overlaps(rA, rL) || overlaps(rL, rS) || overlaps(rA, rS)) return CHOL_EALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dtype == CHOL_F32 ? fwd_impl<float>(batch, n, A, L, status, tile, s)
                             : fwd_impl<double>(batch, n, A, L, status, tile, s);
}

int chol_fwd(int64_t batch, int32_t n, int32_t dtype, const void* A, void* L, int32_t* status,
             void* stream) {
    return chol_fwd_ex(batch, n, dtype, A, L, status, 0, stream);
}

}  // extern "C"

namespace chol {

int check_adj_args(int64_t batch, int32_t n, int32_t dtype, const void* L, const void* adj_L,
                   const void* adj_A, const int32_t* status, int32_t tile, size_t* bytes) {
    int rc = check_shape(batch, n, dtype, bytes);
    if (rc != CHOL_OK) return rc;
    if ((rc = check_tile(tile)) != CHOL_OK) return rc;
    if (batch == 0) return CHOL_OK;
    if (L == nullptr || adj_L == nullptr || adj_A == nullptr) return CHOL_EINVAL;
    const size_t es = (size_t)elem_size(dtype);
    if (!aligned(L, es) || !aligned(adj_L, es) || !aligned(adj_A, es)) return CHOL_EINVAL;
    if (status != nullptr && !aligned(status, 4)) return CHOL_EINVAL;
    if (!is_device_pointer(L) || !is_device_pointer(adj_L) || !is_device_pointer(adj_A) ||
        (status != nullptr && !is_device_pointer(status)))
        return CHOL_EINVAL;
    const Range rL = range_of(L, *bytes), rLb = range_of(adj_L, *bytes),
                rAb = range_of(adj_A, *bytes);
    if (overlaps(rAb, rL) || overlaps(rAb, rLb)) return CHOL_EALIAS;
    if (status != nullptr && overlaps(rAb, range_of(status, (size_t)batch * 4)))
        return CHOL_EALIAS;
    return CHOL_OK;
}

}  // namespace chol

extern "C" {

int chol_adj_ex(int64_t batch, int32_t n, int32_t dtype, const void* L, const void* adj_L,
                void* adj_A, const int32_t* status, int32_t tile, void* stream) {
    size_t bytes = 0;
    const int rc = chol::check_adj_args(batch, n, dtype, L, adj_L, adj_A, status, tile, &bytes);
    if (rc != CHOL_OK || batch == 0) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dtype == CHOL_F32
               ? adj_impl<float>(batch, n, L, adj_L, adj_A, status, tile, bytes, true, s)
               : adj_impl<double>(batch, n, L, adj_L, adj_A, status, tile, bytes, true, s);
}

int chol_adj(int64_t batch, int32_t n, int32_t dtype, const void* L, const void* adj_L,
             void* adj_A, const int32_t* status, void* stream) {
    return chol_adj_ex(batch, n, dtype, L, adj_L, adj_A, status, 0, stream);
}

// In place: the kernels read every matrix (or, on the blocked path, a stage
// copies it) in full before anything of it is written, so the output may be
// the input buffer itself.
int chol_fwd_inplace(int64_t batch, int32_t n, int32_t dtype, void* A, int32_t* status,
                     int32_t tile, void* stream) {
    size_t bytes = 0;
    int rc = check_shape(batch, n, dtype, &bytes);
    if (rc != CHOL_OK) return rc;
    if ((rc = check_tile(tile)) != CHOL_OK) return rc;
    if (batch == 0) return CHOL_OK;
    if (A == nullptr || status == nullptr) return CHOL_EINVAL;
    if (!aligned(A, (size_t)elem_size(dtype)) || !aligned(status, 4)) return CHOL_EINVAL;
    if (!is_device_pointer(A) || !is_device_pointer(status)) return CHOL_EINVAL;
    if (overlaps(range_of(A, bytes), range_of(status, (size_t)batch * 4))) return CHOL_EALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dtype == CHOL_F32 ? fwd_impl<float>(batch, n, A, A, status, tile, s)
                             : fwd_impl<double>(batch, n, A, A, status, tile, s);
}

int chol_adj_inplace(int64_t batch, int32_t n, int32_t dtype, const void* L, void* adj,
                     const int32_t* status, int32_t tile, void* stream) {
    size_t bytes = 0;
    int rc = check_shape(batch, n, dtype, &bytes);
    if (rc != CHOL_OK) return rc;
    if ((rc = check_tile(tile)) != CHOL_OK) return rc;
    if (batch == 0) return CHOL_OK;
    if (L == nullptr || adj == nullptr) return CHOL_EINVAL;
    const size_t es = (size_t)elem_size(dtype);
    if (!aligned(L, es) || !aligned(adj, es)) return CHOL_EINVAL;
    if (status != nullptr && !aligned(status, 4)) return CHOL_EINVAL;
    if (!is_device_pointer(L) || !is_device_pointer(adj) ||
        (status != nullptr && !is_device_pointer(status)))
        return CHOL_EINVAL;
    const Range rL = range_of(L, bytes), rX = range_of(adj, bytes);
    if (overlaps(rX, rL)) return CHOL_EALIAS;
    if (status != nullptr && overlaps(rX, range_of(status, (size_t)batch * 4)))
        return CHOL_EALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dtype == CHOL_F32 ? adj_impl<float>(batch, n, L, adj, adj, status, tile, bytes, false, s)
                             : adj_impl<double>(batch, n, L, adj, adj, status, tile, bytes, false, s);
}

int chol_selftest_wait_timeout(int64_t batch, const void* A, void* L, int32_t* status,
                               uint32_t max_polls, void* stream) {
    size_t bytes = 0;
    int rc = check_shape(batch, 16, CHOL_F32, &bytes);
    if (rc != CHOL_OK) return rc;
    if (batch == 0) return CHOL_OK;
    if (max_polls < 1 || max_polls > (1u << 22)) return CHOL_EINVAL;
    if (A == nullptr || L == nullptr || status == nullptr) return CHOL_EINVAL;
    if (!aligned(A, 16) || !aligned(L, 16) || !aligned(status, 4)) return CHOL_EINVAL;
    if (!is_device_pointer(A) || !is_device_pointer(L) || !is_device_pointer(status))
        return CHOL_EINVAL;
    const Range rA = range_of(A, bytes), rL = range_of(L, bytes),
                rS = range_of(status, (size_t)batch * 4);
    if (overlaps(rA, rL) || overlaps(rL, rS) || overlaps(rA, rS)) return CHOL_EALIAS;
    return to_code(chol::tpm_fwd_wait_selftest(static_cast<const float*>(A), static_cast<float*>(L),
                                               status, batch, max_polls,
                                               static_cast<cudaStream_t>(stream)));
}

const char* chol_strerror(int code) {
    switch (code) {
        case CHOL_OK: return "success";
        case CHOL_EINVAL: return "invalid argument (shape, tile, null, misaligned or non-device pointer)";
        case CHOL_EDTYPE: return "unsupported dtype (expected CHOL_F32 or CHOL_F64)";
        case CHOL_EALIAS: return "an output buffer overlaps an input buffer";
        case CHOL_ENOMEM: return "device workspace allocation failed";
        case CHOL_ECUDA: return "CUDA launch or runtime error";
        default: return "unknown error code";
    }
}

int32_t chol_abi_version(void) { return CHOL_ABI_VERSION; }

}  // extern "C"
