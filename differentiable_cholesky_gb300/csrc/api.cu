// C ABI of the library (declared in include/chol.h): argument checks, the
// small/blocked dispatch and workspace handling.  No kernel code lives here.

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <initializer_list>
#include <type_traits>

#include "chol.h"
#include "chol_tile.cuh"
#include "chol_selftest.h"
#include "common.cuh"
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

int elem_size(int32_t dtype) {
    switch (dtype) {
        case CHOL_F32: return 4;
        case CHOL_F64: return 8;
        case CHOL_C64: return 8;
        case CHOL_C128: return 16;
        default: return 0;
    }
}

using chol_tile::cplx;

template <typename T> struct is_cplx : std::false_type {};
template <typename R> struct is_cplx<cplx<R>> : std::true_type {};
template <typename T> constexpr bool is_complex() { return is_cplx<T>::value; }

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

int check_tile(int32_t tile, int32_t dtype) {
    if (!(tile == 0 || tile == 32 || tile == 64 || tile == 128)) return CHOL_EINVAL;
    if (tile > chol::blocked_max_tile(elem_size(dtype))) return CHOL_EINVAL;
    return CHOL_OK;
}

// The default tile for a shape, capped by what the element type allows.
// The blocked tile when the caller leaves it to the library (tile == 0).
// tensor_ok: a float64 call that may take workspace, so 128-wide tiles run
// the tensor-core products, the cluster diagonal factor and the literal
// diagonal-tile adjoint; for a few such matrices that beats every FMA-pipe
// tiling (one 512 x 512 matrix, forward + adjoint: 1.65 ms at 128, 3.99 ms at
// 32, 5.54 ms at 64).
int pick_tile(int32_t tile, int n, int64_t batch, int esize, bool tensor_ok) {
    if (tile != 0) return tile;
    if (tensor_ok && n > 128 && batch * 8 <= chol::device_sm_count()) return 128;
    return std::min(chol::blocked_default_tile(n, batch), chol::blocked_max_tile(esize));
}

int to_code(cudaError_t e) { return e == cudaSuccess ? CHOL_OK : CHOL_ECUDA; }

// f(T{}) for the element type of a (checked) dtype.
template <typename F>
int dispatch(int32_t dtype, F&& f) {
    switch (dtype) {
        case CHOL_F32: return f(float{});
        case CHOL_F64: return f(double{});
        case CHOL_C64: return f(cplx<float>{});
        case CHOL_C128: return f(cplx<double>{});
        default: return CHOL_EDTYPE;
    }
}

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
        if constexpr (is_complex<T>()) {
            return to_code(chol::hsmall_fwd<T>(a, l, status, batch, n, stream));
        } else {
            const bool vec = vec_ok(n, sizeof(T), {A, L});
            if constexpr (sizeof(T) == 4) {
                if (vec && chol::tpm_supported(n))
                    return to_code(chol::tpm_fwd(a, l, status, batch, n, stream));
            }
            return to_code(chol::small_fwd<T>(a, l, status, batch, n, vec, stream));
        }
    }
    tile = pick_tile(tile, n, batch, sizeof(T), std::is_same<T, double>::value);
    const size_t wbytes =
        chol::blocked_fwd_workspace_bytes(std::is_same<T, double>::value, batch, n, tile);
    void* work = nullptr;
    if (wbytes > 0 && cudaMallocAsync(&work, wbytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return CHOL_ENOMEM;
    }
    const int rc = to_code(chol::blocked_fwd<T>(a, l, status, batch, n, tile, work, stream));
    if (work != nullptr && cudaFreeAsync(work, stream) != cudaSuccess) return CHOL_ECUDA;
    return rc;
}

template <typename T>
int adj_impl(int64_t batch, int32_t n, const void* L, const void* Lbar, void* Abar,
             const int32_t* status, int32_t tile, size_t bytes, bool accumulate,
             cudaStream_t stream) {
    const T* l = static_cast<const T*>(L);
    const T* lb = static_cast<const T*>(Lbar);
    T* ab = static_cast<T*>(Abar);
    if (n <= kSmallMax) {
        if constexpr (is_complex<T>()) {
            return to_code(chol::hsmall_adj<T>(l, lb, ab, status, batch, n, accumulate, stream));
        } else {
            const bool vec = vec_ok(n, sizeof(T), {L, Lbar, Abar});
            return to_code(
                chol::small_adj<T>(l, lb, ab, status, batch, n, vec, accumulate, stream));
        }
    }
    const bool in_place = !accumulate && Lbar == Abar;
    tile = pick_tile(tile, n, batch, sizeof(T), std::is_same<T, double>::value);
    // float64 with 128-wide tiles takes the tensor-core updates' operand
    // slices, after the batch * n * n working matrices (256-byte aligned)
    const size_t oz_bytes = (std::is_same<T, double>::value && tile == 128)
                                ? chol::ozaki_adj_workspace_bytes(batch, n)
                                : 0;
    // in place the sweep runs on the caller's buffer: no working matrices,
    // and no workspace at all for the FMA-pipe updates
    if (in_place && oz_bytes == 0)
        return to_code(chol::blocked_adj<T>(l, lb, ab, status, batch, n, tile, nullptr, false,
                                            nullptr, stream));
    const size_t wbytes = in_place ? 0 : (bytes + 255) / 256 * 256;
    void* work = nullptr;
    if (cudaMallocAsync(&work, wbytes + oz_bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return CHOL_ENOMEM;
    }
    void* oz = oz_bytes > 0 ? static_cast<void*>(static_cast<char*>(work) + wbytes) : nullptr;
    const int rc = to_code(chol::blocked_adj<T>(l, lb, ab, status, batch, n, tile,
                                                in_place ? nullptr : static_cast<T*>(work),
                                                accumulate, oz, stream));
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
    if ((rc = check_tile(tile, dtype)) != CHOL_OK) return rc;
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
    return dispatch(dtype, [&](auto t) {
        return fwd_impl<decltype(t)>(batch, n, A, L, status, tile, s);
    });
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
    if ((rc = check_tile(tile, dtype)) != CHOL_OK) return rc;
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
    return dispatch(dtype, [&](auto t) {
        return adj_impl<decltype(t)>(batch, n, L, adj_L, adj_A, status, tile, bytes, true, s);
    });
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
    if ((rc = check_tile(tile, dtype)) != CHOL_OK) return rc;
    if (batch == 0) return CHOL_OK;
    if (A == nullptr || status == nullptr) return CHOL_EINVAL;
    if (!aligned(A, (size_t)elem_size(dtype)) || !aligned(status, 4)) return CHOL_EINVAL;
    if (!is_device_pointer(A) || !is_device_pointer(status)) return CHOL_EINVAL;
    if (overlaps(range_of(A, bytes), range_of(status, (size_t)batch * 4))) return CHOL_EALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dispatch(dtype, [&](auto t) {
        return fwd_impl<decltype(t)>(batch, n, A, A, status, tile, s);
    });
}

int chol_adj_inplace(int64_t batch, int32_t n, int32_t dtype, const void* L, void* adj,
                     const int32_t* status, int32_t tile, void* stream) {
    size_t bytes = 0;
    int rc = check_shape(batch, n, dtype, &bytes);
    if (rc != CHOL_OK) return rc;
    if ((rc = check_tile(tile, dtype)) != CHOL_OK) return rc;
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
    return dispatch(dtype, [&](auto t) {
        return adj_impl<decltype(t)>(batch, n, L, adj, adj, status, tile, bytes, false, s);
    });
}

int chol_solve(int64_t batch, int32_t n, int32_t nrhs, int32_t dtype, const void* L,
               const void* B, void* X, const int32_t* status, void* stream) {
    size_t bytes = 0;
    int rc = check_shape(batch, n, dtype, &bytes);
    if (rc != CHOL_OK) return rc;
    if (nrhs < 0) return CHOL_EINVAL;
    const size_t es = (size_t)elem_size(dtype);
    const unsigned __int128 rb = (unsigned __int128)batch * n * (unsigned)nrhs * es;
    if (rb > ((unsigned __int128)1 << 62)) return CHOL_EINVAL;
    if (batch == 0 || nrhs == 0) return CHOL_OK;
    if (L == nullptr || B == nullptr || X == nullptr) return CHOL_EINVAL;
    if (!aligned(L, es) || !aligned(B, es) || !aligned(X, es)) return CHOL_EINVAL;
    if (status != nullptr && !aligned(status, 4)) return CHOL_EINVAL;
    if (!is_device_pointer(L) || !is_device_pointer(B) || !is_device_pointer(X) ||
        (status != nullptr && !is_device_pointer(status)))
        return CHOL_EINVAL;
    const Range rL = range_of(L, bytes), rB = range_of(B, (size_t)rb), rX = range_of(X, (size_t)rb);
    if (overlaps(rX, rL) || (X != B && overlaps(rX, rB))) return CHOL_EALIAS;
    if (status != nullptr && overlaps(rX, range_of(status, (size_t)batch * 4))) return CHOL_EALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dispatch(dtype, [&](auto t) {
        using T = decltype(t);
        return to_code(chol::potrs_solve<T>(static_cast<const T*>(L), static_cast<const T*>(B),
                                            static_cast<T*>(X), status, batch, n, nrhs, s));
    });
}

int chol_solve_adj(int64_t batch, int32_t n, int32_t nrhs, int32_t dtype, const void* L,
                   const void* X, const void* adj_X, void* adj_B, void* adj_L,
                   const int32_t* status, void* stream) {
    size_t bytes = 0;
    int rc = check_shape(batch, n, dtype, &bytes);
    if (rc != CHOL_OK) return rc;
    if (nrhs < 0) return CHOL_EINVAL;
    const size_t es = (size_t)elem_size(dtype);
    const unsigned __int128 rb = (unsigned __int128)batch * n * (unsigned)nrhs * es;
    if (rb > ((unsigned __int128)1 << 62)) return CHOL_EINVAL;
    if (batch == 0 || nrhs == 0 || (adj_B == nullptr && adj_L == nullptr)) return CHOL_OK;
    if (L == nullptr || X == nullptr || adj_X == nullptr) return CHOL_EINVAL;
    for (const void* p : {L, X, adj_X, (const void*)adj_B, (const void*)adj_L})
        if (p != nullptr && (!aligned(p, es) || !is_device_pointer(p))) return CHOL_EINVAL;
    if (status != nullptr && (!aligned(status, 4) || !is_device_pointer(status)))
        return CHOL_EINVAL;
    const Range rL = range_of(L, bytes), rX = range_of(X, (size_t)rb),
                rXb = range_of(adj_X, (size_t)rb);
    if (adj_B != nullptr) {
        const Range r = range_of(adj_B, (size_t)rb);
        if (overlaps(r, rL) || overlaps(r, rX) || overlaps(r, rXb)) return CHOL_EALIAS;
        if (status != nullptr && overlaps(r, range_of(status, (size_t)batch * 4)))
            return CHOL_EALIAS;
    }
    if (adj_L != nullptr) {
        const Range r = range_of(adj_L, bytes);
        if (overlaps(r, rL) || overlaps(r, rX) || overlaps(r, rXb)) return CHOL_EALIAS;
        if (adj_B != nullptr && overlaps(r, range_of(adj_B, (size_t)rb))) return CHOL_EALIAS;
        if (status != nullptr && overlaps(r, range_of(status, (size_t)batch * 4)))
            return CHOL_EALIAS;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t welems = chol::potrs_adj_workspace_elems(batch, n, nrhs, adj_L != nullptr);
    void* work = nullptr;
    if (cudaMallocAsync(&work, welems * es, s) != cudaSuccess) {
        cudaGetLastError();
        return CHOL_ENOMEM;
    }
    rc = dispatch(dtype, [&](auto t) {
        using T = decltype(t);
        return to_code(chol::potrs_adj<T>(static_cast<const T*>(L), static_cast<const T*>(X),
                                          static_cast<const T*>(adj_X), static_cast<T*>(adj_B),
                                          static_cast<T*>(adj_L), status, batch, n, nrhs,
                                          static_cast<T*>(work), s));
    });
    if (cudaFreeAsync(work, s) != cudaSuccess) return CHOL_ECUDA;
    return rc;
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
