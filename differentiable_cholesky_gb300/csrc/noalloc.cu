// chol_adj_noalloc: the Cholesky adjoint for callers that cannot allocate GPU
// memory while they run.
//
// chol_adj takes the blocked path's workspace (one n x n matrix per batch
// entry) from the stream-ordered allocator on every call.  Some callers cannot
// do that: code running inside a CUDA-graph capture that must not grow the
// graph's memory pool, real-time or embedded hosts that forbid device
// allocation after start-up, and plug-ins whose host application owns every
// allocation.  This entry point runs the same kernels on a fixed scratch area
// that lives in the library itself: a file-scope __device__ array of
// kScratchBytes (16 MiB), which every GPU that loads the library holds until
// the process exits.
//
// Rules for callers:
//   - batch * n * n * sizeof(element) must fit in the 16 MiB scratch for n > 64
//     (n <= 64 needs no scratch at all); larger problems get CHOL_ENOMEM and
//     nothing is enqueued -- use chol_adj for them.
//   - The first call on each device looks up the device address of the scratch
//     array (cudaGetSymbolAddress, with that device current) and remembers it
//     with the context it belongs to; a call in another context of that
//     device (after cudaDeviceReset, say) looks it up again.  Make the first
//     call in a context before any stream capture begins.
//   - Every call on a device shares the one scratch array and leaves its last
//     contents there.  The kernels write every scratch element they read, so
//     nothing needs clearing between calls, but calls that overlap on the GPU
//     (on different streams, or from several host threads without ordering
//     between their streams) race on the scratch and corrupt each other.

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "chol.h"
#include "chol_tile.cuh"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = (size_t)16 << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_adj_scratch[kScratchBytes];

// The scratch address belongs to the CUDA context it was looked up in: after
// cudaDeviceReset, or with another context made current on the same device,
// the array lives somewhere else.  The cache therefore remembers the context
// beside the address and looks the address up again when the context changes.
struct ScratchEntry {
    CUcontext ctx;
    void* ptr;
};
std::mutex g_scratch_mutex;
ScratchEntry g_scratch[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry-point lookup, so the
// library needs no link-time dependency on the driver library.
CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return (CtxGetCurrentFn) nullptr;
        }
        return reinterpret_cast<CtxGetCurrentFn>(p);
    }();
    return fn;
}

// Device address of the scratch array in the current device's current
// context (looked up on the first call there).  Returns nullptr if the lookup
// fails.
void* scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    CtxGetCurrentFn get = ctx_get_current();
    CUcontext ctx = nullptr;
    if (get == nullptr || get(&ctx) != CUDA_SUCCESS) return nullptr;
    if (ctx == nullptr) {
        // the runtime makes its context current lazily; the symbol lookup
        // (no allocation) does that
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_adj_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchEntry& e = g_scratch[dev];
    if (e.ptr == nullptr || e.ctx != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_adj_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return nullptr;
        }
        e.ctx = ctx;
        e.ptr = p;
    }
    return e.ptr;
}

using chol_tile::cplx;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename T>
int run(int64_t batch, int32_t n, const void* L, const void* Lbar, void* Abar,
        const int32_t* status, int32_t tile, cudaStream_t stream) {
    const T* l = static_cast<const T*>(L);
    const T* lb = static_cast<const T*>(Lbar);
    T* ab = static_cast<T*>(Abar);
    cudaError_t e;
    if (n <= 64) {
        if constexpr (std::is_same<T, float>::value || std::is_same<T, double>::value) {
            const bool vec = (n * (int)sizeof(T)) % 16 == 0 && aligned16(L) && aligned16(Lbar) &&
                             aligned16(Abar);
            e = chol::small_adj<T>(l, lb, ab, status, batch, n, vec, true, stream);
        } else {
            e = chol::hsmall_adj<T>(l, lb, ab, status, batch, n, true, stream);
        }
        return e == cudaSuccess ? CHOL_OK : CHOL_ECUDA;
    }
    const unsigned __int128 need =
        (unsigned __int128)batch * (unsigned __int128)n * (unsigned __int128)n * sizeof(T);
    if (need > kScratchBytes) return CHOL_ENOMEM;
    void* work = scratch_on_current_device();
    if (work == nullptr) return CHOL_ECUDA;
    if (tile == 0)
        tile = std::min(chol::blocked_default_tile(n, batch),
                        chol::blocked_max_tile((int)sizeof(T)));
    e = chol::blocked_adj<T>(l, lb, ab, status, batch, n, tile, static_cast<T*>(work), true,
                             nullptr, stream);
    return e == cudaSuccess ? CHOL_OK : CHOL_ECUDA;
}

}  // namespace

extern "C" CHOL_API int chol_adj_noalloc(int64_t batch, int32_t n, int32_t dtype, const void* L,
                                         const void* adj_L, void* adj_A, const int32_t* status,
                                         int32_t tile, void* stream) {
    // the same checks, in the same order, as chol_adj_ex
    size_t bytes = 0;
    const int rc = chol::check_adj_args(batch, n, dtype, L, adj_L, adj_A, status, tile, &bytes);
    if (rc != CHOL_OK || batch == 0) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (dtype) {
        case CHOL_F32: return run<float>(batch, n, L, adj_L, adj_A, status, tile, s);
        case CHOL_F64: return run<double>(batch, n, L, adj_L, adj_A, status, tile, s);
        case CHOL_C64: return run<cplx<float>>(batch, n, L, adj_L, adj_A, status, tile, s);
        case CHOL_C128: return run<cplx<double>>(batch, n, L, adj_L, adj_A, status, tile, s);
        default: return CHOL_EDTYPE;
    }
}
