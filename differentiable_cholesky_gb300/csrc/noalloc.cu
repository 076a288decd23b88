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
//     array (cudaGetSymbolAddress, with that device current).  Make that first
//     call before any stream capture begins.
//   - Every call on a device shares the one scratch array and leaves its last
//     contents there.  The kernels write every scratch element they read, so
//     nothing needs clearing between calls, but calls that overlap on the GPU
//     (on different streams, or from several host threads without ordering
//     between their streams) race on the scratch and corrupt each other.

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "chol.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = (size_t)16 << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_adj_scratch[kScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on first
// use per device).  Returns nullptr if the lookup fails.
void* scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_adj_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return nullptr;
        }
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

bool on_device(const void* p) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged;
}

bool disjoint(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x + na <= y || y + nb <= x;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename T>
int run(int64_t batch, int32_t n, const void* L, const void* Lbar, void* Abar,
        const int32_t* status, int32_t tile, cudaStream_t stream) {
    const T* l = static_cast<const T*>(L);
    const T* lb = static_cast<const T*>(Lbar);
    T* ab = static_cast<T*>(Abar);
    cudaError_t e;
    if (n <= 64) {
        const bool vec = (n * (int)sizeof(T)) % 16 == 0 && aligned16(L) && aligned16(Lbar) &&
                         aligned16(Abar);
        e = chol::small_adj<T>(l, lb, ab, status, batch, n, vec, true, stream);
        return e == cudaSuccess ? CHOL_OK : CHOL_ECUDA;
    }
    const unsigned __int128 need =
        (unsigned __int128)batch * (unsigned __int128)n * (unsigned __int128)n * sizeof(T);
    if (need > kScratchBytes) return CHOL_ENOMEM;
    void* work = scratch_on_current_device();
    if (work == nullptr) return CHOL_ECUDA;
    if (tile == 0) tile = chol::blocked_default_tile(n, batch);
    e = chol::blocked_adj<T>(l, lb, ab, status, batch, n, tile, static_cast<T*>(work), true,
                             stream);
    return e == cudaSuccess ? CHOL_OK : CHOL_ECUDA;
}

}  // namespace

extern "C" CHOL_API int chol_adj_noalloc(int64_t batch, int32_t n, int32_t dtype, const void* L,
                                         const void* adj_L, void* adj_A, const int32_t* status,
                                         int32_t tile, void* stream) {
    const size_t es = dtype == CHOL_F32 ? 4 : dtype == CHOL_F64 ? 8 : 0;
    if (es == 0) return CHOL_EDTYPE;
    if (batch < 0 || n <= 0) return CHOL_EINVAL;
    if (!(tile == 0 || tile == 32 || tile == 64 || tile == 128)) return CHOL_EINVAL;
    const unsigned __int128 total =
        (unsigned __int128)batch * (unsigned __int128)n * (unsigned __int128)n * es;
    if (total > ((unsigned __int128)1 << 62)) return CHOL_EINVAL;
    if (batch == 0) return CHOL_OK;
    if (L == nullptr || adj_L == nullptr || adj_A == nullptr) return CHOL_EINVAL;
    const uintptr_t mask = es - 1;
    if ((reinterpret_cast<uintptr_t>(L) & mask) || (reinterpret_cast<uintptr_t>(adj_L) & mask) ||
        (reinterpret_cast<uintptr_t>(adj_A) & mask) ||
        (status != nullptr && (reinterpret_cast<uintptr_t>(status) & 3u)))
        return CHOL_EINVAL;
    if (!on_device(L) || !on_device(adj_L) || !on_device(adj_A) ||
        (status != nullptr && !on_device(status)))
        return CHOL_EINVAL;
    const size_t bytes = (size_t)total;
    if (!disjoint(adj_A, bytes, L, bytes) || !disjoint(adj_A, bytes, adj_L, bytes) ||
        (status != nullptr && !disjoint(adj_A, bytes, status, (size_t)batch * 4)))
        return CHOL_EALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dtype == CHOL_F32 ? run<float>(batch, n, L, adj_L, adj_A, status, tile, s)
                             : run<double>(batch, n, L, adj_L, adj_A, status, tile, s);
}
