// Thread-per-matrix Cholesky forward for float32 matrices of order N = 8 or
// 16 (the batched 65536 x 16x16 workload).  jaxmg docs "Cholesky
// factorization": lower factor and status.
//
// One warp handles 32 matrices per round, one per lane, with no communication
// between lanes: every lane keeps the lower triangle of its own matrix in
// registers and runs the right-looking column recurrence on it
// (l_jj = d * rsqrt(d), column scaled by rsqrt(d), which keeps the per-column
// latency chain short).  Matrices move between HBM and shared memory by TMA
// bulk copies (cp.async.bulk, one per matrix, completion on an mbarrier) into
// per-lane slots skewed by 16 bytes, so each lane's 16-byte row reads and
// writes fall in distinct bank groups, and L leaves by bulk stores from the
// same slots.  Each warp owns two slot sets, so the copy for its next round is
// in flight while it factors the current one.  A block is one warp; blocks are
// persistent (resident blocks per SM x SMs).

#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace chol {
namespace {

template <int N>
struct Tpm {
    static constexpr uint32_t kBytes = N * N * 4;   // one matrix
    static constexpr int kSlot = N * N + 4;         // floats per lane slot (16-byte skew)
    static constexpr size_t kSlotsBytes = 32 * (size_t)kSlot * 4;
    static_assert(kBytes % 16 == 0, "bulk copies move multiples of 16 bytes");
};

constexpr int kBarBytes = 128;  // mbarrier area in front of the slots

// Lower triangle of row i of the slot into registers.
template <int N>
__device__ __forceinline__ void slot_load_lower(const float* slot, float (&a)[N][N]) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
#pragma unroll
        for (int c = 0; c < N / 4; ++c) {
            if (4 * c > i) continue;
            const float4 v = reinterpret_cast<const float4*>(slot + i * N)[c];
            a[i][4 * c + 0] = v.x;
            if (4 * c + 1 <= i) a[i][4 * c + 1] = v.y;
            if (4 * c + 2 <= i) a[i][4 * c + 2] = v.z;
            if (4 * c + 3 <= i) a[i][4 * c + 3] = v.w;
        }
    }
}

// Issue the bulk loads of matrices [m0, m0 + nvalid) into the lanes' slots,
// completion on `bar`.  Every lane of the warp calls this.
template <int N>
__device__ __forceinline__ void issue_round_load(const float* __restrict__ src, int64_t m0,
                                                 int nvalid, float* slot, uint64_t* bar,
                                                 int lane) {
    fence_proxy_async_smem();  // earlier generic accesses to the slot come first
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)nvalid * Tpm<N>::kBytes);
    __syncwarp();
    if (lane < nvalid) bulk_load(slot, src + (m0 + lane) * (N * N), Tpm<N>::kBytes, bar);
}

__device__ __forceinline__ int round_count(int64_t batch, int64_t w) {
    return batch - w * 32 < 32 ? (int)(batch - w * 32) : 32;
}

template <int N>
__global__ void __launch_bounds__(32)
tpm_potrf_kernel(const float* __restrict__ A, float* __restrict__ L, int32_t* __restrict__ status,
                 int64_t batch) {
    using C = Tpm<N>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);  // bar[0], bar[1]
    const int lane = threadIdx.x;
    float* slots = reinterpret_cast<float*>(smem + kBarBytes);
    float* slot_of[2] = {slots + lane * C::kSlot, slots + (32 + lane) * C::kSlot};
    if (lane == 0) {
        mbar_init(bar + 0, 1);
        mbar_init(bar + 1, 1);
    }
    fence_mbar_init();
    __syncwarp();

    int64_t w = blockIdx.x;
    if (w * 32 >= batch) return;
    issue_round_load<N>(A, w * 32, round_count(batch, w), slot_of[0], bar + 0, lane);
    uint32_t phase[2] = {0u, 0u};
#pragma unroll 1
    for (int r = 0; w * 32 < batch; ++r, w += gridDim.x) {
        const int b = r & 1;
        const int64_t m0 = w * 32;
        const int nvalid = round_count(batch, w);
        const int64_t m = m0 + lane;
        const int64_t wn = w + gridDim.x;
        if (wn * 32 < batch) {
            bulk_wait_read_all();  // the other slot's last store has left shared memory
            issue_round_load<N>(A, wn * 32, round_count(batch, wn), slot_of[b ^ 1], bar + (b ^ 1),
                                lane);
        }
        if (!__all_sync(0xffffffffu, mbar_wait(bar + b, phase[b], kMbarPolls))) {
            // The copies did not complete: mark this round's matrices and stop
            // (after one more bounded wait for the copies in flight).
            if (lane < nvalid) status[m] = -1;
            mbar_wait(bar + b, phase[b], kMbarPolls);
            mbar_wait(bar + (b ^ 1), phase[b ^ 1], kMbarPolls);
            break;
        }
        phase[b] ^= 1u;
        float* slot = slot_of[b];

        float a[N][N];
        if (lane < nvalid) {
            slot_load_lower<N>(slot, a);
        } else {
#pragma unroll
            for (int i = 0; i < N; ++i)
#pragma unroll
                for (int k = 0; k <= i; ++k) a[i][k] = (i == k) ? 1.f : 0.f;
        }

        int st = 0;
#pragma unroll
        for (int j = 0; j < N; ++j) {
            float d = a[j][j];
            if (!(d > 0.f)) {
                if (st == 0) st = j + 1;
                d = 1.f;
            }
            const float inv = rsqrtf(d);  // 1 / l_jj
            a[j][j] = d * inv;
#pragma unroll
            for (int i = j + 1; i < N; ++i) a[i][j] *= inv;
#pragma unroll
            for (int k = j + 1; k < N; ++k)
#pragma unroll
                for (int i = k; i < N; ++i) a[i][k] = fmaf(-a[i][j], a[k][j], a[i][k]);
        }

        if (lane < nvalid) {
#pragma unroll
            for (int i = 0; i < N; ++i) {
#pragma unroll
                for (int c = 0; c < N / 4; ++c) {
                    float4 v;
                    v.x = (4 * c + 0 <= i) ? a[i][4 * c + 0] : 0.f;
                    v.y = (4 * c + 1 <= i) ? a[i][4 * c + 1] : 0.f;
                    v.z = (4 * c + 2 <= i) ? a[i][4 * c + 2] : 0.f;
                    v.w = (4 * c + 3 <= i) ? a[i][4 * c + 3] : 0.f;
                    reinterpret_cast<float4*>(slot + i * N)[c] = v;
                }
            }
            fence_proxy_async_smem();
            bulk_store(L + m * (N * N), slot, C::kBytes);
            bulk_commit();
            status[m] = st;
        }
    }
    bulk_wait_all();
}

// Persistent grid: resident blocks per SM (queried once per kernel) times the
// SM count of the current device, capped by the number of rounds.
template <typename K>
int tpm_grid(K kern, size_t smem, int64_t rounds, int* per_sm_cache) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (*per_sm_cache <= 0) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32, smem) !=
                cudaSuccess || per_sm < 1) {
            cudaGetLastError();
            per_sm = 1;
        }
        *per_sm_cache = per_sm;
    }
    return (int)std::max<int64_t>(
        1, std::min<int64_t>((int64_t)std::max(sms, 1) * *per_sm_cache, rounds));
}

template <int N>
cudaError_t tpm_fwd_n(const float* A, float* L, int32_t* status, int64_t batch,
                      cudaStream_t stream) {
    const size_t smem = kBarBytes + 2 * Tpm<N>::kSlotsBytes;
    auto kern = tpm_potrf_kernel<N>;
    static int smem_set = 0, per_sm = 0;
    if (!smem_set) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        smem_set = 1;
    }
    const int grid = tpm_grid(kern, smem, (batch + 31) / 32, &per_sm);
    kern<<<grid, 32, smem, stream>>>(A, L, status, batch);
    return cudaGetLastError();
}

}  // namespace

bool tpm_supported(int n) { return n == 8 || n == 16; }

cudaError_t tpm_fwd(const float* A, float* L, int32_t* status, int64_t batch, int n,
                    cudaStream_t stream) {
    if (n == 16) return tpm_fwd_n<16>(A, L, status, batch, stream);
    if (n == 8) return tpm_fwd_n<8>(A, L, status, batch, stream);
    return cudaErrorInvalidValue;
}

}  // namespace chol
