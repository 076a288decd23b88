// Thread-per-matrix Cholesky forward for float32 matrices of order N = 8 or
// 16 (the batched 65536 x 16x16 workload).  jaxmg docs "Cholesky
// factorization": lower factor and status.
//
// One warp handles up to 32 matrices per round, one per lane, with no communication
// between lanes: every lane keeps the lower triangle of its own matrix in
// registers and runs the right-looking column recurrence on it
// (l_jj = d * rsqrt(d), column scaled by rsqrt(d), which keeps the per-column
// latency chain short).  Matrices move between HBM and shared memory by TMA
// bulk copies (cp.async.bulk, one per matrix, completion on an mbarrier) into
// per-lane slots skewed by 16 bytes, so each lane's 16-byte row reads and
// writes fall in distinct bank groups, and L leaves by bulk stores from the
// same slots.  Each warp owns two slot sets, so the copy for its next round is
// in flight while it factors the current one.  A block is one warp; blocks are
// persistent (resident blocks per SM x SMs).  At n = 16 a round takes 27
// matrices, so that four blocks (one per SM scheduler) fit in shared memory.

#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace chol {
namespace {

// M matrices per round (lanes 0..M-1 of the warp; the others idle), NSETS
// slot sets: up to NSETS - 1 rounds' loads are in flight while one round is
// factored.
template <int N, int M, int NSETS>
struct Tpm {
    static constexpr uint32_t kBytes = N * N * 4;   // one matrix
    static constexpr int kSlot = N * N + 4;         // floats per lane slot (16-byte skew)
    static constexpr size_t kSetBytes = (size_t)M * kSlot * 4;
    static constexpr size_t kSmem = 128 + NSETS * kSetBytes;
    static_assert(kBytes % 16 == 0, "bulk copies move multiples of 16 bytes");
    static_assert(M >= 1 && M <= 32 && NSETS >= 2 && NSETS <= 8, "one warp, 2..8 slot sets");
};

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
__device__ __forceinline__ void issue_round_load(const float* src, int64_t m0,
                                                 int nvalid, float* slot, uint64_t* bar,
                                                 int lane, int drop_lane) {
    fence_proxy_async_smem();  // earlier generic accesses to the slot come first
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)nvalid * (N * N * 4));
    __syncwarp();
    // (drop_lane >= 0 only in the self-test: that lane's copy is held back,
    //  so the round's barrier cannot complete until the lane issues it late)
    if (lane < nvalid && lane != drop_lane) bulk_load(slot, src + (m0 + lane) * (N * N), N * N * 4, bar);
}

template <int M>
__device__ __forceinline__ int round_count(int64_t batch, int64_t w) {
    return batch - w * M < M ? (int)(batch - w * M) : M;
}

template <int N, int M, int NSETS>
__global__ void __launch_bounds__(32)
tpm_potrf_kernel(const float* A, float* L, int32_t* __restrict__ status, int64_t batch,
                 uint32_t max_polls, int drop_lane) {
    using C = Tpm<N, M, NSETS>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);  // one per slot set
    const int lane = threadIdx.x;
    float* slots = reinterpret_cast<float*>(smem + 128);
    // this lane's slot in set s (lanes >= M have none)
    auto slot_of = [&](int s) { return slots + ((size_t)s * M + (lane < M ? lane : 0)) * C::kSlot; };
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < NSETS; ++s) mbar_init(bar + s, 1);
    }
    fence_mbar_init();
    __syncwarp();

    const int64_t rounds = (batch + M - 1) / M;
    const int64_t w0 = blockIdx.x;
    if (w0 >= rounds) return;
    uint32_t phase_bits = 0u;  // bit s: parity of set s's next completion
    uint32_t inflight = 0u;    // bit s: set s has a load in flight
    // the first NSETS - 1 rounds of this warp go out at once (in the
    // self-test, the first of them without the dropped lane's copy)
#pragma unroll
    for (int s = 0; s < NSETS - 1; ++s) {
        const int64_t w = w0 + (int64_t)s * gridDim.x;
        if (w < rounds) {
            issue_round_load<N>(A, w * M, round_count<M>(batch, w), slot_of(s), bar + s, lane,
                                s == 0 ? drop_lane : -1);
            inflight |= 1u << s;
        }
    }
#pragma unroll 1
    for (int64_t r = 0, w = w0; w < rounds; ++r, w += gridDim.x) {
        const int b = (int)(r % NSETS);
        const int64_t m0 = w * M;
        const int nvalid = round_count<M>(batch, w);
        const int64_t m = m0 + lane;
        // refill the set that the previous round used, NSETS - 1 rounds ahead
        const int64_t wn = w + (int64_t)(NSETS - 1) * gridDim.x;
        if (wn < rounds) {
            const int bn = (int)((r + NSETS - 1) % NSETS);
            bulk_wait_read_all();  // that set's last store has left shared memory
            issue_round_load<N>(A, wn * M, round_count<M>(batch, wn), slot_of(bn), bar + bn, lane,
                                -1);
            inflight |= 1u << bn;
        }
        const uint32_t par = (phase_bits >> b) & 1u;
        if (!__all_sync(0xffffffffu, mbar_wait(bar + b, par, max_polls))) {
            // The copies did not complete: mark this round's matrices and stop,
            // after one more bounded wait for every set's copies in flight so
            // that none lands in shared memory after the block has retired.
            // In the self-test the held-back copy (only ever in a warp's first
            // round) is issued now, so that wait can complete.
            if (lane < nvalid) status[m] = -1;
            if (r == 0 && lane == drop_lane && lane < nvalid)
                bulk_load(slot_of(b), A + m * (N * N), N * N * 4, bar + b);
#pragma unroll
            for (int s = 0; s < NSETS; ++s)
                if ((inflight >> s) & 1u) mbar_wait(bar + s, (phase_bits >> s) & 1u, max_polls);
            break;
        }
        phase_bits ^= 1u << b;
        inflight &= ~(1u << b);
        float* slot = slot_of(b);

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

// Persistent grid: resident blocks per SM (queried once per kernel and
// device) times the SM count of the current device, capped by the number of
// rounds.
template <typename K>
int tpm_grid(K kern, size_t smem, int64_t rounds, PerDeviceInt& per_sm_cache) {
    const int per_sm = per_sm_cache.get([&] {
        int x = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&x, kern, 32, smem) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        return x;
    });
    return (int)std::max<int64_t>(
        1, std::min<int64_t>((int64_t)device_sm_count() * std::max(per_sm, 1), rounds));
}

// Matrices per round and slot sets of the n = 16 kernel: 27 lanes with two
// sets fit four one-warp blocks per SM (one per scheduler) in 228 KB of
// shared memory, where 32 lanes fit three.
constexpr int kM16 = 27;
constexpr int kSets16 = 2;

template <int N, int M, int NSETS>
cudaError_t tpm_fwd_n(const float* A, float* L, int32_t* status, int64_t batch,
                      cudaStream_t stream, uint32_t max_polls = kMbarPolls, int drop_lane = -1) {
    const size_t smem = Tpm<N, M, NSETS>::kSmem;
    auto kern = tpm_potrf_kernel<N, M, NSETS>;
    static std::atomic<uint64_t> smem_set{0};
    static PerDeviceInt per_sm;
    cudaError_t e = allow_smem_once(kern, smem, smem_set);
    if (e != cudaSuccess) return e;
    const int grid = tpm_grid(kern, smem, (batch + M - 1) / M, per_sm);
    kern<<<grid, 32, smem, stream>>>(A, L, status, batch, max_polls, drop_lane);
    return cudaGetLastError();
}

}  // namespace

bool tpm_supported(int n) { return n == 8 || n == 16; }

cudaError_t tpm_fwd_wait_selftest(const float* A, float* L, int32_t* status, int64_t batch,
                                  uint32_t max_polls, cudaStream_t stream) {
    return tpm_fwd_n<16, kM16, kSets16>(A, L, status, batch, stream, max_polls, 0);
}

cudaError_t tpm_fwd(const float* A, float* L, int32_t* status, int64_t batch, int n,
                    cudaStream_t stream) {
    if (n == 16) return tpm_fwd_n<16, kM16, kSets16>(A, L, status, batch, stream);
    if (n == 8) return tpm_fwd_n<8, 32, 2>(A, L, status, batch, stream);
    return cudaErrorInvalidValue;
}

}  // namespace chol
