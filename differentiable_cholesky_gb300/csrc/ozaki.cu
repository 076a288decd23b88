// FP64 trailing update of the blocked Cholesky forward on the bf16 tensor
// cores (tcgen05), for 128-wide tiles.
//
// The trailing update L_IJ -= L_Ik L_Jk^T (jaxmg docs "Cholesky
// factorization": the tiled factorisation with tile size T_A = 128) is the
// only dense contraction of the forward.  On sm_103a the FP64 pipes (FMA and
// the f64 mma.sync path) deliver about 1.1 TFLOP/s in all, while the bf16
// tensor cores deliver about 2 PFLOP/s.  The update is therefore computed as
// an exact sum of bf16 products (the splitting scheme of Ozaki et al., with
// one power-of-two scale per row):
//
//   1. slice_kernel: every row x of the panel L_{.,k} (128 values) is scaled
//      by 2^-e, e = 1 + floor(log2 ||x||_2), so that ||x 2^-e||_2 < 1, and
//      written as 7 signed base-256 digits, x 2^-e = sum_p d_p 2^(-7-8p) with
//      integers |d_p| <= 128 (exact in bf16) and a remainder below 2^-56.
//      The digits go to a workspace in the tensor cores' shared-memory tile
//      layout, so that one bulk copy moves a whole stage.
//   2. trail_kernel (one CTA per 128 x 64 half of an output tile): for
//      d = 0..6 the products of digit slices p + q = d are accumulated in one
//      fp32 TMEM accumulator, acc_d = sum_{p+q=d} D_p(I) D_q(J)^T over the
//      128-long reduction.  Every product is an integer of at most 2^14 and
//      an accumulator sums at most 7 * 128 of them (< 2^24), so fp32 holds it
//      exactly.  The epilogue combines v = sum_d acc_d 256^(6-d) in int64
//      (exact: by Cauchy-Schwarz |v| <= 2^62) and applies
//      L_IJ -= v 2^(e_r + e_c - 62) with one FP64 fused multiply-add.
//
// The result differs from an FP64 GEMM only by the dropped digit products
// (p + q >= 7) and the digit remainders, both below 2^-53 of the row-norm
// scale 2^(e_r + e_c); the one rounding is that of the final FMA.  A row with
// a non-finite value keeps its NaN/Inf: its exponent is a sentinel and the
// epilogue writes NaN into every entry that row touches.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace chol {
namespace {

constexpr int kT = 128;                      // tile: rows per block, reduction length
constexpr int kS = 7;                        // digit slices
constexpr int kKC = 32;                      // reduction per pipeline stage
constexpr int kChunks = kT / kKC;            // stages per output tile
constexpr int kN = 64;                       // output columns per CTA
constexpr int kSliceElems = kT * kKC;        // one slice of one block, one stage: 8 KB
constexpr int kBlockElems = kChunks * kS * kSliceElems;  // one 128-row block: 224 KB
constexpr uint32_t kStageA = kS * kSliceElems * 2;       // 56 KB
constexpr uint32_t kStageB = kS * kN * kKC * 2;          // 28 KB
constexpr uint32_t kStageBytes = kStageA + kStageB;
constexpr int kStages = 2;
constexpr int kTmemCols = 512;               // 7 accumulators x 64 columns, rounded up
constexpr size_t kTrailSmem = 128 + (size_t)kStages * kStageBytes + 128;
constexpr int32_t kNonFinite = INT_MIN;      // exponent sentinel of a non-finite row

// Offset (elements) of element (r, kk) of a 128 x 32 slice: 8 x 8 core
// matrices (8 rows of 16 bytes), four along the reduction per row group.
__host__ __device__ constexpr int core_offset(int r, int kk) {
    return ((r >> 3) * (kKC / 8) + (kk >> 3)) * 64 + (r & 7) * 8 + (kk & 7);
}

// ---------------------------------------------------------------------------
// Digit slices of the panel: rows [r_begin, nt * 128) of column block k.
// One warp per row; lane l holds columns l, l + 32, l + 64, l + 96, i.e.
// reduction index l of each of the four stages.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
slice_kernel(const double* __restrict__ L, __nv_bfloat16* __restrict__ ws,
             int32_t* __restrict__ ex, const int32_t* __restrict__ status, int64_t batch, int n,
             int nt, int k0, int r_begin) {
    const int lane = threadIdx.x & 31;
    const int row = r_begin + (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    if (row >= nt * kT) return;
    for (int64_t b = blockIdx.y; b < batch; b += gridDim.y) {
        if (status != nullptr && status[b] != 0) continue;
        double v[kChunks];
        double ss = 0.0;
        bool finite = true;
#pragma unroll
        for (int j = 0; j < kChunks; ++j) {
            v[j] = row < n ? L[(size_t)b * n * n + (size_t)row * n + k0 + lane + 32 * j] : 0.0;
            finite = finite && isfinite(v[j]);
            ss = fma(v[j], v[j], ss);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        finite = __all_sync(0xffffffffu, finite) && isfinite(ss);
        int e = 0;
        if (!finite) {
            e = kNonFinite;
        } else if (ss > 0.0) {
            e = ilogb(sqrt(ss)) + 1;  // 2^e > ||row||_2 >= every |x|
        }
        const double scale = (finite && ss > 0.0) ? ldexp(128.0, -e) : 0.0;
        const int I = row / kT, r = row % kT;
        __nv_bfloat16* blk = ws + ((size_t)b * nt + I) * kBlockElems;
#pragma unroll
        for (int j = 0; j < kChunks; ++j) {
            double t = v[j] * scale;  // in [-128, 128]
            __nv_bfloat16* dst = blk + (size_t)j * kS * kSliceElems + core_offset(r, lane);
#pragma unroll
            for (int p = 0; p < kS; ++p) {
                const double d = rint(t);
                dst[p * kSliceElems] = __double2bfloat16(d);
                t = (t - d) * 256.0;
            }
        }
        if (lane == 0) ex[(size_t)b * nt * kT + row] = e;
    }
}

// ---------------------------------------------------------------------------
// tcgen05 helpers (inline PTX, sm_100 family)
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor, K-major, no swizzle: 14-bit fields of
// (address >> 4), the leading-dimension byte offset (between core matrices
// along the reduction) and the stride byte offset (between 8-row groups),
// and the descriptor version 1 at bit 46.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), bf16
// A and B (bits 7-9 and 10-12 = 1), both K-major, N >> 3 at bit 17, M >> 4 at
// bit 24.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kN >> 3) << 17) |
                            ((uint32_t)(kT >> 4) << 24);

__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(kIdesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// (i, j) of the t-th entry of a row-major enumeration of a lower triangle.
__device__ __forceinline__ void tri_index(int t, int& i, int& j) {
    int r = (int)((sqrt(8.0 * t + 1.0) - 1.0) * 0.5);
    while ((r + 1) * (r + 2) / 2 <= t) ++r;
    while (r * (r + 1) / 2 > t) --r;
    i = r;
    j = t - r * (r + 1) / 2;
}

// 2^E as a double for E in the normal range, 0 below it (such a contribution
// is under 2^-1022 and lost in any entry it meets).
__device__ __forceinline__ double pow2(int E) {
    if (E < -1022) return 0.0;
    if (E > 1023) return __longlong_as_double(0x7ff0000000000000LL);
    return __longlong_as_double((long long)(E + 1023) << 52);
}

// ---------------------------------------------------------------------------
// One CTA: the 128 x 64 half h of lower output tile (I, J), I >= J > k.
// Warp 0 owns TMEM and (lane 0) issues the MMAs; warp 1 lane 0 issues the
// bulk copies; all four warps run the epilogue (warp w reads TMEM lanes
// 32w .. 32w + 31, i.e. rows 32w .. of the tile).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128, 1)
trail_kernel(double* __restrict__ L, const __nv_bfloat16* __restrict__ ws,
             const int32_t* __restrict__ ex, int32_t* __restrict__ status, int64_t batch, int n,
             int nt, int k, uint32_t max_polls) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char* base = smem_raw;
    uint64_t* bars = reinterpret_cast<uint64_t*>(base);  // full[2], empty[2], done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + 64);
    unsigned char* stages = base + 128;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int job = blockIdx.x;
    const int h = job & 1;
    int ti, tj;
    tri_index(job >> 1, ti, tj);
    const int I = k + 1 + ti, J = k + 1 + tj;
    const int col0 = J * kT + h * kN;  // first output column
    if (col0 >= n) return;             // (uniform over the block)

    if (tid == 0) {
        for (int i = 0; i < 5; ++i) mbar_init(bars + i, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    uint32_t it = 0;  // output tiles handled by this CTA (one per matrix)
    bool failed = false;
    for (int64_t b = blockIdx.y; b < batch; b += gridDim.y, ++it) {
        if (status != nullptr && status[b] != 0) continue;  // uniform
        const __nv_bfloat16* blkA = ws + ((size_t)b * nt + I) * kBlockElems;
        const __nv_bfloat16* blkB = ws + ((size_t)b * nt + J) * kBlockElems + h * (kN * kKC);
        if (tid == 32) {
            // producer: the four stages of this tile
            for (int kc = 0; kc < kChunks; ++kc) {
                const uint32_t g = it * kChunks + kc, s = g & 1, u = g >> 1;
                if (u > 0 && !mbar_wait(bars + 2 + s, (u - 1) & 1, max_polls)) {
                    failed = true;
                    break;
                }
                unsigned char* st = stages + s * kStageBytes;
                mbar_arrive_expect_tx(bars + s, kStageBytes);
                bulk_load(st, blkA + (size_t)kc * kS * kSliceElems, kStageA, bars + s);
                for (int q = 0; q < kS; ++q)
                    bulk_load(st + kStageA + q * (kN * kKC * 2),
                              blkB + (size_t)kc * kS * kSliceElems + (size_t)q * kSliceElems,
                              kN * kKC * 2, bars + s);
            }
        } else if (tid == 0) {
            // MMA issuer: acc_d += D_p(I) D_q(J)^T for p + q = d
            for (int kc = 0; kc < kChunks && !failed; ++kc) {
                const uint32_t g = it * kChunks + kc, s = g & 1, u = g >> 1;
                if (!mbar_wait(bars + s, u & 1, max_polls)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = smem_u32(stages + s * kStageBytes);
                const uint32_t sb = sa + kStageA;
#pragma unroll
                for (int d = 0; d < kS; ++d) {
#pragma unroll
                    for (int p = 0; p <= d; ++p) {
                        const int q = d - p;
#pragma unroll
                        for (int ks = 0; ks < kKC / 16; ++ks) {
                            const uint64_t da =
                                smem_desc(sa + p * (kSliceElems * 2) + ks * 256, 128, 512);
                            const uint64_t db =
                                smem_desc(sb + q * (kN * kKC * 2) + ks * 256, 128, 512);
                            tc_mma(tmem + d * kN, da, db, (kc | p | ks) != 0);
                        }
                    }
                }
                tc_commit(bars + 2 + s);  // the stage may be refilled once these finish
            }
            if (!failed) tc_commit(bars + 4);
        }
        // epilogue: every thread waits for the accumulators
        const bool ok = __syncthreads_and(!failed) && mbar_wait(bars + 4, it & 1, max_polls);
        tc_fence_after();
        const int rl = warp * 32 + lane;
        const int row = I * kT + rl;
        if (!__all_sync(0xffffffffu, ok)) {
            if (tid == 0) status[b] = -1;  // a device wait ran out: reported, not hung
            failed = true;
        } else {
            const int er = row < n ? ex[(size_t)b * nt * kT + row] : 0;
            double* Lrow = L + (size_t)b * n * n + (size_t)row * n;
#pragma unroll 1
            for (int cc = 0; cc < kN / 16; ++cc) {
                uint32_t acc[kS][16];
#pragma unroll
                for (int d = 0; d < kS; ++d)
                    tc_ld16(tmem + ((uint32_t)(warp * 32) << 16) + d * kN + cc * 16, acc[d]);
                tc_wait_ld();
                if (row >= n) continue;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int col = col0 + cc * 16 + j;
                    if (col >= n || (I == J && col > row)) continue;
                    const int ec = ex[(size_t)b * nt * kT + col];
                    // sum_d acc_d 256^(6-d), modulo 2^64 (exact: |sum| <= 2^62)
                    unsigned long long v = 0;
#pragma unroll
                    for (int d = 0; d < kS; ++d)
                        v = v * 256ull +
                            (unsigned long long)(long long)__float2int_rn(__uint_as_float(acc[d][j]));
                    double c;
                    if (er == kNonFinite || ec == kNonFinite) {
                        c = __longlong_as_double(0x7ff8000000000000LL);  // NaN
                        Lrow[col] = c;
                    } else {
                        const double scale = pow2(er + ec - 62);
                        Lrow[col] = fma(-__ll2double_rn((long long)v), scale, Lrow[col]);
                    }
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (failed) break;
    }
    if (failed && tid == 32) {
        // let copies still in flight land before the block retires
        for (int s = 0; s < 2; ++s) mbar_wait(bars + s, 0, max_polls);
    }
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

}  // namespace

size_t ozaki_workspace_bytes(int64_t batch, int n) {
    const int64_t nt = (n + kT - 1) / kT;
    return (size_t)batch * nt * kBlockElems * sizeof(__nv_bfloat16) +
           (size_t)batch * nt * kT * sizeof(int32_t);
}

cudaError_t ozaki_trailing_update(double* L, void* work, int32_t* status, int64_t batch, int n,
                                  int k, cudaStream_t stream) {
    const int nt = (n + kT - 1) / kT;
    const int m = nt - k - 1;
    if (m <= 0) return cudaSuccess;
    __nv_bfloat16* ws = static_cast<__nv_bfloat16*>(work);
    int32_t* ex = reinterpret_cast<int32_t*>(ws + (size_t)batch * nt * kBlockElems);
    const unsigned gy = (unsigned)std::min<int64_t>(batch, 65535);
    {
        const int rows = m * kT;  // rows (k + 1) * 128 .. nt * 128
        const unsigned blocks = (unsigned)((rows * 32 + 255) / 256);
        slice_kernel<<<dim3(blocks, gy), 256, 0, stream>>>(L, ws, ex, status, batch, n, nt,
                                                           k * kT, (k + 1) * kT);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    static std::atomic<uint64_t> smem_set{0};
    cudaError_t e = allow_smem_once(trail_kernel, kTrailSmem, smem_set);
    if (e != cudaSuccess) return e;
    const unsigned jobs = (unsigned)(m * (m + 1) / 2 * 2);
    trail_kernel<<<dim3(jobs, gy), 128, kTrailSmem, stream>>>(L, ws, ex, status, batch, n, nt, k,
                                                              kMbarPolls);
    return cudaGetLastError();
}

}  // namespace chol
