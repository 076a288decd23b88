// FP64 GEMM-shaped steps of the blocked Cholesky (128-wide tiles) on the bf16
// tensor cores (tcgen05): the forward's trailing update and the adjoint's
// two large updates.
//
// The trailing update L_IJ -= L_Ik L_Jk^T (jaxmg docs "Cholesky
// factorization": the tiled factorisation with tile size T_A = 128) is the
// only dense contraction of the forward, and Murray's blocked reverse sweep
// (the adjoint NVIDIA/warp issue #1316's closing comment states, evaluated
// blockwise) spends its flops in two more: W_JK -= C^T L_{below J, K} and
// W_IK -= C_I L_JK (+ the symmetric diagonal term).  On sm_103a the FP64 pipes
// (FMA and the f64 mma.sync path) deliver about 1.1 TFLOP/s in all, while the
// bf16 tensor cores deliver about 2 PFLOP/s.  Each contraction is therefore
// computed as an exact sum of bf16 products (the splitting scheme of Ozaki et
// al., with one power-of-two scale per operand row):
//
//   1. Slicing: every 128-long operand vector x (a row of a panel, or a
//      column of a 128-row chunk) is scaled by 2^-e, e = 1 + floor(log2
//      ||x||_2), so that ||x 2^-e||_2 < 1, truncated to a multiple of 2^-55
//      and written as 7 balanced base-256 digits, x 2^-e ~ sum_p d_p
//      2^(-7-8p), integers |d_p| <= 128 (exact in bf16), by integer
//      arithmetic on the float64 bits.  The digits go to a workspace in the
//      tensor cores' shared-memory tile layout (8 x 8 core matrices), so that
//      one bulk copy moves a whole pipeline stage.
//   2. oz_gemm_kernel (one CTA per 128 x 32 quarter of an output tile): per
//      128-long reduction chunk, for d = 0..6 the products of digit slices
//      p + q = d are accumulated in one fp32 TMEM accumulator,
//      acc_d = sum_{p+q=d} D_p(A) D_q(B)^T.  Every product is an integer of at
//      most 2^14 and an accumulator sums at most 7 * 128 of them (< 2^24), so
//      fp32 holds it exactly.  The epilogue combines v = sum_d acc_d
//      256^(6-d) in int64 (exact: by Cauchy-Schwarz |v| <= 2^62), forms the
//      float64 v 2^(e_r + e_c - 62) from v's bits (one rounding) and applies
//      out -= that with one FP64 subtraction per chunk.
//
// The result differs from an FP64 GEMM only by the dropped digit products
// (p + q >= 7) and the truncation below 2^-55, both below 2^-53 of the
// row-norm scale 2^(e_r + e_c); the one rounding per chunk is that of the FMA.
// An operand vector with a non-finite value keeps its NaN/Inf: its exponent
// is a sentinel and the epilogue writes NaN into every entry it touches.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace chol {
namespace {

constexpr int kT = 128;                      // tile: rows per block, reduction chunk
constexpr int kS = 7;                        // digit slices
// Two CTAs share an SM, so that one's MMAs overlap the other's epilogue: each
// takes 128 x 32 outputs (7 accumulators x 32 TMEM columns = 224, 256
// allocated) and three pipeline stages of 16 reduction steps (105 KB).
constexpr int kKC = 16;                      // reduction per pipeline stage
constexpr int kChunks = kT / kKC;            // stages per reduction chunk
constexpr int kLaneElems = kT / 32;          // a 128-long vector's elements per lane (slicing)
constexpr int kN = 32;                       // output columns per CTA
constexpr int kParts = kT / kN;              // CTAs per 128 x 128 output tile
constexpr int kSliceElems = kT * kKC;        // one slice of one block, one stage: 4 KB
constexpr int kBlockElems = kChunks * kS * kSliceElems;  // one 128 x 128 operand block: 224 KB
constexpr uint32_t kStageA = kS * kSliceElems * 2;       // 28 KB
constexpr uint32_t kStageB = kS * kN * kKC * 2;          // 7 KB
constexpr uint32_t kStageBytes = kStageA + kStageB;
constexpr int kStages = 3;
constexpr int kTmemCols = 256;               // 7 accumulators x 32 columns, rounded up
constexpr uint32_t kSbo = kKC / 8 * 128;     // bytes between 8-row core-matrix groups
constexpr size_t kGemmSmem = 128 + (size_t)kStages * kStageBytes + 128;
constexpr int32_t kNonFinite = INT_MIN;      // exponent sentinel of a non-finite vector
constexpr int kOzThreads = 256;              // 8 warps: two per TMEM lane quadrant
constexpr int kColHalves = kOzThreads / 128;  // column groups per lane quadrant
constexpr int kWarpCols = kN / kColHalves;    // output columns per epilogue warp: 16
constexpr int kEC = 8;                       // output columns per epilogue pass
constexpr int kEpP = kEC + 1;                // pitch (doubles) of the epilogue's staged rows
constexpr int kEpR = 32 / kEC;               // rows per warp-wide access of a pass

using bf16 = __nv_bfloat16;

// Offset (elements) of element (r, kk) of a 128 x kKC slice: 8 x 8 core
// matrices (8 rows of 16 bytes), kKC / 8 along the reduction per row group.
__host__ __device__ constexpr int core_offset(int r, int kk) {
    return ((r >> 3) * (kKC / 8) + (kk >> 3)) * 64 + (r & 7) * 8 + (kk & 7);
}

// Offset of element (m, k) (operand index m, reduction index k, both < 128)
// of digit slice p inside one operand block.
__device__ __forceinline__ int block_offset(int m, int k, int p) {
    return (k / kKC) * (kS * kSliceElems) + p * kSliceElems + core_offset(m, k % kKC);
}

// v * 2^E for an integer |v| <= 2^62, rounded to the nearest float64 (ties
// to even).  Where the result is a normal number it is assembled from v's
// bits by integer instructions (leading-zero count, shift, round on the 11
// bits below the 53 kept): an int64 -> float64 conversion would occupy the
// FP64 pipe, the scarce one here, once per output entry.  Otherwise (a
// result outside the normal range) the conversion and ldexp, which give the
// same value wherever both apply.
__device__ __forceinline__ double scale_int(long long v, int E) {
    if (v == 0) return 0.0;
    const unsigned long long sgn = (unsigned long long)v & 0x8000000000000000ull;
    unsigned long long a = v < 0 ? 0ull - (unsigned long long)v : (unsigned long long)v;
    const int lz = __clzll((long long)a);
    const int ex = 63 - lz + E;  // exponent of v's leading bit, scaled
    if (ex < -1022 || ex > 1022) return ldexp(__ll2double_rn(v), E);
    a <<= lz;                                   // leading bit at bit 63
    unsigned long long m = a >> 11;             // 53 bits, bit 52 set
    const unsigned rem = (unsigned)a & 0x7ffu;  // the bits rounded off
    m += (rem > 0x400u || (rem == 0x400u && (m & 1ull))) ? 1ull : 0ull;
    // bit 52 of m (and a carry out of the rounding, m = 2^53) adds to the
    // biased exponent ex + 1022, giving ex + 1023 (or ex + 1024, mantissa 0)
    return __longlong_as_double(
        (long long)(sgn | (((unsigned long long)(ex + 1022) << 52) + m)));
}

// v = sum_d acc_d 256^(6-d) from the 7 fp32 accumulators of one entry (exact
// integers below 2^24 in magnitude), modulo 2^64, which is exact since
// |v| <= 2^62: digits 3..6 by 64-bit multiply-adds of 32-bit values, digits
// 0..2 in 32 bits (their sum is only needed modulo 2^32 once shifted by 32).
template <int W>
__device__ __forceinline__ long long combine_acc(const uint32_t (&acc)[kS][W], int j) {
    int a[kS];
#pragma unroll
    for (int d = 0; d < kS; ++d) a[d] = __float2int_rn(__uint_as_float(acc[d][j]));
    const long long lo = (long long)a[3] * (1 << 24) + (long long)a[4] * (1 << 16) +
                         (long long)a[5] * (1 << 8) + (long long)a[6];
    const unsigned hi = (unsigned)a[0] * 65536u + (unsigned)a[1] * 256u + (unsigned)a[2];
    return (long long)((unsigned long long)lo + ((unsigned long long)hi << 32));
}

// Scale exponent of the 128-long vector a warp holds four values per lane:
// 2^e > ||x||_2, 0 for a vector below 2^-1022 (its digits are all zero) and
// the sentinel for a non-finite one.  Integer and fp32 arithmetic only (the
// FP64 pipe is the scarce one): the largest binary exponent by an integer
// warp maximum, then the squares of the values relative to it in fp32, whose
// sum is inflated by 2^-16 so that rounding cannot place 2^e at or below the
// exact norm.  A slightly large e only costs the last fraction of a bit.
__device__ __forceinline__ int warp_scale_exponent(const double (&v)[kLaneElems],
                                                   bool finite_lane) {
    if (!__all_sync(0xffffffffu, finite_lane)) return kNonFinite;
    unsigned emax = 0;
#pragma unroll
    for (int j = 0; j < kLaneElems; ++j) {
        const unsigned E = (unsigned)((__double_as_longlong(v[j]) >> 52) & 0x7ff);
        emax = E > emax ? E : emax;
    }
    emax = __reduce_max_sync(0xffffffffu, emax);
    if (emax == 0) return 0;  // zeros and subnormals only
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kLaneElems; ++j) {
        const long long bits = __double_as_longlong(v[j]);
        const int E = (int)((bits >> 52) & 0x7ff);
        const int fe = E - (int)emax + 127;  // |x| 2^-(emax-1023) as a float, in [2^-126, 2)
        if (E == 0 || fe < 1) continue;      // below 2^-126 of the largest: negligible
        const unsigned fbits = ((unsigned)fe << 23) | (unsigned)((bits >> 29) & 0x7fffff);
        const float xs = __uint_as_float(fbits);
        ss = fmaf(xs, xs, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    // the truncated mantissas and the fp32 sums only lose: a margin keeps 2^e above
    ss *= 1.0f + 0x1p-16f;
    return (int)emax - 1023 + ilogbf(sqrtf(ss)) + 1;  // ss in [1, 512)
}

// The 7 balanced base-256 digits of v 2^(55-e) (|v| < 2^e), truncated toward
// zero below 2^(e-55), most significant first, from the float64's bits.
__device__ __forceinline__ void to_digits(double v, int e, int (&d)[kS]) {
    const long long bits = __double_as_longlong(v);
    const int E = (int)((bits >> 52) & 0x7ff);
    long long X = 0;
    if (E != 0 && e != kNonFinite) {  // zeros and subnormals (< 2^-1022) give 0
        const long long M = (bits & ((1ll << 52) - 1)) | (1ll << 52);
        const int s = E - 1075 + 55 - e;  // X = M 2^s, s <= 2 since |v| < 2^e
        X = s >= 0 ? (M << s) : (s > -64 ? (M >> -s) : 0);
        if (bits < 0) X = -X;
    }
#pragma unroll
    for (int p = kS - 1; p >= 1; --p) {
        const int lo = (int)(signed char)(X & 0xff);  // in [-128, 127]
        d[p] = lo;
        X = (X - lo) >> 8;                            // exact
    }
    d[0] = (int)X;  // |d_0| <= 128
}

// Balancing of the reduction index.  A product sum_r a_r b_r is unchanged
// when a_r is multiplied and b_r divided by the same power of two 2^s_r.
// Cholesky operands carry the factor's row scales along the reduction (rows
// of L scale like sqrt(a_rr), the panel before its solve like a_rr, the
// gradient like 1 / sqrt(a_rr)), so each term is balanced with
// s_r = ilogb(L_rr) before the per-vector scaling: the digits then resolve
// every term to the same relative precision even when the rows span many
// binades.  sign = +1 multiplies, -1 divides, 0 leaves the operand as it is.
struct Bal {
    const int32_t* exp;  // s_r per reduction index (per batch entry: stride)
    size_t stride;
    int off;             // reduction index of the slicer's element 0
    int sign;
};

// x 2^s, exact: an integer add to the exponent field where x and the result
// are normal numbers, ldexp otherwise (zeros, subnormals, non-finite values,
// results out of the normal range).
__device__ __forceinline__ double balance(double x, const Bal& bal, int64_t b, int r) {
    if (bal.sign == 0) return x;
    const int s = bal.sign * bal.exp[b * bal.stride + bal.off + r];
    const long long bits = __double_as_longlong(x);
    const int E = (int)((bits >> 52) & 0x7ff);
    if (E != 0 && E != 0x7ff && E + s >= 1 && E + s <= 0x7fe)
        return __longlong_as_double(bits + ((long long)s << 52));
    return ldexp(x, s);
}

// ---------------------------------------------------------------------------
// Row slicing: rows [row0, row0 + nrows) of the 128 columns [col0, col0+128)
// of src (n x n, row-major); one warp per row, lane l holding reduction
// indices l, l + 32, l + 64, l + 96.  Row r goes to operand block r / 128 at
// position r % 128, its exponent to ex[r].  With sym_blocks, the first 128 rows
// (block row0 / 128, which must equal col0 / 128) are read as the Hermitian
// matrix S + S^T of the lower triangle of that diagonal block: the upper half
// mirrors the lower one and the diagonal is doubled.  Rows >= n are zeros.
// ---------------------------------------------------------------------------
// One launch may slice two such row ranges (of two matrices): the warps
// past the first range's rows take the second's.
struct RowSlice {
    const double* src;
    bf16* dst;
    int32_t* ex;
    int n, row0, nrows, col0;
    bool sym_first;
    size_t dst_stride, ex_stride;
    Bal bal;
};

__global__ void __launch_bounds__(256)
slice_rows_kernel(RowSlice s0, RowSlice s1, const int32_t* __restrict__ status, int64_t batch) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    int rl = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const bool second = rl >= s0.nrows;
    if (second) rl -= s0.nrows;
    const RowSlice sl = second ? s1 : s0;
    if (rl >= sl.nrows) return;
    const double* __restrict__ src = sl.src;
    bf16* __restrict__ dst = sl.dst;
    int32_t* __restrict__ ex = sl.ex;
    const int n = sl.n, col0 = sl.col0;
    const bool sym_first = sl.sym_first;
    const size_t dst_stride = sl.dst_stride, ex_stride = sl.ex_stride;
    const Bal bal = sl.bal;
    const int row = sl.row0 + rl;
    for (int64_t b = blockIdx.y; b < batch; b += gridDim.y) {
        if (status != nullptr && status[b] != 0) continue;
        const double* S = src + (size_t)b * n * n;
        double v[kLaneElems];
        bool finite = true;
#pragma unroll
        for (int j = 0; j < kLaneElems; ++j) {
            const int col = col0 + lane + 32 * j;
            double x = 0.0;
            if (row < n && col < n) {
                if (sym_first && rl < kT) {
                    x = col <= row ? S[(size_t)row * n + col] : S[(size_t)col * n + row];
                    if (col == row) x += x;
                } else {
                    x = S[(size_t)row * n + col];
                }
                x = balance(x, bal, b, col);
            }
            v[j] = x;
            finite = finite && isfinite(x);
        }
        const int e = warp_scale_exponent(v, finite);
        bf16* blk = dst + b * dst_stride + (size_t)(row / kT) * kBlockElems;
#pragma unroll
        for (int j = 0; j < kLaneElems; ++j) {
            int d[kS];
            to_digits(v[j], e, d);
#pragma unroll
            for (int p = 0; p < kS; ++p)
                blk[block_offset(row % kT, lane + 32 * j, p)] = __int2bfloat16_rn(d[p]);
        }
        if (lane == 0) ex[b * ex_stride + row] = e;
    }
}

// ---------------------------------------------------------------------------
// Column slicing: for every 128-row chunk c of a list and every column block
// K of it, the columns x = src[c*128 .. c*128+127, K*128 + m] (the reduction
// runs down the rows) go to operand block blk(c, K) at position m.  With
// lower_only, entries above the diagonal (row < column) read as zero (the
// upper triangle of a factor is never read).  One block of 256 threads per
// (chunk, column block): the 128 x 128 tile goes through shared memory, read
// by rows (coalesced), sliced by columns.
// Chunk list: chunks c = c_begin .. c_end - 1; column blocks K = 0 .. kmax(c)
// where kmax(c) = (tri ? c : k_fixed), so blocks are (c, K <= c) packed
// lower-triangle-wise (tri) or (c, k_fixed) one per chunk.  Each (c, K) is
// split over kColGroups blocks of 32 columns (more blocks than chunks: one
// matrix's few chunks would leave most SMs idle).
// ---------------------------------------------------------------------------
constexpr int kColThreads = 256;
constexpr int kColGroups = 4;
constexpr int kColW = kT / kColGroups;  // columns per block

__global__ void __launch_bounds__(kColThreads)
slice_cols_kernel(const double* __restrict__ src, bf16* __restrict__ dst,
                  int32_t* __restrict__ ex, const int32_t* __restrict__ status, int64_t batch,
                  int n, int c_begin, bool tri, int k_fixed, bool lower_only, size_t dst_stride,
                  size_t ex_stride, Bal bal) {
    pdl_wait();
    extern __shared__ __align__(128) unsigned char smem_raw[];
    double* tile = reinterpret_cast<double*>(smem_raw);  // 128 x (kColW + 1)
    constexpr int P = kColW + 1;
    // which (c, K) and which group of its columns: blockIdx.x enumerates them
    const int grp = (int)blockIdx.x % kColGroups;
    const int item = (int)blockIdx.x / kColGroups;
    int c, K, slot;
    if (tri) {
        // slot t = c (c + 1) / 2 + K over c >= c_begin: t0 = c_begin (c_begin + 1) / 2
        const int t = c_begin * (c_begin + 1) / 2 + item;
        int r = (int)((sqrt(8.0 * t + 1.0) - 1.0) * 0.5);
        while ((r + 1) * (r + 2) / 2 <= t) ++r;
        while (r * (r + 1) / 2 > t) --r;
        c = r;
        K = t - r * (r + 1) / 2;
        slot = t;
    } else {
        c = c_begin + item;
        K = k_fixed;
        slot = c;
    }
    const int r0 = c * kT, q0 = K * kT + grp * kColW;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t b = blockIdx.y; b < batch; b += gridDim.y) {
        if (status != nullptr && status[b] != 0) continue;
        const double* S = src + (size_t)b * n * n;
        __syncthreads();
        for (int e = threadIdx.x; e < kT * kColW; e += kColThreads) {
            const int i = e / kColW, j = e % kColW;
            const int row = r0 + i, col = q0 + j;
            double x = 0.0;
            if (row < n && col < n && (!lower_only || col <= row))
                x = balance(S[(size_t)row * n + col], bal, b, row);
            tile[i * P + j] = x;
        }
        __syncthreads();
        bf16* blk = dst + b * dst_stride + (size_t)slot * kBlockElems;
        // warp w takes columns w, w + 8, ...; lane l holds rows l, l+32, l+64, l+96
        for (int m = warp; m < kColW; m += kColThreads / 32) {
            const int mb = grp * kColW + m;  // position in the operand block
            double v[kLaneElems];
            bool finite = true;
#pragma unroll
            for (int j = 0; j < kLaneElems; ++j) {
                v[j] = tile[(lane + 32 * j) * P + m];
                finite = finite && isfinite(v[j]);
            }
            const int e = warp_scale_exponent(v, finite);
#pragma unroll
            for (int j = 0; j < kLaneElems; ++j) {
                int d[kS];
                to_digits(v[j], e, d);
#pragma unroll
                for (int p = 0; p < kS; ++p)
                    blk[block_offset(mb, lane + 32 * j, p)] = __int2bfloat16_rn(d[p]);
            }
            if (lane == 0) ex[b * ex_stride + (size_t)slot * kT + mb] = e;
        }
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

// Instruction descriptor of kind::f16 for an M = 128, N-wide product: fp32
// accumulator (bits 4-5 = 1), bf16 A and B (bits 7-9 and 10-12 = 1), both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t mma_idesc(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(kT >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
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

// 8 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tc_ld8(uint32_t taddr, uint32_t (&v)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                   "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32-byte global accesses (four doubles; the address 32-byte aligned).
__device__ __forceinline__ void ld_global_v4(const double* p, double (&v)[4]) {
    asm volatile("ld.global.v4.f64 {%0, %1, %2, %3}, [%4];"
                 : "=d"(v[0]), "=d"(v[1]), "=d"(v[2]), "=d"(v[3])
                 : "l"(p));
}
__device__ __forceinline__ void st_global_v4(double* p, const double (&v)[4]) {
    asm volatile("st.global.v4.f64 [%0], {%1, %2, %3, %4};" ::"l"(p), "d"(v[0]), "d"(v[1]),
                 "d"(v[2]), "d"(v[3])
                 : "memory");
}

// (i, j) of the t-th entry of a row-major enumeration of a lower triangle.
__device__ __forceinline__ void tri_index(int t, int& i, int& j) {
    int r = (int)((sqrt(8.0 * t + 1.0) - 1.0) * 0.5);
    while ((r + 1) * (r + 2) / 2 <= t) ++r;
    while (r * (r + 1) / 2 > t) --r;
    i = r;
    j = t - r * (r + 1) / 2;
}


// ---------------------------------------------------------------------------
// The contractions.  Per output quarter tile (128 rows x 32 columns) a CTA
// runs one or more 128-long reduction chunks, each with its own operand
// blocks and scales.
// ---------------------------------------------------------------------------
enum OzMode {
    OZ_FWD_TRAIL = 0,  // L_IJ -= L_Ik L_Jk^T, I >= J > k           (A, B: row slices of the panel)
    OZ_REV_ROW = 1,    // W_JK -= sum_{c > J} C_c^T L_cK, K <= J     (A: column slices of C per chunk,
                       //                                             B: column slices of L per chunk)
    OZ_REV_UPD = 2,    // W_IK -= Chat_I L_JK, I >= J, K < J         (A: row slices of Chat,
                       //                                             B: column slices of L, chunk J)
    OZ_ASSIGN = 3      // X_I = P_I G^T, I > step: a panel solve by the inverse of its diagonal
                       // tile (A: row slices of the panel, B: slices of the inverse, written
                       // over the panel)
};

struct OzArgs {
    double* out;          // the matrix updated (L or W), n x n per batch entry
    const bf16* a;        // A operand blocks
    const int32_t* ea;    // their exponents (128 per block)
    const bf16* b;        // B operand blocks
    const int32_t* eb;
    size_t a_stride, ea_stride, b_stride, eb_stride;  // per batch entry (elements)
    const int32_t* status;  // matrices with status != 0 are skipped
    int32_t* fail;          // where a device wait that ran out is reported (or null)
    int64_t batch;
    int n, nt, step;      // step: k (forward) or J (adjoint)
    int splits;           // OZ_REV_ROW: the reduction split over this many CTAs
    double* part;         // ... each writing its partial sum here (splits > 1)
    int sub;              // OZ_FWD_TRAIL: 0 every trailing tile, 1 only block column
                          // step + 1, 2 only block columns >= step + 2; OZ_REV_UPD:
                          // 0 every K < J, 1 only K = J - 1, 2 only K < J - 1
    int k_lo, k_n;        // OZ_REV_ROW: output block columns K = k_lo .. k_lo + k_n - 1
};

struct OzJob {
    int out_r0, out_c0;   // output half tile origin
    bool lower;           // diagonal tile: only entries with col <= row
    int ch_begin, ch_end; // reduction chunks of this CTA
    int h;                // which 32-column quarter of the B block
    int split;            // which part of a split reduction (OZ_REV_ROW)
};

template <int MODE>
__device__ __forceinline__ OzJob oz_job(const OzArgs& g, int job, int& p0, int& p1) {
    OzJob o{};
    o.h = job % kParts;
    const int t = job / kParts;
    if (MODE == OZ_FWD_TRAIL) {
        int i, j;
        if (g.sub == 1) {
            i = t;
            j = 0;
        } else {
            tri_index(t, i, j);
        }
        const int off = g.sub == 2 ? 1 : 0;
        const int I = g.step + 1 + off + i, J = g.step + 1 + off + j;
        o.out_r0 = I * kT;
        o.out_c0 = J * kT + o.h * kN;
        o.lower = I == J;
        o.ch_begin = 0;
        o.ch_end = 1;
        p0 = I;  // A: row-slice block I, B: row-slice block J
        p1 = J;
    } else if (MODE == OZ_REV_ROW) {
        const int K = g.k_lo + t / g.splits;  // K <= J
        o.split = t % g.splits;
        o.out_r0 = g.step * kT;
        o.out_c0 = K * kT + o.h * kN;
        o.lower = K == g.step;
        const int chunks = g.nt - g.step - 1;
        const int per = (chunks + g.splits - 1) / g.splits;
        o.ch_begin = o.split * per;
        o.ch_end = min(chunks, o.ch_begin + per);
        p0 = K;
        p1 = 0;
    } else if (MODE == OZ_ASSIGN) {
        const int I = g.step + 1 + t;
        o.out_r0 = I * kT;
        o.out_c0 = g.step * kT + o.h * kN;
        o.lower = false;
        o.ch_begin = 0;
        o.ch_end = 1;
        p0 = I;
        p1 = 0;
    } else {
        const int J = g.step;
        // I >= J and K < J; or only K = J - 1 (sub 1); or only K < J - 1 (sub 2)
        const int kw = g.sub == 0 ? J : (g.sub == 1 ? 1 : J - 1);
        const int I = J + t / kw, K = t % kw + (g.sub == 1 ? J - 1 : 0);
        o.out_r0 = I * kT;
        o.out_c0 = K * kT + o.h * kN;
        o.lower = false;
        o.ch_begin = 0;
        o.ch_end = 1;
        p0 = I;
        p1 = K;
    }
    return o;
}

// Operand blocks of chunk `ch` of a job (element offsets within a batch entry).
template <int MODE>
__device__ __forceinline__ void oz_chunk(const OzArgs& g, int p0, int p1, int ch, size_t& ablk,
                                         size_t& eaoff, size_t& bblk, size_t& eboff) {
    if (MODE == OZ_FWD_TRAIL) {
        ablk = (size_t)p0 * kBlockElems;
        eaoff = (size_t)p0 * kT;
        bblk = (size_t)p1 * kBlockElems;
        eboff = (size_t)p1 * kT;
    } else if (MODE == OZ_REV_ROW) {
        const int c = g.step + 1 + ch;       // reduction chunk: rows c*128 ..
        ablk = (size_t)c * kBlockElems;      // column slices of C, chunk c
        eaoff = (size_t)c * kT;
        const size_t slot = (size_t)c * (c + 1) / 2 + p0;  // column slices of L, (c, K)
        bblk = slot * kBlockElems;
        eboff = slot * kT;
    } else if (MODE == OZ_ASSIGN) {
        ablk = (size_t)p0 * kBlockElems;     // row slices of the panel, block I
        eaoff = (size_t)p0 * kT;
        bblk = 0;                            // slices of the inverse (one block)
        eboff = 0;
    } else {
        ablk = (size_t)p0 * kBlockElems;     // row slices of Chat, block I
        eaoff = (size_t)p0 * kT;
        const size_t slot = (size_t)g.step * (g.step + 1) / 2 + p1;  // L (J, K)
        bblk = slot * kBlockElems;
        eboff = slot * kT;
    }
}

// Warp 0 owns TMEM and (lane 0) issues the MMAs; warp 1 lane 0 issues the
// bulk copies; all eight warps run the epilogue: warp w reads TMEM lanes
// 32 (w % 4) .. + 31 (output rows 32 (w % 4) .. of the tile), columns
// 16 (w / 4) .. + 15 of the CTA's 32, so that four warps per scheduler hide
// the epilogue's latencies (two CTAs per SM, at most 128 registers a thread).
template <int MODE>
__global__ void __launch_bounds__(kOzThreads, 2)
oz_gemm_kernel(OzArgs g, uint32_t max_polls) {
    pdl_wait();
    extern __shared__ __align__(128) unsigned char smem_raw[];
    // full[kStages], empty[kStages], done
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw);
    uint64_t* full = bars;
    uint64_t* empty = bars + kStages;
    uint64_t* done = bars + 2 * kStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + 64);
    unsigned char* stages = smem_raw + 128;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3;                // TMEM lane quadrant
    const int cw = (warp >> 2) * kWarpCols;   // first of this warp's output columns
    const int rl = quad * 32 + lane;          // this thread's row of the tile
    const uint32_t tlane = (uint32_t)(quad * 32) << 16;

    int p0 = 0, p1 = 0;
    const OzJob job = oz_job<MODE>(g, blockIdx.x, p0, p1);
    if (job.out_c0 >= g.n || job.out_r0 >= g.n || job.ch_begin >= job.ch_end) return;  // uniform
    // A split reduction writes its partial sums (positive) to its own 128 x 128
    // tile of g.part; otherwise the product is subtracted from the output.
    const bool partial = MODE == OZ_REV_ROW && g.splits > 1;

    if (tid == 0) {
        for (int i = 0; i < 2 * kStages + 1; ++i) mbar_init(bars + i, 1);
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

    uint32_t it = 0;   // reduction chunks handled by this CTA
    bool failed = false;
    for (int64_t b = blockIdx.y; b < g.batch && !failed; b += gridDim.y) {
        if (g.status != nullptr && g.status[b] != 0) continue;  // uniform
        double* out = g.out + (size_t)b * g.n * g.n;
        size_t ld = (size_t)g.n;
        int dst_r0 = 0, dst_c0 = 0;
        if (partial) {
            out = g.part +
                  (((size_t)b * g.splits + job.split) * g.k_n + (p0 - g.k_lo)) * kT * kT;
            ld = kT;
            dst_r0 = job.out_r0;
            dst_c0 = p0 * kT;
        }
        // The single-chunk updates (row per lane, below) read each lane's
        // output row segment (cold rows of L or W) before the MMAs finish: an
        // L2 prefetch of it here, which blocks no thread, then the loads into
        // registers just before the wait for the accumulators, so the
        // read-modify-write no longer waits on HBM after the MMAs.
        constexpr bool kRowMode = !(MODE == OZ_REV_ROW || MODE == OZ_ASSIGN);
        double rowv[kRowMode ? kWarpCols : 1];
        if constexpr (kRowMode) {
            // one 128-byte line: 16 doubles from a multiple of 16 columns
            const int row = job.out_r0 + rl;
            if (row < g.n && job.out_c0 + cw < g.n)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(out + (size_t)row * ld +
                                                              job.out_c0 + cw));
        }
        // staged modes: the running values of this thread's outputs across the
        // reduction chunks of the job (the old value minus the chunks so far, or
        // the partial sum), in registers: the output is read before the first
        // chunk and written after the last one
        constexpr bool kStagedMode = MODE == OZ_REV_ROW || MODE == OZ_ASSIGN;
        constexpr int kPasses = kWarpCols / kEC;
        double ov[kStagedMode ? kPasses : 1][kEC];
        for (int ch = job.ch_begin; ch < job.ch_end; ++ch, ++it) {
            const bool first = ch == job.ch_begin;
            const bool last = ch == job.ch_end - 1;
            size_t ablk, eaoff, bblk, eboff;
            oz_chunk<MODE>(g, p0, p1, ch, ablk, eaoff, bblk, eboff);
            const bf16* blkA = g.a + b * g.a_stride + ablk;
            const bf16* blkB = g.b + b * g.b_stride + bblk + job.h * (kN * kKC);
            if (tid == 32) {
                // producer: the stages of this chunk, through a ring of kStages
                for (int kc = 0; kc < kChunks; ++kc) {
                    const uint32_t i_ = it * kChunks + kc;
                    const uint32_t s_ = i_ % kStages, u = i_ / kStages;
                    if (u > 0 && !mbar_wait(empty + s_, (u - 1) & 1, max_polls)) {
                        failed = true;
                        break;
                    }
                    unsigned char* st = stages + s_ * kStageBytes;
                    mbar_arrive_expect_tx(full + s_, kStageBytes);
                    bulk_load(st, blkA + (size_t)kc * kS * kSliceElems, kStageA, full + s_);
                    for (int q = 0; q < kS; ++q)
                        bulk_load(st + kStageA + q * (kN * kKC * 2),
                                  blkB + (size_t)kc * kS * kSliceElems + (size_t)q * kSliceElems,
                                  kN * kKC * 2, full + s_);
                }
            } else if (tid == 0) {
                // MMA issuer: acc_d = sum_{p+q=d} D_p(A) D_q(B)^T over the chunk
                for (int kc = 0; kc < kChunks && !failed; ++kc) {
                    const uint32_t i_ = it * kChunks + kc;
                    const uint32_t s_ = i_ % kStages, u = i_ / kStages;
                    if (!mbar_wait(full + s_, u & 1, max_polls)) {
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(stages + s_ * kStageBytes);
                    const uint32_t sb = sa + kStageA;
                    // The stage holds B's slices stacked (slice q in rows
                    // 32q .. 32q + 31 of one K-major operand), so the product
                    // of D_p(A) with slices 0 .. 6-p (N = 32 (7 - p)) puts
                    // slice q's part in TMEM columns 32 (p + q) .., which is
                    // accumulator p + q: 7 MMAs per 16-step instead of 28,
                    // each reading its A slice from shared memory once.  The
                    // first (p = 0) initialises all 7 accumulators.
#pragma unroll
                    for (int p = 0; p < kS; ++p) {
#pragma unroll
                        for (int ks = 0; ks < kKC / 16; ++ks) {
                            const uint64_t da =
                                smem_desc(sa + p * (kSliceElems * 2) + ks * 256, 128, kSbo);
                            const uint64_t db = smem_desc(sb + ks * 256, 128, kSbo);
                            tc_mma(tmem + p * kN, da, db, mma_idesc((kS - p) * kN),
                                   (kc | p | ks) != 0);
                        }
                    }
                    tc_commit(empty + s_);  // the stage may be refilled once these finish
                }
                if (!failed) tc_commit(done);
            }
            // epilogue.  Two layouts of the output accesses, chosen per mode
            // by measurement (8192 x 8192 float64 step, ncu launch lists):
            // - the trailing and adjoint updates (one chunk per CTA, a
            //   read-modify-write of rows of L or W that come cold from HBM)
            //   keep the accumulators' row-per-lane layout: each lane walks
            //   its own row, so after the first access of a line the next
            //   ones hit in L1;
            // - the split row update (partial tiles, hot in L2 or written
            //   without a read) and the panel solves (written without a read)
            //   go through the stage buffers in passes of kEC = 8 columns, so
            //   the output is written by whole 64-byte row segments, after the
            //   job's last chunk; the old values are read 8 at a time (lane l
            //   on column l % 8 of row l / 8 of each group of 4 rows), all of
            //   them before the first chunk's accumulators are ready.
            constexpr bool kStaged = MODE == OZ_REV_ROW || MODE == OZ_ASSIGN;
            // Row per lane, a whole 16-column segment of an off-diagonal tile
            // with 32-byte aligned rows: the old values and the results move
            // four doubles at a time (each warp-wide access touches 32 rows'
            // lines, so fewer accesses mean fewer L1 wavefronts).
            const bool vec = !kStaged && !job.lower && job.out_c0 + cw + kWarpCols <= g.n &&
                             ld % 4 == 0 && (reinterpret_cast<uintptr_t>(out) & 31) == 0;
            const int wrow0 = job.out_r0 + quad * 32;
            const int ecol = lane % kEC;
            const bool need_old = MODE != OZ_ASSIGN && !partial;
            auto out_at = [&](int cc, int i, bool& ok) -> double* {
                const int r = wrow0 + kEpR * i + lane / kEC;
                const int col = job.out_c0 + cw + cc * kEC + ecol;
                ok = r < g.n && col < g.n && !(job.lower && col > r);
                return out + (size_t)(r - dst_r0) * ld + (col - dst_c0);
            };
            // (the MMA-issuing and copy-issuing lanes finish their loops first,
            // so their warps do not split between those loops and these loads)
            __syncwarp();
            if constexpr (kStaged) {
                // every pass's old values, in flight while the first chunk's
                // MMAs finish
                if (first) {
#pragma unroll
                    for (int cc = 0; cc < kPasses; ++cc)
#pragma unroll
                        for (int i = 0; i < kEC; ++i) {
                            bool okf;
                            const double* o = out_at(cc, i, okf);
                            ov[cc][i] = (need_old && okf) ? *o : 0.0;
                        }
                }
            } else if (vec) {
                const int row = job.out_r0 + rl;
                const double* seg = out + (size_t)row * ld + job.out_c0 + cw;
#pragma unroll
                for (int q = 0; q < kWarpCols / 4; ++q) {
                    double t[4] = {0.0, 0.0, 0.0, 0.0};
                    if (row < g.n) ld_global_v4(seg + 4 * q, t);
#pragma unroll
                    for (int e = 0; e < 4; ++e) rowv[4 * q + e] = t[e];
                }
            } else {
                const int row = job.out_r0 + rl;
                const double* orow = out + (size_t)row * ld;
#pragma unroll
                for (int j = 0; j < kWarpCols; ++j) {
                    const int col = job.out_c0 + cw + j;
                    rowv[j] =
                        (row < g.n && col < g.n && !(job.lower && col > row)) ? orow[col] : 0.0;
                }
            }
            const bool ok = __syncthreads_and(!failed) && mbar_wait(done, it & 1, max_polls);
            tc_fence_after();
            if (!__all_sync(0xffffffffu, ok)) {
                if (tid == 0 && g.fail != nullptr) g.fail[b] = -1;  // reported, not hung
                failed = true;
            } else if constexpr (kStaged) {
                const int32_t* ea = g.ea + b * g.ea_stride + eaoff;
                const int32_t* eb = g.eb + b * g.eb_stride + eboff + job.h * kN + cw;
                const int er = ea[rl];
                double* stg = reinterpret_cast<double*>(stages) + warp * (32 * kEpP);
#pragma unroll
                for (int cc = 0; cc < kPasses; ++cc) {
                    int ecv[kEC];
#pragma unroll
                    for (int j = 0; j < kEC; ++j) ecv[j] = eb[cc * kEC + j];
                    uint32_t acc[kS][kEC];
#pragma unroll
                    for (int d = 0; d < kS; ++d)
                        tc_ld8(tmem + tlane + d * kN + cw + cc * kEC, acc[d]);
                    tc_wait_ld();
#pragma unroll
                    for (int j = 0; j < kEC; ++j)
                        stg[lane * kEpP + j] =
                            (er == kNonFinite || ecv[j] == kNonFinite)
                                ? __longlong_as_double(0x7ff8000000000000LL)  // NaN
                                : scale_int(combine_acc(acc, j), er + ecv[j] - 62);
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < kEC; ++i) {
                        bool oks;
                        double* o = out_at(cc, i, oks);
                        const double t = stg[(kEpR * i + lane / kEC) * kEpP + ecol];
                        ov[cc][i] = MODE == OZ_ASSIGN
                                        ? t
                                        : (partial ? (first ? t : ov[cc][i] + t) : ov[cc][i] - t);
                        if (oks && last) *o = ov[cc][i];
                    }
                    __syncwarp();
                }
                // the staging writes and reads (generic proxy) come before the
                // next chunk's bulk copies into the same buffers (async proxy)
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            } else {
                // out = old - v 2^E, row per lane, the old values from rowv
                const int32_t* ea = g.ea + b * g.ea_stride + eaoff;
                const int32_t* eb = g.eb + b * g.eb_stride + eboff + job.h * kN + cw;
                const int er = ea[rl];
                const int row = job.out_r0 + rl;
                double* orow = out + (size_t)row * ld;
#pragma unroll
                for (int cc = 0; cc < kWarpCols / kEC; ++cc) {
                    // the column exponents first: their loads overlap the TMEM reads
                    int ecv[kEC];
#pragma unroll
                    for (int j = 0; j < kEC; ++j) ecv[j] = eb[cc * kEC + j];
                    uint32_t acc[kS][kEC];
#pragma unroll
                    for (int d = 0; d < kS; ++d) tc_ld8(tmem + tlane + d * kN + cw + cc * kEC, acc[d]);
                    tc_wait_ld();
                    if (row >= g.n) continue;
                    if (vec) {
                        double* seg = orow + job.out_c0 + cw + cc * kEC;
#pragma unroll
                        for (int q = 0; q < kEC / 4; ++q) {
                            double nv[4];
                            bool changed = false;
#pragma unroll
                            for (int h2 = 0; h2 < 4; ++h2) {
                                const int j = 4 * q + h2;
                                const long long v = combine_acc(acc, j);
                                nv[h2] = rowv[cc * kEC + j];
                                if (er == kNonFinite || ecv[j] == kNonFinite) {
                                    nv[h2] = __longlong_as_double(0x7ff8000000000000LL);  // NaN
                                    changed = true;
                                } else if (v != 0) {
                                    nv[h2] -= scale_int(v, er + ecv[j] - 62);
                                    changed = true;
                                }
                            }
                            if (changed) st_global_v4(seg + 4 * q, nv);
                        }
                        continue;
                    }
#pragma unroll
                    for (int j = 0; j < kEC; ++j) {
                        const int col = job.out_c0 + cw + cc * kEC + j;
                        if (col >= g.n || (job.lower && col > row)) continue;
                        const long long v = combine_acc(acc, j);
                        if (er == kNonFinite || ecv[j] == kNonFinite)
                            orow[col] = __longlong_as_double(0x7ff8000000000000LL);  // NaN
                        else if (v != 0)
                            orow[col] = rowv[cc * kEC + j] - scale_int(v, er + ecv[j] - 62);
                    }
                }
            }
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            if (failed) break;
        }
    }
    if (failed && tid == 32) {
        // let copies still in flight land before the block retires
        for (int s = 0; s < kStages; ++s) mbar_wait(full + s, 0, max_polls);
    }
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

inline unsigned gy(int64_t batch) { return (unsigned)std::min<int64_t>(batch, 65535); }

template <int MODE>
cudaError_t launch_oz(const OzArgs& g, unsigned jobs, cudaStream_t stream) {
    if (jobs == 0) return cudaSuccess;
    static std::atomic<uint64_t> attr_set{0};
    cudaError_t e = once_per_device(attr_set, [] {
        cudaError_t r = cudaFuncSetAttribute(oz_gemm_kernel<MODE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kGemmSmem);
        // the whole unified L1 / shared array as shared memory, so two CTAs fit
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(oz_gemm_kernel<MODE>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        return r;
    });
    if (e != cudaSuccess) return e;
    return launch_pdl(oz_gemm_kernel<MODE>, dim3(jobs, gy(g.batch)), dim3(kOzThreads), kGemmSmem,
                      stream, g, (uint32_t)kMbarPolls);
}

constexpr size_t kColSmem = (size_t)kT * (kColW + 1) * sizeof(double);

cudaError_t launch_slice_rows2(const RowSlice& s0, const RowSlice& s1, const int32_t* status,
                               int64_t batch, cudaStream_t stream) {
    const int64_t rows = (int64_t)std::max(s0.nrows, 0) + std::max(s1.nrows, 0);
    if (rows <= 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((rows * 32 + 255) / 256);
    return launch_pdl(slice_rows_kernel, dim3(blocks, gy(batch)), dim3(256), 0, stream, s0, s1,
                      status, batch);
}

cudaError_t launch_slice_rows(const double* src, bf16* dst, int32_t* ex, const int32_t* status,
                              int64_t batch, int n, int row0, int nrows, int col0, bool sym,
                              size_t dst_stride, size_t ex_stride, Bal bal, cudaStream_t stream) {
    if (nrows <= 0) return cudaSuccess;
    const RowSlice s0{src, dst, ex, n, row0, nrows, col0, sym, dst_stride, ex_stride, bal};
    const RowSlice s1{nullptr, nullptr, nullptr, 0, 0, 0, 0, false, 0, 0, Bal{nullptr, 0, 0, 0}};
    return launch_slice_rows2(s0, s1, status, batch, stream);
}

cudaError_t launch_slice_cols(const double* src, bf16* dst, int32_t* ex, const int32_t* status,
                              int64_t batch, int n, int c_begin, unsigned count, bool tri,
                              int k_fixed, bool lower_only, size_t dst_stride, size_t ex_stride,
                              Bal bal, cudaStream_t stream) {
    if (count == 0) return cudaSuccess;
    static std::atomic<uint64_t> smem_set{0};
    cudaError_t e = allow_smem_once(slice_cols_kernel, kColSmem, smem_set);
    if (e != cudaSuccess) return e;
    return launch_pdl(slice_cols_kernel, dim3(count * kColGroups, gy(batch)), dim3(kColThreads),
                      kColSmem, stream, src, dst, ex, status, batch, n, c_begin, tri, k_fixed,
                      lower_only, dst_stride, ex_stride, bal);
}

inline int tiles_of(int n) { return (n + kT - 1) / kT; }

// W_JK -= sum_s part[s][K] for K <= J (lower part of the diagonal tile),
// the partial sums added in split order, so the result does not depend on
// which CTA finished first.
__global__ void __launch_bounds__(256)
split_reduce_kernel(double* __restrict__ W, const double* __restrict__ part,
                    const int32_t* __restrict__ status, int64_t batch, int n, int J, int splits,
                    int k_lo, int k_n) {
    pdl_wait();
    const int64_t per = (int64_t)k_n * kT * kT;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < batch * per;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = e / per;
        if (status != nullptr && status[b] != 0) continue;
        const int64_t w = e % per;
        const int K = k_lo + (int)(w / (kT * kT)), m = (int)((w / kT) % kT), c = (int)(w % kT);
        const int row = J * kT + m, col = K * kT + c;
        if (row >= n || col >= n || (K == J && c > m)) continue;
        double s = 0.0;
        for (int sp = 0; sp < splits; ++sp) s += part[((b * splits + sp) * k_n) * kT * kT + w];
        W[(size_t)b * n * n + (size_t)row * n + col] -= s;
    }
}

// Split of OZ_REV_ROW's reduction: about one split tile per SM (four
// quarter-tile CTAs per SM, two waves at two CTAs per SM; half as many
// measured slower), the partial tiles bounded by 2 * SMs per call.
inline int row_splits(int64_t batch, int k_n, int chunks) {
    const int64_t tiles = batch * k_n;
    const int64_t want = (2 * (int64_t)device_sm_count() + 2 * tiles - 1) / (2 * tiles);
    return (int)std::max<int64_t>(1, std::min<int64_t>(want, chunks));
}

inline size_t part_elems() { return (size_t)2 * (device_sm_count() + 1) * kT * kT; }

// Adjoint workspace, per batch entry: column slices of L (all (c, K <= c)),
// column slices of C (one block per chunk), row slices of Chat (one block per
// row block), then the three exponent arrays.
// Bump layout of a workspace: every region 256-byte aligned.
struct Carve {
    uintptr_t p;
    template <typename X>
    X* take(size_t count) {
        X* r = reinterpret_cast<X*>(p);
        p += (count * sizeof(X) + 255) / 256 * 256;
        return r;
    }
};

// Inverses of diagonal tiles and what slices them (per batch entry: `count`
// 128 x 128 float64 matrices, operand blocks and their exponents), and the
// balancing exponents of every row (nt * 128 per batch entry).
struct InvWs {
    double* inv;
    bf16* sl;
    int32_t* ex;
    int32_t* bal;
};

template <typename C>
InvWs carve_inv(C& c, int64_t batch, int nt, int count) {
    InvWs w;
    w.inv = c.template take<double>((size_t)batch * count * kT * kT);
    w.sl = c.template take<bf16>((size_t)batch * count * kBlockElems);
    w.ex = c.template take<int32_t>((size_t)batch * count * kT);
    w.bal = c.template take<int32_t>((size_t)batch * nt * kT);
    return w;
}

// Forward workspace: row slices of the panel (nt blocks per batch entry) and
// their exponents, twice (step k uses set k % 2, so the trailing update of
// one step may still read its slices while the next step slices its panel),
// and the inverse parts.
struct FwdWs {
    bf16* rs[2];
    int32_t* ers[2];
    InvWs iv;
};

FwdWs fwd_layout(Carve& c, int64_t batch, int n) {
    const int nt = tiles_of(n);
    FwdWs w;
    for (int s = 0; s < 2; ++s) {
        w.rs[s] = c.take<bf16>((size_t)batch * nt * kBlockElems);
        w.ers[s] = c.take<int32_t>((size_t)batch * nt * kT);
    }
    w.iv = carve_inv(c, batch, nt, 1);
    return w;
}

FwdWs fwd_ws(void* work, int64_t batch, int n) {
    Carve c{reinterpret_cast<uintptr_t>(work)};
    return fwd_layout(c, batch, n);
}

// Adjoint workspace, per batch entry: column slices of L (all (c, K <= c)),
// column slices of C (one block per chunk), row slices of Chat (one block per
// row block), their exponents, the inverses of the diagonal tiles and their
// slices, and the partial sums of the split reduction.
struct AdjWs {
    // C column slices and Chat / C row slices: set J % 2 for tile column J
    bf16 *lc, *cc[2], *ch[2];
    int32_t *elc, *ecc[2], *ech[2];
    InvWs iv;
    double* part;   // partial sums of split reductions (part_elems()), the caller's stream
    double* part2;  // the same for the row update's part on the side stream
    double* lit;    // S and T of the literal diagonal-tile adjoint (2 x 128 x 128 per matrix)
    size_t lc_stride, cc_stride, ch_stride, elc_stride, ecc_stride, ech_stride;
};

// The adjoint inverts every diagonal tile up front, since L is fixed: one
// launch instead of one per tile column.  The inverses serve the panel solves
// (tiles 0 .. nt - 2) and the literal diagonal-tile adjoint (every tile).
inline int adj_inverses(int nt) { return nt; }

AdjWs adj_layout(uintptr_t base, int64_t batch, int n) {
    const size_t nt = tiles_of(n), ntri = nt * (nt + 1) / 2;
    AdjWs w{};
    w.lc_stride = ntri * kBlockElems;
    w.cc_stride = nt * kBlockElems;
    w.ch_stride = nt * kBlockElems;
    w.elc_stride = ntri * kT;
    w.ecc_stride = nt * kT;
    w.ech_stride = nt * kT;
    Carve c{base};
    w.lc = c.take<bf16>(batch * w.lc_stride);
    for (int s = 0; s < 2; ++s) w.cc[s] = c.take<bf16>(batch * w.cc_stride);
    for (int s = 0; s < 2; ++s) w.ch[s] = c.take<bf16>(batch * w.ch_stride);
    w.elc = c.take<int32_t>(batch * w.elc_stride);
    for (int s = 0; s < 2; ++s) w.ecc[s] = c.take<int32_t>(batch * w.ecc_stride);
    for (int s = 0; s < 2; ++s) w.ech[s] = c.take<int32_t>(batch * w.ech_stride);
    w.iv = carve_inv(c, batch, (int)nt, adj_inverses((int)nt));
    w.part = c.take<double>(part_elems());
    w.part2 = c.take<double>(part_elems());
    w.lit = c.take<double>((size_t)2 * batch * kT * kT);
    return w;
}

AdjWs adj_ws(void* work, int64_t batch, int n) {
    return adj_layout(reinterpret_cast<uintptr_t>(work), batch, n);
}

// ---------------------------------------------------------------------------
// Inverses of diagonal tiles G = L[k0 .. k0+kb, k0 .. k0+kb] (lower,
// kb <= 128), X = G^-1, tiles k = tile0 + blockIdx.z.  Column c of X solves
// G x = e_c by forward substitution in its right-looking (column) form on
// the rows scaled by 1 / g_ii: with H_im = g_im / g_ii and x_c = 1 / g_cc,
// x_m is final at step m and every row i > m takes acc_i -= H_im x_m, the lane
// owning row m handing x_m to the others by a shuffle.  The dependent chain
// per row is one shuffle and one fused multiply-add.  One warp per column at
// a time: an FP64 instruction occupies an SM sub-partition's FP64 unit for
// its whole warp, so columns spread over warps (and, for few matrices, over
// blocks) rather than rows over more lanes.  X is written as a 128 x 128
// matrix (zeros above the diagonal and beyond kb; all zeros for a matrix
// whose status is set).  With bal, block x = 0 also writes the balancing
// exponents ilogb(g_ii) of the tile's rows to bal[k0 + i].
// ---------------------------------------------------------------------------
constexpr size_t kInvSmem = ((size_t)kT * (kT + 1) + kT) * sizeof(double);

template <int WARPS>
__global__ void __launch_bounds__(WARPS * 32)
tri_inverse_kernel(const double* __restrict__ L, double* __restrict__ Inv,
                   int32_t* __restrict__ bal, const int32_t* __restrict__ status, int64_t batch,
                   int n, int nt, int tile0) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    constexpr int P = kT + 1;
    constexpr int Q = kT / 32;                        // rows per lane
    double* H = reinterpret_cast<double*>(smem_raw);  // kb x kb, pitch P
    double* rinv = H + (size_t)kT * P;                // 1 / g_ii
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k0 = (tile0 + (int)blockIdx.z) * kT;
    const int kb = min(kT, n - k0);
    // columns of this warp: blockIdx.x + gridDim.x * (warp + WARPS * t)
    const int cstep = (int)gridDim.x * WARPS;
    const int cfirst = (int)blockIdx.x + (int)gridDim.x * warp;
    for (int64_t b = blockIdx.y; b < batch; b += gridDim.y) {
        double* Ib = Inv + ((size_t)b * gridDim.z + blockIdx.z) * kT * kT;
        if (status != nullptr && status[b] != 0) {
            for (int c = cfirst; c < kT; c += cstep)
                for (int i = lane; i < kT; i += 32) Ib[(size_t)i * kT + c] = 0.0;
            continue;
        }
        const double* Lb = L + (size_t)b * n * n;
        __syncthreads();
        for (int i = threadIdx.x; i < kb; i += blockDim.x) {
            const double d = Lb[(size_t)(k0 + i) * n + k0 + i];
            rinv[i] = 1.0 / d;
            if (bal != nullptr && blockIdx.x == 0)
                bal[b * (size_t)nt * kT + k0 + i] = (d > 0.0 && isfinite(d)) ? ilogb(d) : 0;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < kb * kT; e += blockDim.x) {
            const int i = e / kT, j = e % kT;
            H[i * P + j] = j < i ? Lb[(size_t)(k0 + i) * n + k0 + j] * rinv[i] : 0.0;
        }
        __syncthreads();
        for (int c = cfirst; c < kT; c += cstep) {
            // acc[q] holds row lane + 32 q: 1 / g_cc at row c, then the
            // partial solve, then (from its own step on) the solution
            double acc[Q];
#pragma unroll
            for (int q = 0; q < Q; ++q) acc[q] = (lane + 32 * q == c && c < kb) ? rinv[c] : 0.0;
            for (int m = c; m < kb - 1; ++m) {
                const int slot = m >> 5;
                double v = acc[0];
#pragma unroll
                for (int q = 1; q < Q; ++q) v = slot == q ? acc[q] : v;
                const double xm = __shfl_sync(0xffffffffu, v, m & 31);
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    if (32 * q + 31 <= m) continue;  // (warp-uniform) no row of this slot is left
                    const int i = lane + 32 * q;
                    if (i > m && i < kb) acc[q] = fma(-H[i * P + m], xm, acc[q]);
                }
            }
#pragma unroll
            for (int q = 0; q < Q; ++q) {
                const int i = lane + 32 * q;
                Ib[(size_t)i * kT + c] = (c < kb && i >= c && i < kb) ? acc[q] : 0.0;
            }
        }
    }
}

// Inverts tiles tile0 .. tile0 + count - 1 of every matrix into
// Inv[b][t][128][128].  Few matrices: 4-warp blocks, the columns of a tile
// spread over up to 32 blocks (the dependent chains run side by side on
// different SMs); many: one 8-warp block per tile.
cudaError_t launch_tri_inverse(const double* L, double* Inv, int32_t* bal, const int32_t* status,
                               int64_t batch, int n, int tile0, int count, cudaStream_t stream) {
    const int64_t tiles = batch * count;
    int gx = 1;
    while (gx < 32 && tiles * gx * 2 <= device_sm_count()) gx *= 2;
    const dim3 grid((unsigned)gx, gy(batch), (unsigned)count);
    if (gx > 1) {
        static std::atomic<uint64_t> smem_set{0};
        cudaError_t e = allow_smem_once(tri_inverse_kernel<4>, kInvSmem, smem_set);
        if (e != cudaSuccess) return e;
        tri_inverse_kernel<4><<<grid, 128, kInvSmem, stream>>>(L, Inv, bal, status, batch, n,
                                                              tiles_of(n), tile0);
    } else {
        static std::atomic<uint64_t> smem_set{0};
        cudaError_t e = allow_smem_once(tri_inverse_kernel<8>, kInvSmem, smem_set);
        if (e != cudaSuccess) return e;
        tri_inverse_kernel<8><<<grid, 256, kInvSmem, stream>>>(L, Inv, bal, status, batch, n,
                                                              tiles_of(n), tile0);
    }
    return cudaGetLastError();
}

// bal[b][r] = ilogb(L_rr) (0 where L_rr is not a positive number, and for
// r >= n), r < nt * 128.
__global__ void __launch_bounds__(256)
diag_exp_kernel(const double* __restrict__ L, int32_t* __restrict__ bal,
                const int32_t* __restrict__ status, int64_t batch, int n, int nt) {
    const int64_t per = (int64_t)nt * kT;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < batch * per;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = e / per;
        const int r = (int)(e % per);
        int s = 0;
        if (r < n && !(status != nullptr && status[b] != 0)) {
            const double d = L[(size_t)b * n * n + (size_t)r * n + r];
            if (d > 0.0 && isfinite(d)) s = ilogb(d);
        }
        bal[e] = s;
    }
}

// ---------------------------------------------------------------------------
// Adjoint of one diagonal tile by its literal formula (warp issue #1316,
// closing comment): with G = L_JJ, X = G^-1 (inverted up front) and W_JJ the
// gradient with respect to G's lower entries,
//   S = Phi(G^T W_JJ),  T = S X,  M = X^T T,  W_JJ <- Phi(M + M^T),
// Phi keeping the lower triangle and halving the diagonal.  This is the
// gradient the reverse sweep reaches column by column, but as three products
// with no dependent chain: for few matrices the sweep's 128-step chain on one
// SM costs far more than the formula's 2.5x larger FP64 work spread over
// 136 blocks.  S, T and every operand are lower triangular, so each sum runs
// only where both factors can be non-zero.
//
// One block per 8 x 8 output block (ba, bb), ba >= bb, of the tile's lower
// part; 256 threads = 64 outputs x 4 groups that split the reduction index
// (interleaved) and add their partial sums in a fixed order.  The operand
// strips the block needs (at most 128 x 8 per operand) are staged in shared
// memory first.  S and T live in a scratch area of 128 x 128 per matrix.
// ---------------------------------------------------------------------------
constexpr int kLB = 8;
constexpr int kLitThreads = 256;
enum LitStep { LIT_S = 0, LIT_T = 1, LIT_A = 2 };

template <int STEP>
__global__ void __launch_bounds__(kLitThreads)
lit_diag_kernel(const double* __restrict__ L, double* __restrict__ W,
                const double* __restrict__ X, size_t x_stride, double* __restrict__ S,
                double* __restrict__ Tm, const int32_t* __restrict__ status, int64_t batch, int n,
                int j0, int kb) {
    pdl_wait();
    __shared__ double sA[kT * kLB], sB[kT * kLB], sC[kT * kLB], sD[kT * kLB];
    __shared__ double red[4][kLB * kLB];
    int ba, bb;
    tri_index((int)blockIdx.x, ba, bb);
    const int tid = threadIdx.x, g = tid >> 6, o = tid & 63, ty = o >> 3, tx = o & 7;
    const int a = kLB * ba + ty, bcol = kLB * bb + tx;
    const int a0 = kLB * ba, b0 = kLB * bb;
    // reduction range [c_lo, c_hi)
    const int c_lo = STEP == LIT_T ? b0 : a0;
    const int c_hi = STEP == LIT_T ? min(a0 + kLB, kb) : kb;
    const int len = c_hi - c_lo;
    for (int64_t b = blockIdx.y; b < batch; b += gridDim.y) {
        if (status != nullptr && status[b] != 0) continue;
        const double* Lb = L + b * (size_t)n * n;
        double* Wb = W + b * (size_t)n * n;
        const double* Xb = X + b * x_stride;
        double* Sb = S + b * (size_t)kT * kT;
        double* Tb = Tm + b * (size_t)kT * kT;
        __syncthreads();
        // strips: element [c'][i] for c = c_lo + c', i < 8
        for (int e = tid; e < len * kLB; e += kLitThreads) {
            const int cc = e / kLB, i = e % kLB, c = c_lo + cc;
            const int ra = a0 + i, rb = b0 + i;
            if (STEP == LIT_S) {
                // G_c,a (c >= a) and W_c,b (c >= b), inside the tile
                sA[e] = (ra < kb && c >= ra) ? Lb[(size_t)(j0 + c) * n + j0 + ra] : 0.0;
                sB[e] = (rb < kb && c >= rb) ? Wb[(size_t)(j0 + c) * n + j0 + rb] : 0.0;
            } else if (STEP == LIT_T) {
                // S_a,c (c <= a) and X_c,b (c >= b)
                sA[e] = (ra < kb && c <= ra) ? Sb[(size_t)ra * kT + c] : 0.0;
                sB[e] = (rb < kb && c >= rb) ? Xb[(size_t)c * kT + rb] : 0.0;
            } else {
                // X_c,a, T_c,b, X_c,b, T_c,a (all lower: zero for c above)
                sA[e] = (ra < kb && c >= ra) ? Xb[(size_t)c * kT + ra] : 0.0;
                sB[e] = (rb < kb && c >= rb) ? Tb[(size_t)c * kT + rb] : 0.0;
                sC[e] = (rb < kb && c >= rb) ? Xb[(size_t)c * kT + rb] : 0.0;
                sD[e] = (ra < kb && c >= ra) ? Tb[(size_t)c * kT + ra] : 0.0;
            }
        }
        __syncthreads();
        double acc = 0.0;
        if (STEP == LIT_A) {
            const bool diag = a == bcol;
            for (int cc = g; cc < len; cc += 4) {
                acc = fma(sA[cc * kLB + ty], sB[cc * kLB + tx], acc);
                if (!diag) acc = fma(sC[cc * kLB + tx], sD[cc * kLB + ty], acc);
            }
        } else {
            for (int cc = g; cc < len; cc += 4) acc = fma(sA[cc * kLB + ty], sB[cc * kLB + tx], acc);
        }
        red[g][o] = acc;
        __syncthreads();
        if (g == 0 && a < kb && bcol < kb) {
            const double v = (red[0][o] + red[1][o]) + (red[2][o] + red[3][o]);
            if (STEP == LIT_S) {
                Sb[(size_t)a * kT + bcol] = a > bcol ? v : (a == bcol ? 0.5 * v : 0.0);
            } else if (STEP == LIT_T) {
                Tb[(size_t)a * kT + bcol] = a >= bcol ? v : 0.0;
            } else if (a >= bcol) {
                Wb[(size_t)(j0 + a) * n + j0 + bcol] = v;
            }
        }
    }
}

}  // namespace

// ---------------------------------------------------------------------------
// Forward, step k: the panel solve and the trailing update.  Workspace: row
// slices of the panel, their exponents, the inverse of the diagonal tile and
// its slices, the balancing exponents.
// ---------------------------------------------------------------------------
size_t ozaki_workspace_bytes(int64_t batch, int n) {
    Carve c{0};
    fwd_layout(c, batch, n);
    return (size_t)c.p;
}

void ozaki_fwd_inverse(void* work, int64_t batch, int n, double** inv, int32_t** bal) {
    const FwdWs w = fwd_ws(work, batch, n);
    *inv = w.iv.inv;
    *bal = w.iv.bal;
}

cudaError_t ozaki_panel_solve(double* L, void* work, int32_t* status, int64_t batch, int n,
                              int k, bool have_inverse, cudaStream_t stream) {
    const int nt = tiles_of(n);
    const int m = nt - k - 1;
    if (m <= 0) return cudaSuccess;
    const FwdWs w = fwd_ws(work, batch, n);
    const size_t stride = (size_t)nt * kBlockElems, estride = (size_t)nt * kT;
    const size_t bstride = (size_t)nt * kT;
    // G^-1 of the (full) diagonal tile, and the balancing exponents of its rows
    cudaError_t e = have_inverse
                        ? cudaSuccess
                        : launch_tri_inverse(L, w.iv.inv, w.iv.bal, status, batch, n, k, 1, stream);
    if (e != cudaSuccess) return e;
    // L_Ik <- L_Ik G^-T: A = the panel's rows (reduction over the tile's
    // columns, divided by the balancing factors), B = rows of G^-1 (multiplied)
    // (both in one launch: the panel's rows, then the inverse's)
    bf16* rs = w.rs[k & 1];
    int32_t* ers = w.ers[k & 1];
    const RowSlice panel{L, rs, ers, n, (k + 1) * kT, m * kT, k * kT, false, stride, estride,
                         Bal{w.iv.bal, bstride, 0, -1}};
    const RowSlice ginv{w.iv.inv, w.iv.sl, w.iv.ex, kT, 0, kT, 0, false, kBlockElems, kT,
                        Bal{w.iv.bal, bstride, k * kT, 1}};
    e = launch_slice_rows2(panel, ginv, status, batch, stream);
    if (e != cudaSuccess) return e;
    OzArgs g{L, rs, ers, w.iv.sl, w.iv.ex, stride, estride, kBlockElems, kT, status, status,
             batch, n, nt, k, 1, nullptr};
    return launch_oz<OZ_ASSIGN>(g, (unsigned)(kParts * m), stream);
}

cudaError_t ozaki_trailing_slice(double* L, void* work, int32_t* status, int64_t batch, int n,
                                 int k, cudaStream_t stream) {
    const int nt = tiles_of(n);
    const int m = nt - k - 1;
    if (m <= 0) return cudaSuccess;
    const FwdWs w = fwd_ws(work, batch, n);
    const size_t stride = (size_t)nt * kBlockElems, estride = (size_t)nt * kT;
    return launch_slice_rows(L, w.rs[k & 1], w.ers[k & 1], status, batch, n, (k + 1) * kT,
                             m * kT, k * kT, false, stride, estride, Bal{nullptr, 0, 0, 0},
                             stream);
}

cudaError_t ozaki_trailing_gemm(double* L, void* work, int32_t* status, int64_t batch, int n,
                                int k, int part, cudaStream_t stream) {
    const int nt = tiles_of(n);
    const int m = nt - k - 1;
    // tiles: all m (m + 1) / 2, the m of block column k + 1, or the rest
    const int tiles = part == 0 ? m * (m + 1) / 2 : (part == 1 ? m : (m - 1) * m / 2);
    if (m <= 0 || tiles <= 0) return cudaSuccess;
    const FwdWs w = fwd_ws(work, batch, n);
    const size_t stride = (size_t)nt * kBlockElems, estride = (size_t)nt * kT;
    OzArgs g{L, w.rs[k & 1], w.ers[k & 1], w.rs[k & 1], w.ers[k & 1], stride, estride, stride,
             estride, status, status, batch, n, nt, k, 1, nullptr, part};
    return launch_oz<OZ_FWD_TRAIL>(g, (unsigned)(kParts * tiles), stream);
}

cudaError_t ozaki_trailing_update(double* L, void* work, int32_t* status, int64_t batch, int n,
                                  int k, cudaStream_t stream) {
    cudaError_t e = ozaki_trailing_slice(L, work, status, batch, n, k, stream);
    if (e != cudaSuccess) return e;
    return ozaki_trailing_gemm(L, work, status, batch, n, k, 0, stream);
}

// ---------------------------------------------------------------------------
// Adjoint (Murray's blocked reverse sweep, see blocked_adj): the column
// slices of L and the balancing exponents once, then per tile column J the
// panel solve and the two contractions.
// ---------------------------------------------------------------------------
size_t ozaki_adj_workspace_bytes(int64_t batch, int n) {
    const AdjWs w = adj_layout(0, batch, n);
    return reinterpret_cast<uintptr_t>(w.lit + (size_t)2 * batch * kT * kT) + 256;
}

cudaError_t ozaki_adj_prepare(const double* L, void* work, const int32_t* status, int64_t batch,
                              int n, cudaStream_t stream) {
    const int nt = tiles_of(n);
    const AdjWs w = adj_ws(work, batch, n);
    const size_t bstride = (size_t)nt * kT;
    const int64_t total = batch * (int64_t)bstride;
    diag_exp_kernel<<<(unsigned)std::min<int64_t>((total + 255) / 256,
                                                  (int64_t)device_sm_count() * 16),
                      256, 0, stream>>>(L, w.iv.bal, status, batch, n, nt);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // L's rows divided by their balancing factors (the gradient operands are
    // multiplied by the same ones)
    e = launch_slice_cols(L, w.lc, w.elc, status, batch, n, 0, (unsigned)(nt * (nt + 1) / 2),
                          true, 0, true, w.lc_stride, w.elc_stride,
                          Bal{w.iv.bal, bstride, 0, -1}, stream);
    if (e != cudaSuccess) return e;
    // L_JJ^-1 for every tile column J and its column slices (the inverses,
    // batch * nt matrices of order 128, are zeros for a matrix whose status
    // is set)
    const int cnt = adj_inverses(nt);
    e = launch_tri_inverse(L, w.iv.inv, nullptr, status, batch, n, 0, cnt, stream);
    if (e != cudaSuccess) return e;
    return launch_slice_cols(w.iv.inv, w.iv.sl, w.iv.ex, nullptr, batch * cnt, kT, 0, 1, false, 0,
                             false, kBlockElems, kT, Bal{nullptr, 0, 0, 0}, stream);
}

cudaError_t ozaki_adj_solve(const double* L, double* W, void* work, const int32_t* status,
                            int64_t batch, int n, int J, cudaStream_t stream) {
    const int nt = tiles_of(n);
    const int m = nt - J - 1;
    if (m <= 0) return cudaSuccess;
    const AdjWs w = adj_ws(work, batch, n);
    // C <- C L_JJ^-1: A = C's rows (reduction over the tile's columns), B =
    // columns of L_JJ^-1 (sliced up front); the inverse scales like C along
    // the reduction, so no balancing is needed here
    cudaError_t e = launch_slice_rows(W, w.ch[J & 1], w.ech[J & 1], status, batch, n,
                                      (J + 1) * kT, m * kT, J * kT, false, w.ch_stride,
                                      w.ech_stride,
                                      Bal{nullptr, 0, 0, 0}, stream);
    if (e != cudaSuccess) return e;
    const size_t cnt = (size_t)adj_inverses(nt);
    OzArgs g{W, w.ch[J & 1], w.ech[J & 1], w.iv.sl + (size_t)J * kBlockElems,
             w.iv.ex + (size_t)J * kT,
             w.ch_stride, w.ech_stride, cnt * kBlockElems, cnt * kT, status, nullptr, batch, n,
             nt, J, 1, nullptr};
    return launch_oz<OZ_ASSIGN>(g, (unsigned)(kParts * m), stream);
}

cudaError_t ozaki_adj_row(const double* L, double* W, void* work, const int32_t* status,
                          int64_t batch, int n, int J, int part, cudaStream_t stream) {
    (void)L;
    const int nt = tiles_of(n);
    if (J >= nt - 1) return cudaSuccess;
    // output block columns: all K <= J (part 0), K = J - 1 .. J (part 1), K < J - 1 (part 2)
    const int k_lo = part == 1 ? std::max(0, J - 1) : 0;
    const int k_hi = part == 2 ? J - 2 : J;
    if (k_hi < k_lo) return cudaSuccess;
    const int k_n = k_hi - k_lo + 1;
    const AdjWs w = adj_ws(work, batch, n);
    const size_t bstride = (size_t)nt * kT;
    cudaError_t e = cudaSuccess;
    if (part != 2) {
        // C (W's rows below tile J, block column J), sliced by columns per chunk
        e = launch_slice_cols(W, w.cc[J & 1], w.ecc[J & 1], status, batch, n, J + 1,
                              (unsigned)(nt - J - 1), false, J, false, w.cc_stride, w.ecc_stride,
                              Bal{w.iv.bal, bstride, 0, 1}, stream);
        if (e != cudaSuccess) return e;
    }
    double* pbuf = part == 2 ? w.part2 : w.part;
    const int splits = row_splits(batch, k_n, nt - J - 1);
    OzArgs g{W, w.cc[J & 1], w.ecc[J & 1], w.lc, w.elc, w.cc_stride, w.ecc_stride, w.lc_stride,
             w.elc_stride, status, nullptr, batch, n, nt, J, splits, pbuf, 0, k_lo, k_n};
    e = launch_oz<OZ_REV_ROW>(g, (unsigned)(kParts * k_n * splits), stream);
    if (e != cudaSuccess || splits == 1) return e;
    const int64_t total = batch * (int64_t)k_n * kT * kT;
    const unsigned blocks = (unsigned)std::min<int64_t>((total + 255) / 256,
                                                        (int64_t)device_sm_count() * 16);
    return launch_pdl(split_reduce_kernel, dim3(blocks), dim3(256), 0, stream, W, pbuf, status,
                      batch, n, J, splits, k_lo, k_n);
}

cudaError_t ozaki_adj_upd_slice(double* W, void* work, const int32_t* status, int64_t batch,
                                int n, int J, cudaStream_t stream) {
    const int nt = tiles_of(n);
    if (J <= 0) return cudaSuccess;
    const AdjWs w = adj_ws(work, batch, n);
    const size_t bstride = (size_t)nt * kT;
    // Chat = [W_JJ + W_JJ^T; C], rows J*128 .., block column J, sliced by rows
    return launch_slice_rows(W, w.ch[J & 1], w.ech[J & 1], status, batch, n, J * kT,
                             (nt - J) * kT, J * kT, true, w.ch_stride, w.ech_stride,
                             Bal{w.iv.bal, bstride, 0, 1}, stream);
}

cudaError_t ozaki_adj_upd_gemm(double* W, void* work, const int32_t* status, int64_t batch,
                               int n, int J, int part, cudaStream_t stream) {
    const int nt = tiles_of(n);
    const int kw = part == 0 ? J : (part == 1 ? 1 : J - 1);
    if (J <= 0 || kw <= 0) return cudaSuccess;
    const AdjWs w = adj_ws(work, batch, n);
    OzArgs g{W, w.ch[J & 1], w.ech[J & 1], w.lc, w.elc, w.ch_stride, w.ech_stride, w.lc_stride,
             w.elc_stride, status, nullptr, batch, n, nt, J, 1, nullptr, part};
    return launch_oz<OZ_REV_UPD>(g, (unsigned)(kParts * (nt - J) * kw), stream);
}

cudaError_t ozaki_adj_upd(const double* L, double* W, void* work, const int32_t* status,
                          int64_t batch, int n, int J, cudaStream_t stream) {
    (void)L;
    cudaError_t e = ozaki_adj_upd_slice(W, work, status, batch, n, J, stream);
    if (e != cudaSuccess) return e;
    return ozaki_adj_upd_gemm(W, work, status, batch, n, J, 0, stream);
}


bool ozaki_adj_lit_pays(int64_t batch) {
    // the literal form's products fill the GPU from one matrix on; its FP64
    // work is 2.5x the sweep's, which wins once the sweeps alone fill it
    return batch * 4 <= device_sm_count();
}

cudaError_t ozaki_adj_diag(const double* L, double* W, void* work, const int32_t* status,
                           int64_t batch, int n, int J, cudaStream_t stream) {
    const int nt = tiles_of(n);
    const AdjWs w = adj_ws(work, batch, n);
    const int j0 = J * kT, kb = std::min(kT, n - j0);
    const int nb = (kb + kLB - 1) / kLB;
    const dim3 grid((unsigned)(nb * (nb + 1) / 2), gy(batch));
    const size_t cnt = (size_t)adj_inverses(nt);
    const double* X = w.iv.inv + (size_t)J * kT * kT;
    const size_t xs = cnt * kT * kT;
    double* S = w.lit;
    double* T = w.lit + (size_t)batch * kT * kT;
    cudaError_t e = launch_pdl(lit_diag_kernel<LIT_S>, grid, dim3(kLitThreads), 0, stream, L, W, X,
                               xs, S, T, status, batch, n, j0, kb);
    if (e == cudaSuccess)
        e = launch_pdl(lit_diag_kernel<LIT_T>, grid, dim3(kLitThreads), 0, stream, L, W, X, xs, S,
                       T, status, batch, n, j0, kb);
    if (e == cudaSuccess)
        e = launch_pdl(lit_diag_kernel<LIT_A>, grid, dim3(kLitThreads), 0, stream, L, W, X, xs, S,
                       T, status, batch, n, j0, kb);
    return e;
}

}  // namespace chol
