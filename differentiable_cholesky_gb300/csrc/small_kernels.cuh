// Kernels of the small path (n <= 64): included by the translation units
// that instantiate them, one per element type and padded order, so that
// they compile in parallel.
//
// Batched Cholesky forward and adjoint for small matrices (n <= 64).
//
// A group of LPG lanes owns one matrix of padded order NT = 8, 16, 32 or 64
// (the next size >= n); each lane owns two rows (or columns) of it, t and
// NT-1-t, where registers allow (LPG = NT / 2), else one.  A block holds
// several groups: 128 threads, or one warp for the adjoint at NT <= 16.  A
// matrix of order n < NT is padded to
// blockdiag(A, I), whose factor is blockdiag(L, I) and whose adjoint (with a
// zero-padded adj_L) is blockdiag(adj_A, 0): the padding changes no result.
// Every loop over matrix indices is fully unrolled, so each lane keeps its
// rows (or columns) in registers.
//
// Forward (jaxmg docs "Cholesky factorization": lower factor and status;
// NVIDIA/warp issue #1316: out-of-place tile factor, one block per tile).
//   Right-looking column recurrence, one group barrier per column: at step j
//   every lane publishes its current a_ij to a double-buffered shared column,
//   then reads the pivot d = a_jj, computes r = 1/sqrt(d) itself (no second
//   broadcast), sets l_ij = a_ij * r and updates its trailing entries
//   a_ik -= (l_ij r) a_kj.  A pivot that is not > 0 records status j + 1
//   (first failure only) and is replaced by 1 so the rest of the (unspecified)
//   factor stays finite and the group stays convergent.  A lane's low row
//   (t < LPG) skips the columns k >= LPG, which lie above its diagonal.
//   Full-order matrices with rows of 128 bytes or more move as contiguous
//   16-byte chunks through a shared staging area (cp.async in, chunk stores
//   out) instead of row by row.
//
// Adjoint (Murray 2016 as NVIDIA/warp issue #1316's closing comment states it:
// S = Phi(L^T adj_L), then solves against L^T and L, accumulated into the lower
// triangle of adj_A).  L is staged in shared memory with packed rows and read
// by broadcast; the reciprocals of its diagonal sit in the transpose buffer's
// padding.
//   1. each lane takes its columns of tril(adj_L) and forms the same columns
//      of P = L^T tril(adj_L) in place (outer-product order over rows of L);
//   2. S = Phi(P) on those columns;
//   3. X = L^-T S: back substitution on the columns (rows of L broadcast);
//   4. transpose through shared memory: the lane takes the same rows of X;
//   5. M = X L^-1: back substitution on the rows (rows of L broadcast);
//   6. transpose once more and add M_tk + M_kt (k < t) and M_tt into the
//      lane's rows of adj_A's lower triangle (or write them there, for the
//      in-place form).  Matrices with status != 0 are skipped (or zeroed).
// Full-order matrices move as contiguous chunks (cp.async into their shared
// places, chunk stores out); blocks take the batch from its end, so right
// after the forward the factors still in L2 are read first.

#pragma once

#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace chol {
namespace {

constexpr int kBlock = 128;

// Load the lower part of row `row` (row < n) into r[0..NT): zeros above the
// diagonal.  Only the 16-byte chunks that hold lower-triangle elements are read.
// Plain (coherent) loads: the in-place forms read rows of the very buffer the
// kernel later writes.
template <typename T, int NT, bool VEC>
__device__ __forceinline__ void load_lower_row(const T* rowp, int row, int n, T (&r)[NT]) {
    if constexpr (VEC) {
        using V = typename Vec16<T>::type;
        constexpr int W = Vec16<T>::N;
        const V* vp = reinterpret_cast<const V*>(rowp);
#pragma unroll
        for (int c = 0; c < NT / W; ++c) {
            V v;
            if (c * W <= row) {
                v = vp[c];
            } else {
                v = V{};
            }
#pragma unroll
            for (int e = 0; e < W; ++e) r[c * W + e] = (c * W + e <= row) ? vget<T>(v, e) : T(0);
        }
    } else {
#pragma unroll
        for (int k = 0; k < NT; ++k) r[k] = (k <= row && k < n) ? rowp[k] : T(0);
    }
}

// Element offset that shifts a group's shared-memory region by NT 4-byte
// words modulo 32 banks, so the groups that share a warp (NT < 32) never hit
// the same bank with their broadcast reads.
template <typename T, int NT>
__host__ __device__ constexpr int group_stride(int base_elems) {
    constexpr int wpe = (int)sizeof(T) / 4;  // words per element
    const int words = base_elems * wpe;
    const int target = NT < 32 ? NT : 0;
    const int pad_words = ((target - words % 32) % 32 + 32) % 32;
    return base_elems + pad_words / wpe;
}

// Row `row` of matrix b for the forward: lower part of A, or an identity row
// for padding rows and for slots past the end of the batch.
template <typename T, int NT, bool VEC>
__device__ __forceinline__ void fetch_fwd_row(const T* A, int64_t b, int64_t batch,
                                              int row, int n, T (&r)[NT]) {
    if (b < batch && row < n) {
        load_lower_row<T, NT, VEC>(A + (size_t)b * n * n + (size_t)row * n, row, n, r);
    } else {
#pragma unroll
        for (int k = 0; k < NT; ++k) r[k] = (k == row) ? T(1) : T(0);
    }
}

// Lanes per matrix LPG = NT / RPL: each lane owns RPL rows, t and NT-1-t for
// RPL = 2 (balanced triangle rows).  Every broadcast read of the published
// column then feeds RPL rows.
__host__ __device__ constexpr int owned_index(int t, int q, int lpg) {
    return (q & 1) ? (q + 1) * lpg - 1 - t : q * lpg + t;
}

template <int LPG>
__device__ __forceinline__ void lanes_sync(int group) {
    if constexpr (LPG <= 32) {
        __syncwarp();
    } else {
        // Named barrier per group of LPG (a multiple of 32) threads; id 0 is
        // __syncthreads.
        asm volatile("bar.sync %0, %1;" ::"r"(1 + group), "r"(LPG) : "memory");
    }
}

// Row r[0..NT) to / from a 16-byte aligned shared-memory row, as vectors.
template <typename T, int NT>
__device__ __forceinline__ void store_row(T* dst, const T (&r)[NT]) {
    using V = typename Vec16<T>::type;
    constexpr int W = Vec16<T>::N;
#pragma unroll
    for (int u = 0; u < NT / W; ++u) {
        V v;
#pragma unroll
        for (int e = 0; e < W; ++e) vset<T>(v, e, r[u * W + e]);
        reinterpret_cast<V*>(dst)[u] = v;
    }
}
template <typename T, int NT>
__device__ __forceinline__ void load_row(const T* src, T (&r)[NT]) {
    using V = typename Vec16<T>::type;
    constexpr int W = Vec16<T>::N;
#pragma unroll
    for (int u = 0; u < NT / W; ++u) {
        const V v = reinterpret_cast<const V*>(src)[u];
#pragma unroll
        for (int e = 0; e < W; ++e) r[u * W + e] = vget<T>(v, e);
    }
}

// Whole matrices of the padded order (n == NT) move between HBM and the group
// as contiguous 16-byte chunks: lane t of a group takes chunks t, t + LPG,
// t + 2 LPG, ... of each matrix, so one warp-wide access covers whole 128-byte
// lines (a row-wise access spreads over a line per row).  Chunk c holds
// elements u W .. u W + W - 1 of row r, with u = c % (NT / W) fixed per lane
// when LPG is a multiple of NT / W.
template <typename T, int NT, int LPG>
struct Chunks {
    static constexpr int W = 16 / (int)sizeof(T);
    static constexpr int PER_ROW = NT / W;
    static constexpr int PER_LANE = NT * PER_ROW / LPG;
    static constexpr int ROW_STEP = LPG / PER_ROW;  // rows between a lane's chunks
    static constexpr bool OK = LPG % PER_ROW == 0 && (NT * PER_ROW) % LPG == 0 && PER_LANE <= 16;
    static constexpr int BATCH = PER_LANE < 8 ? PER_LANE : 8;  // output chunks held at once
};

// Rows of at least 128 bytes: the forward also moves whole-order matrices
// as chunks, staged through shared memory (row pitch NT + W elements).
template <typename T, int NT>
constexpr bool fwd_chunks() {
    return NT * (int)sizeof(T) >= 128;
}

// A and L may be the same buffer (the in-place forward): a group reads its
// matrix in full before it writes any of it, and no other group touches it.
template <typename T, int NT, int RPL, bool VEC, bool FULL>
__global__ void __launch_bounds__(kBlock)
small_potrf_kernel(const T* A, T* L, int32_t* __restrict__ status, int64_t batch, int n) {
    constexpr int LPG = NT / RPL;
    constexpr int G = kBlock / LPG;
    constexpr int CS = group_stride<T, LPG>(2 * NT);
    __shared__ __align__(16) T colbuf[G * CS];
    using V = typename Vec16<T>::type;
    constexpr int W = Vec16<T>::N;

    const int g = threadIdx.x / LPG;
    const int t = threadIdx.x % LPG;
    const int64_t b = (int64_t)blockIdx.x * G + g;
    int rows[RPL];
#pragma unroll
    for (int q = 0; q < RPL; ++q) rows[q] = owned_index(t, q, LPG);

    T a[RPL][NT];
    using CK = Chunks<T, NT, LPG>;
    constexpr int SP = NT + W;  // staging row pitch (FULL)
    T* Sg = nullptr;
    const int cu = t % CK::PER_ROW, cr = t / CK::PER_ROW;
    if constexpr (FULL) {
        // A's chunks straight into the group's staging area by cp.async;
        // what lies above the diagonal (and all of a matrix past the end of
        // the batch) is zero-filled, then each lane reads its rows
        static_assert(LPG % CK::PER_ROW == 0 && (NT * CK::PER_ROW) % LPG == 0, "chunk layout");
        extern __shared__ __align__(16) unsigned char stage_raw[];
        Sg = reinterpret_cast<T*>(stage_raw) + (size_t)g * NT * SP;
        const bool in_batch = b < batch;
        const V* Am = reinterpret_cast<const V*>(in_batch ? A + (size_t)b * NT * NT : A) + t;
#pragma unroll
        for (int i = 0; i < CK::PER_LANE; ++i) {
            const int r = cr + CK::ROW_STEP * i;
            const int lower = r - cu * W + 1;
            const uint32_t nb =
                in_batch ? (uint32_t)(lower <= 0 ? 0 : lower >= W ? 16 : lower * (int)sizeof(T)) : 0u;
            cp_async16(Sg + r * SP + cu * W, in_batch ? Am + i * LPG : Am, nb);
        }
        cp_async_wait_all();
        lanes_sync<LPG>(g);
#pragma unroll
        for (int q = 0; q < RPL; ++q) {
            load_row<T, NT>(Sg + rows[q] * SP, a[q]);
            if (!in_batch) {
#pragma unroll
                for (int k = 0; k < NT; ++k) a[q][k] = (k == rows[q]) ? T(1) : T(0);
            }
        }
        // a lane's low row (t < LPG) holds nothing at k >= LPG: constants,
        // not registers, through the recurrence (else they stay live to the
        // end and cost ~80 registers at order 64)
        if constexpr (RPL == 2) {
#pragma unroll
            for (int k = LPG; k < NT; ++k) a[0][k] = T(0);
        }
    } else {
#pragma unroll
        for (int q = 0; q < RPL; ++q) fetch_fwd_row<T, NT, VEC>(A, b, batch, rows[q], n, a[q]);
    }

    int st = 0;
    static_for<0, NT>([&](auto jc) {
        constexpr int j = decltype(jc)::value;
        T* buf = colbuf + g * CS + (j & 1) * NT;
#pragma unroll
        for (int q = 0; q < RPL; ++q) buf[rows[q]] = a[q][j];
        lanes_sync<LPG>(g);
        T d = buf[j];
        if (!(d > T(0))) {
            if (st == 0) st = j + 1;
            d = T(1);
        }
        const T r = rsqrt_t(d);
        T coef[RPL];
#pragma unroll
        for (int q = 0; q < RPL; ++q) {
            const T lij = a[q][j] * r;
            coef[q] = T(rows[q] > j) * (lij * r);
            a[q][j] = lij;
        }
        // trailing update with the published column, read as aligned vectors.
        // Row q = 0 of a lane (t < LPG) only ever needs columns k <= t < LPG:
        // its entries at k >= LPG lie above the diagonal and are left stale.
        static_for<(j + 1) / W, NT / W>([&](auto cc) {
            constexpr int c = decltype(cc)::value;
            const V v = reinterpret_cast<const V*>(buf)[c];
            static_for<0, W>([&](auto ec) {
                constexpr int e = decltype(ec)::value;
                constexpr int k = c * W + e;
                if constexpr (k > j) {
                    static_for<0, RPL>([&](auto qc) {
                        constexpr int q = decltype(qc)::value;
                        if constexpr (!(RPL == 2 && q == 0 && k >= LPG))
                            a[q][k] = fma(-coef[q], vget<T>(v, e), a[q][k]);
                    });
                }
            });
        });
    });

    if constexpr (FULL) {
        // rows back into the staging area (zeros above the diagonal), then
        // out to L as whole chunks
#pragma unroll
        for (int q = 0; q < RPL; ++q) {
            const int i = rows[q];
            V* dst = reinterpret_cast<V*>(Sg + i * SP);
#pragma unroll
            for (int c = 0; c < NT / W; ++c) {
                V v;
#pragma unroll
                for (int e = 0; e < W; ++e) vset<T>(v, e, (c * W + e <= i) ? a[q][c * W + e] : T(0));
                dst[c] = v;
            }
        }
        lanes_sync<LPG>(g);
        if (b >= batch) return;
        V* Lm = reinterpret_cast<V*>(L + (size_t)b * NT * NT) + t;
#pragma unroll
        for (int i = 0; i < CK::PER_LANE; ++i)
            Lm[i * LPG] = *reinterpret_cast<const V*>(Sg + (cr + CK::ROW_STEP * i) * SP + cu * W);
        if (t == 0) status[b] = st;
        return;
    }
    if (b >= batch) return;
#pragma unroll
    for (int q = 0; q < RPL; ++q) {
        const int i = rows[q];
        if (i >= n) continue;
        T* rowp = L + (size_t)b * n * n + (size_t)i * n;
        if constexpr (VEC) {
            V* vp = reinterpret_cast<V*>(rowp);
#pragma unroll
            for (int c = 0; c < NT / W; ++c) {
                if (c * W < n) {
                    V v;
#pragma unroll
                    for (int e = 0; e < W; ++e)
                        vset<T>(v, e, (c * W + e <= i) ? a[q][c * W + e] : T(0));
                    vp[c] = v;
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < NT; ++k)
                if (k < n) rowp[k] = (k <= i) ? a[q][k] : T(0);
        }
    }
    if (t == 0) status[b] = st;
}

// Adjoint layout: a group of LPG = NT / CPL lanes per matrix, each lane owning
// CPL columns (and, after the transpose, CPL rows): columns t and NT-1-t for
// CPL = 2, which balances the triangular work.  Every broadcast read of a row
// of L then feeds CPL columns.

// Phi's factor for row i of column col: 1 below the diagonal, 1/2 on it,
// 0 above; and the strict-lower indicator k < col.  float uses one saturated
// add each; double compares.
__device__ __forceinline__ float phi_factor(int i, float colf) {
    return __saturatef((float(i) + 0.5f) - colf);
}
__device__ __forceinline__ float below(int k, float colf) { return __saturatef(colf - float(k)); }

// L is staged with its rows packed: row r keeps only the 16-byte vectors that
// hold its lower part, W * (r / W + 1) elements (W per vector), and starts
// where row r - 1 ends.  Every read of a row has a compile-time r.
template <typename T>
__host__ __device__ constexpr int lrow_off(int r) {
    constexpr int W = 16 / (int)sizeof(T);
    const int a = r / W, b = r % W;
    return W * (W * a * (a + 1) / 2 + b * (a + 1));
}

// Row `row` (runtime) of L into its packed place: the vectors up to the diagonal.
template <typename T, int NT>
__device__ __forceinline__ void store_lrow(T* Ls, int row, const T (&r)[NT]) {
    using V = typename Vec16<T>::type;
    constexpr int W = Vec16<T>::N;
    V* dst = reinterpret_cast<V*>(Ls + lrow_off<T>(row));
#pragma unroll
    for (int u = 0; u < NT / W; ++u) {
        if (u * W <= row) {
            V v;
#pragma unroll
            for (int e = 0; e < W; ++e) vset<T>(v, e, r[u * W + e]);
            dst[u] = v;
        }
    }
}

template <typename T, int NT, int CPL>
struct AdjCfg {
    // short matrices run in one-warp blocks: more, smaller blocks per SM hide
    // the global-load latency at their start and end better (batched
    // 65536 x 16x16: 128 threads 70.0 us, 64 threads 68.2 us, and with the
    // later kernel 49.1 -> 48.4 us from 64 to 32 threads)
    static constexpr int BLOCK = NT <= 16 ? 32 : kBlock;
    static constexpr int LPG = NT / CPL;                   // lanes per matrix
    static constexpr int G = BLOCK / LPG;                  // matrices per block
    static constexpr int LSIZE = lrow_off<T>(NT);          // packed L (rows read by broadcast)
    static constexpr int RP = NT + 16 / (int)sizeof(T);    // transpose pitch (16-byte rows)
    // The reciprocals of L's diagonal live in R's padding columns (NT .. RP-1,
    // never touched by the transposes): 1/l_ii at row i / W, column NT + i % W.
    // They are read into registers when they are few, else as used.
    static constexpr bool RV = NT * sizeof(T) <= 64;
    static constexpr int per_group = group_stride<T, LPG>(LSIZE + NT * RP);
    // Murray's reverse sweep instead of the literal P / Phi / two solves:
    // n^3 / 3 multiply-adds, the column of W being retired handed to the
    // group by shuffles (or, when the group spans warps, shared memory) once
    // per column instead of rows of L read by broadcast for every step; the
    // gradient is the same up to rounding (pinned against the literal
    // oracle).  Used where a lane owns two columns and the group fits in a
    // warp (order <= 32 for float, <= 16 for double).  With one column per
    // lane the owner's serial diagonal sum and scaling sit on the critical
    // path of every column (batched 8192 x 64x64 float: 0.27 ms literal,
    // 0.92 ms swept through shared memory), so those orders keep the literal
    // form.
    static constexpr bool SWEEP = CPL == 2 && LPG <= 32 && NT * CPL * 2 * sizeof(T) <= 512;
    static constexpr size_t bytes = (size_t)G * per_group * sizeof(T);
};


// Row `row` of one of the adjoint's inputs, or its padding: identity rows of
// L, zero rows of adj_L.
template <typename T, int NT, bool VEC>
__device__ __forceinline__ void fetch_adj_row(const T* src, bool active, int64_t b,
                                              int row, int n, T pad_diag, T (&r)[NT]) {
    if (active && row < n) {
        load_lower_row<T, NT, VEC>(src + (size_t)b * n * n + (size_t)row * n, row, n, r);
    } else {
#pragma unroll
        for (int k = 0; k < NT; ++k) r[k] = (k == row) ? pad_diag : T(0);
    }
}

// Padding rows in place of rows that were read: identity rows of L, zero
// rows of adj_L (for matrices whose status turned out non-zero).
template <typename T, int NT>
__device__ __forceinline__ void pad_row(int row, T pad_diag, T (&r)[NT]) {
#pragma unroll
    for (int k = 0; k < NT; ++k) r[k] = (k == row) ? pad_diag : T(0);
}

// adj_A is read only at the adjoint's end: one lane per matrix starts bringing
// it into L2 at the start, so that read finds it there (orders up to 32; at 64
// the extra L2 traffic cost more than it saved).
template <typename T, int NT, bool VEC>
__device__ __forceinline__ void prefetch_abar(const T* Abar, int64_t b, int n, bool issue) {
    if constexpr (VEC && NT <= 32) {
        if (issue) l2_prefetch(Abar + (size_t)b * n * n, (uint32_t)((size_t)n * n * sizeof(T)));
    }
}

// Lbar and Abar may be the same buffer (the in-place adjoint, not
// accumulating): a group reads its matrix in full before it writes any of it.
template <typename T, int NT, int CPL, bool VEC, bool FULL>
__global__ void __launch_bounds__(AdjCfg<T, NT, CPL>::BLOCK)
small_potrf_adj_kernel(const T* __restrict__ Lg, const T* Lbar, T* Abar,
                       const int32_t* __restrict__ status, int64_t batch, int n, bool accumulate) {
    using S = AdjCfg<T, NT, CPL>;
    using V = typename Vec16<T>::type;
    constexpr int W = Vec16<T>::N;
    constexpr int RP = S::RP;
    constexpr int LPG = S::LPG;
    extern __shared__ __align__(16) unsigned char smem_raw[];

    const int g = threadIdx.x / LPG;
    const int t = threadIdx.x % LPG;
    // Blocks take the batch from its end: called right after the forward,
    // whose last-written factors are the ones still in L2, the adjoint reads
    // those first (batched 65536 x 16x16: 50.8 -> 49.0 us).
    const int64_t b = (int64_t)(gridDim.x - 1 - blockIdx.x) * S::G + g;
    // The status word is read beside the rows, not before them, so the row
    // loads never wait for it; a matrix with status != 0 (skipped) has its
    // rows replaced by padding once they arrive.
    const bool in_batch = b < batch;
    const int32_t st = (in_batch && status != nullptr) ? __ldg(status + b) : 0;

    T* Ls = reinterpret_cast<T*>(smem_raw) + (size_t)g * S::per_group;
    T* R = Ls + S::LSIZE;
    auto rinv = [&](int i) -> T& { return R[(i / W) * RP + NT + i % W]; };
    int col[CPL];
#pragma unroll
    for (int q = 0; q < CPL; ++q) col[q] = owned_index(t, q, LPG);

    // When they are short, the lane's rows of adj_A are read now, so their
    // latency overlaps the solves; otherwise just before they are updated.
    constexpr bool kEarly = !FULL && NT * CPL * sizeof(T) <= 64;
    T old[CPL][NT];
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
        if (!kEarly) break;
        if (accumulate && in_batch && col[q] < n) {
            load_lower_row<T, NT, VEC>(Abar + (size_t)b * n * n + (size_t)col[q] * n, col[q], n,
                                       old[q]);
        } else {
#pragma unroll
            for (int k = 0; k < NT; ++k) old[q][k] = T(0);
        }
    }

    // Rows col[q] of L into shared memory (identity rows for padding or
    // skipped matrices) and rows col[q] of tril(adj_L) into the transpose buffer.
    using CK = Chunks<T, NT, LPG>;
    const int cu = t % CK::PER_ROW;  // the lane's chunk column (FULL)
    const int cr = t / CK::PER_ROW;  // row of the lane's first chunk (FULL)
    if constexpr (FULL) {
        // whole chunks copied straight into their places (L packed, adj_L
        // into R), no registers in between; a chunk of adj_L that reaches
        // above the diagonal copies only its lower part and is zero-filled
        static_assert(CK::OK, "chunk layout");
        const V* Lm = reinterpret_cast<const V*>(in_batch ? Lg + (size_t)b * NT * NT : Lg) + t;
        const V* Bm = reinterpret_cast<const V*>(in_batch ? Lbar + (size_t)b * NT * NT : Lbar) + t;
#pragma unroll
        for (int i = 0; i < CK::PER_LANE; ++i) {
            const int r = cr + CK::ROW_STEP * i;
            const int lower = r - cu * W + 1;  // elements of the chunk on or below the diagonal
            const uint32_t nb =
                in_batch ? (uint32_t)(lower <= 0 ? 0 : lower >= W ? 16 : lower * (int)sizeof(T)) : 0u;
            if (lower > 0) cp_async16(Ls + lrow_off<T>(r) + cu * W, in_batch ? Lm + i * LPG : Lm, nb ? 16u : 0u);
            cp_async16(R + r * RP + cu * W, in_batch ? Bm + i * LPG : Bm, nb);
        }
        prefetch_abar<T, NT, VEC>(Abar, b, n, accumulate && t == 0 && in_batch);
        cp_async_wait_all();
        if (!in_batch || st != 0) {
            // skipped matrix: identity rows of L, zero rows of adj_L
#pragma unroll
            for (int i = 0; i < CK::PER_LANE; ++i) {
                const int r = cr + CK::ROW_STEP * i;
                V l, z{};
#pragma unroll
                for (int e = 0; e < W; ++e) vset<T>(l, e, T(cu * W + e == r));
                if (cu * W <= r) *reinterpret_cast<V*>(Ls + lrow_off<T>(r) + cu * W) = l;
                *reinterpret_cast<V*>(R + r * RP + cu * W) = z;
            }
        }
    } else if constexpr (NT * CPL * sizeof(T) <= 128) {
        // short rows: all of the lane's row loads are issued before any store
        T lr[CPL][NT], br[CPL][NT];
#pragma unroll
        for (int q = 0; q < CPL; ++q) {
            fetch_adj_row<T, NT, VEC>(Lg, in_batch, b, col[q], n, T(1), lr[q]);
            fetch_adj_row<T, NT, VEC>(Lbar, in_batch, b, col[q], n, T(0), br[q]);
        }
        prefetch_abar<T, NT, VEC>(Abar, b, n, accumulate && t == 0 && in_batch);
        if (st != 0) {
#pragma unroll
            for (int q = 0; q < CPL; ++q) {
                pad_row<T, NT>(col[q], T(1), lr[q]);
                pad_row<T, NT>(col[q], T(0), br[q]);
            }
        }
#pragma unroll
        for (int q = 0; q < CPL; ++q) {
            store_lrow<T, NT>(Ls, col[q], lr[q]);
            store_row<T, NT>(R + col[q] * RP, br[q]);
        }
    } else {
        prefetch_abar<T, NT, VEC>(Abar, b, n, accumulate && t == 0 && in_batch);
#pragma unroll
        for (int q = 0; q < CPL; ++q) {
            T r[NT];
            fetch_adj_row<T, NT, VEC>(Lg, in_batch, b, col[q], n, T(1), r);
            if (st != 0) pad_row<T, NT>(col[q], T(1), r);
            store_lrow<T, NT>(Ls, col[q], r);
            fetch_adj_row<T, NT, VEC>(Lbar, in_batch, b, col[q], n, T(0), r);
            if (st != 0) pad_row<T, NT>(col[q], T(0), r);
            store_row<T, NT>(R + col[q] * RP, r);
        }
    }
    const bool active = in_batch && st == 0;
    lanes_sync<LPG>(g);
#pragma unroll
    for (int q = 0; q < CPL; ++q) rinv(col[q]) = rcp_t(Ls[lrow_off<T>(col[q]) + col[q]]);

    // Columns col[q] of tril(adj_L).
    T c[CPL][NT];
#pragma unroll
    for (int q = 0; q < CPL; ++q)
#pragma unroll
        for (int k = 0; k < NT; ++k) c[q][k] = R[k * RP + col[q]];

    constexpr bool kSweep = S::SWEEP;
    if constexpr (kSweep) {
        // Murray's unblocked reverse sweep, column-per-lane (see AdjCfg::SWEEP):
        // c[q] holds column col[q] of W = tril(adj_L), l[q] the same column of L.
        T l[CPL][NT];
#pragma unroll
        for (int q = 0; q < CPL; ++q)
#pragma unroll
            for (int i = 0; i < NT; ++i) l[q][i] = i >= col[q] ? Ls[lrow_off<T>(i) + col[q]] : T(0);
        lanes_sync<LPG>(g);  // rinv visible to the group; every lane is done with R's columns
        static_for<0, NT>([&](auto jc) {
            constexpr int j = NT - 1 - decltype(jc)::value;
            // the lane that owns column j, and which of its columns it is
            constexpr int qo = (CPL == 2 && j >= LPG) ? 1 : 0;
            constexpr int towner = (CPL == 2 && j >= LPG) ? NT - 1 - j : j;
            const bool own = t == towner;
            const T rj = rinv(j);
            if (own) {
                // the diagonal from s = sum_{i > j} l_ij w_ij, the column scaled
                T s0 = T(0), s1 = T(0);
                static_for<j + 1, NT>([&](auto ic) {
                    constexpr int i = decltype(ic)::value;
                    if constexpr ((i - j) & 1) s0 = fma(l[qo][i], c[qo][i], s0);
                    else s1 = fma(l[qo][i], c[qo][i], s1);
                });
                static_for<j + 1, NT>([&](auto ic) {
                    constexpr int i = decltype(ic)::value;
                    c[qo][i] *= rj;
                });
                c[qo][j] = (c[qo][j] - (s0 + s1) * rj) * rj;
            }
            // column j of W (rows i >= j) to the group; lanes whose columns lie
            // left of j take  w_jk -= sum_{i >= j} w_ij l_ik  and
            // w_ik -= w_ij l_jk (i > j)
            T acc[CPL];
#pragma unroll
            for (int q = 0; q < CPL; ++q) acc[q] = T(0);
            static_for<j, NT>([&](auto ic) {
                constexpr int i = decltype(ic)::value;
                const T v = __shfl_sync(0xffffffffu, c[qo][i], towner, LPG);
#pragma unroll
                for (int q = 0; q < CPL; ++q) {
                    if (col[q] < j) {
                        acc[q] = fma(v, l[q][i], acc[q]);
                        if constexpr (i > j) c[q][i] = fma(-v, l[q][j], c[q][i]);
                    }
                }
            });
#pragma unroll
            for (int q = 0; q < CPL; ++q)
                if (col[q] < j) c[q][j] -= acc[q];
            if (own) c[qo][j] *= T(0.5);
        });
        // the columns of the gradient through R, so rows come back out
        lanes_sync<LPG>(g);
#pragma unroll
        for (int q = 0; q < CPL; ++q)
#pragma unroll
            for (int i = 0; i < NT; ++i) R[i * RP + col[q]] = c[q][i];
        lanes_sync<LPG>(g);
        if constexpr (!FULL) {
#pragma unroll
            for (int q = 0; q < CPL; ++q) load_row<T, NT>(R + col[q] * RP, c[q]);
        }
    } else {

    // 1. columns of P = L^T tril(adj_L), in place: slot k is finished once
    //    row k of L has been applied, so it can take p_k's first term.
    static_for<0, NT>([&](auto kc) {
        constexpr int k = decltype(kc)::value;
        T ck[CPL];
#pragma unroll
        for (int q = 0; q < CPL; ++q) ck[q] = c[q][k];
        const T* lrow = Ls + lrow_off<T>(k);
        static_for<0, k / W + 1>([&](auto uc) {
            constexpr int u = decltype(uc)::value;
            const V v = reinterpret_cast<const V*>(lrow)[u];
            static_for<0, W>([&](auto ec) {
                constexpr int i = u * W + decltype(ec)::value;
#pragma unroll
                for (int q = 0; q < CPL; ++q) {
                    if constexpr (i < k) c[q][i] = fma(vget<T>(v, i - u * W), ck[q], c[q][i]);
                    else if constexpr (i == k) c[q][i] = vget<T>(v, i - u * W) * ck[q];
                }
            });
        });
    });
    // 2. S = Phi(P): keep rows below the column, halve the diagonal, clear above.
    // (a factor rather than a select: a select chain on a lane-dependent index
    //  is turned into an indexed store, which moves c out of registers)
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
        const float colf = float(col[q]);
#pragma unroll
        for (int i = 0; i < NT; ++i) c[q][i] *= T(phi_factor(i, colf));
    }
    lanes_sync<LPG>(g);  // rinv visible to the group
    constexpr bool kRv = S::RV;
    T rv[kRv ? NT : 1];
    if constexpr (kRv) {
#pragma unroll
        for (int u = 0; u < NT / W; ++u) {
            const V v = *reinterpret_cast<const V*>(R + u * RP + NT);
#pragma unroll
            for (int e = 0; e < W; ++e) rv[u * W + e] = vget<T>(v, e);
        }
    }

    // 3. X = L^-T S (back substitution, rows of L broadcast).
    static_for<0, NT>([&](auto ic) {
        constexpr int i = NT - 1 - decltype(ic)::value;
        T ri;
        if constexpr (kRv) ri = rv[i]; else ri = rinv(i);
        T xi[CPL];
#pragma unroll
        for (int q = 0; q < CPL; ++q) {
            xi[q] = c[q][i] * ri;
            c[q][i] = xi[q];
        }
        const T* lrow = Ls + lrow_off<T>(i);
        static_for<0, (i + W - 1) / W>([&](auto uc) {
            constexpr int u = decltype(uc)::value;
            const V v = reinterpret_cast<const V*>(lrow)[u];
            static_for<0, W>([&](auto ec) {
                constexpr int k = u * W + decltype(ec)::value;
                if constexpr (k < i) {
#pragma unroll
                    for (int q = 0; q < CPL; ++q)
                        c[q][k] = fma(-vget<T>(v, k - u * W), xi[q], c[q][k]);
                }
            });
        });
    });
    // 4. transpose: columns col[q] of X out, rows col[q] in.
#pragma unroll
    for (int q = 0; q < CPL; ++q)
#pragma unroll
        for (int i = 0; i < NT; ++i) R[i * RP + col[q]] = c[q][i];
    lanes_sync<LPG>(g);
#pragma unroll
    for (int q = 0; q < CPL; ++q) load_row<T, NT>(R + col[q] * RP, c[q]);

    // 5. M = X L^-1 (back substitution on the rows).
    static_for<0, NT>([&](auto jc) {
        constexpr int j = NT - 1 - decltype(jc)::value;
        T rj;
        if constexpr (kRv) rj = rv[j]; else rj = rinv(j);
        T mj[CPL];
#pragma unroll
        for (int q = 0; q < CPL; ++q) {
            mj[q] = c[q][j] * rj;
            c[q][j] = mj[q];
        }
        const T* lrow = Ls + lrow_off<T>(j);
        static_for<0, (j + W - 1) / W>([&](auto uc) {
            constexpr int u = decltype(uc)::value;
            const V v = reinterpret_cast<const V*>(lrow)[u];
            static_for<0, W>([&](auto ec) {
                constexpr int k = u * W + decltype(ec)::value;
                if constexpr (k < j) {
#pragma unroll
                    for (int q = 0; q < CPL; ++q)
                        c[q][k] = fma(-vget<T>(v, k - u * W), mj[q], c[q][k]);
                }
            });
        });
    });
    // 6. Phi(M + M^T) into rows col[q] of adj_A's lower triangle.  Each lane
    //    only rewrites the rows it has read.
#pragma unroll
    for (int q = 0; q < CPL; ++q) store_row<T, NT>(R + col[q] * RP, c[q]);
    lanes_sync<LPG>(g);
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
        const float colf = float(col[q]);
#pragma unroll
        for (int k = 0; k < NT; ++k) c[q][k] = fma(T(below(k, colf)), R[k * RP + col[q]], c[q][k]);
    }
    if constexpr (FULL) {
        // rows col[q] of the result through R once more
        lanes_sync<LPG>(g);  // every lane is done with R's columns
#pragma unroll
        for (int q = 0; q < CPL; ++q) store_row<T, NT>(R + col[q] * RP, c[q]);
        lanes_sync<LPG>(g);
    }
    }  // literal form

    if constexpr (FULL) {
        // the result's rows (in R) out as chunks added to adj_A's; chunks
        // wholly above the diagonal are not touched, and a chunk that
        // straddles it is written element by element
        if (!in_batch || (accumulate && !active)) return;
        V* Am = reinterpret_cast<V*>(Abar + (size_t)b * NT * NT) + t;
        // keep the adj_A loads here: hoisted into the solves they hold
        // registers that cost occupancy
        asm volatile("" ::: "memory");
        static_for<0, CK::PER_LANE / CK::BATCH>([&](auto hc) {
            constexpr int i0 = decltype(hc)::value * CK::BATCH;
            V av[CK::BATCH];
#pragma unroll
            for (int ii = 0; ii < CK::BATCH; ++ii) {
                const int i = i0 + ii;
                av[ii] = (accumulate && cu * W <= cr + CK::ROW_STEP * i) ? Am[i * LPG] : V{};
            }
#pragma unroll
            for (int ii = 0; ii < CK::BATCH; ++ii) {
                const int i = i0 + ii;
                const int r = cr + CK::ROW_STEP * i;
                if (cu * W > r) continue;
                const V x = *reinterpret_cast<const V*>(R + r * RP + cu * W);
                V v;
#pragma unroll
                for (int e = 0; e < W; ++e) vset<T>(v, e, vget<T>(av[ii], e) + vget<T>(x, e));
                if (cu * W + W - 1 <= r) {
                    Am[i * LPG] = v;
                } else {
                    T* ap = reinterpret_cast<T*>(Am + i * LPG);
#pragma unroll
                    for (int e = 0; e < W; ++e)
                        if (cu * W + e <= r) ap[e] = vget<T>(v, e);
                }
            }
        });
        return;
    }

    // Accumulating, a skipped matrix keeps adj_A as it was; overwriting, it
    // gets the zeros its padding rows produce.
    if (!in_batch || (accumulate && !active)) return;
    static_for<0, CPL>([&](auto qc) {
        constexpr int q = decltype(qc)::value;
        const int row = col[q];
        if (row >= n) return;
        T* rowp = Abar + (size_t)b * n * n + (size_t)row * n;
        if constexpr (!kEarly) {
            if (accumulate) {
                load_lower_row<T, NT, VEC>(rowp, row, n, old[q]);
            } else {
#pragma unroll
                for (int k = 0; k < NT; ++k) old[q][k] = T(0);
            }
        }
        if constexpr (VEC) {
            V* vp = reinterpret_cast<V*>(rowp);
            static_for<0, NT / W>([&](auto uc) {
                constexpr int u = decltype(uc)::value;
                if (u * W + W - 1 <= row) {
                    V v;
#pragma unroll
                    for (int e = 0; e < W; ++e)
                        vset<T>(v, e, old[q][u * W + e] + c[q][u * W + e]);
                    vp[u] = v;
                } else if (u * W <= row) {
                    // chunk straddling the diagonal: write only k <= row
#pragma unroll
                    for (int e = 0; e < W; ++e) {
                        const int k = u * W + e;
                        if (k <= row) rowp[k] = old[q][k] + c[q][k];
                    }
                }
            });
        } else {
#pragma unroll
            for (int k = 0; k < NT; ++k)
                if (k <= row && k < n) rowp[k] = old[q][k] + c[q][k];
        }
    });
}

// Rows (forward) / columns (adjoint) per lane: two where the registers allow.
template <typename T, int NT>
constexpr int per_lane() {
    return (NT * (int)sizeof(T) <= 128) ? 2 : 1;
}

template <typename T, int NT, bool VEC>
cudaError_t launch_fwd_nt(const T* A, T* L, int32_t* status, int64_t batch, int n,
                          cudaStream_t stream) {
    constexpr int RPL = (NT * (int)sizeof(T) <= 256) ? 2 : 1;
    constexpr int G = kBlock / (NT / RPL);
    const int64_t blocks = (batch + G - 1) / G;
    if constexpr (VEC && fwd_chunks<T, NT>()) {
        if (n == NT) {
            constexpr size_t smem = (size_t)G * NT * (NT + 16 / sizeof(T)) * sizeof(T);
            auto kern = small_potrf_kernel<T, NT, RPL, VEC, true>;
            static std::atomic<uint64_t> smem_set{0};
            if (smem > 48 * 1024) {
                cudaError_t e = allow_smem_once(kern, smem, smem_set);
                if (e != cudaSuccess) return e;
            }
            kern<<<(unsigned)blocks, kBlock, smem, stream>>>(A, L, status, batch, n);
            return cudaGetLastError();
        }
    }
    small_potrf_kernel<T, NT, RPL, VEC, false><<<(unsigned)blocks, kBlock, 0, stream>>>(
        A, L, status, batch, n);
    return cudaGetLastError();
}

template <typename T, int NT, bool VEC>
cudaError_t launch_adj_nt(const T* L, const T* Lbar, T* Abar, const int32_t* status,
                          int64_t batch, int n, bool accumulate, cudaStream_t stream) {
    constexpr int CPL = per_lane<T, NT>();
    using S = AdjCfg<T, NT, CPL>;
    const int64_t blocks = (batch + S::G - 1) / S::G;
    // whole-chunk accesses for matrices of exactly the padded order
    constexpr bool kChunks = VEC && Chunks<T, NT, S::LPG>::OK;
    if constexpr (kChunks) {
        if (n == NT) {
            auto kern = small_potrf_adj_kernel<T, NT, CPL, VEC, true>;
            static std::atomic<uint64_t> smem_set{0};
            if (S::bytes > 48 * 1024) {
                cudaError_t e = allow_smem_once(kern, S::bytes, smem_set);
                if (e != cudaSuccess) return e;
            }
            kern<<<(unsigned)blocks, S::BLOCK, S::bytes, stream>>>(L, Lbar, Abar, status, batch,
                                                                   n, accumulate);
            return cudaGetLastError();
        }
    }
    auto kern = small_potrf_adj_kernel<T, NT, CPL, VEC, false>;
    static std::atomic<uint64_t> smem_set{0};
    if (S::bytes > 48 * 1024) {
        cudaError_t e = allow_smem_once(kern, S::bytes, smem_set);
        if (e != cudaSuccess) return e;
    }
    kern<<<(unsigned)blocks, S::BLOCK, S::bytes, stream>>>(L, Lbar, Abar, status, batch, n,
                                                           accumulate);
    return cudaGetLastError();
}

}  // namespace

template <typename T, int NT, bool VEC>
cudaError_t small_fwd_nt(const T* A, T* L, int32_t* status, int64_t batch, int n,
                         cudaStream_t stream) {
    return launch_fwd_nt<T, NT, VEC>(A, L, status, batch, n, stream);
}

template <typename T, int NT, bool VEC>
cudaError_t small_adj_nt(const T* L, const T* Lbar, T* Abar, const int32_t* status,
                         int64_t batch, int n, bool accumulate, cudaStream_t stream) {
    return launch_adj_nt<T, NT, VEC>(L, Lbar, Abar, status, batch, n, accumulate, stream);
}

// Explicit instantiations, one macro per kernel kind.
#define CHOL_SMALL_FWD(T, NT, VEC)                                                   \
    template cudaError_t small_fwd_nt<T, NT, VEC>(const T*, T*, int32_t*, int64_t, int, \
                                                  cudaStream_t);
#define CHOL_SMALL_ADJ(T, NT, VEC)                                                  \
    template cudaError_t small_adj_nt<T, NT, VEC>(const T*, const T*, T*, const int32_t*, \
                                                  int64_t, int, bool, cudaStream_t);

}  // namespace chol
