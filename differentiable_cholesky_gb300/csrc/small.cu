// Batched Cholesky forward and adjoint for small matrices (n <= 64).
//
// One group of NT threads (NT = 8, 16, 32 or 64, the next size >= n) owns one
// matrix; a 128-thread block holds 128 / NT groups.  A matrix of order n < NT
// is padded to blockdiag(A, I), whose factor is blockdiag(L, I) and whose
// adjoint (with a zero-padded adj_L) is blockdiag(adj_A, 0): the padding
// changes no result.  Every loop over matrix indices is fully unrolled, so each
// thread keeps its row (or column) of the matrix in registers.
//
// Forward (jaxmg docs "Cholesky factorization": lower factor and status;
// NVIDIA/warp issue #1316: out-of-place tile factor, one block per tile).
//   Thread i holds row i.  Right-looking column recurrence, one group barrier
//   per column: at step j every thread publishes its current a_ij to a
//   double-buffered shared column, then reads the pivot d = a_jj, computes
//   r = 1/sqrt(d) itself (no second broadcast), sets l_ij = a_ij * r and
//   updates its trailing entries a_ik -= (l_ij r) a_kj.  A pivot that is not
//   > 0 records status j + 1 (first failure only) and is replaced by 1 so the
//   rest of the (unspecified) factor stays finite and the group stays
//   convergent.
//
// Adjoint (Murray 2016 as NVIDIA/warp issue #1316's closing comment states it:
// S = Phi(L^T adj_L), then solves against L^T and L, accumulated into the lower
// triangle of adj_A).  L is staged in shared memory and read by broadcast.
//   1. thread t takes column t of tril(adj_L) and forms column t of
//      P = L^T tril(adj_L) in place (outer-product order over the rows of L);
//   2. S = Phi(P) on that column;
//   3. X = L^-T S: back substitution on the column (rows of L broadcast);
//   4. transpose through shared memory: thread t takes row t of X;
//   5. M = X L^-1: back substitution on the row (rows of L broadcast);
//   6. transpose once more and add M_tk + M_kt (k < t) and M_tt into row t of
//      adj_A's lower triangle.  Matrices with status != 0 are skipped.

#include <cuda_runtime.h>

#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace chol {
namespace {

constexpr int kBlock = 128;

template <int NT>
__device__ __forceinline__ void group_sync(int group) {
    if constexpr (NT <= 32) {
        __syncwarp();
    } else {
        // Named barrier per 64-thread group (id 0 is __syncthreads).
        asm volatile("bar.sync %0, %1;" ::"r"(1 + group), "r"(NT) : "memory");
    }
}

// Load the lower part of row `row` (row < n) into r[0..NT): zeros above the
// diagonal.  Only the 16-byte chunks that hold lower-triangle elements are read.
template <typename T, int NT, bool VEC>
__device__ __forceinline__ void load_lower_row(const T* __restrict__ rowp, int row, int n,
                                               T (&r)[NT]) {
    if constexpr (VEC) {
        using V = typename Vec16<T>::type;
        constexpr int W = Vec16<T>::N;
        const V* vp = reinterpret_cast<const V*>(rowp);
#pragma unroll
        for (int c = 0; c < NT / W; ++c) {
            V v;
            if (c * W <= row) {
                v = __ldg(vp + c);
            } else {
                v = V{};
            }
#pragma unroll
            for (int e = 0; e < W; ++e) r[c * W + e] = (c * W + e <= row) ? vget<T>(v, e) : T(0);
        }
    } else {
#pragma unroll
        for (int k = 0; k < NT; ++k) r[k] = (k <= row && k < n) ? __ldg(rowp + k) : T(0);
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
__device__ __forceinline__ void fetch_fwd_row(const T* __restrict__ A, int64_t b, int64_t batch,
                                              int row, int n, T (&r)[NT]) {
    if (b < batch && row < n) {
        load_lower_row<T, NT, VEC>(A + (size_t)b * n * n + (size_t)row * n, row, n, r);
    } else {
#pragma unroll
        for (int k = 0; k < NT; ++k) r[k] = (k == row) ? T(1) : T(0);
    }
}

// Persistent kernel: block c handles groups of G matrices c, c + gridDim.x, ...
// and fetches the next group's rows while it factors the current one.
template <typename T, int NT, bool VEC>
__global__ void __launch_bounds__(kBlock)
small_potrf_kernel(const T* __restrict__ A, T* __restrict__ L, int32_t* __restrict__ status,
                   int64_t batch, int n) {
    constexpr int G = kBlock / NT;
    constexpr int CS = group_stride<T, NT>(2 * NT);
    __shared__ __align__(16) T colbuf[G * CS];
    using V = typename Vec16<T>::type;
    constexpr int W = Vec16<T>::N;

    const int g = threadIdx.x / NT;
    const int i = threadIdx.x % NT;
    const int64_t ntasks = (batch + G - 1) / G;
    int64_t task = blockIdx.x;
    if (task >= ntasks) return;  // uniform for the whole block

    // the next group's row is held in registers while the current one is
    // factored, when that costs few registers
    constexpr bool kPrefetch = NT * sizeof(T) <= 64;
    T nxt[kPrefetch ? NT : 1];
    if constexpr (kPrefetch) fetch_fwd_row<T, NT, VEC>(A, task * G + g, batch, i, n, nxt);

#pragma unroll 1
    for (; task < ntasks; task = kPrefetch ? task + gridDim.x : ntasks) {
        const int64_t b = task * G + g;
        T a[NT];
        if constexpr (kPrefetch) {
#pragma unroll
            for (int k = 0; k < NT; ++k) a[k] = nxt[k];
            if (task + gridDim.x < ntasks)
                fetch_fwd_row<T, NT, VEC>(A, (task + gridDim.x) * G + g, batch, i, n, nxt);
        } else {
            fetch_fwd_row<T, NT, VEC>(A, b, batch, i, n, a);
        }

        int st = 0;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            T* buf = colbuf + g * CS + (j & 1) * NT;
            buf[i] = a[j];
            group_sync<NT>(g);
            T d = buf[j];
            if (!(d > T(0))) {
                if (st == 0) st = j + 1;
                d = T(1);
            }
            const T r = rsqrt_t(d);
            const T lij = a[j] * r;
            const T coef = (i > j) ? lij * r : T(0);
            a[j] = lij;
            // trailing update with the published column, read as aligned
            // vectors (constant trip counts: inner loops unroll first)
#pragma unroll
            for (int c = 0; c < NT / W; ++c) {
                if (c < (j + 1) / W) continue;
                const V v = reinterpret_cast<const V*>(buf)[c];
#pragma unroll
                for (int e = 0; e < W; ++e) {
                    const int k = c * W + e;
                    if (k > j) a[k] = fma(-coef, vget<T>(v, e), a[k]);
                }
            }
        }

        if (b < batch && i < n) {
            T* rowp = L + (size_t)b * n * n + (size_t)i * n;
            if constexpr (VEC) {
                V* vp = reinterpret_cast<V*>(rowp);
#pragma unroll
                for (int c = 0; c < NT / W; ++c) {
                    if (c * W < n) {
                        V v;
#pragma unroll
                        for (int e = 0; e < W; ++e)
                            vset<T>(v, e, (c * W + e <= i) ? a[c * W + e] : T(0));
                        vp[c] = v;
                    }
                }
            } else {
#pragma unroll
                for (int k = 0; k < NT; ++k)
                    if (k < n) rowp[k] = (k <= i) ? a[k] : T(0);
            }
        }
        if (b < batch && i == 0) status[b] = st;
    }
}

template <typename T, int NT>
struct AdjSmem {
    static constexpr int G = kBlock / NT;
    static constexpr int LP = NT + 16 / (int)sizeof(T);  // L row pitch: 16-byte skew per row
    static constexpr int RP = NT + 1;                     // transpose pitch
    static constexpr int per_group =
        group_stride<T, NT>(NT * LP + NT * RP + ((NT + 3) / 4) * 4);
    static constexpr size_t bytes = (size_t)G * per_group * sizeof(T);
    // rows of L, adj_L and adj_A for the next group are held in registers
    // while the current group is processed, when that costs few registers
    static constexpr bool prefetch = NT * sizeof(T) <= 64;
};

// Whether matrix b takes part in the adjoint (in the batch, status == 0).
__device__ __forceinline__ bool adj_active(const int32_t* __restrict__ status, int64_t b,
                                           int64_t batch) {
    bool active = b < batch;
    if (active && status != nullptr) active = (__ldg(status + b) == 0);
    return active;
}

// Row `row` of one of the adjoint's inputs, or its padding: identity rows of
// L, zero rows of adj_L / adj_A.
template <typename T, int NT, bool VEC>
__device__ __forceinline__ void fetch_adj_row(const T* __restrict__ src, bool active, int64_t b,
                                              int row, int n, T pad_diag, T (&r)[NT]) {
    if (active && row < n) {
        load_lower_row<T, NT, VEC>(src + (size_t)b * n * n + (size_t)row * n, row, n, r);
    } else {
#pragma unroll
        for (int k = 0; k < NT; ++k) r[k] = (k == row) ? pad_diag : T(0);
    }
}

// The three rows of the next matrix, held in registers while the current
// matrix is processed (used when rows are short).
template <typename T, int NT, bool VEC>
struct AdjRows {
    T l[NT], lb[NT], ab[NT];
    bool active;

    __device__ __forceinline__ void fetch(const T* __restrict__ Lg, const T* __restrict__ Lbar,
                                          const T* __restrict__ Abar,
                                          const int32_t* __restrict__ status, int64_t b,
                                          int64_t batch, int row, int n) {
        active = adj_active(status, b, batch);
        fetch_adj_row<T, NT, VEC>(Lg, active, b, row, n, T(1), l);
        fetch_adj_row<T, NT, VEC>(Lbar, active, b, row, n, T(0), lb);
        fetch_adj_row<T, NT, VEC>(Abar, active, b, row, n, T(0), ab);
    }
};

template <typename T, int NT, bool VEC>
__global__ void __launch_bounds__(kBlock)
small_potrf_adj_kernel(const T* __restrict__ Lg, const T* __restrict__ Lbar,
                       T* __restrict__ Abar, const int32_t* __restrict__ status,
                       int64_t batch, int n) {
    using S = AdjSmem<T, NT>;
    using V = typename Vec16<T>::type;
    constexpr int W = Vec16<T>::N;
    constexpr int LP = S::LP;
    constexpr int RP = S::RP;
    constexpr int G = S::G;
    extern __shared__ __align__(16) unsigned char smem_raw[];

    const int g = threadIdx.x / NT;
    const int t = threadIdx.x % NT;
    const int64_t ntasks = (batch + G - 1) / G;
    int64_t task = blockIdx.x;
    if (task >= ntasks) return;  // uniform for the whole block

    T* Ls = reinterpret_cast<T*>(smem_raw) + (size_t)g * S::per_group;
    T* R = Ls + (size_t)NT * LP;
    T* rinv = R + (size_t)NT * RP;

    struct Empty {};
    using Pf = typename std::conditional<S::prefetch, AdjRows<T, NT, VEC>, Empty>::type;
    Pf pf;
    if constexpr (S::prefetch) pf.fetch(Lg, Lbar, Abar, status, task * G + g, batch, t, n);

#pragma unroll 1
    for (; task < ntasks; task = S::prefetch ? task + gridDim.x : ntasks) {
        const int64_t b = task * G + g;
        T c[NT];
        T ab[S::prefetch ? NT : 1];
        bool active;
        group_sync<NT>(g);  // the previous matrix's readers are done with Ls, R, rinv
        if constexpr (S::prefetch) {
            const AdjRows<T, NT, VEC> cur = pf;
            if (task + gridDim.x < ntasks)
                pf.fetch(Lg, Lbar, Abar, status, (task + gridDim.x) * G + g, batch, t, n);
            active = cur.active;
#pragma unroll
            for (int q = 0; q < NT / W; ++q) {
                V v;
#pragma unroll
                for (int e = 0; e < W; ++e) vset<T>(v, e, cur.l[q * W + e]);
                reinterpret_cast<V*>(Ls + (size_t)t * LP)[q] = v;
            }
#pragma unroll
            for (int k = 0; k < NT; ++k) R[t * RP + k] = cur.lb[k];
#pragma unroll
            for (int k = 0; k < NT; ++k) ab[k] = cur.ab[k];
        } else {
            active = adj_active(status, b, batch);
            // Row t of L into shared memory (identity rows for padding / skipped).
            fetch_adj_row<T, NT, VEC>(Lg, active, b, t, n, T(1), c);
#pragma unroll
            for (int q = 0; q < NT / W; ++q) {
                V v;
#pragma unroll
                for (int e = 0; e < W; ++e) vset<T>(v, e, c[q * W + e]);
                reinterpret_cast<V*>(Ls + (size_t)t * LP)[q] = v;
            }
            // Row t of tril(adj_L) into the transpose buffer.
            fetch_adj_row<T, NT, VEC>(Lbar, active, b, t, n, T(0), c);
#pragma unroll
            for (int k = 0; k < NT; ++k) R[t * RP + k] = c[k];
        }
        group_sync<NT>(g);
        rinv[t] = rcp_t(Ls[t * LP + t]);
        // Column t of tril(adj_L).
#pragma unroll
        for (int k = 0; k < NT; ++k) c[k] = R[k * RP + t];

        // 1. column t of P = L^T tril(adj_L), in place: slot k is finished
        //    once row k of L has been applied, so it can take p_k's first term.
#pragma unroll
        for (int k = 0; k < NT; ++k) {
            const T ck = c[k];
            const T* lrow = Ls + k * LP;
#pragma unroll
            for (int q = 0; q < NT / W; ++q) {
                if (q > k / W) continue;
                const V v = reinterpret_cast<const V*>(lrow)[q];
#pragma unroll
                for (int e = 0; e < W; ++e) {
                    const int i = q * W + e;
                    if (i < k) c[i] = fma(vget<T>(v, e), ck, c[i]);
                    else if (i == k) c[i] = vget<T>(v, e) * ck;
                }
            }
        }
        // 2. S = Phi(P): keep rows below t, halve row t, clear rows above.
#pragma unroll
        for (int i = 0; i < NT; ++i) c[i] = (i > t) ? c[i] : ((i == t) ? c[i] * T(0.5) : T(0));
        group_sync<NT>(g);  // rinv visible to the group

        // 3. X = L^-T S (back substitution, rows of L broadcast).
#pragma unroll
        for (int i = NT - 1; i >= 0; --i) {
            const T xi = c[i] * rinv[i];
            c[i] = xi;
            const T* lrow = Ls + i * LP;
#pragma unroll
            for (int q = 0; q < NT / W; ++q) {
                if (q * W >= i) continue;
                const V v = reinterpret_cast<const V*>(lrow)[q];
#pragma unroll
                for (int e = 0; e < W; ++e) {
                    const int k = q * W + e;
                    if (k < i) c[k] = fma(-vget<T>(v, e), xi, c[k]);
                }
            }
        }
        // 4. transpose: thread t writes column t of X and reads row t.
#pragma unroll
        for (int i = 0; i < NT; ++i) R[i * RP + t] = c[i];
        group_sync<NT>(g);
#pragma unroll
        for (int k = 0; k < NT; ++k) c[k] = R[t * RP + k];

        // 5. M = X L^-1 (back substitution on row t).
#pragma unroll
        for (int j = NT - 1; j >= 0; --j) {
            const T mj = c[j] * rinv[j];
            c[j] = mj;
            const T* lrow = Ls + j * LP;
#pragma unroll
            for (int q = 0; q < NT / W; ++q) {
                if (q * W >= j) continue;
                const V v = reinterpret_cast<const V*>(lrow)[q];
#pragma unroll
                for (int e = 0; e < W; ++e) {
                    const int k = q * W + e;
                    if (k < j) c[k] = fma(-vget<T>(v, e), mj, c[k]);
                }
            }
        }
        // 6. Phi(M + M^T) into row t of adj_A's lower triangle.  Thread t only
        //    rewrites row t, which only it has read.
#pragma unroll
        for (int k = 0; k < NT; ++k) R[t * RP + k] = c[k];
        group_sync<NT>(g);
#pragma unroll
        for (int k = 0; k < NT; ++k) c[k] += (k < t) ? R[k * RP + t] : T(0);

        if (active && t < n) {
            T* rowp = Abar + (size_t)b * n * n + (size_t)t * n;
            if constexpr (!S::prefetch) {
                // add the old values in place (no row held across the solve)
                T old[NT];
                load_lower_row<T, NT, VEC>(rowp, t, n, old);
#pragma unroll
                for (int k = 0; k < NT; ++k) c[k] += old[k];
            } else {
#pragma unroll
                for (int k = 0; k < NT; ++k) c[k] += ab[k];
            }
            if constexpr (VEC) {
                V* vp = reinterpret_cast<V*>(rowp);
#pragma unroll
                for (int q = 0; q < NT / W; ++q) {
                    if (q * W + W - 1 <= t) {
                        V v;
#pragma unroll
                        for (int e = 0; e < W; ++e) vset<T>(v, e, c[q * W + e]);
                        vp[q] = v;
                    } else if (q * W <= t) {
                        // chunk straddling the diagonal: write only k <= t
#pragma unroll
                        for (int e = 0; e < W; ++e) {
                            const int k = q * W + e;
                            if (k <= t) rowp[k] = c[k];
                        }
                    }
                }
            } else {
#pragma unroll
                for (int k = 0; k < NT; ++k)
                    if (k <= t && k < n) rowp[k] = c[k];
            }
        }
    }
}

// Persistent grid: resident blocks per SM (queried once per kernel) times the
// SM count of the current device, capped by the number of tasks.
template <typename K>
int persistent_grid(K kern, size_t smem, int64_t tasks, int* per_sm_cache) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (*per_sm_cache <= 0) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kBlock, smem) !=
                cudaSuccess || per_sm < 1) {
            cudaGetLastError();
            per_sm = 1;
        }
        *per_sm_cache = per_sm;
    }
    const int64_t full = (int64_t)std::max(sms, 1) * *per_sm_cache;
    return (int)std::max<int64_t>(1, std::min<int64_t>(full, tasks));
}

template <typename T, int NT, bool VEC>
cudaError_t launch_fwd_nt(const T* A, T* L, int32_t* status, int64_t batch, int n,
                          cudaStream_t stream) {
    constexpr int G = kBlock / NT;
    const int64_t tasks = (batch + G - 1) / G;
    auto kern = small_potrf_kernel<T, NT, VEC>;
    // persistent blocks when the kernel prefetches, else one block per group
    static int per_sm = 0;
    const int64_t grid = NT * sizeof(T) <= 64 ? persistent_grid(kern, 0, tasks, &per_sm) : tasks;
    kern<<<(unsigned)grid, kBlock, 0, stream>>>(A, L, status, batch, n);
    return cudaGetLastError();
}

template <typename T, int NT, bool VEC>
cudaError_t launch_adj_nt(const T* L, const T* Lbar, T* Abar, const int32_t* status,
                          int64_t batch, int n, cudaStream_t stream) {
    using S = AdjSmem<T, NT>;
    const int64_t tasks = (batch + S::G - 1) / S::G;
    auto kern = small_potrf_adj_kernel<T, NT, VEC>;
    static int per_sm = 0;
    if (S::bytes > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)S::bytes);
        if (e != cudaSuccess) return e;
    }
    const int64_t grid = S::prefetch ? persistent_grid(kern, S::bytes, tasks, &per_sm) : tasks;
    kern<<<(unsigned)grid, kBlock, S::bytes, stream>>>(L, Lbar, Abar, status, batch, n);
    return cudaGetLastError();
}

}  // namespace

int small_nt(int n) { return n <= 8 ? 8 : n <= 16 ? 16 : n <= 32 ? 32 : 64; }

template <typename T>
cudaError_t small_fwd(const T* A, T* L, int32_t* status, int64_t batch, int n, bool vec,
                      cudaStream_t stream) {
    const int nt = small_nt(n);
#define CHOL_FWD_CASE(NT)                                                                  \
    if (nt == NT) return vec ? launch_fwd_nt<T, NT, true>(A, L, status, batch, n, stream)  \
                             : launch_fwd_nt<T, NT, false>(A, L, status, batch, n, stream);
    CHOL_FWD_CASE(8)
    CHOL_FWD_CASE(16)
    CHOL_FWD_CASE(32)
    CHOL_FWD_CASE(64)
#undef CHOL_FWD_CASE
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t small_adj(const T* L, const T* Lbar, T* Abar, const int32_t* status, int64_t batch,
                      int n, bool vec, cudaStream_t stream) {
    const int nt = small_nt(n);
#define CHOL_ADJ_CASE(NT)                                                                    \
    if (nt == NT)                                                                            \
        return vec ? launch_adj_nt<T, NT, true>(L, Lbar, Abar, status, batch, n, stream)     \
                   : launch_adj_nt<T, NT, false>(L, Lbar, Abar, status, batch, n, stream);
    CHOL_ADJ_CASE(8)
    CHOL_ADJ_CASE(16)
    CHOL_ADJ_CASE(32)
    CHOL_ADJ_CASE(64)
#undef CHOL_ADJ_CASE
    return cudaErrorInvalidValue;
}

template cudaError_t small_fwd<float>(const float*, float*, int32_t*, int64_t, int, bool,
                                      cudaStream_t);
template cudaError_t small_fwd<double>(const double*, double*, int32_t*, int64_t, int, bool,
                                       cudaStream_t);
template cudaError_t small_adj<float>(const float*, const float*, float*, const int32_t*,
                                      int64_t, int, bool, cudaStream_t);
template cudaError_t small_adj<double>(const double*, const double*, double*, const int32_t*,
                                       int64_t, int, bool, cudaStream_t);

}  // namespace chol
