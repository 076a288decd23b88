/*
 * chol_tile.cuh -- device-side tile API: the Cholesky factor of one tile and
 * its adjoint, computed by all threads of a thread block on a tile in shared
 * memory, for use inside a caller's own kernel (CUDA C++17, sm_103a).
 *
 * NVIDIA/warp issue #1316 uses the factorisation this way: wp.tile_cholesky
 * on a tile inside a kernel launched with launch_tiled (block_dim = 64), with
 * adj_tile_cholesky as its reverse mode (its closing comment: the symmetric-
 * matrix derivative of Murray 2016, gradients accumulated into the lower
 * triangle of A).  These are the same operations for a CUDA kernel; the
 * library's blocked path factors and differentiates its diagonal tiles with
 * them.
 *
 * Rules for both calls
 *   - Every thread of the block calls the function, with the same arguments;
 *     THREADS == blockDim.x, a multiple of 32.  The tile is in shared memory
 *     and must be visible to all threads on entry (a __syncthreads after it
 *     was written); the results are visible to all threads on return.
 *   - `at(i, j)` gives the offset of element (i, j), i >= j, in the tile's
 *     storage: RowMajor{ld} (row-major, leading dimension ld) or PackedLower
 *     (the lower triangle packed by rows, n (n + 1) / 2 elements).  Only
 *     elements on and below the diagonal are read or written.
 *   - Arithmetic is in T: float, double, or the complex types
 *     chol_tile::cplx<float> / cplx<double> (interleaved real and imaginary
 *     parts, the layout of C99 complex and torch complex64/128), for which
 *     the factor is the Hermitian A = L L^H (jaxmg docs "Cholesky
 *     factorization", intro: "symmetric or Hermitian positive-definite"):
 *     conjugates appear where the real recurrence transposes, the pivot is
 *     the real part of the diagonal and L's diagonal is real.  For a pivot d
 *     the factor takes 1 / l_jj = rsqrt(d) from CUDA's reciprocal square root
 *     and l_jj = d * rsqrt(d): one transcendental per column on the serial
 *     chain, within a few ulp of the correctly rounded values.  The adjoint
 *     divides by l_jj.  No wait is unbounded and nothing traps.
 */
#ifndef CHOL_TILE_CUH
#define CHOL_TILE_CUH

#include <cuda_runtime.h>

namespace chol_tile {

struct RowMajor {
    int ld;
    __device__ __forceinline__ int operator()(int i, int j) const { return i * ld + j; }
};

struct PackedLower {
    __device__ __forceinline__ int operator()(int i, int j) const { return i * (i + 1) / 2 + j; }
};

// Complex element: real part, then imaginary part.
template <typename R>
struct __align__(2 * sizeof(R)) cplx {
    R re, im;
};

namespace detail {
__device__ __forceinline__ float rsqrt_t(float x) { return rsqrtf(x); }
__device__ __forceinline__ double rsqrt_t(double x) { return rsqrt(x); }

// Scalar helpers that make one recurrence serve real and complex elements.
template <typename T> struct real_of { using type = T; };
template <typename R> struct real_of<cplx<R>> { using type = R; };

template <typename T> __device__ __forceinline__ T zero() { return T{}; }
__device__ __forceinline__ float re(float x) { return x; }
__device__ __forceinline__ double re(double x) { return x; }
template <typename R> __device__ __forceinline__ R re(cplx<R> x) { return x.re; }
__device__ __forceinline__ float conj(float x) { return x; }
__device__ __forceinline__ double conj(double x) { return x; }
template <typename R> __device__ __forceinline__ cplx<R> conj(cplx<R> x) { return {x.re, -x.im}; }
// a * r for real r
__device__ __forceinline__ float scale(float a, float r) { return a * r; }
__device__ __forceinline__ double scale(double a, double r) { return a * r; }
template <typename R> __device__ __forceinline__ cplx<R> scale(cplx<R> a, R r) {
    return {a.re * r, a.im * r};
}
template <typename T> __device__ __forceinline__ T from_real(typename real_of<T>::type r) {
    T x{};
    if constexpr (sizeof(T) == sizeof(r)) {
        x = r;
    } else {
        x.re = r;
    }
    return x;
}
// c + a * b and c - a * b (complex: four fused multiply-adds)
__device__ __forceinline__ float madd(float a, float b, float c) { return fmaf(a, b, c); }
__device__ __forceinline__ double madd(double a, double b, double c) { return fma(a, b, c); }
template <typename R>
__device__ __forceinline__ cplx<R> madd(cplx<R> a, cplx<R> b, cplx<R> c) {
    return {fma(-a.im, b.im, fma(a.re, b.re, c.re)), fma(a.im, b.re, fma(a.re, b.im, c.im))};
}
__device__ __forceinline__ float msub(float a, float b, float c) { return fmaf(-a, b, c); }
__device__ __forceinline__ double msub(double a, double b, double c) { return fma(-a, b, c); }
template <typename R>
__device__ __forceinline__ cplx<R> msub(cplx<R> a, cplx<R> b, cplx<R> c) {
    return {fma(a.im, b.im, fma(-a.re, b.re, c.re)), fma(-a.im, b.re, fma(-a.re, b.im, c.im))};
}
__device__ __forceinline__ float add(float a, float b) { return a + b; }
__device__ __forceinline__ double add(double a, double b) { return a + b; }
template <typename R> __device__ __forceinline__ cplx<R> add(cplx<R> a, cplx<R> b) {
    return {a.re + b.re, a.im + b.im};
}
__device__ __forceinline__ float sub(float a, float b) { return a - b; }
__device__ __forceinline__ double sub(double a, double b) { return a - b; }
template <typename R> __device__ __forceinline__ cplx<R> sub(cplx<R> a, cplx<R> b) {
    return {a.re - b.re, a.im - b.im};
}
// Re(conj(a) * b) + acc
__device__ __forceinline__ float re_dot(float a, float b, float acc) { return fmaf(a, b, acc); }
__device__ __forceinline__ double re_dot(double a, double b, double acc) { return fma(a, b, acc); }
template <typename R> __device__ __forceinline__ R re_dot(cplx<R> a, cplx<R> b, R acc) {
    return fma(a.im, b.im, fma(a.re, b.re, acc));
}
__device__ __forceinline__ float shfl_xor(float x, int o) { return __shfl_xor_sync(0xffffffffu, x, o); }
__device__ __forceinline__ double shfl_xor(double x, int o) { return __shfl_xor_sync(0xffffffffu, x, o); }
template <typename R> __device__ __forceinline__ cplx<R> shfl_xor(cplx<R> x, int o) {
    return {__shfl_xor_sync(0xffffffffu, x.re, o), __shfl_xor_sync(0xffffffffu, x.im, o)};
}
}  // namespace detail

namespace detail {

// Element (i, j) of the diagonal sub-tile that starts at (o, o).
template <typename Idx>
struct Shift {
    Idx at;
    int o;
    __device__ __forceinline__ int operator()(int i, int j) const { return at(o + i, o + j); }
};

// The column recurrence of potrf (below), one column per step.
template <int THREADS, typename T, typename Idx>
__device__ int potrf_columns(T* a, int n, Idx at) {
    static_assert(THREADS % 32 == 0, "THREADS is a whole number of warps");
    using R = typename detail::real_of<T>::type;
    __shared__ R s_inv;
    const int tid = threadIdx.x;
    for (int j = 0; j < n; ++j) {
        const R d = detail::re(a[at(j, j)]);
        if (!(d > R(0))) {  // every thread read the same value: a uniform exit
            __syncthreads();
            return j + 1;
        }
        // one thread takes 1 / l_jj (the transcendental is the slowest step
        // of the column's chain and the same for every thread), the others
        // read it after the barrier
        if (tid == 0) s_inv = detail::rsqrt_t(d);
        __syncthreads();                     // every thread has read the pivot
        const R inv = s_inv;
        for (int i = j + 1 + tid; i < n; i += THREADS) a[at(i, j)] = detail::scale(a[at(i, j)], inv);
        if (tid == 0) a[at(j, j)] = detail::from_real<T>(d * inv);
        __syncthreads();
        // trailing update of the lower part, 16 x THREADS/16 threads over (i, c):
        // a_ic -= l_ij conj(l_cj)
        const int ty = tid / 16, tx = tid % 16;
        for (int i = j + 1 + ty; i < n; i += THREADS / 16) {
            const T lij = a[at(i, j)];
            for (int c = j + 1 + tx; c <= i; c += 16)
                a[at(i, c)] = detail::msub(lij, detail::conj(a[at(c, j)]), a[at(i, c)]);
        }
        __syncthreads();
    }
    return 0;
}

// The unblocked reverse sweep of potrf_adj (below), one column per step.
template <int THREADS, typename T, typename Idx>
__device__ void potrf_adj_columns(const T* l, T* w, int n, Idx at) {
    static_assert(THREADS % 32 == 0, "THREADS is a whole number of warps");
    using R = typename detail::real_of<T>::type;
    constexpr int kRinv = 128;  // reciprocals of the diagonal kept for tiles up to this order
    __shared__ R red[THREADS / 32];
    __shared__ R rinv[kRinv];
    const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
    // 1 / l_jj for every column up front, one division per thread, so no
    // column's chain waits for one
    const bool pre = n <= kRinv;
    if (pre) {
        for (int j = tid; j < n; j += THREADS) rinv[j] = R(1) / detail::re(l[at(j, j)]);
        __syncthreads();
    }
    for (int j = n - 1; j >= 0; --j) {
        // s = Re sum_{i > j} conj(l_ij) w_ij
        R part = R(0);
        for (int i = j + 1 + tid; i < n; i += THREADS) part = detail::re_dot(l[at(i, j)], w[at(i, j)], part);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) red[warp] = part;
        __syncthreads();
        const R inv = pre ? rinv[j] : R(1) / detail::re(l[at(j, j)]);
        // column j: the diagonal (real) from the sum (one thread forms it),
        // the rest scaled
        for (int i = j + 1 + tid; i < n; i += THREADS) w[at(i, j)] = detail::scale(w[at(i, j)], inv);
        if (tid == 0) {
            R sum = R(0);
#pragma unroll
            for (int k = 0; k < THREADS / 32; ++k) sum += red[k];
            w[at(j, j)] = detail::from_real<T>((detail::re(w[at(j, j)]) - sum * inv) * inv);
        }
        __syncthreads();
        // row j left of the diagonal: w_jk -= sum_{i >= j} conj(w_ij) l_ik
        // (two partial sums halve the dependent chain)
        for (int k = tid; k < j; k += THREADS) {
            T acc0 = detail::zero<T>(), acc1 = detail::zero<T>();
            int i = j;
            for (; i + 1 < n; i += 2) {
                acc0 = detail::madd(detail::conj(w[at(i, j)]), l[at(i, k)], acc0);
                acc1 = detail::madd(detail::conj(w[at(i + 1, j)]), l[at(i + 1, k)], acc1);
            }
            if (i < n) acc0 = detail::madd(detail::conj(w[at(i, j)]), l[at(i, k)], acc0);
            w[at(j, k)] = detail::sub(w[at(j, k)], detail::add(acc0, acc1));
        }
        // rows below, left of column j: w_ik -= w_ij l_jk
        const int ty = tid / 16, tx = tid % 16;
        for (int i = j + 1 + ty; i < n; i += THREADS / 16) {
            const T wij = w[at(i, j)];
            for (int k = tx; k < j; k += 16) w[at(i, k)] = detail::msub(wij, l[at(j, k)], w[at(i, k)]);
        }
        __syncthreads();
        if (tid == 0) w[at(j, j)] = detail::scale(w[at(j, j)], R(0.5));
        // (the next column's first barrier orders this write; nothing before
        //  it reads w_jj)
    }
    __syncthreads();
}

constexpr int kSub = 32;  // sub-tile of the blocked forms

// Right-looking blocked factor for larger tiles: per 32-column sub-tile the
// column recurrence on the diagonal sub-tile, a panel solve of the rows below
// (one thread per row, the row in registers) and the trailing update of the
// lower part; the two bulk steps keep every warp busy between barriers.
template <int THREADS, typename T, typename Idx>
__device__ int potrf_blocked(T* a, int n, Idx at) {
    using R = typename real_of<T>::type;
    __shared__ R rinv[kSub];
    const int tid = threadIdx.x;
    for (int q0 = 0; q0 < n; q0 += kSub) {
        const int m = min(kSub, n - q0);
        const int st = potrf_columns<THREADS>(a, m, Shift<Idx>{at, q0});
        if (st != 0) return q0 + st;  // the same in every thread
        const int r0 = q0 + m;
        if (r0 >= n) break;
        for (int c = tid; c < m; c += THREADS) rinv[c] = R(1) / re(a[at(q0 + c, q0 + c)]);
        __syncthreads();
        // rows below: x L_S^H = a_r (forward substitution), L_S the sub-tile's
        // factor (rows below exist only under a full sub-tile: m == kSub)
        for (int r = r0 + tid; r < n; r += THREADS) {
            T x[kSub];
#pragma unroll
            for (int c = 0; c < kSub; ++c) {
                T s = a[at(r, q0 + c)];
#pragma unroll
                for (int k = 0; k < c; ++k) s = msub(x[k], conj(a[at(q0 + c, q0 + k)]), s);
                x[c] = scale(s, rinv[c]);
            }
#pragma unroll
            for (int c = 0; c < kSub; ++c) a[at(r, q0 + c)] = x[c];
        }
        __syncthreads();
        // trailing lower part: a_rc -= sum_k l_rk conj(l_ck), r >= c >= r0
        const int ty = tid / 16, tx = tid % 16;
        for (int r = r0 + ty; r < n; r += THREADS / 16) {
            for (int c = r0 + tx; c <= r; c += 16) {
                T s0 = zero<T>(), s1 = zero<T>();
                int k = 0;
                for (; k + 1 < m; k += 2) {
                    s0 = madd(a[at(r, q0 + k)], conj(a[at(c, q0 + k)]), s0);
                    s1 = madd(a[at(r, q0 + k + 1)], conj(a[at(c, q0 + k + 1)]), s1);
                }
                if (k < m) s0 = madd(a[at(r, q0 + k)], conj(a[at(c, q0 + k)]), s0);
                a[at(r, c)] = sub(a[at(r, c)], add(s0, s1));
            }
        }
        __syncthreads();
    }
    return 0;
}

// Murray's blocked reverse sweep over 32-column sub-tiles, the same steps as
// the library's blocked adjoint inside one tile: for sub-tile columns J from
// the last, with C the rows of w below the sub-tile:
//   C <- C L_JJ^-1; w_JK -= C^H L_{below, K} (K <= J); w_IK -= C L_JK
//   (I > J, K < J); the column sweep of w_JJ; w_JK -= (w_JJ + w_JJ^H) L_JK.
template <int THREADS, typename T, typename Idx>
__device__ void potrf_adj_blocked(const T* l, T* w, int n, Idx at) {
    using R = typename real_of<T>::type;
    __shared__ R rinv[kSub];
    const int tid = threadIdx.x;
    const int nb = (n + kSub - 1) / kSub;
    for (int jb = nb - 1; jb >= 0; --jb) {
        const int j0 = jb * kSub, m = min(kSub, n - j0), r0 = j0 + m;
        for (int c = tid; c < m; c += THREADS) rinv[c] = R(1) / re(l[at(j0 + c, j0 + c)]);
        __syncthreads();
        // C <- C L_JJ^-1, one row per thread: m_c = (c_c - sum_{k>c} m_k l_kc) / l_cc
        // (rows below exist only under a full sub-tile: m == kSub)
        for (int r = r0 + tid; r < n; r += THREADS) {
            T x[kSub];
#pragma unroll
            for (int c = 0; c < kSub; ++c) x[c] = w[at(r, j0 + c)];
#pragma unroll
            for (int cc = 0; cc < kSub; ++cc) {
                const int c = kSub - 1 - cc;
                T s = x[c];
#pragma unroll
                for (int k = c + 1; k < kSub; ++k) s = msub(x[k], l[at(j0 + k, j0 + c)], s);
                x[c] = scale(s, rinv[c]);
            }
#pragma unroll
            for (int c = 0; c < kSub; ++c) w[at(r, j0 + c)] = x[c];
        }
        __syncthreads();
        // w_JK -= C^H L_{below, K} for columns b < j0 + m (lower part inside
        // the sub-tile), and w_IK -= C L_JK for rows r >= r0, columns b < j0:
        // the two touch different entries and only read C, so they share a phase
        const int wb = j0 + m;
        const int n_row = m * wb;
        const int n_upd = (n - r0) * j0;
        for (int t = tid; t < n_row + n_upd; t += THREADS) {
            if (t < n_row) {
                const int a = t / wb, b = t % wb;
                if (b > j0 + a) continue;
                T s0 = zero<T>(), s1 = zero<T>();
                int r = r0;
                for (; r + 1 < n; r += 2) {
                    s0 = madd(conj(w[at(r, j0 + a)]), l[at(r, b)], s0);
                    s1 = madd(conj(w[at(r + 1, j0 + a)]), l[at(r + 1, b)], s1);
                }
                if (r < n) s0 = madd(conj(w[at(r, j0 + a)]), l[at(r, b)], s0);
                w[at(j0 + a, b)] = sub(w[at(j0 + a, b)], add(s0, s1));
            } else {
                const int u = t - n_row;
                const int r = r0 + u / j0, b = u % j0;
                T s0 = zero<T>(), s1 = zero<T>();
                int c = 0;
                for (; c + 1 < m; c += 2) {
                    s0 = madd(w[at(r, j0 + c)], l[at(j0 + c, b)], s0);
                    s1 = madd(w[at(r, j0 + c + 1)], l[at(j0 + c + 1, b)], s1);
                }
                if (c < m) s0 = madd(w[at(r, j0 + c)], l[at(j0 + c, b)], s0);
                w[at(r, b)] = sub(w[at(r, b)], add(s0, s1));
            }
        }
        __syncthreads();
        // the diagonal sub-tile's own sweep
        potrf_adj_columns<THREADS>(l, w, m, Shift<Idx>{at, j0});
        // w_JK -= (w_JJ + w_JJ^H) L_JK, K < J: the lower part of w_JJ, mirrored
        // (conjugated) above the diagonal, doubled on it
        for (int t = tid; t < m * j0; t += THREADS) {
            const int a = t / j0, b = t % j0;
            T s = zero<T>();
            for (int c = 0; c < m; ++c) {
                T x;
                if (c < a) {
                    x = w[at(j0 + a, j0 + c)];
                } else if (c > a) {
                    x = conj(w[at(j0 + c, j0 + a)]);
                } else {
                    x = w[at(j0 + a, j0 + a)];
                    x = add(x, x);
                }
                s = madd(x, l[at(j0 + c, b)], s);
            }
            w[at(j0 + a, b)] = sub(w[at(j0 + a, b)], s);
        }
        __syncthreads();
    }
}

}  // namespace detail

/*
 * potrf -- in place, a = chol(a), lower: the right-looking column recurrence
 * (jaxmg docs "Cholesky factorization": the lower factor and a status), in
 * 32-column blocks for n > 64.  Returns 0, or j + 1 for the first column j
 * whose pivot is not > 0 (zero, negative or NaN), the same value in every
 * thread; the tile from column j on is then unspecified.
 */
template <int THREADS, typename T, typename Idx>
__device__ int potrf(T* a, int n, Idx at) {
    static_assert(THREADS % 32 == 0, "THREADS is a whole number of warps");
    if (n > 64) return detail::potrf_blocked<THREADS>(a, n, at);
    return detail::potrf_columns<THREADS>(a, n, at);
}

/*
 * potrf_adj -- Murray's (2016) unblocked reverse sweep, in place on w:
 * l is the factor from potrf (read only); on entry w holds the gradient of
 * the loss with respect to l's lower entries, on return the gradient with
 * respect to the lower entries a_ij (i >= j) that potrf read.  That is
 * Phi(M + M^T) with M = l^-T Phi(l^T w) l^-1, Phi keeping the lower triangle
 * and halving the diagonal (warp issue #1316's closing comment), reached
 * column by column from j = n - 1 down to 0 in n^3 / 3 multiply-adds (for
 * n > 64 in 32-column blocks, the same steps as the library's blocked
 * adjoint, so that the bulk of the work runs between few barriers).
 * Complex elements: w holds dLoss/dRe + i dLoss/dIm of a real loss; on
 * return the entries below the diagonal hold M_ij + conj(M_ji) and the
 * diagonal Re(M_ii) (imaginary part 0), with M = l^-H Phi(l^H w) l^-1; the
 * sweep reads only the real part of w's diagonal.
 */
template <int THREADS, typename T, typename Idx>
__device__ void potrf_adj(const T* l, T* w, int n, Idx at) {
    static_assert(THREADS % 32 == 0, "THREADS is a whole number of warps");
    if (n > 64) {
        detail::potrf_adj_blocked<THREADS>(l, w, n, at);
        return;
    }
    detail::potrf_adj_columns<THREADS>(l, w, n, at);
}

}  // namespace chol_tile

#endif  // CHOL_TILE_CUH
