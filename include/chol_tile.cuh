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
 *   - Arithmetic is in T (float or double).  For a pivot d the factor takes
 *     1 / l_jj = rsqrt(d) from CUDA's reciprocal square root and
 *     l_jj = d * rsqrt(d): one transcendental per column on the serial chain,
 *     within a few ulp of the correctly rounded values.  The adjoint divides
 *     by l_jj.  No wait is unbounded and nothing traps.
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

namespace detail {
__device__ __forceinline__ float rsqrt_t(float x) { return rsqrtf(x); }
__device__ __forceinline__ double rsqrt_t(double x) { return rsqrt(x); }
}  // namespace detail

/*
 * potrf -- in place, a = chol(a), lower: the right-looking column recurrence
 * (jaxmg docs "Cholesky factorization": the lower factor and a status).
 * Returns 0, or j + 1 for the first column j whose pivot is not > 0 (zero,
 * negative or NaN), the same value in every thread; the tile from column j on
 * is then unspecified.
 */
template <int THREADS, typename T, typename Idx>
__device__ int potrf(T* a, int n, Idx at) {
    static_assert(THREADS % 32 == 0, "THREADS is a whole number of warps");
    const int tid = threadIdx.x;
    for (int j = 0; j < n; ++j) {
        const T d = a[at(j, j)];
        if (!(d > T(0))) {  // every thread read the same value: a uniform exit
            __syncthreads();
            return j + 1;
        }
        const T inv = detail::rsqrt_t(d);  // 1 / l_jj, then products
        const T ljj = d * inv;
        __syncthreads();                     // every thread has read the pivot
        for (int i = j + 1 + tid; i < n; i += THREADS) a[at(i, j)] *= inv;
        if (tid == 0) a[at(j, j)] = ljj;
        __syncthreads();
        // trailing update of the lower part, 16 x THREADS/16 threads over (i, c)
        const int ty = tid / 16, tx = tid % 16;
        for (int i = j + 1 + ty; i < n; i += THREADS / 16) {
            const T lij = a[at(i, j)];
            for (int c = j + 1 + tx; c <= i; c += 16) a[at(i, c)] = fma(-lij, a[at(c, j)], a[at(i, c)]);
        }
        __syncthreads();
    }
    return 0;
}

/*
 * potrf_adj -- Murray's (2016) unblocked reverse sweep, in place on w:
 * l is the factor from potrf (read only); on entry w holds the gradient of
 * the loss with respect to l's lower entries, on return the gradient with
 * respect to the lower entries a_ij (i >= j) that potrf read.  That is
 * Phi(M + M^T) with M = l^-T Phi(l^T w) l^-1, Phi keeping the lower triangle
 * and halving the diagonal (warp issue #1316's closing comment), reached
 * column by column from j = n - 1 down to 0 in n^3 / 3 multiply-adds.
 */
template <int THREADS, typename T, typename Idx>
__device__ void potrf_adj(const T* l, T* w, int n, Idx at) {
    static_assert(THREADS % 32 == 0, "THREADS is a whole number of warps");
    __shared__ T red[THREADS / 32];
    const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
    for (int j = n - 1; j >= 0; --j) {
        // s = sum_{i > j} l_ij w_ij
        T part = T(0);
        for (int i = j + 1 + tid; i < n; i += THREADS) part = fma(l[at(i, j)], w[at(i, j)], part);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) red[warp] = part;
        __syncthreads();
        T sum = T(0);
#pragma unroll
        for (int k = 0; k < THREADS / 32; ++k) sum += red[k];
        const T inv = T(1) / l[at(j, j)];
        // column j: the diagonal from the sum, the rest scaled
        for (int i = j + 1 + tid; i < n; i += THREADS) w[at(i, j)] *= inv;
        if (tid == 0) w[at(j, j)] = (w[at(j, j)] - sum * inv) * inv;
        __syncthreads();
        // row j left of the diagonal: w_jk -= sum_{i >= j} w_ij l_ik
        // (two partial sums halve the dependent chain)
        for (int k = tid; k < j; k += THREADS) {
            T acc0 = T(0), acc1 = T(0);
            int i = j;
            for (; i + 1 < n; i += 2) {
                acc0 = fma(w[at(i, j)], l[at(i, k)], acc0);
                acc1 = fma(w[at(i + 1, j)], l[at(i + 1, k)], acc1);
            }
            if (i < n) acc0 = fma(w[at(i, j)], l[at(i, k)], acc0);
            w[at(j, k)] -= acc0 + acc1;
        }
        // rows below, left of column j: w_ik -= w_ij l_jk
        const int ty = tid / 16, tx = tid % 16;
        for (int i = j + 1 + ty; i < n; i += THREADS / 16) {
            const T wij = w[at(i, j)];
            for (int k = tx; k < j; k += 16) w[at(i, k)] = fma(-wij, l[at(j, k)], w[at(i, k)]);
        }
        __syncthreads();
        if (tid == 0) w[at(j, j)] *= T(0.5);
        // (the next column's first barrier orders this write; nothing before
        //  it reads w_jj)
    }
    __syncthreads();
}

}  // namespace chol_tile

#endif  // CHOL_TILE_CUH
