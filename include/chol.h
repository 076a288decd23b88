/*
 * chol.h -- C ABI of the GB300 (sm_103a) differentiable Cholesky library.
 *
 * Two calls make up the path (chol_fwd_inplace / chol_adj_inplace are their
 * in-place forms):
 *
 *   chol_fwd  the Cholesky factorisation A = L L^T of symmetric positive-
 *             definite matrices, lower factor, out of place, with a per-matrix
 *             status.  Defined by the jaxmg docs "Cholesky factorization"
 *             (intro: potrf returns the lower-triangular factor without a
 *             solve; "Advanced: control the outer jax.jit": the call returns
 *             `factor, status`) and by NVIDIA/warp issue #1316's closing
 *             comment (wp.tile_cholesky, the out-of-place variant).
 *
 *   chol_adj  its reverse-mode adjoint, the symmetric-matrix derivative of
 *             Cholesky (Murray 2016) as NVIDIA/warp issue #1316's closing
 *             comment states it: S = Phi(L^T adj_L), two triangular solves
 *             against L^T and L, accumulation into the lower triangle of A's
 *             gradient.  Phi keeps the lower triangle and halves the diagonal.
 *
 * Conventions shared by every call
 *   - Matrices are dense, row-major, contiguous: element (i, j) of matrix b
 *     lives at offset (b * n + i) * n + j.  dtype selects float32 or float64.
 *   - Every pointer is a DEVICE pointer (cudaMalloc'd, stream-ordered or
 *     managed memory) owned by the caller; the library keeps no state and
 *     never frees or retains caller memory.  Element pointers must be aligned
 *     to their element size; 16-byte alignment (with n a multiple of 16 / the
 *     element size) selects vectorised loads.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     only enqueue work on it and return without synchronising; results are
 *     stream-ordered.  No kernel traps, asserts or waits without bound.
 *   - Invalid arguments are reported synchronously by a negative return code
 *     (chol_strerror gives the text) and nothing is enqueued.  A matrix that
 *     is not positive definite is data, not an error: it sets its status.
 *   - batch == 0 is a no-op that returns CHOL_OK.
 *   - Complex Hermitian matrices (CHOL_C64, CHOL_C128; the jaxmg docs
 *     "Cholesky factorization" intro factor "a symmetric or Hermitian
 *     positive-definite matrix"): A = L L^H with conjugate transposes where
 *     the real case transposes.  The forward reads the lower triangle and
 *     only the real part of the diagonal; L's diagonal is real (imaginary
 *     part 0).  The adjoint takes adj_L as dLoss/dRe(L) + i dLoss/dIm(L) of a
 *     real loss and adds to adj_A the derivative with respect to the entries
 *     the forward reads: dLoss/dRe(a_ij) + i dLoss/dIm(a_ij) below the
 *     diagonal and dLoss/dRe(a_ii) on it, i.e. M_ij + conj(M_ji) and Re(M_ii)
 *     with M = L^-H Phi(L^H tril(adj_L)) L^-1.  The blocked tile of CHOL_C128
 *     is at most 64 (tile 128 returns CHOL_EINVAL; the default caps at 64).
 */
#ifndef CHOL_GB300_H
#define CHOL_GB300_H

#include <stdint.h>

#if defined(__GNUC__)
#define CHOL_API __attribute__((visibility("default")))
#else
#define CHOL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element types.  The complex types hold interleaved (real, imaginary) pairs,
 * the layout of C99 float/double complex and torch complex64/complex128; for
 * them every call works on Hermitian matrices, A = L L^H (see below). */
typedef enum { CHOL_F32 = 0, CHOL_F64 = 1, CHOL_C64 = 2, CHOL_C128 = 3 } chol_dtype_t;

enum {
    CHOL_OK = 0,
    CHOL_EINVAL = -1,  /* null/misaligned/host pointer, n <= 0, batch < 0, bad tile, size overflow */
    CHOL_EDTYPE = -2,  /* dtype is not one of chol_dtype_t                                           */
    CHOL_EALIAS = -3,  /* an output overlaps an input it must not overlap                            */
    CHOL_ENOMEM = -4,  /* workspace allocation failed                                                */
    CHOL_ECUDA = -5    /* a CUDA call or kernel launch failed (see cudaGetLastError)                 */
};

/*
 * chol_fwd -- L_b = chol(A_b) for b in [0, batch).
 *   A       in : dtype[batch][n][n].  Only the lower triangle (j <= i) is
 *                read; the upper triangle may hold anything.  Never written.
 *   L       out: dtype[batch][n][n].  Fully written: the factor on and below
 *                the diagonal, exact zeros above it.  Must not overlap A or
 *                status (CHOL_EALIAS).
 *   status  out: int32[batch].  0 if A_b is positive definite; otherwise
 *                j + 1 for the first column j (0-based) whose pivot
 *                a_jj - sum_k l_jk^2 is not > 0 (zero, negative or NaN), the
 *                LAPACK `info` convention.  For such a matrix the part of L_b
 *                from column j on is unspecified.
 * n <= 64 runs one fused register/shared-memory kernel per batch; larger n
 * runs the blocked right-looking algorithm (diagonal-tile factor, panel
 * triangular solve, trailing update) with the default tile: 128 for
 * float64 with n > 128 and batch * 8 <= SMs of the device, and for
 * n >= 2048; else 64 when batch * ceil(n/64)^2 >= 4 * SMs; else 32
 * (complex double: at most 64).  float64 with 128-wide tiles runs the panel
 * solve and the trailing update on the tensor cores (exact digit products);
 * it takes a workspace of about 450 KB per 128 rows per matrix with
 * cudaMallocAsync/cudaFreeAsync on `stream` (CHOL_ENOMEM on failure).  With
 * at least three tile columns and `stream` not being captured, part of each
 * trailing update runs on a second stream of the library's, beside the next
 * diagonal factor; `stream` waits for it before the call's work ends, so the
 * call is ordered on `stream` like any other.  For batch * 8 <= SMs the
 * diagonal tiles (orders 33 .. 128, float and double) are factored by a
 * thread-block cluster of 8 SMs per matrix (16 for batch * 16 <= SMs where
 * the device schedules a 16-block cluster).
 */
CHOL_API int chol_fwd(int64_t batch, int32_t n, int32_t dtype, const void* A, void* L,
             int32_t* status, void* stream);

/*
 * chol_fwd_ex -- chol_fwd with an explicit tile for the blocked path
 * (n > 64): tile in {32, 64, 128}, or 0 for the default.  Results are
 * tile-independent up to rounding.  Ignored for n <= 64.
 */
CHOL_API int chol_fwd_ex(int64_t batch, int32_t n, int32_t dtype, const void* A, void* L,
                int32_t* status, int32_t tile, void* stream);

/*
 * chol_adj -- adj_A_b += dA for the loss gradient adj_L_b, b in [0, batch).
 *   L       in : dtype[batch][n][n], the factor from chol_fwd.  Only its lower
 *                triangle is read.
 *   adj_L   in : dtype[batch][n][n], the gradient of the loss with respect to
 *                L.  Only its lower triangle is read (the upper is taken as 0).
 *   adj_A   in/out: dtype[batch][n][n].  On the lower triangle, adds the
 *                partial derivatives of the loss with respect to the entries
 *                a_ij (i >= j) that chol_fwd reads:
 *                  M = L^-T Phi(L^T tril(adj_L)) L^-1,
 *                  adj_A_ij += M_ij + M_ji (i > j),  adj_A_ii += M_ii.
 *                The upper triangle is never written.  Must not overlap L,
 *                adj_L or status (CHOL_EALIAS).
 *   status  in : int32[batch] from chol_fwd, or NULL.  Matrices with a non-zero
 *                status are skipped (their adj_A is left unchanged).
 * The gradient of torch.linalg.cholesky (a symmetric matrix G) relates to this
 * one by adj_A = tril(G + G^T) - diag(G).
 * n > 64 needs batch * n * n elements of device workspace, taken with
 * cudaMallocAsync/cudaFreeAsync on `stream` (CHOL_ENOMEM on failure);
 * float64 with 128-wide tiles also takes the operand slices of its
 * tensor-core updates (about 224 KB per 128 x 128 block of L's lower
 * triangle), the inverses of the diagonal tiles and their slices (about
 * 350 KB per tile), plus a few tens of MB.  For batch * 4 <= SMs each
 * diagonal tile's own adjoint is then taken by its literal formula above
 * (three parallel products with the tile's inverse) instead of the serial
 * reverse sweep; the two agree to rounding.  The default tile is chol_fwd's.
 */
CHOL_API int chol_adj(int64_t batch, int32_t n, int32_t dtype, const void* L, const void* adj_L,
             void* adj_A, const int32_t* status, void* stream);

/* chol_adj with an explicit blocked-path tile (as chol_fwd_ex). */
CHOL_API int chol_adj_ex(int64_t batch, int32_t n, int32_t dtype, const void* L, const void* adj_L,
                void* adj_A, const int32_t* status, int32_t tile, void* stream);

/*
 * chol_adj_noalloc -- chol_adj_ex for callers that cannot allocate device
 * memory while they run (inside a CUDA-graph capture that must not grow its
 * memory pool, hosts that forbid device allocation after start-up, plug-ins
 * whose host application owns every allocation).  It has no counterpart in the
 * pages: it exists for those callers only.
 *   Same arguments and error codes as chol_adj_ex, and the same results
 *   except for float64 with 128-wide tiles and n > 128, where chol_adj_ex
 *   takes its tensor-core updates and this call keeps the FMA-pipe ones
 *   (the two agree to about 1e-12 relative).  It calls no allocator: for n > 64 the blocked path's workspace is a fixed 16 MiB
 *   scratch array inside the library (held by every GPU that loads the library
 *   until the process exits), so batch * n * n * element size must be at most
 *   16 MiB, else CHOL_ENOMEM and nothing is enqueued.  n <= 64 needs no
 *   scratch and has no limit.
 *   The first call on a device looks the scratch array's address up; make it
 *   before any stream capture begins.  All calls on a device share the array
 *   and leave their last contents in it (nothing needs clearing: every scratch
 *   element read is first written by the same call), so calls that overlap on
 *   the GPU race and corrupt each other: order them on one stream.
 */
CHOL_API int chol_adj_noalloc(int64_t batch, int32_t n, int32_t dtype, const void* L,
                              const void* adj_L, void* adj_A, const int32_t* status,
                              int32_t tile, void* stream);

/*
 * chol_fwd_inplace -- chol_fwd with the factor written over its input.  The
 * jaxmg docs "Cholesky factorization" donate the input to the factorization
 * (Warning box: do not use the input array after the call) and, under
 * "Advanced: control the outer jax.jit", return a factor that aliases the
 * input work buffer; NVIDIA/warp issue #1316's closing comment names the
 * in-place tile form tile_cholesky_inplace.
 *   A       in/out: dtype[batch][n][n].  On entry its lower triangle is the
 *                matrix (upper triangle ignored); on return the buffer holds
 *                exactly what chol_fwd writes into L: the factor, exact zeros
 *                above the diagonal.
 *   status  out: as chol_fwd.  Must not overlap A (CHOL_EALIAS).
 *   tile    as chol_fwd_ex.
 * Results are bit-identical to chol_fwd_ex with the same tile.
 */
CHOL_API int chol_fwd_inplace(int64_t batch, int32_t n, int32_t dtype, void* A, int32_t* status,
                              int32_t tile, void* stream);

/*
 * chol_adj_inplace -- the adjoint written over its seed: the in-place form's
 * adjoint, which NVIDIA/warp issue #1316's closing comment notes
 * tile_cholesky_inplace lacks.
 *   L       in : as chol_adj.  Must not overlap adj (CHOL_EALIAS).
 *   adj     in/out: dtype[batch][n][n].  On entry its lower triangle is
 *                adj_L (the upper is taken as 0); on return the lower
 *                triangle holds the gradient chol_adj would ADD to a zero
 *                adj_A (M_ij + M_ji below the diagonal, M_ii on it), and a
 *                matrix with non-zero status gets zeros there.  The upper
 *                triangle is never written.
 *   status  in : as chol_adj (or NULL).  Must not overlap adj.
 *   tile    as chol_adj_ex.  The blocked reverse sweep runs on `adj` itself
 *           (it never touches the upper triangle), so no working copy of
 *           the matrices is taken: with the FMA-pipe updates the call
 *           allocates nothing; float64 with 128-wide tiles (the default for
 *           few large matrices) takes only the tensor-core updates' operand
 *           slices and inverses that chol_adj takes beside its working
 *           matrices (cudaMallocAsync/cudaFreeAsync on `stream`,
 *           CHOL_ENOMEM on failure).
 * Results are bit-identical to chol_adj_ex with the same tile into a zeroed
 * adj_A (up to the sign of zeros).
 */
CHOL_API int chol_adj_inplace(int64_t batch, int32_t n, int32_t dtype, const void* L, void* adj,
                              const int32_t* status, int32_t tile, void* stream);

/*
 * chol_solve -- X_b = A_b^-1 B_b = L_b^-H L_b^-1 B_b, the solve with the
 * factor that the jaxmg docs "Cholesky factorization" keep out of potrf
 * (intro: the factor is returned "without performing a solve"): forward
 * substitution L Y = B, then back substitution L^H X = Y (L^T for real
 * types).
 *   L       in : dtype[batch][n][n], the factor from chol_fwd; only its lower
 *                triangle is read (and only the real part of a complex
 *                diagonal).
 *   B       in : dtype[batch][n][nrhs], row-major right-hand sides.
 *   X       out: dtype[batch][n][nrhs].  May be B itself (solved in place);
 *                must not otherwise overlap B, and must not overlap L or
 *                status (CHOL_EALIAS).
 *   status  in : int32[batch] from chol_fwd, or NULL.  A matrix with a
 *                non-zero status gets X_b = 0.
 * nrhs >= 0 (0 is a no-op).  Allocates nothing.
 */
CHOL_API int chol_solve(int64_t batch, int32_t n, int32_t nrhs, int32_t dtype, const void* L,
                        const void* B, void* X, const int32_t* status, void* stream);

/*
 * chol_solve_adj -- reverse mode of chol_solve for a real loss with gradient
 * adj_X = dLoss/dX (dLoss/dRe + i dLoss/dIm for complex types):
 *   adj_B += Bb,  Bb = A^-1 adj_X                       (if adj_B != NULL)
 *   adj_L += tril(-(Bb X^H + X Bb^H) L)  on the lower triangle (if adj_L != NULL)
 * from dX = -A^-1 dA X and dA = dL L^H + L dL^H.  adj_L's upper triangle is
 * never written; chol_adj then carries adj_L on to adj_A.
 *   L      in : as chol_solve.        X     in : the result of chol_solve.
 *   adj_X  in : dtype[batch][n][nrhs].
 *   adj_B  in/out (or NULL): dtype[batch][n][nrhs].
 *   adj_L  in/out (or NULL): dtype[batch][n][n].
 *   status in : as chol_solve; matrices with non-zero status are skipped.
 * The outputs must not overlap each other or any input (CHOL_EALIAS).
 * Workspace: batch * n * nrhs elements (three times that with adj_L), taken
 * with cudaMallocAsync/cudaFreeAsync on `stream` (CHOL_ENOMEM on failure).
 */
CHOL_API int chol_solve_adj(int64_t batch, int32_t n, int32_t nrhs, int32_t dtype, const void* L,
                            const void* X, const void* adj_X, void* adj_B, void* adj_L,
                            const int32_t* status, void* stream);

/* Static text for a return code (never NULL). */
CHOL_API const char* chol_strerror(int code);

/* ABI version of this header: (major << 16) | minor. */
CHOL_API int32_t chol_abi_version(void);

#define CHOL_ABI_VERSION ((1 << 16) | 4)

#ifdef __cplusplus
}
#endif

#endif /* CHOL_GB300_H */
