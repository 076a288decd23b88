/*
 * Oracle for the differentiable Cholesky hot path -- TEST INFRASTRUCTURE ONLY.
 *
 * This file is a plain, slow, obviously correct CPU restatement of what the
 * GPU library computes.  Only the test-suite, the smoke check and the CPU
 * baseline leg of the benchmark may build, load or call it; the product path
 * never does.  It shares no code, header or constant with the CUDA sources.
 *
 * What it computes (both in the element type it is compiled for; `double`
 * and `float` instantiations are generated below):
 *
 *  potrf   -- the Cholesky factor A = L L^T of a symmetric positive-definite
 *             matrix, lower factor, out of place, reading only the lower
 *             triangle of A ("jaxmg.potrf ... returning the lower-triangular
 *             factor", jaxmg docs "Cholesky factorization", intro; the
 *             out-of-place form, NVIDIA/warp issue #1316 closing comment).
 *             Written as the textbook column recurrence
 *                 d_j  = a_jj - sum_{k<j} l_jk^2
 *                 l_jj = sqrt(d_j)
 *                 l_ij = (a_ij - sum_{k<j} l_ik l_jk) / l_jj     (i > j)
 *             The status output (jaxmg docs, "Advanced: control the outer
 *             jax.jit": `factor, status = ...`) is read as LAPACK's info:
 *             0 on success, else j+1 for the first column whose pivot d_j is
 *             not > 0 (zero, negative or NaN), after which the recurrence
 *             stops and the rest of L is left as computed so far.
 *
 *  adjoint -- the symmetric-matrix derivative of Cholesky (Murray 2016) as
 *             NVIDIA/warp issue #1316's closing comment states it, literally:
 *                 P   = L^T tril(Lbar)
 *                 S   = Phi(P)      (lower triangle, diagonal halved)
 *                 X   : solve L^T X = S
 *                 M   : solve M L   = X
 *                 Abar_ij += M_ij + M_ji  (i > j),  Abar_ii += M_ii
 *             i.e. the partial derivatives with respect to the lower-triangle
 *             entries that the forward reads.  Upper triangles of Lbar and L
 *             are treated as zero, the upper triangle of Abar is untouched.
 *
 * zpotrf / zpotrf_adj -- the same two operations for complex Hermitian
 *             positive-definite matrices, A = L L^H ("a symmetric or Hermitian
 *             positive-definite matrix", jaxmg docs "Cholesky factorization",
 *             intro), written with conjugate transposes where the real
 *             formulas have transposes:
 *                 d_j  = Re(a_jj) - sum_{k<j} |l_jk|^2      (real pivot)
 *                 l_jj = sqrt(d_j)                           (real)
 *                 l_ij = (a_ij - sum_{k<j} l_ik conj(l_jk)) / l_jj
 *             and, for a real loss whose gradient with respect to L is
 *             Lbar = dLoss/dRe(L) + i dLoss/dIm(L),
 *                 P = L^H tril(Lbar),  S = Phi(P),
 *                 X : solve L^H X = S,  M : solve M L = X,
 *                 Abar_ij += M_ij + conj(M_ji)  (i > j),  Abar_ii += Re(M_ii),
 *             the derivative with respect to the lower entries the forward
 *             reads (real and imaginary parts below the diagonal, the real
 *             part on it: the forward ignores Im(a_jj)).  The pages state the
 *             adjoint for the real case only; this is its Hermitian form.
 *
 * potrs / potrs_adj -- the solve with the factor that potrf leaves for later
 *             (jaxmg docs "Cholesky factorization", intro: potrf returns the
 *             factor "without performing a solve"): X = A^-1 B = L^-H L^-1 B
 *             for B with nrhs columns, by forward substitution L Y = B then
 *             back substitution L^H X = Y, and its reverse mode for a loss
 *             gradient Xbar: Bbar += A^-1 Xbar (the same two solves) and
 *             Lbar += tril(G + G^H) L restricted to the lower triangle, with
 *             G = -Bbar X^H the gradient with respect to A (from
 *             dX = -A^-1 dA X and dA = dL L^H + L dL^H).  Real types read ^H
 *             as ^T.
 *
 * Row-major storage, matrix b of a batch at offset b*n*n.  No blocking,
 * fusion or reordering beyond the formulas above.  The batched wrappers run
 * independent matrices on OpenMP threads (each matrix's arithmetic is the
 * same as the single-matrix routine); the single-matrix routines may split
 * independent rows/columns across threads without changing any sum's order.
 */
#include <complex.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define IDX(i, j, n) ((size_t)(i) * (size_t)(n) + (size_t)(j))

/* ---------------------------------------------------------------------- */
/* Generic body, instantiated for double (suffix d) and float (suffix s). */
/* ---------------------------------------------------------------------- */
#define DEFINE_ORACLE(T, SFX, SQRT)                                              \
                                                                                 \
/* Forward factor of one matrix; returns the status (0 or j+1).  When         */ \
/* `threads` > 1 the independent rows i > j of column j are shared out.       */ \
static int32_t potrf_one_##SFX(int32_t n, const T* A, T* L, int threads) {       \
    for (size_t e = 0; e < (size_t)n * (size_t)n; ++e) L[e] = (T)0;              \
    for (int32_t j = 0; j < n; ++j) {                                            \
        T d = A[IDX(j, j, n)];                                                   \
        for (int32_t k = 0; k < j; ++k) d -= L[IDX(j, k, n)] * L[IDX(j, k, n)];  \
        if (!(d > (T)0)) return j + 1;                                           \
        const T ljj = SQRT(d);                                                   \
        L[IDX(j, j, n)] = ljj;                                                   \
        _Pragma("omp parallel for if(threads > 1) num_threads(threads) schedule(static)") \
        for (int32_t i = j + 1; i < n; ++i) {                                    \
            T s = A[IDX(i, j, n)];                                               \
            for (int32_t k = 0; k < j; ++k) s -= L[IDX(i, k, n)] * L[IDX(j, k, n)]; \
            L[IDX(i, j, n)] = s / ljj;                                           \
        }                                                                        \
    }                                                                            \
    return 0;                                                                    \
}                                                                                \
                                                                                 \
/* Literal adjoint of one matrix; W must hold 2*n*n elements of scratch.      */ \
static void potrf_adj_one_##SFX(int32_t n, const T* L, const T* Lbar, T* Abar,   \
                                T* W, int threads) {                             \
    T* P = W;                 /* P = L^T tril(Lbar), then S, then X, then M */   \
    T* R = W + (size_t)n * n; /* second buffer                              */   \
    /* P_ij = sum_k L_ki * tril(Lbar)_kj, k ascending.                     */   \
    _Pragma("omp parallel for if(threads > 1) num_threads(threads) schedule(static)") \
    for (int32_t i = 0; i < n; ++i) {                                            \
        for (int32_t j = 0; j < n; ++j) P[IDX(i, j, n)] = (T)0;                  \
        /* L_ki = 0 for k < i and tril(Lbar)_kj = 0 for j > k: those terms   */ \
        /* of the sum are exact zeros and are not formed.                     */ \
        for (int32_t k = i; k < n; ++k) {                                        \
            const T lki = L[IDX(k, i, n)];                                       \
            for (int32_t j = 0; j <= k; ++j)                                     \
                P[IDX(i, j, n)] += lki * Lbar[IDX(k, j, n)];                     \
        }                                                                        \
    }                                                                            \
    /* S = Phi(P): keep the lower triangle, halve the diagonal. */               \
    for (int32_t i = 0; i < n; ++i)                                              \
        for (int32_t j = 0; j < n; ++j) {                                        \
            T v = P[IDX(i, j, n)];                                               \
            R[IDX(i, j, n)] = (j < i) ? v : ((j == i) ? v / (T)2 : (T)0);        \
        }                                                                        \
    /* X: solve L^T X = S by back substitution, each column of S on its own: */  \
    /*   X_ij = (S_ij - sum_{k>i} L_ki X_kj) / L_ii,  i = n-1 .. 0.          */  \
    _Pragma("omp parallel for if(threads > 1) num_threads(threads) schedule(static)") \
    for (int32_t j = 0; j < n; ++j) {                                            \
        for (int32_t i = n - 1; i >= 0; --i) {                                   \
            T s = R[IDX(i, j, n)];                                               \
            for (int32_t k = i + 1; k < n; ++k) s -= L[IDX(k, i, n)] * P[IDX(k, j, n)]; \
            P[IDX(i, j, n)] = s / L[IDX(i, i, n)];                               \
        }                                                                        \
    }                                                                            \
    /* M: solve M L = X by back substitution, each row of X on its own:      */  \
    /*   M_ij = (X_ij - sum_{k>j} M_ik L_kj) / L_jj,  j = n-1 .. 0.          */  \
    _Pragma("omp parallel for if(threads > 1) num_threads(threads) schedule(static)") \
    for (int32_t i = 0; i < n; ++i) {                                            \
        for (int32_t j = n - 1; j >= 0; --j) {                                   \
            T s = P[IDX(i, j, n)];                                               \
            for (int32_t k = j + 1; k < n; ++k) s -= R[IDX(i, k, n)] * L[IDX(k, j, n)]; \
            R[IDX(i, j, n)] = s / L[IDX(j, j, n)];                               \
        }                                                                        \
    }                                                                            \
    /* Accumulate into the lower triangle: M_ij + M_ji off the diagonal,     */  \
    /* M_ii on it.                                                           */  \
    for (int32_t i = 0; i < n; ++i) {                                            \
        for (int32_t j = 0; j < i; ++j)                                          \
            Abar[IDX(i, j, n)] += R[IDX(i, j, n)] + R[IDX(j, i, n)];             \
        Abar[IDX(i, i, n)] += R[IDX(i, i, n)];                                   \
    }                                                                            \
}                                                                                \
                                                                                 \
/* Public entry points.                                                      */  \
int32_t orc_potrf_##SFX(int32_t n, const T* A, T* L, int32_t threads) {          \
    if (n <= 0) return 0;                                                        \
    return potrf_one_##SFX(n, A, L, threads);                                    \
}                                                                                \
                                                                                 \
void orc_potrf_batch_##SFX(int64_t batch, int32_t n, const T* A, T* L,           \
                           int32_t* status, int32_t threads) {                   \
    const size_t nn = (size_t)n * (size_t)n;                                     \
    _Pragma("omp parallel for if(threads > 1) num_threads(threads) schedule(dynamic, 16)") \
    for (int64_t b = 0; b < batch; ++b)                                          \
        status[b] = potrf_one_##SFX(n, A + b * nn, L + b * nn, 1);               \
}                                                                                \
                                                                                 \
int32_t orc_potrf_adj_##SFX(int32_t n, const T* L, const T* Lbar, T* Abar,       \
                            int32_t threads) {                                   \
    if (n <= 0) return 0;                                                        \
    T* W = (T*)malloc(2 * (size_t)n * (size_t)n * sizeof(T));                    \
    if (!W) return -1;                                                           \
    potrf_adj_one_##SFX(n, L, Lbar, Abar, W, threads);                           \
    free(W);                                                                     \
    return 0;                                                                    \
}                                                                                \
                                                                                 \
int32_t orc_potrf_adj_batch_##SFX(int64_t batch, int32_t n, const T* L,          \
                                  const T* Lbar, T* Abar, const int32_t* status, \
                                  int32_t threads) {                             \
    const size_t nn = (size_t)n * (size_t)n;                                     \
    int32_t rc = 0;                                                              \
    _Pragma("omp parallel if(threads > 1) num_threads(threads)")                 \
    {                                                                            \
        T* W = (T*)malloc(2 * nn * sizeof(T));                                   \
        if (!W) {                                                                \
            _Pragma("omp atomic write")                                          \
            rc = -1;                                                             \
        } else {                                                                 \
            _Pragma("omp for schedule(dynamic, 16)")                             \
            for (int64_t b = 0; b < batch; ++b) {                                \
                if (status && status[b] != 0) continue; /* failed factor */     \
                potrf_adj_one_##SFX(n, L + b * nn, Lbar + b * nn, Abar + b * nn, \
                                    W, 1);                                       \
            }                                                                    \
            free(W);                                                             \
        }                                                                        \
    }                                                                            \
    return rc;                                                                   \
}

DEFINE_ORACLE(double, d, sqrt)
DEFINE_ORACLE(float, s, sqrtf)

int32_t orc_max_threads(void) {
#ifdef _OPENMP
    return (int32_t)omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------- */
/* Complex Hermitian instantiation: double complex (z) and float complex  */
/* (c).  Same structure as above with conjugates where the real formulas  */
/* transpose.                                                              */
/* ---------------------------------------------------------------------- */
#define DEFINE_ORACLE_HERMITIAN(T, R, SFX, SQRT, CONJ, CREAL)                    \
                                                                                 \
static int32_t hpotrf_one_##SFX(int32_t n, const T* A, T* L, int threads) {     \
    for (size_t e = 0; e < (size_t)n * (size_t)n; ++e) L[e] = (T)0;              \
    for (int32_t j = 0; j < n; ++j) {                                            \
        R d = CREAL(A[IDX(j, j, n)]);                                            \
        for (int32_t k = 0; k < j; ++k) {                                        \
            const T l = L[IDX(j, k, n)];                                         \
            d -= CREAL(l * CONJ(l));                                             \
        }                                                                        \
        if (!(d > (R)0)) return j + 1;                                           \
        const R ljj = SQRT(d);                                                   \
        L[IDX(j, j, n)] = (T)ljj;                                                \
        _Pragma("omp parallel for if(threads > 1) num_threads(threads) schedule(static)") \
        for (int32_t i = j + 1; i < n; ++i) {                                    \
            T s = A[IDX(i, j, n)];                                               \
            for (int32_t k = 0; k < j; ++k) s -= L[IDX(i, k, n)] * CONJ(L[IDX(j, k, n)]); \
            L[IDX(i, j, n)] = s / ljj;                                           \
        }                                                                        \
    }                                                                            \
    return 0;                                                                    \
}                                                                                \
                                                                                 \
static void hpotrf_adj_one_##SFX(int32_t n, const T* L, const T* Lbar, T* Abar,  \
                                 T* W, int threads) {                            \
    T* P = W;                 /* P = L^H tril(Lbar), then X                 */   \
    T* R_ = W + (size_t)n * n; /* S, then M                                  */  \
    _Pragma("omp parallel for if(threads > 1) num_threads(threads) schedule(static)") \
    for (int32_t i = 0; i < n; ++i) {                                            \
        for (int32_t j = 0; j < n; ++j) P[IDX(i, j, n)] = (T)0;                  \
        for (int32_t k = i; k < n; ++k) {                                        \
            const T lki = CONJ(L[IDX(k, i, n)]);                                 \
            for (int32_t j = 0; j <= k; ++j)                                     \
                P[IDX(i, j, n)] += lki * Lbar[IDX(k, j, n)];                     \
        }                                                                        \
    }                                                                            \
    /* S = Phi(P): keep the lower triangle, halve the diagonal. */               \
    for (int32_t i = 0; i < n; ++i)                                              \
        for (int32_t j = 0; j < n; ++j) {                                        \
            T v = P[IDX(i, j, n)];                                               \
            R_[IDX(i, j, n)] = (j < i) ? v : ((j == i) ? v / (R)2 : (T)0);       \
        }                                                                        \
    /* X: solve L^H X = S, X_ij = (S_ij - sum_{k>i} conj(L_ki) X_kj) / L_ii  */  \
    _Pragma("omp parallel for if(threads > 1) num_threads(threads) schedule(static)") \
    for (int32_t j = 0; j < n; ++j) {                                            \
        for (int32_t i = n - 1; i >= 0; --i) {                                   \
            T s = R_[IDX(i, j, n)];                                              \
            for (int32_t k = i + 1; k < n; ++k)                                  \
                s -= CONJ(L[IDX(k, i, n)]) * P[IDX(k, j, n)];                    \
            P[IDX(i, j, n)] = s / CREAL(L[IDX(i, i, n)]);                        \
        }                                                                        \
    }                                                                            \
    /* M: solve M L = X, M_ij = (X_ij - sum_{k>j} M_ik L_kj) / L_jj          */  \
    _Pragma("omp parallel for if(threads > 1) num_threads(threads) schedule(static)") \
    for (int32_t i = 0; i < n; ++i) {                                            \
        for (int32_t j = n - 1; j >= 0; --j) {                                   \
            T s = P[IDX(i, j, n)];                                               \
            for (int32_t k = j + 1; k < n; ++k) s -= R_[IDX(i, k, n)] * L[IDX(k, j, n)]; \
            R_[IDX(i, j, n)] = s / CREAL(L[IDX(j, j, n)]);                       \
        }                                                                        \
    }                                                                            \
    /* Accumulate: M_ij + conj(M_ji) below the diagonal, Re(M_ii) on it.     */  \
    for (int32_t i = 0; i < n; ++i) {                                            \
        for (int32_t j = 0; j < i; ++j)                                          \
            Abar[IDX(i, j, n)] += R_[IDX(i, j, n)] + CONJ(R_[IDX(j, i, n)]);     \
        Abar[IDX(i, i, n)] += CREAL(R_[IDX(i, i, n)]);                           \
    }                                                                            \
}                                                                                \
                                                                                 \
void orc_hpotrf_batch_##SFX(int64_t batch, int32_t n, const T* A, T* L,          \
                            int32_t* status, int32_t threads) {                  \
    const size_t nn = (size_t)n * (size_t)n;                                     \
    if (batch == 1) {                                                            \
        status[0] = n > 0 ? hpotrf_one_##SFX(n, A, L, threads) : 0;              \
        return;                                                                  \
    }                                                                            \
    _Pragma("omp parallel for if(threads > 1) num_threads(threads) schedule(dynamic, 16)") \
    for (int64_t b = 0; b < batch; ++b)                                          \
        status[b] = hpotrf_one_##SFX(n, A + b * nn, L + b * nn, 1);              \
}                                                                                \
                                                                                 \
int32_t orc_hpotrf_adj_batch_##SFX(int64_t batch, int32_t n, const T* L,         \
                                   const T* Lbar, T* Abar, const int32_t* status, \
                                   int32_t threads) {                            \
    const size_t nn = (size_t)n * (size_t)n;                                     \
    if (n <= 0) return 0;                                                        \
    if (batch == 1) {                                                            \
        if (status && status[0] != 0) return 0;                                  \
        T* W = (T*)malloc(2 * nn * sizeof(T));                                   \
        if (!W) return -1;                                                       \
        hpotrf_adj_one_##SFX(n, L, Lbar, Abar, W, threads);                      \
        free(W);                                                                 \
        return 0;                                                                \
    }                                                                            \
    int32_t rc = 0;                                                              \
    _Pragma("omp parallel if(threads > 1) num_threads(threads)")                 \
    {                                                                            \
        T* W = (T*)malloc(2 * nn * sizeof(T));                                   \
        if (!W) {                                                                \
            _Pragma("omp atomic write")                                          \
            rc = -1;                                                             \
        } else {                                                                 \
            _Pragma("omp for schedule(dynamic, 16)")                             \
            for (int64_t b = 0; b < batch; ++b) {                                \
                if (status && status[b] != 0) continue; /* failed factor */     \
                hpotrf_adj_one_##SFX(n, L + b * nn, Lbar + b * nn, Abar + b * nn, \
                                     W, 1);                                      \
            }                                                                    \
            free(W);                                                             \
        }                                                                        \
    }                                                                            \
    return rc;                                                                   \
}

DEFINE_ORACLE_HERMITIAN(double complex, double, z, sqrt, conj, creal)
DEFINE_ORACLE_HERMITIAN(float complex, float, c, sqrtf, conjf, crealf)

/* ---------------------------------------------------------------------- */
/* Solve with the factor and its adjoint, for all four element types.     */
/* B, X, Xbar, Bbar: [n][nrhs] row-major per matrix; L, Lbar: [n][n].    */
/* ---------------------------------------------------------------------- */
#define RID(x) (x)
#define DEFINE_POTRS(T, R, SFX, CONJ, CREAL)                                     \
                                                                                 \
/* X = L^-H (L^-1 B), column by column; X may be B itself. */                    \
static void potrs_one_##SFX(int32_t n, int32_t nrhs, const T* L, const T* B,     \
                            T* X, T* Y) {                                        \
    for (int32_t r = 0; r < nrhs; ++r) {                                         \
        /* forward: y_i = (b_i - sum_{k<i} L_ik y_k) / L_ii */                   \
        for (int32_t i = 0; i < n; ++i) {                                        \
            T s = B[IDX(i, r, nrhs)];                                            \
            for (int32_t k = 0; k < i; ++k) s -= L[IDX(i, k, n)] * Y[k];         \
            Y[i] = s / CREAL(L[IDX(i, i, n)]);                                   \
        }                                                                        \
        /* back: x_i = (y_i - sum_{k>i} conj(L_ki) x_k) / L_ii */                \
        for (int32_t i = n - 1; i >= 0; --i) {                                   \
            T s = Y[i];                                                          \
            for (int32_t k = i + 1; k < n; ++k) s -= CONJ(L[IDX(k, i, n)]) * Y[n + k]; \
            Y[n + i] = s / CREAL(L[IDX(i, i, n)]);                               \
        }                                                                        \
        for (int32_t i = 0; i < n; ++i) X[IDX(i, r, nrhs)] = Y[n + i];           \
    }                                                                            \
}                                                                                \
                                                                                 \
int32_t orc_potrs_##SFX(int64_t batch, int32_t n, int32_t nrhs, const T* L,      \
                        const T* B, T* X, const int32_t* status, int32_t threads) { \
    const size_t nn = (size_t)n * n, nb = (size_t)n * nrhs;                      \
    int32_t rc = 0;                                                              \
    _Pragma("omp parallel if(threads > 1) num_threads(threads)")                 \
    {                                                                            \
        T* Y = (T*)malloc(2 * (size_t)n * sizeof(T) + 1);                        \
        if (!Y) {                                                                \
            _Pragma("omp atomic write")                                          \
            rc = -1;                                                             \
        } else {                                                                 \
            _Pragma("omp for schedule(dynamic, 4)")                              \
            for (int64_t b = 0; b < batch; ++b) {                                \
                if (status && status[b] != 0) continue;                          \
                potrs_one_##SFX(n, nrhs, L + b * nn, B + b * nb, X + b * nb, Y); \
            }                                                                    \
            free(Y);                                                             \
        }                                                                        \
    }                                                                            \
    return rc;                                                                   \
}                                                                                \
                                                                                 \
/* Bbar += A^-1 Xbar (if Bbar); Lbar += tril((G + G^H) L), G = -Bbar_new X^H */  \
/* with Bbar_new = A^-1 Xbar (if Lbar).                                      */  \
int32_t orc_potrs_adj_##SFX(int64_t batch, int32_t n, int32_t nrhs, const T* L,  \
                            const T* X, const T* Xbar, T* Bbar, T* Lbar,         \
                            const int32_t* status, int32_t threads) {            \
    const size_t nn = (size_t)n * n, nb = (size_t)n * nrhs;                      \
    int32_t rc = 0;                                                              \
    _Pragma("omp parallel if(threads > 1) num_threads(threads)")                 \
    {                                                                            \
        T* Y = (T*)malloc((2 * (size_t)n + nb + 2 * nn) * sizeof(T));            \
        if (!Y) {                                                                \
            _Pragma("omp atomic write")                                          \
            rc = -1;                                                             \
        } else {                                                                 \
            T* Bb = Y + 2 * (size_t)n; /* A^-1 Xbar      */                      \
            T* G = Bb + nb;            /* -Bb X^H        */                      \
            T* H = G + nn;             /* (G + G^H) L    */                      \
            _Pragma("omp for schedule(dynamic, 1)")                              \
            for (int64_t b = 0; b < batch; ++b) {                                \
                if (status && status[b] != 0) continue;                          \
                const T* Lb = L + b * nn;                                        \
                const T* Xb = X + b * nb;                                        \
                potrs_one_##SFX(n, nrhs, Lb, Xbar + b * nb, Bb, Y);              \
                if (Bbar)                                                        \
                    for (size_t e = 0; e < nb; ++e) Bbar[b * nb + e] += Bb[e];   \
                if (!Lbar) continue;                                             \
                for (int32_t i = 0; i < n; ++i)                                  \
                    for (int32_t j = 0; j < n; ++j) {                            \
                        T s = (T)0;                                              \
                        for (int32_t r = 0; r < nrhs; ++r)                       \
                            s += Bb[IDX(i, r, nrhs)] * CONJ(Xb[IDX(j, r, nrhs)]); \
                        G[IDX(i, j, n)] = -s;                                    \
                    }                                                            \
                for (int32_t i = 0; i < n; ++i)                                  \
                    for (int32_t j = 0; j < n; ++j) {                            \
                        T s = (T)0;                                              \
                        for (int32_t k = 0; k < n; ++k)                          \
                            s += (G[IDX(i, k, n)] + CONJ(G[IDX(k, i, n)])) * Lb[IDX(k, j, n)]; \
                        H[IDX(i, j, n)] = s;                                     \
                    }                                                            \
                for (int32_t i = 0; i < n; ++i)                                  \
                    for (int32_t j = 0; j <= i; ++j)                             \
                        Lbar[b * nn + IDX(i, j, n)] += H[IDX(i, j, n)];          \
            }                                                                    \
            free(Y);                                                             \
        }                                                                        \
    }                                                                            \
    return rc;                                                                   \
}

DEFINE_POTRS(double, double, d, RID, RID)
DEFINE_POTRS(float, float, s, RID, RID)
DEFINE_POTRS(double complex, double, z, conj, creal)
DEFINE_POTRS(float complex, float, c, conjf, crealf)
