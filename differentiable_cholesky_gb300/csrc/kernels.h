// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace chol {

// Threads per matrix of the small path for order n (8, 16, 32 or 64).
int small_nt(int n);

// n <= 64.  `vec` selects 16-byte vector accesses (every pointer 16-byte
// aligned and n a multiple of 16 / sizeof(T)).
template <typename T>
cudaError_t small_fwd(const T* A, T* L, int32_t* status, int64_t batch, int n, bool vec,
                      cudaStream_t stream);
// The adjoint adds its gradient into adj_A's lower triangle (accumulate) or
// writes it there (matrices with status != 0 then get zeros); adj_A may be
// adj_L itself when not accumulating, since every matrix is read in full
// before its first write.
template <typename T>
cudaError_t small_adj(const T* L, const T* Lbar, T* Abar, const int32_t* status, int64_t batch,
                      int n, bool vec, bool accumulate, cudaStream_t stream);

// The same for one padded order NT (8, 16, 32 or 64, n <= NT) and access mode
// (VEC: 16-byte vectors).
template <typename T, int NT, bool VEC>
cudaError_t small_fwd_nt(const T* A, T* L, int32_t* status, int64_t batch, int n,
                         cudaStream_t stream);
template <typename T, int NT, bool VEC>
cudaError_t small_adj_nt(const T* L, const T* Lbar, T* Abar, const int32_t* status,
                         int64_t batch, int n, bool accumulate, cudaStream_t stream);

// Complex Hermitian elements (chol_tile::cplx<float> / cplx<double>), n <= 64:
// one block per matrix.  adj as small_adj.
template <typename T>
cudaError_t hsmall_fwd(const T* A, T* L, int32_t* status, int64_t batch, int n,
                       cudaStream_t stream);
template <typename T>
cudaError_t hsmall_adj(const T* L, const T* Lbar, T* Abar, const int32_t* status, int64_t batch,
                       int n, bool accumulate, cudaStream_t stream);

// Solve with the factor, X = A^-1 B (B, X: [batch][n][nrhs]; X may be B),
// any element type; matrices with status != 0 get X = 0.
template <typename T>
cudaError_t potrs_solve(const T* L, const T* B, T* X, const int32_t* status, int64_t batch,
                        int n, int nrhs, cudaStream_t stream);
// Its reverse mode: Bbar += A^-1 Xbar (Bbar may be null); Lbar (may be null)
// += tril(-(Bb X^H + X Bb^H) L), Bb = A^-1 Xbar.  `work` holds
// potrs_adj_workspace_elems() elements.
size_t potrs_adj_workspace_elems(int64_t batch, int n, int nrhs, bool want_L);
template <typename T>
cudaError_t potrs_adj(const T* L, const T* X, const T* Xbar, T* Bbar, T* Lbar,
                      const int32_t* status, int64_t batch, int n, int nrhs, T* work,
                      cudaStream_t stream);

// Largest blocked tile for an element size: 64 for complex double (its
// diagonal-tile kernels would not fit in shared memory at 128), else 128.
inline int blocked_max_tile(int esize) { return esize > 8 ? 64 : 128; }

// Thread-per-matrix float32 forward for n in {8, 16}; A and L 16-byte aligned.
bool tpm_supported(int n);
cudaError_t tpm_fwd(const float* A, float* L, int32_t* status, int64_t batch, int n,
                    cudaStream_t stream);
// The n = 16 kernel with lane 0's copy of every round dropped and `max_polls`
// polls per barrier wait: every warp's first round times out (status -1).
cudaError_t tpm_fwd_wait_selftest(const float* A, float* L, int32_t* status, int64_t batch,
                                  uint32_t max_polls, cudaStream_t stream);

// n > 64, blocked with square tiles of `tile` (32, 64 or 128).  `work`
// (may be null) holds blocked_fwd_workspace_bytes() bytes; with it, float64
// tiles of 128 take the trailing update on the tensor cores.
template <typename T>
cudaError_t blocked_fwd(const T* A, T* L, int32_t* status, int64_t batch, int n, int tile,
                        void* work, cudaStream_t stream);
// Workspace the forward uses for this shape (0: none); real_double: the
// element type is float64.
size_t blocked_fwd_workspace_bytes(bool real_double, int64_t batch, int n, int tile);

// Diagonal-tile factor of the blocked forward on a cluster of 8 blocks
// (8 SMs) per matrix, 16 for one or a few matrices where such a cluster fits: the tile L[k0 .. k0+kb, k0 .. k0+kb] (kb <= 128,
// lower part) factored in place, status[b] = k0 + the failing column + 1.
// With Inv (else null): also the tile's inverse into Inv[b] (128 x 128,
// zeros above the diagonal and beyond kb) and, with bal, the balancing
// exponents ilogb(l_ii) of its rows into bal[b * ceil(n/128) * 128 + k0 + i].
// cluster_diag_pays: few enough matrices that the clusters leave SMs idle.
bool cluster_diag_pays(int64_t batch, int kb);
template <typename T>
cudaError_t cluster_potrf_diag(T* L, int32_t* status, int64_t batch, int n, int k0, int kb,
                               T* Inv, int32_t* bal, cudaStream_t stream);

// Trailing update of step k of the float64 blocked forward with 128-wide
// tiles on the bf16 tensor cores (exact digit-slice products): for every
// lower tile (I, J), I >= J > k, L_IJ -= L_Ik L_Jk^T.  `work` holds
// ozaki_workspace_bytes(batch, n) bytes.
size_t ozaki_workspace_bytes(int64_t batch, int n);
cudaError_t ozaki_trailing_update(double* L, void* work, int32_t* status, int64_t batch, int n,
                                  int k, cudaStream_t stream);
// The same in two parts: slicing the panel's rows, then the products for all
// trailing tiles (part 0), only block column k + 1 (part 1) or the block
// columns right of it (part 2).  Step k's slices stay valid until step k + 2
// slices its panel, so part 2 of step k may run beside step k + 1.
cudaError_t ozaki_trailing_slice(double* L, void* work, int32_t* status, int64_t batch, int n,
                                 int k, cudaStream_t stream);
cudaError_t ozaki_trailing_gemm(double* L, void* work, int32_t* status, int64_t batch, int n,
                                int k, int part, cudaStream_t stream);
// The panel solve of step k on the tensor cores: L_Ik <- L_Ik G^-T, I > k,
// with G^-1 the inverse of the (factored) diagonal tile, computed here unless
// have_inverse (the diagonal factor wrote it to the workspace's inverse and
// balancing arrays, ozaki_fwd_inverse).
cudaError_t ozaki_panel_solve(double* L, void* work, int32_t* status, int64_t batch, int n,
                              int k, bool have_inverse, cudaStream_t stream);
// Where the forward's workspace keeps the diagonal tile's inverse
// (batch x 128 x 128) and the balancing exponents (batch x ceil(n/128) x 128).
void ozaki_fwd_inverse(void* work, int64_t batch, int n, double** inv, int32_t** bal);
// The same for the float64 blocked adjoint with 128-wide tiles: `work` holds
// ozaki_adj_workspace_bytes(batch, n) bytes; prepare slices L once, then per
// tile column J: row (W_JK -= C^T L_{below J, K}, K <= J) before the
// diagonal sweep, upd (W_IK -= Chat_I L_JK, I >= J > K, Chat = [W_JJ + W_JJ^T;
// C]) after it.
size_t ozaki_adj_workspace_bytes(int64_t batch, int n);
cudaError_t ozaki_adj_prepare(const double* L, void* work, const int32_t* status, int64_t batch,
                              int n, cudaStream_t stream);
// The adjoint's panel solve C <- C L_JJ^-1 (rows below tile J).
cudaError_t ozaki_adj_solve(const double* L, double* W, void* work, const int32_t* status,
                            int64_t batch, int n, int J, cudaStream_t stream);
// The adjoint's row update W_JK -= C^T L_{below J, K} for the output block
// columns K <= J (part 0), K = J - 1 .. J only (part 1, which also slices C)
// or K < J - 1 only (part 2, which reuses part 1's slices of C and its own
// partial-sum buffer, so it may run on the side stream beside tile column
// J - 1's solve and row update).
cudaError_t ozaki_adj_row(const double* L, double* W, void* work, const int32_t* status,
                          int64_t batch, int n, int J, int part, cudaStream_t stream);
// Adjoint of diagonal tile J by the literal formula Phi(M + M^T),
// M = X^T Phi(L_JJ^T W_JJ) X with X = L_JJ^-1 from ozaki_adj_prepare, in
// place on W_JJ (three products, no column chain).  ozaki_adj_lit_pays: few
// enough matrices that this beats the one-block reverse sweep.
bool ozaki_adj_lit_pays(int64_t batch);
cudaError_t ozaki_adj_diag(const double* L, double* W, void* work, const int32_t* status,
                           int64_t batch, int n, int J, cudaStream_t stream);
cudaError_t ozaki_adj_upd(const double* L, double* W, void* work, const int32_t* status,
                          int64_t batch, int n, int J, cudaStream_t stream);
// The same in two parts: slicing Chat, then the products for every K < J
// (part 0), only K = J - 1 (part 1) or only K < J - 1 (part 2).  Tile column
// J's slices stay valid until tile column J - 2 slices its own, so part 2 of
// J may run beside the solve, row update and diagonal tile of J - 1.
cudaError_t ozaki_adj_upd_slice(double* W, void* work, const int32_t* status, int64_t batch,
                                int n, int J, cudaStream_t stream);
cudaError_t ozaki_adj_upd_gemm(double* W, void* work, const int32_t* status, int64_t batch,
                               int n, int J, int part, cudaStream_t stream);
// `work` holds batch * n * n elements of scratch.  accumulate as small_adj.
// Not accumulating with adj_A == adj_L (in place), the sweep runs on adj_A
// itself and `work` is not used (may be null).  `oz_work` (may be null) holds
// ozaki_adj_workspace_bytes(batch, n) bytes; with it, float64 tiles of 128
// take the two large updates on the tensor cores.
template <typename T>
cudaError_t blocked_adj(const T* L, const T* Lbar, T* Abar, const int32_t* status,
                        int64_t batch, int n, int tile, T* work, bool accumulate, void* oz_work,
                        cudaStream_t stream);

int blocked_default_tile(int n, int64_t batch);

// Argument checks of chol_adj_ex (shape, dtype, tile, null, alignment,
// device residency, aliasing), shared by every adjoint entry point that
// promises the same error codes.  On CHOL_OK, *bytes is the size of one
// [batch][n][n] array; batch == 0 passes (the caller returns at once).
int check_adj_args(int64_t batch, int32_t n, int32_t dtype, const void* L, const void* adj_L,
                   const void* adj_A, const int32_t* status, int32_t tile, size_t* bytes);

}  // namespace chol
