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

// Thread-per-matrix float32 forward for n in {8, 16}; A and L 16-byte aligned.
bool tpm_supported(int n);
cudaError_t tpm_fwd(const float* A, float* L, int32_t* status, int64_t batch, int n,
                    cudaStream_t stream);
// The n = 16 kernel with lane 0's copy of every round dropped and `max_polls`
// polls per barrier wait: every warp's first round times out (status -1).
cudaError_t tpm_fwd_wait_selftest(const float* A, float* L, int32_t* status, int64_t batch,
                                  uint32_t max_polls, cudaStream_t stream);

// n > 64, blocked with square tiles of `tile` (32, 64 or 128).
template <typename T>
cudaError_t blocked_fwd(const T* A, T* L, int32_t* status, int64_t batch, int n, int tile,
                        cudaStream_t stream);
// `work` holds batch * n * n elements of scratch.  accumulate as small_adj.
// Not accumulating with adj_A == adj_L (in place), the sweep runs on adj_A
// itself and `work` is not used (may be null).
template <typename T>
cudaError_t blocked_adj(const T* L, const T* Lbar, T* Abar, const int32_t* status,
                        int64_t batch, int n, int tile, T* work, bool accumulate,
                        cudaStream_t stream);

int blocked_default_tile(int n, int64_t batch);

// Argument checks of chol_adj_ex (shape, dtype, tile, null, alignment,
// device residency, aliasing), shared by every adjoint entry point that
// promises the same error codes.  On CHOL_OK, *bytes is the size of one
// [batch][n][n] array; batch == 0 passes (the caller returns at once).
int check_adj_args(int64_t batch, int32_t n, int32_t dtype, const void* L, const void* adj_L,
                   const void* adj_A, const int32_t* status, int32_t tile, size_t* bytes);

}  // namespace chol
