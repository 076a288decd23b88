// Dispatch of the small path (n <= 64) on the padded order; the kernels are
// in small_kernels.cuh, instantiated by the small_<type>*.cu translation
// units (the order-64 kernels, the slowest to compile, one per file).

#include <cuda_runtime.h>

#include "kernels.h"

namespace chol {

int small_nt(int n) { return n <= 8 ? 8 : n <= 16 ? 16 : n <= 32 ? 32 : 64; }

template <typename T>
cudaError_t small_fwd(const T* A, T* L, int32_t* status, int64_t batch, int n, bool vec,
                      cudaStream_t stream) {
#define CHOL_FWD_CASE(NT)                                                      \
    case NT:                                                                   \
        return vec ? small_fwd_nt<T, NT, true>(A, L, status, batch, n, stream) \
                   : small_fwd_nt<T, NT, false>(A, L, status, batch, n, stream);
    switch (small_nt(n)) {
        CHOL_FWD_CASE(8)
        CHOL_FWD_CASE(16)
        CHOL_FWD_CASE(32)
        CHOL_FWD_CASE(64)
    }
#undef CHOL_FWD_CASE
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t small_adj(const T* L, const T* Lbar, T* Abar, const int32_t* status, int64_t batch,
                      int n, bool vec, bool accumulate, cudaStream_t stream) {
#define CHOL_ADJ_CASE(NT)                                                                 \
    case NT:                                                                              \
        return vec ? small_adj_nt<T, NT, true>(L, Lbar, Abar, status, batch, n, accumulate, stream) \
                   : small_adj_nt<T, NT, false>(L, Lbar, Abar, status, batch, n, accumulate, stream);
    switch (small_nt(n)) {
        CHOL_ADJ_CASE(8)
        CHOL_ADJ_CASE(16)
        CHOL_ADJ_CASE(32)
        CHOL_ADJ_CASE(64)
    }
#undef CHOL_ADJ_CASE
    return cudaErrorInvalidValue;
}

template cudaError_t small_fwd<float>(const float*, float*, int32_t*, int64_t, int, bool,
                                      cudaStream_t);
template cudaError_t small_fwd<double>(const double*, double*, int32_t*, int64_t, int, bool,
                                       cudaStream_t);
template cudaError_t small_adj<float>(const float*, const float*, float*, const int32_t*,
                                      int64_t, int, bool, bool, cudaStream_t);
template cudaError_t small_adj<double>(const double*, const double*, double*, const int32_t*,
                                       int64_t, int, bool, bool, cudaStream_t);

}  // namespace chol
