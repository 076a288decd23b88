// Blocked Cholesky forward and adjoint for n > 64 (placeholder: not built yet).
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace chol {

int blocked_default_tile(int n, int elem_size) { return 128; }

template <typename T>
cudaError_t blocked_fwd(const T*, T*, int32_t*, int64_t, int, int, cudaStream_t) {
    return cudaErrorNotSupported;
}
template <typename T>
cudaError_t blocked_adj(const T*, const T*, T*, const int32_t*, int64_t, int, int, T*,
                        cudaStream_t) {
    return cudaErrorNotSupported;
}
template cudaError_t blocked_fwd<float>(const float*, float*, int32_t*, int64_t, int, int, cudaStream_t);
template cudaError_t blocked_fwd<double>(const double*, double*, int32_t*, int64_t, int, int, cudaStream_t);
template cudaError_t blocked_adj<float>(const float*, const float*, float*, const int32_t*, int64_t, int, int, float*, cudaStream_t);
template cudaError_t blocked_adj<double>(const double*, const double*, double*, const int32_t*, int64_t, int, int, double*, cudaStream_t);

}  // namespace chol
