// Small-path forward kernel for double matrices of padded order 64,
// scalar accesses.
#include "small_kernels.cuh"

namespace chol {

CHOL_SMALL_FWD(double, 64, false)

}  // namespace chol
