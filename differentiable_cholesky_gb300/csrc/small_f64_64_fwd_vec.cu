// Small-path forward kernel for double matrices of padded order 64,
// 16-byte vector accesses.
#include "small_kernels.cuh"

namespace chol {

CHOL_SMALL_FWD(double, 64, true)

}  // namespace chol
