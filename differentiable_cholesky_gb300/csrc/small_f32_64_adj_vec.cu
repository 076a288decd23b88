// Small-path adjoint kernel for float matrices of padded order 64,
// 16-byte vector accesses.
#include "small_kernels.cuh"

namespace chol {

CHOL_SMALL_ADJ(float, 64, true)

}  // namespace chol
