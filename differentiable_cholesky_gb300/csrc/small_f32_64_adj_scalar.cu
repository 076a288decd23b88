// Small-path adjoint kernel for float matrices of padded order 64,
// scalar accesses.
#include "small_kernels.cuh"

namespace chol {

CHOL_SMALL_ADJ(float, 64, false)

}  // namespace chol
