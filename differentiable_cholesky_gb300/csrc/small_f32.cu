// Small-path kernels for float matrices of padded order 8, 16 and 32.
#include "small_kernels.cuh"

namespace chol {

CHOL_SMALL_FWD(float, 8, true)
CHOL_SMALL_ADJ(float, 8, true)
CHOL_SMALL_FWD(float, 8, false)
CHOL_SMALL_ADJ(float, 8, false)
CHOL_SMALL_FWD(float, 16, true)
CHOL_SMALL_ADJ(float, 16, true)
CHOL_SMALL_FWD(float, 16, false)
CHOL_SMALL_ADJ(float, 16, false)
CHOL_SMALL_FWD(float, 32, true)
CHOL_SMALL_ADJ(float, 32, true)
CHOL_SMALL_FWD(float, 32, false)
CHOL_SMALL_ADJ(float, 32, false)

}  // namespace chol
