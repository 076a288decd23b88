// Small-path kernels for double matrices of padded order 8, 16 and 32.
#include "small_kernels.cuh"

namespace chol {

CHOL_SMALL_FWD(double, 8, true)
CHOL_SMALL_ADJ(double, 8, true)
CHOL_SMALL_FWD(double, 8, false)
CHOL_SMALL_ADJ(double, 8, false)
CHOL_SMALL_FWD(double, 16, true)
CHOL_SMALL_ADJ(double, 16, true)
CHOL_SMALL_FWD(double, 16, false)
CHOL_SMALL_ADJ(double, 16, false)
CHOL_SMALL_FWD(double, 32, true)
CHOL_SMALL_ADJ(double, 32, true)
CHOL_SMALL_FWD(double, 32, false)
CHOL_SMALL_ADJ(double, 32, false)

}  // namespace chol
