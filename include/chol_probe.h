/*
 * chol_probe.h -- measurement utility shipped with the GB300 Cholesky library.
 *
 * Not part of the factorisation path: it measures the denominator that the
 * FP64 (and FP32) rooflines of the blocked path are reported against, since
 * the chip's FMA peaks are not published figures one can rely on.
 */
#ifndef CHOL_PROBE_H
#define CHOL_PROBE_H

#include <stdint.h>

#include "chol.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * chol_probe_fma_peak -- runs a kernel of independent FMA chains on every SM
 * of the current device (dtype CHOL_F32 or CHOL_F64), `iters` FMAs per chain,
 * times it with CUDA events on `stream` (synchronising that stream) and
 * writes the rate in FLOP/s (2 per FMA) to *flops.  `sink` is a device buffer
 * of at least 1 element of dtype that receives a value so the work is kept.
 * Returns CHOL_OK, CHOL_EINVAL, CHOL_EDTYPE or CHOL_ECUDA.
 */
CHOL_API int chol_probe_fma_peak(int32_t dtype, int64_t iters, void* sink, double* flops,
                                 void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CHOL_PROBE_H */
