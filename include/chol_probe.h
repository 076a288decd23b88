/*
 * chol_probe.h -- measurement utility shipped with the GB300 Cholesky library.
 *
 * Not part of the factorisation path: it measures the denominators that the
 * FP64 (and FP32) rooflines of the blocked path are reported against, since
 * the chip's FP64 rates are not published figures one can rely on.  Both
 * FP64 pipes are measured: the FMA pipe and the f64 mma.sync tensor path.
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

/* Shapes of the f64 mma.sync instruction (the FP64 tensor path, DMMA). */
enum {
    CHOL_DMMA_M8N8K4 = 0,
    CHOL_DMMA_M16N8K4 = 1,
    CHOL_DMMA_M16N8K8 = 2,
    CHOL_DMMA_M16N8K16 = 3
};

/*
 * chol_probe_dmma_peak -- the same measurement for the double-precision
 * tensor path: every thread of a full-occupancy grid issues `iters` rounds of
 * 4 independent warp-wide `mma.sync ... .f64` operations of the given shape
 * (CHOL_DMMA_*).  *flops receives the rate in FLOP/s (2 M N K per warp-wide
 * operation).  `sink` is a device buffer of at least one double.  Returns
 * CHOL_OK, CHOL_EINVAL (bad shape, iters <= 0, null pointer) or CHOL_ECUDA.
 */
CHOL_API int chol_probe_dmma_peak(int32_t shape, int64_t iters, void* sink, double* flops,
                                  void* stream);

/*
 * chol_probe_tc_update -- times the dominant kernel of the float64 blocked
 * path, the trailing update on the bf16 tensor cores (exact digit-slice
 * products), alone: for the float64 n x n row-major matrix L on the device
 * (n > 128, 128-wide tiles) it slices the rows of panel k once, then launches
 * `reps` times the update L_IJ -= L_Ik L_Jk^T of every lower tile I >= J > k,
 * timed with CUDA events on `stream` (which it synchronises).  L's trailing
 * tiles are modified: pass a scratch copy.  Writes the average time of one
 * launch in ms, the rate of the bf16 digit products the tensor cores execute
 * (28 products of 2 * 128^3 flops per tile) and the float64-equivalent rate
 * (2 * 128^3 per tile), both in FLOP/s.  Takes a workspace with
 * cudaMallocAsync on `stream`.  Returns CHOL_OK, CHOL_EINVAL (n <= 128, k not
 * in [0, ceil(n/128) - 2], reps <= 0, null pointer), CHOL_ENOMEM or
 * CHOL_ECUDA.
 */
CHOL_API int chol_probe_tc_update(int32_t n, void* L, int32_t k, int32_t reps, double* ms,
                                  double* bf16_flops, double* fp64_equiv_flops, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CHOL_PROBE_H */
