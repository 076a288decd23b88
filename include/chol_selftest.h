/*
 * chol_selftest.h -- self-test of the library's bounded device waits.  Not
 * part of the path: it lets a test check, on the GPU, that a wait which can
 * never complete ends in an error status the host reads, with the CUDA
 * context still usable, instead of hanging.
 */
#ifndef CHOL_GB300_SELFTEST_H
#define CHOL_GB300_SELFTEST_H

#include <stdint.h>

#include "chol.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * chol_selftest_wait_timeout -- runs the batched float32 n = 16 forward kernel
 * (the one chol_fwd uses for 16-byte-aligned float32 16x16 matrices) with one
 * matrix copy of every warp's first round held back, a lost message, so that
 * round's arrival barrier cannot complete, and with `max_polls` polls per
 * barrier wait.  Every warp gives up on its first round and writes status -1
 * for that round's matrices; the held-back copy is then issued late and the
 * warp waits (again at most max_polls polls per barrier) until every copy it
 * issued has landed, so no block retires with a copy in flight, and returns.
 * No other status entry and no part of L is written.
 *   A       in : float[batch][16][16], device, 16-byte aligned.
 *   L       out: float[batch][16][16], device, 16-byte aligned, not
 *                overlapping A or status.
 *   status  out: int32[batch], device.
 *   max_polls  : 1 .. 4194304 (the kernel's own limit).
 * Returns CHOL_OK once enqueued; argument errors as chol_fwd.
 */
CHOL_API int chol_selftest_wait_timeout(int64_t batch, const void* A, void* L, int32_t* status,
                                        uint32_t max_polls, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CHOL_GB300_SELFTEST_H */
