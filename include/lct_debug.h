/*
 * lct_debug.h -- test hooks of liblct.so (not part of the codec itself).
 *
 * The codec's writers place each block's overflow bytes with a single-pass
 * scan in which a block waits for earlier blocks to publish their counts.
 * Every such wait is bounded; these hooks let a test watch a wait run out on
 * the GPU without faulting or hanging it.
 */
#ifndef LCT_DEBUG_H
#define LCT_DEBUG_H

#include <stdint.h>

#include "lct.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Enqueue one tiny kernel (one warp) that clears two scan words at d_work
 * (device, at least 16 bytes, 16-byte aligned) and then waits, as block 1,
 * for block 0 to publish -- which nothing does -- in each form of the wait the
 * writers use (a warp reading every predecessor, a warp walking back window
 * by window, a single thread), one after the other.  Each gives up after
 * limit_ns nanoseconds (1 .. 10^9) of %globaltimer; when all of them have,
 * LCT_ERR_TIMEOUT is latched into the status word of the header at d_header
 * (device, LCT_HEADER_BYTES, 16-byte aligned; the latch only fires if the
 * status is 0).  The kernel returns normally; the CUDA context stays usable.
 * Errors: LCT_ERR_INVALID_ARG for NULL/misaligned pointers or a limit out of
 * range, LCT_ERR_CUDA for a launch failure. */
lct_status lct_debug_wait_timeout(void *d_header, void *d_work, uint64_t limit_ns, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* LCT_DEBUG_H */
