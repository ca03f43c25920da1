/*
 * w4_selftest.h -- a test hook of libw4 (not part of the method; the pages
 * have no counterpart).
 *
 * Every wait inside libw4's kernels is bounded: a wait on an mbarrier, and a
 * split-row-tile owner's wait for a sharer's partial sums, give up after a time
 * limit, set a per-kernel fault word and let the block finish.  A linear whose
 * wait gave up still returned W4_OK when it was enqueued; w4_device_fault is
 * what reports it.  This hook makes those waits run out on purpose, so that the
 * path can be tested without faulting or hanging a GPU.
 */
#ifndef W4_SELFTEST_H
#define W4_SELFTEST_H

#include "w4.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * w4_selftest_bounded_waits -- enqueue one block of 64 threads on `stream` that
 *  - waits on an mbarrier nothing completes (the helper the TMA-fed kernels use
 *    for their ring slots), and
 *  - as the owner of a 16-row split tile, collects the partial sums of a sharer
 *    that never publishes them (the stream-K decode kernels' owner collect):
 *    worker 1's slot in `workspace`, which must hold 256 zero bytes (two
 *    16-row slots of one token, 8 bytes a word).
 * Both waits give up after `limit_ns` nanoseconds (1e5 .. 1e9), raise the
 * device fault word and return.  The owner counts the missing share as zero and
 * writes its own sums to Y[0..15] (bf16): row r gets r + 0.5.  Afterwards
 * w4_device_fault returns W4_ERR_TIMEOUT once, and the workspace is still zero.
 * Errors: W4_ERR_INVALID_ARG (NULL, workspace_bytes < 256, limit out of range),
 * W4_ERR_MISALIGNED (pointers not 16-byte aligned), W4_ERR_CUDA (launch).
 */
W4_API w4_status w4_selftest_bounded_waits(void *workspace, size_t workspace_bytes, uint16_t *Y,
                                           uint64_t limit_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* W4_SELFTEST_H */
