/* fvx_testing.h — test hooks of libfvx.
 *
 * Not part of the library's interface for applications: these entry points
 * exist so that a test can make the library's failure reporting happen on
 * purpose, on a GPU, without faulting it.  The pages have no counterpart;
 * "DriveRT" (Inspection and debugging) asks only that a failure be reported
 * with what failed, which is what these let a test check.
 */
#ifndef FVX_TESTING_H
#define FVX_TESTING_H

#include "fvx.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Runs one bounded device-side wait, of the form the library's kernels use,
 * on something that nothing completes, so that it gives up after limit_ns
 * nanoseconds and records FVX_ERR_DEVICE_TIMEOUT in the device status word,
 * which the next fvx_device_status (or the next call that reads the word at
 * a synchronisation) reports and clears.  The kernel then returns: the
 * context stays usable.
 *   kind 0: an mbarrier phase wait (the convolution kernels' pipeline waits),
 *           one thread, on a barrier with no arrivals.
 *   kind 1: a warp polling a published word (the look-back waits of the scan
 *           and the radix sort) that stays zero.
 * Asynchronous on `stream` (one block of 32 threads).  Read the status with
 * fvx_device_status before launching other work: the library's pipelined
 * kernels give up at once while the word is set.
 * Errors: FVX_ERR_INVALID_ARG unless kind is 0 or 1 and 1000 <= limit_ns <=
 * 2e9; FVX_ERR_CUDA if the status word cannot be set up or the launch fails. */
fvx_status fvx_testing_bounded_wait(int32_t kind, uint64_t limit_ns, fvx_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* FVX_TESTING_H */
