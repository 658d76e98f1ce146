/*
 * pa_timestamps.h -- extra entry point of the instrumented build (libpa_ts.so).
 *
 * The instrumented build is the same library compiled with -DPA_TIMESTAMPS: every
 * kernel records %globaltimer nanoseconds into a caller-owned device buffer, so the
 * gaps between the three stages of a decode step (and how much of them PDL hides)
 * can be measured without a tracing tool.  The production libpa.so does not export
 * this call and its kernels carry none of the instrumentation.
 */
#ifndef PA_TIMESTAMPS_H_
#define PA_TIMESTAMPS_H_

#include <stdint.h>

#include "pa.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Make later launches record stage times into `buffer` (device memory, 9 uint64,
 * NULL stops recording).  Stage k = 0 metadata, 1 split-K producer, 2 reducer:
 *   buffer[3k + 0]  earliest block entry            (atomicMin; preset to UINT64_MAX)
 *   buffer[3k + 1]  earliest return from the wait on the previous grid (atomicMin)
 *   buffer[3k + 2]  latest warp finish              (atomicMax; preset to 0)
 * The buffer pointer is captured into kernel arguments at launch (and so into CUDA
 * graphs captured afterwards).  The caller resets the buffer between steps.
 */
PA_API pa_status pa_set_timestamp_buffer(uint64_t* buffer);

/*
 * Failure-detection test hook: with hold != 0, later tensor-core producer launches
 * issue no copies, so each consumer's wait on its first stage gives up after the wait
 * limit (~2 s), the kernel sets PA_DEVERR_WAIT_TIMEOUT in the error word, drains (also
 * bounded) and returns without writing partials; the context stays usable.  hold = 0
 * restores normal launches.
 */
PA_API pa_status pa_set_test_hold_loads(int32_t hold);

/*
 * A/B test hook: with off != 0, later producer launches keep one block per (request,
 * kv head, split) even where the library would run its persistent form (one CTA per
 * resident slot claiming items of a largest-first work list); off = 0 restores the
 * library's choice.  Both forms give the same bits.
 */
PA_API pa_status pa_set_test_no_persist(int32_t off);

#ifdef __cplusplus
}
#endif

#endif /* PA_TIMESTAMPS_H_ */
