/*
 * tbe_selftest.h -- diagnostics of the TBE library (not part of the computation).
 *
 * Every wait inside the library's kernels is bounded: a kernel that waits on an mbarrier (for a
 * bulk copy, a tensor-core MMA or a cluster-launch-control reply) gives up after a fixed number
 * of polls, counts TBE_STAT_WAIT_TIMEOUT in d_stats and returns, so a lost completion never
 * hangs the GPU ("Modernizing Table Batched Embeddings with FBTriton", section 4, Problem 5: the
 * long-run merge is built so that no block waits on another; the library extends that rule to
 * every wait it has).  This entry point exercises that give-up path on purpose.
 */
#ifndef TBE_SELFTEST_H
#define TBE_SELFTEST_H

#include <stdint.h>

#include "tbe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Launches one CTA that waits, through the library's bounded mbarrier wait, for a phase of a
 * fresh mbarrier that nothing ever completes (no copy, MMA or arrival is pending on it), giving
 * up after `polls` polls (1 <= polls <= 4096; each poll suspends the thread for at most a
 * hardware-chosen time, so the kernel ends within microseconds).  On giving up it adds 1 to
 * d_stats[TBE_STAT_WAIT_TIMEOUT] (d_stats: device int64[TBE_NUM_STATS], caller-owned) and
 * returns.  Asynchronous on `stream`.  TBE_ERR_INVALID_ARG for a NULL d_stats, a misaligned one
 * or polls outside the range; TBE_ERR_CUDA if the launch fails. */
tbe_status tbe_selftest_wait_timeout(uint32_t polls, int64_t* d_stats, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TBE_SELFTEST_H */
