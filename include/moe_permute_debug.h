/*
 * moe_permute_debug.h -- a test hook exported only by the debug build of the
 * library (compiled with -DMOE_DEBUG_HOOKS, libmoe_permute_debug.so).  The
 * production library does not export it.
 *
 * The routing grid of moe_permute (batches above 2048 expanded rows) has
 * every block read every block's row of a per-expert histogram table, waiting
 * for rows that do not carry the current call's tag yet.  Each wait is bounded
 * (2^24 polls or a time limit); when it runs out the block sets
 * MOE_FLAG_BARRIER_TIMEOUT in the workspace status word and returns, so the
 * GPU context stays usable.  This hook makes those waits run out on purpose,
 * without any fault, trap or endless loop: every block also waits for
 * `extra_rows` table rows past the grid that no block ever writes.
 */
#ifndef MOE_PERMUTE_DEBUG_H
#define MOE_PERMUTE_DEBUG_H

#include "moe_permute.h"

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_DEBUG_MAX_EXTRA_ROWS 4

/*
 * moe_debug_set_table_wait: from the next routing launch on, every block of
 * the routing grid also waits for `extra_rows` (0..MOE_DEBUG_MAX_EXTRA_ROWS)
 * table rows past the grid, and a wait gives up after `wait_ns` nanoseconds
 * (or 2^24 polls).  (0, 2000000000) restores the production behaviour.
 *  - A routing launch whose grid plus extra_rows exceeds the workspace's
 *    table (min(max_tokens, 1024) rows) is refused on the host
 *    (MOE_ERR_CUDA), so no wait reads outside the workspace.
 *  - The setting is process-wide and synchronous (it copies to device
 *    symbols); do not change it while routing launches are in flight.
 * Returns MOE_OK, MOE_ERR_INVALID_ARG (extra_rows out of range, wait_ns 0) or
 * MOE_ERR_CUDA.
 */
MOE_API int moe_debug_set_table_wait(int extra_rows, unsigned long long wait_ns);

#ifdef __cplusplus
}
#endif

#endif /* MOE_PERMUTE_DEBUG_H */
