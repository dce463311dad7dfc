/*
 * moe_permute_debug.h -- a test hook exported only by the debug build of the
 * library (compiled with -DMOE_DEBUG_HOOKS, libmoe_permute_debug.so).  The
 * production library does not export it.
 *
 * The routing grid of moe_permute (batches above 3072 expanded rows without an
 * expert map) has every block read every block's row of a per-expert
 * histogram table, waiting for rows that do not carry the current call's tag
 * yet.  Each wait is bounded
 * (2^24 polls or a time limit); when it runs out the block sets
 * MOE_FLAG_BARRIER_TIMEOUT in the workspace status word and returns, so the
 * GPU context stays usable.  This hook makes those waits run out on purpose,
 * without any fault, trap or endless loop: every block also waits for
 * `extra_rows` table rows past the grid that no block ever writes.
 *
 * A second hook checks, on the GPU, the division the fp8 quantiser uses in
 * place of an IEEE division (see moe_debug_check_quant_division).
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

/*
 * moe_debug_check_quant_division: moe_permute_quant_fp8 divides each element
 * x of a 128-column group by the group's scale s = amax / 448 with an
 * fma-corrected reciprocal (quant.cuh, div_by_scale) when s lies in
 * [2^-100, 2^100].  This runs, on the current device, every pair (x, amax) of
 * finite bf16 values with |x| <= amax and amax > 0 through both that division
 * and __fdiv_rn, and writes to the HOST array counts[4]:
 *   counts[0]  pairs checked,
 *   counts[1]  pairs whose e4m3 codes (satfinite, round to nearest even)
 *              differ,
 *   counts[2]  pairs whose fp32 quotients differ while |x / s| >= 2^-12,
 *   counts[3]  pairs outside the scale range (IEEE division there).
 * Synchronous (about a millisecond of GPU time).  Returns MOE_OK,
 * MOE_ERR_INVALID_ARG (counts NULL) or MOE_ERR_CUDA.
 */
MOE_API int moe_debug_check_quant_division(unsigned long long *counts);

#ifdef __cplusplus
}
#endif

#endif /* MOE_PERMUTE_DEBUG_H */
