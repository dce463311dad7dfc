/*
 * moe_permute.h -- C ABI of the GB300 (sm_103a) MoE token permute / unpermute
 * library (libmoe_permute.so).
 *
 * The two operations come from vLLM PR #14568, "permute/unpermute kernel for
 * moe optimization", description: moe_permute expands every token into its K
 * routed rows and orders them by expert, so that each expert's rows are
 * contiguous for the grouped GEMM that follows; moe_unpermute reduces the
 * expanded GEMM output back to tokens, scaling each row by its top-k weight.
 * The output buffers and their shapes follow the vLLM PR #43014 digest,
 * section "key source excerpts" (MoEPermuteScratch): expert_first_token_offset
 * int64 [num_local_experts + 1], permuted_idx and inv_permuted_idx int32
 * [max_tokens * topk], permuted_hidden_states [max_tokens * topk, hidden].
 * The workspace-size query and the caller-owned, reused scratch follow the
 * same digest, sections "implementation breakdown" (items 1 and 3: scratch
 * allocated once and reused, the sort workspace sized by a query op) and
 * "review highlights" (outputs are written into the caller's buffers, never
 * into a copy).
 *
 * Conventions shared by every entry point:
 *  - Every pointer except the ones noted as host pointers is a DEVICE pointer
 *    to caller-owned, contiguous, row-major memory on the current device.
 *    The library never allocates, frees or synchronises (except
 *    moe_read_status, which synchronises the given stream by design;
 *    moe_permute_read_status is its asynchronous form); all
 *    device work is enqueued on `stream` in stream order, so the calls can be
 *    captured into a CUDA graph.
 *  - Return value: MOE_OK (0) or a negative moe_status_t.  Argument errors are
 *    detected on the host before anything is enqueued; nothing is written on
 *    error.  No C++ exception crosses this ABI.
 *  - Conditions found on the device (bad ids, bad map values, bad inverse
 *    indices) never trap: the row is dropped and a MOE_FLAG_* bit is ORed into
 *    the workspace status word (read it with moe_read_status).
 *  - One workspace must not be used by two calls that may run concurrently
 *    (two streams, or overlapping graph branches).
 *  - Row order inside one expert is stable: key = local expert, tie-break =
 *    expanded row id r = t*topk + k.
 */
#ifndef MOE_PERMUTE_H
#define MOE_PERMUTE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL means the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,          /* bad size, NULL or misaligned pointer */
    MOE_ERR_WORKSPACE_TOO_SMALL = -2,  /* workspace_bytes below the requirement */
    MOE_ERR_UNSUPPORTED_DEVICE = -3,   /* current device is not sm_103 family */
    MOE_ERR_CUDA = -4                  /* a CUDA runtime call or launch failed */
} moe_status_t;

/* Element type of the rows moved by moe_permute (rows are moved as bytes). */
typedef enum {
    MOE_DTYPE_BF16 = 0,
    MOE_DTYPE_FP16 = 1,
    MOE_DTYPE_FP8_E4M3 = 2,
    MOE_DTYPE_FP8_E5M2 = 3,
    MOE_DTYPE_FP32 = 4
} moe_dtype_t;

/* Storage type of topk_ids. */
typedef enum { MOE_INDEX_INT32 = 0, MOE_INDEX_INT64 = 1 } moe_index_t;

/* Device status bits (ORed into the workspace status word). */
#define MOE_FLAG_ID_OUT_OF_RANGE  1u  /* a topk id outside [0, num_experts) */
#define MOE_FLAG_MAP_OUT_OF_RANGE 2u  /* expert_map value not -1 and outside [0, num_local_experts) */
#define MOE_FLAG_INV_OUT_OF_RANGE 4u  /* unpermute: inv index >= num_rows or < -1 */
#define MOE_FLAG_BARRIER_TIMEOUT  8u  /* permute: a bounded wait for another block's
                                         histogram gave up.  The outputs of that call
                                         are undefined; the workspace needs no
                                         re-initialisation: every call tags its
                                         histogram entries afresh, so the next call on
                                         the same workspace is exact again */
#define MOE_FLAG_CAPACITY_OVERFLOW 16u /* batched permute: an expert got more rows than
                                          its capacity; the extra rows were dropped */

/* Limits checked on the host. */
#define MOE_MAX_TOPK 32
#define MOE_MAX_LOCAL_EXPERTS 1024

/*
 * moe_permute_supported: 1 if `device` is an sm_103-family GPU this library
 * was built for, 0 if not, MOE_ERR_CUDA if the device cannot be queried.
 * (Digest of vLLM PR #43014, "review highlights": callers check support
 * before sizing the sort workspace.)
 */
MOE_API int moe_permute_supported(int device);

/* Human-readable text for a moe_status_t; never NULL; static storage. */
MOE_API const char *moe_status_string(int status);

/*
 * moe_permute_workspace_size: bytes of device workspace one moe_permute call
 * with at most `max_tokens` tokens needs, for `topk` and `num_experts` (global
 * experts).  Returns 0 for invalid arguments (max_tokens < 0, topk < 1 or
 * > MOE_MAX_TOPK, num_experts < 1, or max_tokens*topk > INT32_MAX).
 * The workspace holds the per-block expert histograms of one call (a table
 * whose entries carry a per-call tag), a call counter and the status word.
 * (Digest of vLLM PR #43014, "implementation breakdown" item 3: the sort
 * workspace is sized by a query op and pre-allocated.)
 */
MOE_API size_t moe_permute_workspace_size(int64_t max_tokens, int32_t topk,
                                  int32_t num_experts);

/*
 * moe_permute_workspace_init: zero the first `workspace_bytes` bytes of the
 * workspace (status word, call counter, histogram table).  Call once after
 * allocating the workspace (async on `stream`), with the size that was
 * allocated; every later call leaves the workspace ready for the next one.
 * `workspace` must be 256-byte aligned and at least
 * moe_permute_workspace_size(...) bytes.
 */
MOE_API int moe_permute_workspace_init(void *workspace, size_t workspace_bytes,
                               moe_stream_t stream);

/*
 * moe_permute: routing metadata plus the row gather.
 *
 *   T = num_tokens, H = hidden_size, K = topk, E = num_experts,
 *   E_L = num_local_experts, R = T*K, r = t*K + k.
 *
 * In:
 *  hidden_states     [T, H] of hidden_dtype.  May be NULL only when
 *                    permuted_hidden_states is NULL (metadata-only call).
 *  hidden_scales     [T, scale_cols] fp32 (e.g. fp8 per-token per-128-column
 *                    scales, scale_cols = H/128) or NULL with scale_cols = 0.
 *  topk_ids          [T, K], int32 or int64 per topk_ids_dtype (4/8-byte aligned).
 *  expert_map        [E] int32 or NULL.  NULL: local expert = global id and
 *                    E_L must equal E.  Otherwise expert_map[g] is the local id
 *                    of global expert g, or -1 if g is not local (its rows are
 *                    dropped).  Single-GPU index filtering only.
 * Out (all written in place, stream-ordered):
 *  permuted_hidden_states [R, H] or NULL.  Row p < N_valid is
 *                    hidden_states[permuted_idx[p] / K]; rows >= N_valid are
 *                    not written.
 *  permuted_scales   [R, scale_cols] fp32, or NULL (must be NULL iff
 *                    hidden_scales is NULL).  Row p is hidden_scales[token].
 *  expert_first_token_offset [E_L + 1] int64 (8-byte aligned): offset[0] = 0,
 *                    offset[e+1] - offset[e] = rows routed to local expert e,
 *                    offset[E_L] = N_valid.
 *  permuted_idx      [R] int32: p -> r for p < N_valid, -1 for p >= N_valid.
 *  inv_permuted_idx  [R] int32: r -> p, or -1 for a dropped row.
 * Workspace: at least moe_permute_workspace_size(T, K, E) bytes, 256-byte
 *  aligned, initialised once by moe_permute_workspace_init.
 * Dropped rows: an id outside [0, E) (flag MOE_FLAG_ID_OUT_OF_RANGE), a map
 *  value of -1 (no flag), or a map value outside [0, E_L) other than -1
 *  (flag MOE_FLAG_MAP_OUT_OF_RANGE).
 * T = 0 is valid: offsets are set to 0 and nothing else is written; every
 *  pointer but expert_first_token_offset may then be NULL.
 * Limits: K <= MOE_MAX_TOPK, E_L <= MOE_MAX_LOCAL_EXPERTS, R <= INT32_MAX.
 */
MOE_API int moe_permute(const void *hidden_states, moe_dtype_t hidden_dtype,
                const float *hidden_scales, int64_t scale_cols,
                const void *topk_ids, moe_index_t topk_ids_dtype,
                const int32_t *expert_map,
                int64_t num_tokens, int64_t hidden_size, int32_t topk,
                int32_t num_experts, int32_t num_local_experts,
                void *permuted_hidden_states, float *permuted_scales,
                int64_t *expert_first_token_offset,
                int32_t *permuted_idx, int32_t *inv_permuted_idx,
                void *workspace, size_t workspace_bytes,
                moe_stream_t stream);

/*
 * moe_permute_batched: moe_permute into the batched activation layout, the
 * second of the two layouts the modular MoE kernel's activation-format enum
 * distinguishes ("[Kernels] MoE refactor" (vLLM PR #19636), description):
 * one fixed-capacity block of rows per local expert instead of contiguous
 * variable-length segments.
 *
 *  max_rows_per_expert  M >= 1, the capacity of each expert's block
 *                       (E_L * M <= INT32_MAX).  M = num_tokens always fits
 *                       when a token's K experts are distinct.
 *  batched_hidden_states [E_L, M, H] of hidden_dtype, or NULL (metadata only).
 *                       Slot e*M + j holds the j-th row (stable, r order)
 *                       routed to local expert e; slots j >= expert_num_tokens[e]
 *                       are not written.
 *  batched_scales       [E_L, M, scale_cols] fp32 or NULL, as for moe_permute.
 *  expert_num_tokens    [E_L] int32: min(rows routed to e, M).
 *  inv_permuted_idx     [T*K] int32: r -> slot e*M + j, or -1 for a dropped
 *                       row.  Rows beyond an expert's capacity are dropped too
 *                       and raise MOE_FLAG_CAPACITY_OVERFLOW.  moe_unpermute
 *                       with num_rows = E_L * M reduces the batched GEMM
 *                       output back to tokens.
 *  Inputs, dropped-row rules, workspace rules and errors are those of
 *  moe_permute; T = 0 sets expert_num_tokens to 0 (other pointers may be NULL).
 */
MOE_API int moe_permute_batched(const void *hidden_states, moe_dtype_t hidden_dtype,
                                const float *hidden_scales, int64_t scale_cols,
                                const void *topk_ids, moe_index_t topk_ids_dtype,
                                const int32_t *expert_map,
                                int64_t num_tokens, int64_t hidden_size, int32_t topk,
                                int32_t num_experts, int32_t num_local_experts,
                                int64_t max_rows_per_expert,
                                void *batched_hidden_states, float *batched_scales,
                                int32_t *expert_num_tokens, int32_t *inv_permuted_idx,
                                void *workspace, size_t workspace_bytes,
                                moe_stream_t stream);

/*
 * moe_permute_quant_fp8: moe_permute for bf16 activations that feed an fp8
 * grouped GEMM, with the quantisation done during the row gather instead of
 * in a separate pass ("[Kernels] MoE refactor" (vLLM PR #19636), bot summary:
 * activation quantisation parameters quant_dtype, per_act_token_quant,
 * block_shape).  Per token and per MOE_QUANT_GROUP-column group:
 *   scale = amax(|x|) / 448 (fp32 division; 1 for an all-zero group),
 *   code  = e4m3(x / scale) (fp32 division, round to nearest even,
 *           saturating at +-448),
 * and permuted row p gets the codes and scales of its token.
 *
 *  hidden_states    [T, H] bf16, 16-byte aligned, H a multiple of MOE_QUANT_GROUP.
 *  permuted_codes   [R, H] fp8 e4m3 (bytes), 8-byte aligned.
 *  permuted_scales  [R, H / MOE_QUANT_GROUP] fp32.
 *  Every other argument, the metadata outputs, the workspace rules and the
 *  dropped-row rules are those of moe_permute.  Rows p >= N_valid of the codes
 *  and scales are not written.
 */
#define MOE_QUANT_GROUP 128
MOE_API int moe_permute_quant_fp8(const void *hidden_states, const void *topk_ids,
                                  moe_index_t topk_ids_dtype, const int32_t *expert_map,
                                  int64_t num_tokens, int64_t hidden_size, int32_t topk,
                                  int32_t num_experts, int32_t num_local_experts,
                                  void *permuted_codes, float *permuted_scales,
                                  int64_t *expert_first_token_offset,
                                  int32_t *permuted_idx, int32_t *inv_permuted_idx,
                                  void *workspace, size_t workspace_bytes,
                                  moe_stream_t stream);

/*
 * moe_unpermute: out[t] = bf16_rne( sum over k = 0..K-1 in order, skipping
 * rows with inv_permuted_idx[t*K+k] == -1, of topk_weights[t,k] *
 * permuted_rows[inv_permuted_idx[t*K+k]] ), accumulated in fp32 with a
 * separately rounded multiply and add per term.  A token whose rows were all
 * dropped gets +0.0.
 *
 *  permuted_rows     [num_rows, H] bf16 (the grouped-GEMM output, in the
 *                    permuted row order).
 *  topk_weights      [T, K] fp32.
 *  inv_permuted_idx  [T*K] int32, as written by moe_permute.  A value >=
 *                    num_rows or < -1 is treated as dropped and, when a
 *                    workspace is given, raises MOE_FLAG_INV_OUT_OF_RANGE.
 *  out               [T, H] bf16.  Must not overlap the inputs.
 *  workspace         optional (may be NULL): only its status word is used.
 * T = 0 is valid and enqueues nothing.
 */
MOE_API int moe_unpermute(const void *permuted_rows, int64_t num_rows,
                  const float *topk_weights, const int32_t *inv_permuted_idx,
                  int64_t num_tokens, int64_t hidden_size, int32_t topk,
                  void *out, void *workspace, moe_stream_t stream);

/*
 * moe_read_status: copy the workspace status word (OR of MOE_FLAG_* bits since
 * the last clear) to the HOST pointer `host_status`.  Synchronises `stream`.
 */
MOE_API int moe_read_status(const void *workspace, uint32_t *host_status,
                    moe_stream_t stream);

/*
 * moe_permute_read_status: the asynchronous form of moe_read_status.  Enqueues
 * on `stream` one tiny kernel that copies the status word to `dst` and, when
 * clear_after_read is non-zero, zeroes the word in the same step; nothing
 * synchronises, so the call captures into a CUDA graph with the permutes it
 * follows, and a serving loop reads each step's flags without a host round
 * trip.  (vLLM PR #43014 digest, "review highlights": results go into the
 * caller's buffers.)
 *  dst  4-byte aligned memory the device can write: device or managed memory,
 *       or page-locked host memory (cudaHostAlloc / cudaHostRegister).
 *       Pageable host memory is refused with MOE_ERR_INVALID_ARG.  The value
 *       is there once the stream has reached this call.
 */
MOE_API int moe_permute_read_status(void *workspace, uint32_t *dst, int clear_after_read,
                                    moe_stream_t stream);

/* moe_clear_status: zero the status word (async on `stream`). */
MOE_API int moe_clear_status(void *workspace, moe_stream_t stream);

/*
 * moe_permute_noalloc: moe_permute for callers that cannot allocate device
 * memory at all, not even the small workspace moe_permute asks for.  Examples:
 * a plugin whose host framework owns every device allocation and only hands
 * over input and output pointers; a serving loop that must not call
 * cudaMalloc once it is running, because cudaMalloc can synchronise the
 * device and grow the memory footprint after start-up.  The pages have no
 * counterpart of this entry point: their scratch buffers are always
 * allocated by the caller.
 *
 * Arguments and results are exactly those of moe_permute without the
 * workspace.  The scratch lives instead in one static device array of
 * MOE_NOALLOC_SCRATCH_BYTES inside this library: every GPU that loads the
 * library holds it until the process exits.  Nothing is allocated or freed.
 *  - The first call on a device looks up that array's device address and
 *    zeroes it (stream-ordered on `stream`).  Make that first
 *    call before capturing any stream into a CUDA graph.
 *  - Every call on a device shares the one array, which keeps the last call's
 *    contents.  Calls that may overlap on the GPU (two streams, or parallel
 *    graph branches) race on it; serialise them.
 *  - Arguments are checked first, exactly as moe_permute checks them, and
 *    before any device is touched.  Then a call whose scratch need,
 *    moe_permute_workspace_size(num_tokens, topk, num_experts), exceeds
 *    MOE_NOALLOC_SCRATCH_BYTES returns MOE_ERR_WORKSPACE_TOO_SMALL and
 *    enqueues nothing: up to 256 experts fit for any token count, 512
 *    experts up to 512 tokens, 1024 up to 256.  num_tokens = 0 always fits.
 *  - Device status flags (MOE_FLAG_*) are kept in the shared array and are
 *    not readable through this entry point; rows with bad ids are still
 *    dropped exactly as moe_permute drops them.  After a bounded wait gave
 *    up (MOE_FLAG_BARRIER_TIMEOUT in moe_permute's terms) the next call is
 *    exact again with no re-initialisation, as for moe_permute.
 */
#define MOE_NOALLOC_SCRATCH_BYTES ((size_t)(1u << 20) + 256u)
MOE_API int moe_permute_noalloc(const void *hidden_states, moe_dtype_t hidden_dtype,
                                const float *hidden_scales, int64_t scale_cols,
                                const void *topk_ids, moe_index_t topk_ids_dtype,
                                const int32_t *expert_map,
                                int64_t num_tokens, int64_t hidden_size, int32_t topk,
                                int32_t num_experts, int32_t num_local_experts,
                                void *permuted_hidden_states, float *permuted_scales,
                                int64_t *expert_first_token_offset,
                                int32_t *permuted_idx, int32_t *inv_permuted_idx,
                                moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_PERMUTE_H */
