/*
 * moe_oracle.c -- plain, slow, single-threaded CPU oracle for the MoE token
 * permute / unpermute path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * loads this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or helper with the CUDA
 * path.  Build with -ffp-contract=off so that every multiply and add below is
 * a separately rounded IEEE fp32 operation.
 *
 * What is computed, and where it is defined:
 *
 *  - "permute/unpermute kernel for moe optimization" (vLLM PR #14568),
 *    description: moe_permute expands every token into its K routed rows and
 *    orders them by expert so that each expert's tokens are contiguous for the
 *    grouped GEMM; moe_unpermute reduces the expanded GEMM output back to
 *    tokens, scaling each row by its top-k weight.
 *  - "MoE permute pre-allocated scratch" digest (vLLM PR #43014), section
 *    "key source excerpts": the output buffers -- expert_first_token_offset
 *    int64 [num_local_experts + 1], permuted_idx and inv_permuted_idx int32
 *    [max_tokens * topk], permuted_hidden_states [max_tokens * topk * hidden],
 *    and token_expert_indices = arange(T*K) viewed [T, K] (so the expanded
 *    row id of (t, k) is r = t*K + k).
 *  - The order inside one expert is not fixed by the pages; it is taken to be
 *    stable by expanded row id r (key = local expert, tie-break = r).  The
 *    oracle therefore computes a stable counting sort written as the plain
 *    cursor loop below, which *is* the stable sort by (expert, r).
 *
 * Readings of points the pages leave open (each is also listed in the design
 * notes):
 *  - permuted_idx[p] holds the expanded row id r (not the token id); the
 *    source token is r / K.  inv_permuted_idx[r] = p.
 *  - An id outside [0, E) is dropped and raises ORC_FLAG_ID_RANGE.  With an
 *    expert_map, map value -1 means "not local" (dropped silently); any other
 *    value outside [0, E_local) is dropped and raises ORC_FLAG_MAP_RANGE.
 *  - Dropped rows get inv_permuted_idx[r] = -1 and do not appear in
 *    [0, N_valid); permuted_idx[p] = -1 for p in [N_valid, T*K).  Rows
 *    p >= N_valid of permuted_hidden are not written.
 *  - Quantise-on-permute (the fp8 activation step before the fp8 grouped
 *    GEMM; "[Kernels] MoE refactor" (vLLM PR #19636), bot summary: quant_dtype,
 *    per_act_token_quant, block_shape): per token and 128-column group,
 *    scale = amax / 448 (1 for an all-zero group), code = e4m3(x / scale) with
 *    round-to-nearest-even and saturation at +-448; the permuted rows are
 *    these codes and scales gathered like any other rows.
 *  - Batched layout (the modular kernel's second activation format, "[Kernels]
 *    MoE refactor" (vLLM PR #19636), description: an activation-format enum
 *    lets prepare/finalize and the experts agree on the layout): rows of local
 *    expert e go to slots e*M + j, j = the row's stable rank inside the expert,
 *    for a per-expert capacity M; rows with j >= M do not fit and are dropped
 *    with ORC_FLAG_CAPACITY; expert_num_tokens[e] = min(count, M).
 *  - Unpermute: acc = 0.0f; for k = 0..K-1 in order, if inv[t*K+k] names a
 *    row (0 <= inv < num_rows), acc = acc + w[t,k] * float(row) (fp32
 *    multiply, then fp32 add); the result is rounded once to bf16,
 *    round-to-nearest-even.  A token with no valid row yields +0.0.  -1 is a
 *    dropped row; any other value outside [0, num_rows) is skipped as well
 *    and raises ORC_FLAG_INV_RANGE.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#define ORC_FLAG_ID_RANGE  1u
#define ORC_FLAG_MAP_RANGE 2u
#define ORC_FLAG_INV_RANGE 4u
#define ORC_FLAG_CAPACITY  16u

/* Expert id of (t, k), widened to 64 bits whatever the storage type. */
static int64_t orc_topk_id(const void *topk_ids, int ids_are_i64, int64_t r)
{
    if (ids_are_i64)
        return ((const int64_t *)topk_ids)[r];
    return (int64_t)((const int32_t *)topk_ids)[r];
}

/* Local expert of expanded row r, or -1 when the row is dropped. */
static int32_t orc_local_expert(const void *topk_ids, int ids_are_i64,
                                const int32_t *expert_map, int32_t E,
                                int32_t E_local, int64_t r, uint32_t *flags)
{
    int64_t g = orc_topk_id(topk_ids, ids_are_i64, r);
    if (g < 0 || g >= (int64_t)E) {
        *flags |= ORC_FLAG_ID_RANGE;
        return -1;
    }
    if (expert_map == NULL)
        return (int32_t)g;
    int32_t e = expert_map[g];
    if (e == -1)
        return -1;
    if (e < 0 || e >= E_local) {
        *flags |= ORC_FLAG_MAP_RANGE;
        return -1;
    }
    return e;
}

/*
 * oracle_permute: routing metadata plus the row (and optional scale-row) copy.
 *
 * hidden:            [T, row_bytes] bytes (any element type: rows are copied
 *                    as raw bytes), may be NULL when permuted_hidden is NULL.
 * scales:            [T, scale_cols] fp32 or NULL.
 * topk_ids:          [T, K] int32 (ids_are_i64 == 0) or int64.
 * expert_map:        [E] int32 or NULL (identity, E_local must equal E).
 * offsets:           [E_local + 1] int64 out.
 * permuted_idx:      [T*K] int32 out.
 * inv_permuted_idx:  [T*K] int32 out.
 * permuted_hidden:   [T*K, row_bytes] out or NULL.
 * permuted_scales:   [T*K, scale_cols] fp32 out or NULL.
 * Returns the OR of the ORC_FLAG_* conditions met; -1 cast to uint32 on a
 * host allocation failure.
 */
uint32_t oracle_permute(const void *hidden, int64_t row_bytes,
                        const float *scales, int64_t scale_cols,
                        const void *topk_ids, int ids_are_i64,
                        const int32_t *expert_map,
                        int64_t T, int32_t K, int32_t E, int32_t E_local,
                        int64_t *offsets, int32_t *permuted_idx,
                        int32_t *inv_permuted_idx,
                        void *permuted_hidden, float *permuted_scales)
{
    uint32_t flags = 0;
    int64_t R = T * (int64_t)K;

    /* Step 1: the local expert of every expanded row r = t*K + k. */
    int32_t *key = (int32_t *)malloc((size_t)(R > 0 ? R : 1) * sizeof(int32_t));
    int64_t *count = (int64_t *)calloc((size_t)E_local + 1, sizeof(int64_t));
    int64_t *cursor = (int64_t *)malloc(((size_t)E_local + 1) * sizeof(int64_t));
    if (!key || !count || !cursor) {
        free(key); free(count); free(cursor);
        return 0xffffffffu;
    }
    for (int64_t t = 0; t < T; ++t)
        for (int32_t k = 0; k < K; ++k) {
            int64_t r = t * K + k;
            key[r] = orc_local_expert(topk_ids, ids_are_i64, expert_map, E,
                                      E_local, r, &flags);
        }

    /* Step 2: histogram over local experts (valid rows only). */
    for (int64_t r = 0; r < R; ++r)
        if (key[r] >= 0)
            count[key[r]] += 1;

    /* Step 3: expert_first_token_offset = exclusive prefix sum of counts. */
    offsets[0] = 0;
    for (int32_t e = 0; e < E_local; ++e)
        offsets[e + 1] = offsets[e] + count[e];
    int64_t n_valid = offsets[E_local];

    /* Step 4: stable scatter, r ascending, one cursor per expert. */
    for (int32_t e = 0; e < E_local; ++e)
        cursor[e] = offsets[e];
    for (int64_t r = 0; r < R; ++r) {
        if (key[r] < 0) {
            inv_permuted_idx[r] = -1;
            continue;
        }
        int64_t p = cursor[key[r]]++;
        permuted_idx[p] = (int32_t)r;
        inv_permuted_idx[r] = (int32_t)p;
        int64_t t = r / K;
        if (permuted_hidden != NULL)
            memcpy((char *)permuted_hidden + p * row_bytes,
                   (const char *)hidden + t * row_bytes, (size_t)row_bytes);
        if (permuted_scales != NULL && scale_cols > 0)
            memcpy(permuted_scales + p * scale_cols, scales + t * scale_cols,
                   (size_t)scale_cols * sizeof(float));
    }
    for (int64_t p = n_valid; p < R; ++p)
        permuted_idx[p] = -1;

    free(key); free(count); free(cursor);
    return flags;
}

/* bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits. */
static float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * fp32 -> bf16, IEEE round-to-nearest, ties to even, on the 16 bits dropped.
 * A carry out of the kept mantissa correctly bumps the exponent (and turns the
 * largest finite values into infinity).  NaN stays NaN, made quiet.
 */
static uint16_t orc_f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xffffu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

/*
 * oracle_unpermute: out[t] = bf16_rne( sum_k w[t,k] * rows[inv[t*K+k]] ),
 * k ascending, fp32 multiply then fp32 add, dropped rows (inv = -1) skipped.
 * An inv value outside [-1, num_rows) -- at or past the end of rows, or below
 * -1 -- names no row and no dropped row: it is skipped too and raises
 * ORC_FLAG_INV_RANGE.
 *
 * rows: [num_rows, H] bf16 bits; w: [T, K] fp32; inv: [T*K] int32;
 * out: [T, H] bf16 bits.
 */
uint32_t oracle_unpermute(const uint16_t *rows, int64_t num_rows,
                          const float *w, const int32_t *inv,
                          int64_t T, int64_t H, int32_t K, uint16_t *out)
{
    uint32_t flags = 0;
    for (int64_t t = 0; t < T; ++t)
        for (int32_t k = 0; k < K; ++k)
            if (inv[t * K + k] < -1 || inv[t * K + k] >= num_rows)
                flags |= ORC_FLAG_INV_RANGE;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int32_t k = 0; k < K; ++k) {
                int32_t p = inv[t * K + k];
                if (p < 0 || p >= num_rows)
                    continue;
                float x = orc_bf16_to_f32(rows[(int64_t)p * H + h]);
                float prod = w[t * K + k] * x;
                acc = acc + prod;
            }
            out[t * H + h] = orc_f32_to_bf16_rne(acc);
        }
    }
    return flags;
}

/* The rounding helper alone, exposed so tests can pin it directly. */
void oracle_f32_to_bf16_rne(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_f32_to_bf16_rne(x[i]);
}

/*
 * fp32 -> fp8 e4m3 ("fn" variant: no infinities, 0x7F/0xFF are NaN, largest
 * finite value 448 = 1.75 * 2^8), round to nearest, ties to even, saturating
 * finite values beyond 448 to +-448.  Written from the format: normal codes
 * are (exponent + 7) << 3 | mantissa for 2^-6 <= |v| < 2^9, subnormal codes
 * count multiples of 2^-9 below 2^-6.  Exact in double: every scaling below
 * is by a power of two.
 */
static double orc_round_half_even(double v) /* v >= 0 */
{
    double fl = (double)(long long)v;
    double frac = v - fl;
    if (frac > 0.5 || (frac == 0.5 && ((long long)fl & 1)))
        fl += 1.0;
    return fl;
}

static uint8_t orc_f32_to_e4m3_satfinite(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint8_t sign = (uint8_t)((u >> 31) << 7);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint8_t)(sign | 0x7f); /* NaN */
    double a = fabs((double)f);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7e); /* saturate (also +-inf) */
    if (a < 0.015625) { /* below 2^-6: subnormal grid of 2^-9 */
        double m = orc_round_half_even(a * 512.0); /* 0..8; 8 is the smallest normal */
        return (uint8_t)(sign | (uint8_t)m);
    }
    int e = 0;
    double t = a;
    while (t >= 2.0) { t *= 0.5; e += 1; }
    while (t < 1.0) { t *= 2.0; e -= 1; }
    double m8 = orc_round_half_even(t * 8.0); /* 8..16 */
    if (m8 == 16.0) { m8 = 8.0; e += 1; }
    if (e > 8 || (e == 8 && m8 > 14.0))
        return (uint8_t)(sign | 0x7e);
    return (uint8_t)(sign | (uint8_t)(((e + 7) << 3) | ((int)m8 - 8)));
}

/* The conversion alone, exposed so tests can pin it directly. */
void oracle_f32_to_e4m3(const float *x, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_f32_to_e4m3_satfinite(x[i]);
}

/*
 * Per-token, per-group fp8 quantisation of bf16 rows (the activation format
 * the fp8 grouped GEMM reads: per-token quantisation in column groups):
 *   amax  = max |x| over the group's elements (0 if all are zero),
 *   scale = amax / 448 (fp32 division), or 1 when amax == 0,
 *   code  = e4m3(x / scale) (fp32 division, then the conversion above).
 * x: [T, H] bf16 bits; codes: [T, H] e4m3; scales: [T, H / group] fp32.
 * H must be a multiple of group.
 */
void oracle_quantize_fp8(const uint16_t *x, int64_t T, int64_t H, int64_t group,
                         uint8_t *codes, float *scales)
{
    int64_t n_groups = H / group;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t g = 0; g < n_groups; ++g) {
            const uint16_t *xg = x + t * H + g * group;
            float amax = 0.0f;
            for (int64_t i = 0; i < group; ++i) {
                float v = fabsf(orc_bf16_to_f32(xg[i]));
                if (v > amax)
                    amax = v;
            }
            float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
            scales[t * n_groups + g] = scale;
            for (int64_t i = 0; i < group; ++i)
                codes[t * H + g * group + i] =
                    orc_f32_to_e4m3_satfinite(orc_bf16_to_f32(xg[i]) / scale);
        }
    }
}

/*
 * oracle_permute_batched: the batched layout.  Slots are [E_local, M] rows.
 * inv_permuted_idx[r] = e*M + j, or -1 (dropped row, or no room: j >= M).
 * expert_num_tokens: [E_local] int32 = min(rows routed to e, M).
 * batched_hidden: [E_local*M, row_bytes] or NULL; batched_scales likewise.
 * Slots j >= expert_num_tokens[e] are not written.
 */
uint32_t oracle_permute_batched(const void *hidden, int64_t row_bytes,
                                const float *scales, int64_t scale_cols,
                                const void *topk_ids, int ids_are_i64,
                                const int32_t *expert_map,
                                int64_t T, int32_t K, int32_t E, int32_t E_local,
                                int64_t M, int32_t *expert_num_tokens,
                                int32_t *inv_permuted_idx,
                                void *batched_hidden, float *batched_scales)
{
    uint32_t flags = 0;
    int64_t R = T * (int64_t)K;
    int64_t *next = (int64_t *)calloc((size_t)E_local + 1, sizeof(int64_t));
    if (!next)
        return 0xffffffffu;
    for (int64_t r = 0; r < R; ++r) {
        int32_t e = orc_local_expert(topk_ids, ids_are_i64, expert_map, E,
                                     E_local, r, &flags);
        if (e < 0) {
            inv_permuted_idx[r] = -1;
            continue;
        }
        int64_t j = next[e]++;
        if (j >= M) {
            inv_permuted_idx[r] = -1;
            flags |= ORC_FLAG_CAPACITY;
            continue;
        }
        int64_t slot = (int64_t)e * M + j;
        inv_permuted_idx[r] = (int32_t)slot;
        int64_t t = r / K;
        if (batched_hidden != NULL)
            memcpy((char *)batched_hidden + slot * row_bytes,
                   (const char *)hidden + t * row_bytes, (size_t)row_bytes);
        if (batched_scales != NULL && scale_cols > 0)
            memcpy(batched_scales + slot * scale_cols, scales + t * scale_cols,
                   (size_t)scale_cols * sizeof(float));
    }
    for (int32_t e = 0; e < E_local; ++e)
        expert_num_tokens[e] = (int32_t)(next[e] < M ? next[e] : M);
    free(next);
    return flags;
}
