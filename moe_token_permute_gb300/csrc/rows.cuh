// rows.cuh -- the row-moving kernels of moe_permute and moe_unpermute.
//
// vLLM PR #14568 ("permute/unpermute kernel for moe optimization",
// description): permute gathers each expert's non-contiguous tokens into
// contiguous rows for the grouped GEMM; unpermute reduces the expanded GEMM
// output back to tokens and scales each row by its top-k weight.
//
// Both are pure HBM traffic.  The unit of work is a (token, chunk) item: one
// warp moves one chunk of 32*V vectors of one token's row (VecT is 16 bytes
// whenever the pointers and the row pitch allow it).  Permute reads the chunk
// once and writes it to each of the token's K destinations; unpermute reads
// the chunk of each of the token's kept rows -- all loads of a group of up to
// four rows in flight at once -- and writes one.  Splitting rows into chunks
// keeps every SM busy at small token counts and bounds the registers per warp
// at large ones.
#pragma once

#include "common.cuh"
#include "quant.cuh"
#include "routing.cuh"

namespace moe {

constexpr int kRowThreads = 256;
constexpr int kRowWarps = kRowThreads / kWarpSize;

template <typename VecT, int V>
__device__ __forceinline__ void load_chunk(const VecT* __restrict__ src, int64_t c0,
                                           int64_t row_vecs, VecT (&v)[V]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int64_t c = c0 + i * 32 + lane;
    if (c < row_vecs) v[i] = ld_stream(src + c);
  }
}

// Write one chunk to every destination row p_k whose bit k is set in `valid`;
// lane k < K holds p_k in `p_lane`.
template <typename VecT, int V>
__device__ __forceinline__ void store_chunk(const VecT (&v)[V], VecT* __restrict__ out,
                                            int64_t c0, int64_t row_vecs, int p_lane,
                                            unsigned valid) {
  const int lane = threadIdx.x & 31;
  unsigned m = valid;
  while (m != 0u) {
    const int k = __ffs(m) - 1;
    m &= m - 1u;
    const int pk = __shfl_sync(kFullMask, p_lane, k);
    VecT* dst = out + static_cast<int64_t>(pk) * row_vecs;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int64_t c = c0 + i * 32 + lane;
      if (c < row_vecs) dst[c] = v[i];
    }
  }
}

// Row gather of the large-batch permute: one warp per (token, chunk) item, one
// item per warp, so the hardware block scheduler balances the work across SMs.
// Launched as the dependent of the routing grid, which lets it start early:
// the caller's hidden rows are complete by then (the routing grid has passed
// its own dependency wait), so the first kEarlyLoadWarps warps of each block
// load their chunk first and only then wait for the routing grid before
// reading inv_permuted_idx; the others wait first.  With every resident warp
// loading early (about 20 MB at once), the routing grid's own reads queue
// behind those loads and it ends about as much later as they gained; with
// half of the warps, measured on GB300: Mixtral T = 16384 permute 2.1% faster,
// Qwen3 T = 8192 2.8%, DeepSeek-V3 T = 32768 unchanged (a quarter to three
// quarters were within 1% of half).
constexpr int kEarlyLoadWarps = kRowWarps / 2;

template <typename VecT, int V>
__global__ void __launch_bounds__(kRowThreads)
k_gather_rows(const VecT* __restrict__ hidden, int64_t row_vecs,
              const float* __restrict__ scales, int64_t scale_cols,
              const int32_t* __restrict__ inv_permuted_idx, int64_t T, int K,
              VecT* __restrict__ permuted_hidden, float* __restrict__ permuted_scales,
              int64_t num_out_rows) {
  constexpr int64_t kChunk = 32 * V;
  const int lane = threadIdx.x & 31;
  const int64_t n_chunks = (row_vecs + kChunk - 1) / kChunk;
  const int64_t item = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (item >= T * n_chunks) return;
  const int64_t t = item / n_chunks;
  const int64_t c0 = (item - t * n_chunks) * kChunk;
  VecT v[V];
  if ((threadIdx.x >> 5) >= kEarlyLoadWarps) pdl_wait();
  load_chunk<VecT, V>(hidden + t * row_vecs, c0, row_vecs, v);
  const bool with_scales = permuted_scales != nullptr && c0 == 0;
  float sc[kPreScaleChunks];
  if (with_scales) load_token_scales(scales + t * scale_cols, scale_cols, sc);
  pdl_wait();
  int p = lane < K ? __ldcg(inv_permuted_idx + t * K + lane) : -1;
  // Positions outside [0, num_out_rows) can only come from a routing grid that
  // gave up (status MOE_FLAG_BARRIER_TIMEOUT); never store through them.
  if (p >= num_out_rows) p = -1;
  const unsigned valid = __ballot_sync(kFullMask, p >= 0);
  if (valid == 0u) return;  // every row of this token was dropped
  store_chunk<VecT, V>(v, permuted_hidden, c0, row_vecs, p, valid);
  if (with_scales)
    store_token_scales(scales + t * scale_cols, scale_cols, sc, permuted_scales, p, valid);
}

// One item's row chunk; the quantising copy zero-fills past the row's end so
// every lane's group maximum is defined.
template <bool kQuant, typename VecT, int V>
__device__ __forceinline__ void load_item(const VecT* __restrict__ src, int64_t c0,
                                          int64_t row_vecs, VecT (&v)[V]) {
  if constexpr (kQuant) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int64_t c = c0 + i * 32 + lane;
      v[i] = c < row_vecs ? ld_stream(src + c) : make_uint4(0, 0, 0, 0);
    }
  } else {
    load_chunk<VecT, V>(src, c0, row_vecs, v);
  }
}

// Single-launch permute for small batches (at most kMetaChunkRows = 2048 expanded rows
// with J = 2 rows per lane, up to 4096 with J = 4; the dispatch takes it where
// it measured faster than the two-kernel path).  Every block
// computes the whole stable counting sort in shared memory (R is small, the
// ids come from L2), block 0 writes the metadata, and all blocks share the
// row copy: no block ever waits for another.
// Shared memory: cnt [n_rank_warps][E_local] | s_base [E_local + 1] | s_p [R].
// kQuant: quantise-on-permute (VecT = uint4 of 8 bf16 values): each row is
// written as fp8 e4m3 codes (permuted_hidden reinterpreted as uint2) plus one
// fp32 scale per 128 columns (permuted_scales), by the same arithmetic as
// k_gather_quant_fp8.
// kEarly: each warp loads the row chunk of its first copy item before the
// ranking, so that load overlaps the routing.  The launch takes it only for
// the quantising copy from kFusedEarlyMinTokens tokens: measured on GB300
// (DeepSeek-V3 shape) 5-10% faster at T = 32 to 128, equal at 256, 5% slower
// at T = 1; for the plain copy it was up to 14% slower at small T and never
// more than 3% faster.
template <typename IdT, typename VecT, int V, bool kQuant = false, bool kEarly = false,
          int J = kMetaRowsPerLane>
__global__ void __launch_bounds__(kMetaThreads, 1)
k_permute_fused(const IdT* __restrict__ ids, const int32_t* __restrict__ emap,
                int64_t T, int K, int E, int E_local,
                const VecT* __restrict__ hidden, int64_t row_vecs,
                const float* __restrict__ scales, int64_t scale_cols,
                VecT* __restrict__ permuted_hidden, float* __restrict__ permuted_scales,
                int64_t* __restrict__ offsets, int32_t* __restrict__ permuted_idx,
                int32_t* __restrict__ inv_permuted_idx, WsHeader* __restrict__ hdr) {
  extern __shared__ int smem[];
  __shared__ int s_warp[32];
  const int64_t R = T * K;
  // warps that own at least one row (each owns 32 * J rows)
  const int n_rank_warps = static_cast<int>((R + 32 * J - 1) / (32 * J));
  int* cnt = smem;
  int* s_base = cnt + n_rank_warps * E_local;
  int* s_p = s_base + E_local + 1;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool writer = blockIdx.x == 0;

  pdl_wait();
  VecT v0[V];  // kEarly: the row chunk of this warp's first copy item
  float sc0[kPreScaleChunks];
  if constexpr (kEarly) {
    const int64_t nc = (row_vecs + 32 * V - 1) / (32 * V);
    const int64_t first = blockIdx.x + static_cast<int64_t>(warp) * gridDim.x;
    if (permuted_hidden != nullptr && first < T * nc) {
      const int64_t t = first / nc;
      const int64_t c0 = (first - t * nc) * (32 * V);
      load_item<kQuant, VecT, V>(hidden + t * row_vecs, c0, row_vecs, v0);
      if (!kQuant && permuted_scales != nullptr && c0 == 0)
        load_token_scales(scales + t * scale_cols, scale_cols, sc0);
    }
  }
  for (int i = threadIdx.x; i < n_rank_warps * E_local; i += blockDim.x) cnt[i] = 0;
  __syncthreads();

  const int64_t slice0 = static_cast<int64_t>(warp) * 32 * J;
  int key[J], rank[J];
  if (warp < n_rank_warps) {
    unsigned flags = 0;
    load_keys<IdT, J>(ids, emap, E, E_local, slice0, R, key, flags);
    rank_warp_slice<J>(key, cnt + warp * E_local, rank);
    if (writer) {
      flags = __reduce_or_sync(kFullMask, flags);
      if (flags != 0 && lane == 0) atomicOr(&hdr->status, flags);
    }
  }
  __syncthreads();
  scan_counts_over_warps(cnt, E_local, n_rank_warps, s_base);
  __syncthreads();
  // Exclusive scan of the per-expert totals (E_local <= blockDim.x).
  {
    const int v = threadIdx.x < E_local ? s_base[threadIdx.x] : 0;
    int total;
    const int excl = block_exclusive_sum(v, s_warp, &total);
    if (threadIdx.x < E_local) s_base[threadIdx.x] = excl;
    if (threadIdx.x == 0) s_base[E_local] = total;
  }
  __syncthreads();
  if (writer)
    for (int e = threadIdx.x; e <= E_local; e += blockDim.x) offsets[e] = s_base[e];

  if (warp < n_rank_warps) {
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int64_t r = slice0 + j * 32 + lane;
      if (r < R) {
        const int e = key[j];
        const int p = e >= 0 ? s_base[e] + cnt[warp * E_local + e] + rank[j] : -1;
        s_p[r] = p;
        if (writer) {
          inv_permuted_idx[r] = p;
          if (p >= 0) permuted_idx[p] = static_cast<int32_t>(r);
        }
      }
    }
  }
  if (writer)
    for (int64_t p = s_base[E_local] + threadIdx.x; p < R; p += blockDim.x) permuted_idx[p] = -1;
  if (permuted_hidden == nullptr) return;
  __syncthreads();

  // Items go round-robin over the blocks first (item i -> block i % G), so a
  // small batch still spreads its copy over every block's SM.  A token's
  // scales are loaded with its first row chunk, before any store.
  constexpr int64_t kChunk = 32 * V;
  const int64_t n_chunks = (row_vecs + kChunk - 1) / kChunk;
  const int64_t n_items = T * n_chunks;
  const int64_t G = gridDim.x;
  const int64_t item0 = blockIdx.x + warp * G;
  for (int64_t item = item0; item < n_items; item += kMetaWarps * G) {
    const int64_t t = item / n_chunks;
    const int64_t c0 = (item - t * n_chunks) * kChunk;
    const int p = lane < K ? s_p[t * K + lane] : -1;
    const unsigned valid = __ballot_sync(kFullMask, p >= 0);
    if (valid == 0u) continue;
    const bool with_scales = !kQuant && permuted_scales != nullptr && c0 == 0;
    VecT v[V];
    float sc[kPreScaleChunks];
    if (kEarly && item == item0) {  // loaded before the ranking
#pragma unroll
      for (int i = 0; i < V; ++i) v[i] = v0[i];
#pragma unroll
      for (int i = 0; i < kPreScaleChunks; ++i) sc[i] = sc0[i];
    } else {
      load_item<kQuant, VecT, V>(hidden + t * row_vecs, c0, row_vecs, v);
      if (with_scales) load_token_scales(scales + t * scale_cols, scale_cols, sc);
    }
    if constexpr (kQuant) {
      // (quantising the early chunk before the ranking as well measured 6-8%
      // slower at T = 32-256: the ranking warps carry the quantiser's
      // registers and latency)
      uint2 codes[V];
      float qs[V];
      quant_chunk<V>(v, codes, qs);
      store_quant_chunk<V>(codes, qs, c0, row_vecs, p, valid,
                           reinterpret_cast<uint2*>(permuted_hidden), permuted_scales);
    } else {
      store_chunk<VecT, V>(v, permuted_hidden, c0, row_vecs, p, valid);
      if (with_scales)
        store_token_scales(scales + t * scale_cols, scale_cols, sc, permuted_scales, p, valid);
    }
  }
}

// bf16 lanes (raw bits) of a vector register.
template <typename VecT>
struct Bf16Vec {
  static constexpr int kElems = sizeof(VecT) / 2;
  union {
    VecT v;
    unsigned short e[kElems];
  };
};

// Unpermute: warp per (token, chunk).  k ascending, fp32 multiply then fp32
// add per term (no contraction), one bf16 round-to-nearest-even at the end.
// The loads of up to KG kept rows are in flight together; KG * V is kept near
// 8 vectors per lane whatever K is.  With V <= 2 the kernel fits 64 registers
// without spilling, so 4 blocks of 256 threads can share an SM (the launch
// decides whether to use the fourth).  V = 4 keeps 3 blocks (80 registers;
// without a bound the compiler spends 122 and only 2 fit), V = 8 needs 2.
template <typename VecT, int KG, int V>
__global__ void __launch_bounds__(kRowThreads, V <= 2 ? 4 : (V <= 4 ? 3 : 2))
k_unpermute(const VecT* __restrict__ rows, int64_t num_rows, int64_t row_vecs,
            const float* __restrict__ topk_weights, const int32_t* __restrict__ inv_permuted_idx,
            int64_t T, int K, VecT* __restrict__ out, unsigned* __restrict__ status) {
  constexpr int kE = Bf16Vec<VecT>::kElems;
  constexpr int kG = KG;
  constexpr int64_t kChunk = 32 * V;
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t n_chunks = (row_vecs + kChunk - 1) / kChunk;
  const int64_t n_items = T * n_chunks;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t item = warp0; item < n_items; item += n_warps) {
    const int64_t t = item / n_chunks;
    const int64_t c0 = (item - t * n_chunks) * kChunk;
    int p = -1;
    float w = 0.f;
    bool bad = false;
    if (lane < K) {
      p = __ldg(inv_permuted_idx + t * K + lane);
      w = __ldg(topk_weights + t * K + lane);
      if (p < -1 || p >= num_rows) {
        bad = true;
        p = -1;
      }
    }
    if (status != nullptr && c0 == 0 && __any_sync(kFullMask, bad) && lane == 0)
      atomicOr(status, MOE_FLAG_INV_OUT_OF_RANGE);
    float acc[V][kE];
#pragma unroll
    for (int i = 0; i < V; ++i)
#pragma unroll
      for (int e = 0; e < kE; ++e) acc[i][e] = 0.f;
    unsigned m = __ballot_sync(kFullMask, p >= 0);  // kept rows, k ascending
    while (m != 0u) {
      int ks[kG];
#pragma unroll
      for (int j = 0; j < kG; ++j) {
        ks[j] = m != 0u ? __ffs(m) - 1 : -1;
        m &= m - 1u;  // no-op once m is 0
      }
      Bf16Vec<VecT> x[kG][V];
#pragma unroll
      for (int j = 0; j < kG; ++j) {
        if (ks[j] < 0) continue;
        const int pk = __shfl_sync(kFullMask, p, ks[j]);
        const VecT* src = rows + static_cast<int64_t>(pk) * row_vecs;
#pragma unroll
        for (int i = 0; i < V; ++i) {
          const int64_t c = c0 + i * 32 + lane;
          if (c < row_vecs) x[j][i].v = ld_stream(src + c);
        }
      }
#pragma unroll
      for (int j = 0; j < kG; ++j) {
        if (ks[j] < 0) continue;
        const float wk = __shfl_sync(kFullMask, w, ks[j]);
#pragma unroll
        for (int i = 0; i < V; ++i)
#pragma unroll
          for (int e = 0; e < kE; ++e)
            acc[i][e] = __fadd_rn(
                acc[i][e], __fmul_rn(wk, __bfloat162float(__ushort_as_bfloat16(x[j][i].e[e]))));
      }
    }
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int64_t c = c0 + i * 32 + lane;
      if (c < row_vecs) {
        Bf16Vec<VecT> y;
#pragma unroll
        for (int e = 0; e < kE; ++e) y.e[e] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[i][e]));
        out[t * row_vecs + c] = y.v;
      }
    }
  }
}

// T = 0: offsets all zero.
__global__ void k_zero_offsets(int64_t* __restrict__ offsets, int n) {
  pdl_wait();
  for (int i = threadIdx.x; i < n; i += blockDim.x) offsets[i] = 0;
}

}  // namespace moe
