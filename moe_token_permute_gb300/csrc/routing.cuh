// routing.cuh -- device helpers of the stable counting sort behind moe_permute.
//
// vLLM PR #14568 ("permute/unpermute kernel for moe optimization",
// description): permute orders the expanded rows r = t*K + k by expert so each
// expert's rows are contiguous for the grouped GEMM.  The prior art sorts with
// a generic radix sort and a sort workspace (vLLM PR #43014 digest,
// "implementation breakdown" item 3).  Here the key range is only the number
// of local experts, so the sort is a counting sort: a per-expert histogram,
// an exclusive scan of the counts, and a stable scatter whose ranks come from
// match_any peer groups inside a warp plus per-warp counts scanned across the
// warps of a block.  Warp w of a block owns a contiguous slice of 32*J rows,
// so ranks computed warp by warp in row order are stable.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kMetaThreads = 1024;
constexpr int kMetaWarps = kMetaThreads / kWarpSize;
// Rows per lane the single-launch kernel ranks (J).  2 puts up to 32 warps on
// the ranking of at most 2048 rows; with 8, only R / 256 warps ranked while the
// rest waited at the block barriers (measured on GB300: 7-18% faster per call
// from T = 1 up to R = 1024, equal at R = 2048).
constexpr int kMetaRowsPerLane = 2;  // J
constexpr int kMetaChunkRows = kMetaThreads * kMetaRowsPerLane;  // rows one block ranks: 2048
// J = 4 lets one block rank up to 4096 rows: the single-launch permute serves
// batches a little above 2048 rows with it (the dispatch says which).
constexpr int kMetaRowsPerLaneWide = 4;
constexpr int kMetaChunkRowsWide = kMetaThreads * kMetaRowsPerLaneWide;  // 4096

// Local expert of one global id, or -1 when the row is dropped.
template <typename IdT>
__device__ __forceinline__ int local_expert(IdT raw, const int32_t* __restrict__ emap,
                                            int E, int E_local, unsigned& flags) {
  const int64_t g = static_cast<int64_t>(raw);
  if (g < 0 || g >= E) {
    flags |= MOE_FLAG_ID_OUT_OF_RANGE;
    return -1;
  }
  if (emap == nullptr) return static_cast<int>(g);
  const int e = emap[g];  // global memory (read-only path) or a shared-memory copy
  if (e == -1) return -1;
  if (e < 0 || e >= E_local) {
    flags |= MOE_FLAG_MAP_OUT_OF_RANGE;
    return -1;
  }
  return e;
}

// Keys of this lane's J rows of the warp slice starting at slice0.
template <typename IdT, int J>
__device__ __forceinline__ void load_keys(const IdT* __restrict__ ids,
                                          const int32_t* __restrict__ emap, int E,
                                          int E_local, int64_t slice0, int64_t row_end,
                                          int (&key)[J], unsigned& flags) {
  const int lane = threadIdx.x & 31;
  IdT raw[J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int64_t r = slice0 + j * 32 + lane;
    raw[j] = r < row_end ? __ldg(ids + r) : IdT(-1);
  }
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int64_t r = slice0 + j * 32 + lane;
    key[j] = r < row_end ? local_expert(raw[j], emap, E, E_local, flags) : -1;
  }
}

// Stable ranks inside one warp slice.  cnt_w: this warp's [E_local] counters
// in shared memory, zero on entry; on exit cnt_w[e] = rows of the slice with
// key e.  rank[j] = number of earlier rows of the slice with the same key.
template <int J>
__device__ __forceinline__ void rank_warp_slice(const int (&key)[J], int* cnt_w,
                                                int (&rank)[J]) {
  const unsigned lt = lanemask_lt();
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int e = key[j];
    const unsigned peers = __match_any_sync(kFullMask, e);
    int prev = 0;
    if (e >= 0) prev = cnt_w[e];
    __syncwarp();
    if (e >= 0 && (peers & lt) == 0) cnt_w[e] = prev + __popc(peers);
    __syncwarp();
    rank[j] = prev + __popc(peers & lt);
  }
}

// Turn cnt[w][e] (w < n_warps) into exclusive prefixes over w, in place;
// s_total[e] receives the block's count of expert e.
__device__ __forceinline__ void scan_counts_over_warps(int* cnt, int E_local, int n_warps,
                                                       int* s_total) {
  for (int e = threadIdx.x; e < E_local; e += blockDim.x) {
    int run = 0;
#pragma unroll 8
    for (int w = 0; w < n_warps; ++w) {
      const int c = cnt[w * E_local + e];
      cnt[w * E_local + e] = run;
      run += c;
    }
    s_total[e] = run;
  }
}

}  // namespace moe
