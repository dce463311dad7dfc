// routing.cuh -- routing metadata of moe_permute as a stable counting sort.
//
// vLLM PR #14568 ("permute/unpermute kernel for moe optimization",
// description): permute orders the expanded rows r = t*K + k by expert so each
// expert's rows are contiguous for the grouped GEMM.  The prior art sorts with
// a generic radix sort and a sort workspace (vLLM PR #43014 digest,
// "implementation breakdown" item 3).  Here the key range is only the number
// of local experts, so the sort is a counting sort:
//   k_route_hist     per-block expert histogram (warp-aggregated shared
//                    atomics); the last block to finish scans all histograms
//                    into per-(expert, block) bases and writes
//                    expert_first_token_offset.
//   k_route_scatter  per-block stable ranks (match_any peer groups inside a
//                    warp, per-warp counts scanned across warps), then
//                    p = base[e][b] + rank; writes permuted_idx / inv_permuted_idx.
// Chunks: block b owns rows [b*C, (b+1)*C), C = kMetaWarps * 32 * kMetaRowsPerLane;
// warp w of a block owns the contiguous rows [w*32*J, (w+1)*32*J) of the chunk,
// so ranks computed warp by warp in row order are stable.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kMetaThreads = 1024;
constexpr int kMetaWarps = kMetaThreads / kWarpSize;
constexpr int kMetaRowsPerLane = 8;  // J
constexpr int kMetaChunkRows = kMetaThreads * kMetaRowsPerLane;  // C = 8192

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
  const int e = __ldg(emap + g);
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

// Kernel 1: per-block histogram; the last block scans every histogram.
// hist: [E_local][B] ints in the workspace; on exit (last block) it holds the
// exclusive prefix over (e-major, b-minor) order, i.e. the first output
// position of expert e's rows from block b.
template <typename IdT>
__global__ void __launch_bounds__(kMetaThreads)
k_route_hist(const IdT* __restrict__ ids, const int32_t* __restrict__ emap,
             int64_t R, int E, int E_local, int* __restrict__ hist,
             int64_t* __restrict__ offsets, WsHeader* __restrict__ hdr) {
  extern __shared__ int s_hist[];  // [E_local]
  __shared__ int s_warp[32];
  __shared__ int s_is_last;
  pdl_wait();
  pdl_launch_dependents();

  const int B = gridDim.x;
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E_local; e += blockDim.x) s_hist[e] = 0;
  __syncthreads();

  const int64_t chunk0 = static_cast<int64_t>(b) * kMetaChunkRows;
  const int64_t row_end = min(R, chunk0 + kMetaChunkRows);
  const int64_t slice0 = chunk0 + static_cast<int64_t>(threadIdx.x >> 5) * 32 * kMetaRowsPerLane;
  int key[kMetaRowsPerLane];
  unsigned flags = 0;
  load_keys<IdT, kMetaRowsPerLane>(ids, emap, E, E_local, slice0, row_end, key, flags);
#pragma unroll
  for (int j = 0; j < kMetaRowsPerLane; ++j) {
    const int e = key[j];
    const unsigned peers = __match_any_sync(kFullMask, e);
    if (e >= 0 && (peers & lanemask_lt()) == 0) atomicAdd(&s_hist[e], __popc(peers));
  }
  flags = __reduce_or_sync(kFullMask, flags);
  if (flags != 0 && lane == 0) atomicOr(&hdr->status, flags);
  __syncthreads();
  for (int e = threadIdx.x; e < E_local; e += blockDim.x)
    hist[static_cast<int64_t>(e) * B + b] = s_hist[e];

  // Last block to finish does the scan (no block ever waits for another).
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_is_last = atomicAdd(&hdr->ticket, 1u) == static_cast<unsigned>(B - 1);
  __syncthreads();
  if (!s_is_last) return;
  __threadfence();

  const int64_t n = static_cast<int64_t>(E_local) * B;
  const int64_t seg = (n + blockDim.x - 1) / blockDim.x;
  const int64_t i0 = min(n, static_cast<int64_t>(threadIdx.x) * seg);
  const int64_t i1 = min(n, i0 + seg);
  int sum = 0;
#pragma unroll 8
  for (int64_t i = i0; i < i1; ++i) sum += __ldcg(hist + i);
  int total;
  int run = block_exclusive_sum(sum, s_warp, &total);
  for (int64_t i = i0; i < i1; ++i) {
    const int c = __ldcg(hist + i);
    hist[i] = run;
    if (i % B == 0) offsets[i / B] = run;
    run += c;
  }
  if (threadIdx.x == 0) {
    offsets[E_local] = total;
    hdr->ticket = 0u;  // ready for the next call on this workspace
  }
}

// Kernel 2: stable scatter of the indices.  Ranks are computed before waiting
// on kernel 1 (they depend only on the caller's ids), then combined with the
// bases kernel 1 produced.
template <typename IdT>
__global__ void __launch_bounds__(kMetaThreads)
k_route_scatter(const IdT* __restrict__ ids, const int32_t* __restrict__ emap,
                int64_t R, int E, int E_local, const int* __restrict__ base,
                const int64_t* __restrict__ offsets, int32_t* __restrict__ permuted_idx,
                int32_t* __restrict__ inv_permuted_idx) {
  extern __shared__ int smem[];  // cnt [kMetaWarps][E_local], s_base [E_local]
  int* cnt = smem;
  int* s_base = smem + kMetaWarps * E_local;
  const int B = gridDim.x;
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kMetaWarps * E_local; i += blockDim.x) cnt[i] = 0;
  __syncthreads();

  const int64_t chunk0 = static_cast<int64_t>(b) * kMetaChunkRows;
  const int64_t row_end = min(R, chunk0 + kMetaChunkRows);
  const int64_t slice0 = chunk0 + static_cast<int64_t>(warp) * 32 * kMetaRowsPerLane;
  int key[kMetaRowsPerLane], rank[kMetaRowsPerLane];
  unsigned flags = 0;  // already reported by kernel 1
  load_keys<IdT, kMetaRowsPerLane>(ids, emap, E, E_local, slice0, row_end, key, flags);
  rank_warp_slice<kMetaRowsPerLane>(key, cnt + warp * E_local, rank);
  __syncthreads();
  scan_counts_over_warps(cnt, E_local, kMetaWarps, s_base);  // s_base: scratch for totals

  pdl_wait();  // kernel 1's bases and offsets are visible from here on
  pdl_launch_dependents();
  __syncthreads();
  for (int e = threadIdx.x; e < E_local; e += blockDim.x)
    s_base[e] = __ldcg(base + static_cast<int64_t>(e) * B + b);
  __syncthreads();

#pragma unroll
  for (int j = 0; j < kMetaRowsPerLane; ++j) {
    const int64_t r = slice0 + j * 32 + lane;
    if (r < row_end) {
      const int e = key[j];
      int p = -1;
      if (e >= 0) {
        p = s_base[e] + cnt[warp * E_local + e] + rank[j];
        permuted_idx[p] = static_cast<int32_t>(r);
      }
      inv_permuted_idx[r] = p;
    }
  }
  // Tail of permuted_idx: positions [N_valid, R) hold -1.
  const int64_t n_valid = __ldcg(offsets + E_local);
  for (int64_t p = n_valid + static_cast<int64_t>(b) * blockDim.x + threadIdx.x; p < R;
       p += static_cast<int64_t>(B) * blockDim.x)
    permuted_idx[p] = -1;
}

}  // namespace moe
