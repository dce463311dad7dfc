// permute_coop.cuh -- moe_permute as one persistent, cooperatively launched
// kernel: routing metadata and row gather in a single grid.
//
// vLLM PR #14568 ("permute/unpermute kernel for moe optimization",
// description): expand each token to its K rows, order the rows by expert,
// gather the rows for the grouped GEMM.  Order inside an expert is stable by
// expanded row id r = t*K + k.
//
// Block b owns the contiguous tokens [b*tpb, (b+1)*tpb) and so the contiguous
// rows [b*tpb*K, (b+1)*tpb*K).  Phases:
//   1. histogram of the block's rows -> table[b][e] (workspace);
//   2. one grid barrier (every block is resident: cooperative launch);
//   3. every block reads the whole [B][E_local] table: offsets (block 0
//      writes them) and its bases base[e] = offset[e] + sum_{b'<b} table[b'][e];
//   4. stable ranks of the block's rows in rounds of kCoopRoundRows (warp w
//      owns a contiguous slice of each round) -> permuted_idx, inv_permuted_idx;
//   5. the block copies its own tokens' rows: their positions were written by
//      this block in phase 4, so no further synchronisation is needed.
// The barrier spin is bounded: on timeout the status word gets
// MOE_FLAG_BARRIER_TIMEOUT and the kernel returns (outputs undefined).
#pragma once

#include "common.cuh"
#include "routing.cuh"
#include "rows.cuh"

namespace moe {

constexpr int kCoopThreads = 1024;
constexpr int kCoopWarps = kCoopThreads / kWarpSize;
constexpr int kCoopRowsPerLane = 4;
constexpr int kCoopRoundRows = kCoopThreads * kCoopRowsPerLane;  // 4096
constexpr unsigned kBarrierSpinLimit = 1u << 26;  // ~ seconds with the back-off below

// Grid-wide barrier for a cooperatively launched grid.  hdr->arrive counts
// arrivals (the last one resets it), hdr->gen is bumped once per barrier.
// Returns false (and flags the status word) if the wait gave up.
__device__ __forceinline__ bool grid_barrier(WsHeader* hdr) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const unsigned gen = *reinterpret_cast<volatile unsigned*>(&hdr->gen);
    __threadfence();
    const unsigned arrived = atomicAdd(&hdr->arrive, 1u);
    if (arrived == gridDim.x - 1) {
      hdr->arrive = 0u;
      __threadfence();
      atomicAdd(&hdr->gen, 1u);
    } else {
      unsigned spins = 0;
      while (true) {
        unsigned now;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(now) : "l"(&hdr->gen) : "memory");
        if (now != gen) break;
        if (++spins == kBarrierSpinLimit) {
          atomicOr(&hdr->status, MOE_FLAG_BARRIER_TIMEOUT);
          ok = 0;
          break;
        }
        __nanosleep(32);
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// Shared memory: s_base [E_local + 1] | s_run [E_local] | cnt [kCoopWarps][E_local]
template <typename IdT, typename VecT, int V>
__global__ void __launch_bounds__(kCoopThreads, 1)
k_permute_coop(const IdT* __restrict__ ids, const int32_t* __restrict__ emap,
               int64_t T, int K, int E, int E_local,
               const VecT* __restrict__ hidden, int64_t row_vecs,
               const float* __restrict__ scales, int64_t scale_cols,
               VecT* __restrict__ permuted_hidden, float* __restrict__ permuted_scales,
               int64_t* __restrict__ offsets, int32_t* __restrict__ permuted_idx,
               int32_t* __restrict__ inv_permuted_idx, WsHeader* __restrict__ hdr,
               int* __restrict__ table) {
  extern __shared__ int smem[];
  __shared__ int s_warp[32];
  int* s_base = smem;                   // [E_local + 1]
  int* s_run = s_base + E_local + 1;    // [E_local]
  int* cnt = s_run + E_local;           // [kCoopWarps][E_local]
  const int B = gridDim.x;
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t R = T * K;
  const int64_t tpb = (T + B - 1) / B;
  const int64_t t0 = min(T, static_cast<int64_t>(b) * tpb);
  const int64_t t1 = min(T, t0 + tpb);
  const int64_t r0 = t0 * K, r1 = t1 * K;

  pdl_wait();
  // The first chunk of each warp's first gather item does not depend on the
  // routing: start loading it now so HBM is busy during phases 1-4.
  constexpr int64_t kChunk = 32 * V;
  const int64_t n_chunks = (row_vecs + kChunk - 1) / kChunk;
  const int64_t n_items = permuted_hidden != nullptr ? (t1 - t0) * n_chunks : 0;
  VecT v[V];
  if (warp < n_items) {
    const int64_t t = t0 + warp / n_chunks;
    load_chunk<VecT, V>(hidden + t * row_vecs, (warp % n_chunks) * kChunk, row_vecs, v);
  }
  // Phase 1: histogram of rows [r0, r1) (warp-aggregated shared atomics).
  for (int e = threadIdx.x; e < E_local; e += blockDim.x) s_run[e] = 0;
  __syncthreads();
  unsigned flags = 0;
  for (int64_t g0 = r0 + warp * 32; g0 < r1; g0 += kCoopThreads) {
    const int64_t r = g0 + lane;
    const int e = r < r1 ? local_expert(__ldg(ids + r), emap, E, E_local, flags) : -1;
    const unsigned peers = __match_any_sync(kFullMask, e);
    if (e >= 0 && (peers & lanemask_lt()) == 0) atomicAdd(&s_run[e], __popc(peers));
  }
  flags = __reduce_or_sync(kFullMask, flags);
  if (flags != 0 && lane == 0) atomicOr(&hdr->status, flags);
  __syncthreads();
  const int e_pad = (E_local + 3) & ~3;  // table rows padded to whole int4s
  for (int e = threadIdx.x; e < e_pad; e += blockDim.x)
    table[static_cast<int64_t>(b) * e_pad + e] = e < E_local ? s_run[e] : 0;

  // Phase 2: every block's histogram is in the table after this.
  if (!grid_barrier(hdr)) return;

  // Phase 3: totals, offsets and this block's bases from the whole table.
  // Thread i reads 4 experts (quad i % n_quads) of the table rows
  // bb = i / n_quads, i / n_quads + n_groups, ... with 16-byte loads.
  for (int e = threadIdx.x; e < E_local; e += blockDim.x) {
    s_base[e] = 0;
    s_run[e] = 0;
  }
  __syncthreads();
  {
    const int n_quads = e_pad / 4;
    const int n_groups = max(1, static_cast<int>(blockDim.x) / n_quads);
    for (int i = threadIdx.x; i < n_quads * n_groups; i += blockDim.x) {
      const int q = i % n_quads;
      const int g = i / n_quads;
      int4 tot = make_int4(0, 0, 0, 0), bef = make_int4(0, 0, 0, 0);
#pragma unroll 4
      for (int bb = g; bb < B; bb += n_groups) {
        const int4 c = __ldcg(reinterpret_cast<const int4*>(table + static_cast<int64_t>(bb) * e_pad) + q);
        tot.x += c.x; tot.y += c.y; tot.z += c.z; tot.w += c.w;
        if (bb < b) { bef.x += c.x; bef.y += c.y; bef.z += c.z; bef.w += c.w; }
      }
      const int e0 = q * 4;
      const int tv[4] = {tot.x, tot.y, tot.z, tot.w};
      const int bv[4] = {bef.x, bef.y, bef.z, bef.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (e0 + u < E_local) {
          atomicAdd(&s_base[e0 + u], tv[u]);
          atomicAdd(&s_run[e0 + u], bv[u]);
        }
      }
    }
  }
  __syncthreads();
  {
    const int v = threadIdx.x < E_local ? s_base[threadIdx.x] : 0;
    int n_valid;
    const int excl = block_exclusive_sum(v, s_warp, &n_valid);
    if (threadIdx.x < E_local) s_base[threadIdx.x] = excl + s_run[threadIdx.x];
    if (b == 0 && threadIdx.x < E_local) offsets[threadIdx.x] = excl;
    if (threadIdx.x == 0) {
      s_base[E_local] = n_valid;
      if (b == 0) offsets[E_local] = n_valid;
    }
  }
  __syncthreads();
  // Tail of permuted_idx: positions [N_valid, R) hold -1 (spread over blocks).
  for (int64_t p = s_base[E_local] + static_cast<int64_t>(b) * blockDim.x + threadIdx.x; p < R;
       p += static_cast<int64_t>(B) * blockDim.x)
    permuted_idx[p] = -1;

  // Phase 4: stable ranks in rounds; s_run[e] = this block's rows of expert e
  // placed so far.
  for (int e = threadIdx.x; e < E_local; e += blockDim.x) s_run[e] = 0;
  for (int64_t q0 = r0; q0 < r1; q0 += kCoopRoundRows) {
    const int64_t q1 = min(r1, q0 + kCoopRoundRows);
    const int n_rank_warps =
        static_cast<int>((q1 - q0 + 32 * kCoopRowsPerLane - 1) / (32 * kCoopRowsPerLane));
    for (int i = threadIdx.x; i < n_rank_warps * E_local; i += blockDim.x) cnt[i] = 0;
    __syncthreads();
    const int64_t slice0 = q0 + static_cast<int64_t>(warp) * 32 * kCoopRowsPerLane;
    int key[kCoopRowsPerLane], rank[kCoopRowsPerLane];
    if (warp < n_rank_warps) {
      unsigned f = 0;  // already reported in phase 1
      load_keys<IdT, kCoopRowsPerLane>(ids, emap, E, E_local, slice0, q1, key, f);
      rank_warp_slice<kCoopRowsPerLane>(key, cnt + warp * E_local, rank);
    }
    __syncthreads();
    // exclusive prefix over warps, then the round's totals go into s_run
    for (int e = threadIdx.x; e < E_local; e += blockDim.x) {
      int run = s_run[e];
      for (int w = 0; w < n_rank_warps; ++w) {
        const int c = cnt[w * E_local + e];
        cnt[w * E_local + e] = run;
        run += c;
      }
      s_run[e] = run;
    }
    __syncthreads();
    if (warp < n_rank_warps) {
#pragma unroll
      for (int j = 0; j < kCoopRowsPerLane; ++j) {
        const int64_t r = slice0 + j * 32 + lane;
        if (r < q1) {
          const int e = key[j];
          int p = -1;
          if (e >= 0) {
            p = s_base[e] + cnt[warp * E_local + e] + rank[j];
            permuted_idx[p] = static_cast<int32_t>(r);
          }
          inv_permuted_idx[r] = p;
        }
      }
    }
    __syncthreads();
  }
  // Phase 5: gather this block's tokens (their inv entries were written above
  // by this block; bar.sync orders them for every thread of the block).
  for (int64_t item = warp; item < n_items; item += kCoopWarps) {
    const int64_t t = t0 + item / n_chunks;
    const int64_t c0 = (item % n_chunks) * kChunk;
    const int p = lane < K ? inv_permuted_idx[t * K + lane] : -1;
    const unsigned valid = __ballot_sync(kFullMask, p >= 0);
    if (valid == 0u) continue;
    if (item != warp) load_chunk<VecT, V>(hidden + t * row_vecs, c0, row_vecs, v);
    store_chunk<VecT, V>(v, permuted_hidden, c0, row_vecs, p, valid);
    if (permuted_scales != nullptr && c0 == 0)
      copy_token_scales(scales + t * scale_cols, scale_cols, permuted_scales, p, valid);
  }
}

}  // namespace moe
