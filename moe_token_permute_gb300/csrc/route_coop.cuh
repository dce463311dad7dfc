// route_coop.cuh -- routing metadata of moe_permute for large batches: one
// cooperatively launched grid with a single grid barrier.
//
// vLLM PR #14568 ("permute/unpermute kernel for moe optimization",
// description): expand each token to its K rows and order the rows by expert
// for the grouped GEMM.  Order inside an expert is stable by expanded row id
// r = t*K + k.
//
// Block b owns the contiguous tokens [b*tpb, (b+1)*tpb), i.e. the contiguous
// rows [r0, r1).  Phases:
//   1. histogram of the block's rows -> table[b][e] (workspace).  When the
//      block's rows fit one round (kRouteRoundRows), the stable in-block ranks
//      are computed in the same pass and kept in registers;
//   2. one grid barrier (every block is resident: cooperative launch);
//   3. every block reads the whole [B][E_local] table with 16-byte loads:
//      offsets (block 0 writes them) and its bases
//      base[e] = offset[e] + sum_{b'<b} table[b'][e];
//   4. positions p = base[e] + (rows of expert e before r in the block) ->
//      permuted_idx, inv_permuted_idx (in rounds when the block has more rows).
// The kernel lets the row-gather kernel that follows launch as soon as it
// starts: those blocks load their source rows while routing runs and wait for
// this grid before they read inv_permuted_idx.
// The barrier wait is bounded (2^24 polls or 2 s): on timeout the status word
// gets MOE_FLAG_BARRIER_TIMEOUT and the kernel returns (outputs undefined; the
// gather that follows never stores through an out-of-range position).
#pragma once

#include "common.cuh"
#include "routing.cuh"

namespace moe {

constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / kWarpSize;
constexpr int kRouteRowsPerLane = 4;
constexpr int kRouteRoundRows = kRouteThreads * kRouteRowsPerLane;  // 1024
constexpr unsigned kBarrierSpinLimit = 1u << 24;                  // polls before giving up
constexpr unsigned long long kBarrierTimeLimitNs = 2000000000ull;  // or 2 s, whichever first

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Grid-wide barrier for a cooperatively launched grid.  hdr->arrive counts
// arrivals (the last one resets it); hdr->gen is bumped once per barrier.
// `gen` is the generation thread 0 read at kernel start: it cannot move before
// every block of this grid has arrived.  Ordering: bar.sync gathers the
// block's writes into thread 0, whose arrival is an acquire-release atomic;
// the last block publishes with a release add on gen; waiters read gen with
// acquire loads.  Returns false (and flags the status word) if the wait gave
// up.
__device__ __forceinline__ bool grid_barrier(WsHeader* hdr, unsigned gen) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    unsigned arrived;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
                 : "=r"(arrived) : "l"(&hdr->arrive) : "memory");
    if (arrived == gridDim.x - 1) {
      asm volatile("st.relaxed.gpu.global.u32 [%0], 0;" :: "l"(&hdr->arrive) : "memory");
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(&hdr->gen) : "memory");
    } else {
      unsigned spins = 0;
      const unsigned long long t_start = global_ns();
      while (true) {
        unsigned now;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(now) : "l"(&hdr->gen) : "memory");
        if (now != gen) break;
        if (++spins == kBarrierSpinLimit ||
            ((spins & 1023u) == 0u && global_ns() - t_start > kBarrierTimeLimitNs)) {
          atomicOr(&hdr->status, MOE_FLAG_BARRIER_TIMEOUT);
          ok = 0;
          break;
        }
        if (spins > 4096u) __nanosleep(64);
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// Final position of a kept row whose contiguous position is p.  Contiguous
// layout: p itself (and permuted_idx[p] = r).  Batched layout: slot
// e*M + (p - first[e]), or -1 when the expert's capacity M is exceeded.
__device__ __forceinline__ int place_row(int p, int e, int64_t r, int64_t M, const int* first,
                                         int32_t* __restrict__ permuted_idx,
                                         WsHeader* __restrict__ hdr) {
  if (M == 0) {
    permuted_idx[p] = static_cast<int32_t>(r);
    return p;
  }
  const int64_t j = p - first[e];
  if (j >= M) {
    atomicOr(&hdr->status, MOE_FLAG_CAPACITY_OVERFLOW);
    return -1;
  }
  return static_cast<int>(static_cast<int64_t>(e) * M + j);
}

// Shared memory: s_base [E_local + 1] | s_run [E_local] | s_tot [E_local] |
//                s_bef [E_local] | cnt [kRouteWarps][E_local]
// Batched layout (M > 0): instead of the contiguous segments, rows of local
// expert e go to slots e*M + j, j = the row's stable rank inside the expert;
// rows with j >= M are dropped (MOE_FLAG_CAPACITY_OVERFLOW).  Block 0 writes
// expert_num_tokens[e] = min(rows of e, M); offsets and permuted_idx are not
// used.
template <typename IdT>
__global__ void __launch_bounds__(kRouteThreads, 4)
k_route_coop(const IdT* __restrict__ ids, const int32_t* __restrict__ emap,
             int64_t T, int K, int E, int E_local,
             int64_t* __restrict__ offsets, int32_t* __restrict__ permuted_idx,
             int32_t* __restrict__ inv_permuted_idx, WsHeader* __restrict__ hdr,
             int* __restrict__ table, int64_t M, int32_t* __restrict__ expert_num_tokens) {
  extern __shared__ int smem[];
  __shared__ int s_warp[32];
  int* s_base = smem;                 // [E_local + 1]
  int* s_run = s_base + E_local + 1;  // [E_local]
  int* s_tot = s_run + E_local;       // [E_local] all blocks' rows per expert
  int* s_bef = s_tot + E_local;       // [E_local] rows per expert in blocks before b
  int* cnt = s_bef + E_local;         // [kRouteWarps][E_local]
  __shared__ unsigned s_gen;
  const int B = gridDim.x;
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t R = T * K;
  const int64_t tpb = (T + B - 1) / B;
  const int64_t t0 = min(T, static_cast<int64_t>(b) * tpb);
  const int64_t t1 = min(T, t0 + tpb);
  const int64_t r0 = t0 * K, r1 = t1 * K;
  const bool one_round = r1 - r0 <= kRouteRoundRows;
  constexpr int J = kRouteRowsPerLane;

  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    unsigned g;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(g) : "l"(&hdr->gen) : "memory");
    s_gen = g;
  }
  for (int e = threadIdx.x; e < E_local; e += blockDim.x) {
    s_tot[e] = 0;
    s_bef[e] = 0;
  }

  // Phase 1: histogram (and, for one round, the ranks).
  int key[J], rank[J];
  const int64_t slice0 = r0 + static_cast<int64_t>(warp) * 32 * J;
  unsigned flags = 0;
  if (one_round) {
    for (int i = threadIdx.x; i < kRouteWarps * E_local; i += blockDim.x) cnt[i] = 0;
    __syncthreads();
    load_keys<IdT, J>(ids, emap, E, E_local, slice0, r1, key, flags);
    rank_warp_slice<J>(key, cnt + warp * E_local, rank);
    __syncthreads();
    scan_counts_over_warps(cnt, E_local, kRouteWarps, s_run);  // s_run = block totals
  } else {
    for (int e = threadIdx.x; e < E_local; e += blockDim.x) s_run[e] = 0;
    __syncthreads();
    for (int64_t g0 = r0 + warp * 32; g0 < r1; g0 += kRouteThreads) {
      const int64_t r = g0 + lane;
      const int e = r < r1 ? local_expert(__ldg(ids + r), emap, E, E_local, flags) : -1;
      const unsigned peers = __match_any_sync(kFullMask, e);
      if (e >= 0 && (peers & lanemask_lt()) == 0) atomicAdd(&s_run[e], __popc(peers));
    }
  }
  flags = __reduce_or_sync(kFullMask, flags);
  if (flags != 0 && lane == 0) atomicOr(&hdr->status, flags);
  __syncthreads();
  const int e_pad = (E_local + 3) & ~3;  // table rows padded to whole int4s
  for (int e = threadIdx.x; e < e_pad; e += blockDim.x)
    table[static_cast<int64_t>(b) * e_pad + e] = e < E_local ? s_run[e] : 0;

  // Phase 2: every block's histogram is in the table after this.
  if (!grid_barrier(hdr, s_gen)) return;

  // Phase 3: totals, offsets and this block's bases from the whole table.
  // Thread i reads 4 experts (quad i % n_quads) of the table rows
  // bb = i / n_quads, i / n_quads + n_groups, ... with 16-byte loads.
  {
    const int n_quads = e_pad / 4;
    const int n_groups = max(1, static_cast<int>(blockDim.x) / n_quads);
    for (int i = threadIdx.x; i < n_quads * n_groups; i += blockDim.x) {
      const int q = i % n_quads;
      const int g = i / n_quads;
      int4 tot = make_int4(0, 0, 0, 0), bef = make_int4(0, 0, 0, 0);
#pragma unroll 8
      for (int bb = g; bb < B; bb += n_groups) {
        const int4 c =
            __ldcg(reinterpret_cast<const int4*>(table + static_cast<int64_t>(bb) * e_pad) + q);
        tot.x += c.x; tot.y += c.y; tot.z += c.z; tot.w += c.w;
        if (bb < b) { bef.x += c.x; bef.y += c.y; bef.z += c.z; bef.w += c.w; }
      }
      const int e0 = q * 4;
      const int tv[4] = {tot.x, tot.y, tot.z, tot.w};
      const int bv[4] = {bef.x, bef.y, bef.z, bef.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (e0 + u < E_local) {
          atomicAdd(&s_tot[e0 + u], tv[u]);
          atomicAdd(&s_bef[e0 + u], bv[u]);
        }
      }
    }
  }
  __syncthreads();
  // Exclusive scan of the totals; E_local <= MOE_MAX_LOCAL_EXPERTS, i.e. at
  // most kPer consecutive experts per thread.
  {
    constexpr int kPer = MOE_MAX_LOCAL_EXPERTS / kRouteThreads;
    int tot[kPer], sum = 0;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = threadIdx.x * kPer + u;
      tot[u] = e < E_local ? s_tot[e] : 0;
      sum += tot[u];
    }
    int n_valid;
    int run = block_exclusive_sum(sum, s_warp, &n_valid);
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = threadIdx.x * kPer + u;
      if (e < E_local) {
        s_base[e] = run + s_bef[e];
        s_tot[e] = run;  // from here on: the expert's first contiguous position
        if (b == 0) {
          if (M > 0)
            expert_num_tokens[e] = static_cast<int32_t>(min(static_cast<int64_t>(tot[u]), M));
          else
            offsets[e] = run;
        }
      }
      run += tot[u];
    }
    if (threadIdx.x == 0) {
      s_base[E_local] = n_valid;
      if (b == 0 && M == 0) offsets[E_local] = n_valid;
    }
  }
  __syncthreads();
  // Tail of permuted_idx: positions [N_valid, R) hold -1 (spread over blocks).
  if (M == 0)
    for (int64_t p = s_base[E_local] + static_cast<int64_t>(b) * blockDim.x + threadIdx.x;
         p < R; p += static_cast<int64_t>(B) * blockDim.x)
      permuted_idx[p] = -1;

  // Phase 4: positions.
  if (one_round) {
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int64_t r = slice0 + j * 32 + lane;
      if (r < r1) {
        const int e = key[j];
        int p = -1;
        if (e >= 0) {
          p = s_base[e] + cnt[warp * E_local + e] + rank[j];
          p = place_row(p, e, r, M, s_tot, permuted_idx, hdr);
        }
        inv_permuted_idx[r] = p;
      }
    }
    return;
  }
  // More rows than one round: rank round by round; s_run[e] = this block's
  // rows of expert e placed so far.
  for (int e = threadIdx.x; e < E_local; e += blockDim.x) s_run[e] = 0;
  for (int64_t q0 = r0; q0 < r1; q0 += kRouteRoundRows) {
    const int64_t q1 = min(r1, q0 + kRouteRoundRows);
    for (int i = threadIdx.x; i < kRouteWarps * E_local; i += blockDim.x) cnt[i] = 0;
    __syncthreads();
    const int64_t s0 = q0 + static_cast<int64_t>(warp) * 32 * J;
    unsigned f = 0;  // already reported in phase 1
    load_keys<IdT, J>(ids, emap, E, E_local, s0, q1, key, f);
    rank_warp_slice<J>(key, cnt + warp * E_local, rank);
    __syncthreads();
    for (int e = threadIdx.x; e < E_local; e += blockDim.x) {
      int run = s_run[e];
      for (int w = 0; w < kRouteWarps; ++w) {
        const int c = cnt[w * E_local + e];
        cnt[w * E_local + e] = run;
        run += c;
      }
      s_run[e] = run;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int64_t r = s0 + j * 32 + lane;
      if (r < q1) {
        const int e = key[j];
        int p = -1;
        if (e >= 0) {
          p = s_base[e] + cnt[warp * E_local + e] + rank[j];
          p = place_row(p, e, r, M, s_tot, permuted_idx, hdr);
        }
        inv_permuted_idx[r] = p;
      }
    }
    __syncthreads();
  }
}

}  // namespace moe
