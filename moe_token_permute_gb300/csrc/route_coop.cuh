// route_coop.cuh -- routing metadata of moe_permute for large batches: one
// cooperatively launched grid whose blocks exchange per-expert histograms
// through a tagged table instead of a grid barrier.
//
// vLLM PR #14568 ("permute/unpermute kernel for moe optimization",
// description): expand each token to its K rows and order the rows by expert
// for the grouped GEMM.  Order inside an expert is stable by expanded row id
// r = t*K + k.
//
// Block b owns the contiguous tokens [b*tpb, (b+1)*tpb), i.e. the contiguous
// rows [r0, r1).  Phases:
//   1. histogram of the block's rows -> row b of the table (workspace), each
//      entry tagged with this call's tag.  When the block's rows fit one
//      round (kRouteThreads * J rows), the stable in-block ranks are computed in the
//      same pass and kept in registers;
//   2. every block reads the whole [B][E_local] table with 16-byte loads,
//      re-reading entries that do not carry this call's tag yet (every block
//      is resident: cooperative launch), and forms the offsets (block 0 writes
//      them) and its bases base[e] = offset[e] + sum_{b'<b} table[b'][e];
//   3. positions p = base[e] + (rows of expert e before r in the block) ->
//      permuted_idx, inv_permuted_idx (in rounds when the block has more rows).
// A tagged entry is its own completion flag, so no block waits on a counter,
// a fence or another block's arrival: each waits only until the rows it reads
// have landed.
// Tags: entry = tag << 24 | count, tag = 0x80 | (gen & 0x7f), gen a word of
// the workspace header that block 0 advances by one per call (after it has
// seen every row, i.e. after every block has read gen).  Block 0 also zeroes
// the entries past this call's extent that an earlier call left.  So while a
// call runs, every entry holds zero, the previous call's tag or this call's:
// a stale entry can never pass for a fresh one.
// The kernel lets the row-gather kernel that follows launch as soon as it
// starts: those blocks load their source rows while routing runs and wait for
// this grid before they read inv_permuted_idx.
// Every wait for a table entry is bounded (2^24 polls or 2 s): on timeout the
// status word gets MOE_FLAG_BARRIER_TIMEOUT and the kernel returns (outputs
// undefined; the gather that follows never stores through an out-of-range
// position).  Block 0 still advances gen on that path, so the next call tags
// its entries afresh and is exact without re-initialising the workspace.
#pragma once

#include "common.cuh"
#include "routing.cuh"

namespace moe {

// 512 threads x 2 rows per lane: 1024 rows per round, with short per-lane
// ranking loops and twice the threads for reading the table (measured on
// GB300 against 256 x 4: permute 0.4-2.9% faster on every workload shape).
constexpr int kRouteThreads = 512;
constexpr int kRouteWarps = kRouteThreads / kWarpSize;
// Rows per lane in one round (J): 2 (1024 rows per round) normally; 4, with
// half the blocks, when the [B][E] table every block reads is large.
constexpr int kRouteRowsPerLane = 2;
constexpr int kRouteRowsPerLaneLargeTable = 4;
constexpr unsigned kTablePollLimit = 1u << 24;                   // polls before giving up
constexpr unsigned long long kTableTimeLimitNs = 2000000000ull;  // or 2 s, whichever first
constexpr int kTagShift = 24;
constexpr unsigned kCountMask = (1u << kTagShift) - 1u;  // per-entry counts stay below 2^24
constexpr int kPollBatch = 4;                            // table rows a thread loads at once

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

#ifdef MOE_DEBUG_HOOKS
// Debug builds only (moe_debug_set_table_wait): table rows past the grid
// that every block also waits for -- rows no block writes, so the waits run
// out -- and the time limit of a wait.
__device__ int g_debug_extra_rows = 0;
__device__ unsigned long long g_debug_table_wait_ns = kTableTimeLimitNs;
__device__ __forceinline__ int debug_extra_rows() { return g_debug_extra_rows; }
__device__ __forceinline__ unsigned long long table_time_limit_ns() {
  return g_debug_table_wait_ns;
}
#else
__device__ __forceinline__ int debug_extra_rows() { return 0; }
__device__ __forceinline__ unsigned long long table_time_limit_ns() { return kTableTimeLimitNs; }
#endif

__device__ __forceinline__ unsigned call_tag(unsigned gen) { return 0x80u | (gen & 0x7fu); }

__device__ __forceinline__ void st_relaxed(unsigned* p, unsigned v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint4 ld_relaxed_quad(const unsigned* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ bool has_tag(uint4 v, unsigned tag) {
  return ((v.x >> kTagShift) == tag) & ((v.y >> kTagShift) == tag) &
         ((v.z >> kTagShift) == tag) & ((v.w >> kTagShift) == tag);
}

// Re-read four table entries until all carry `tag`.  Bounded: false after
// kTablePollLimit reads or kTableTimeLimitNs.
__device__ __forceinline__ bool poll_quad(const unsigned* p, unsigned tag, uint4& v) {
  unsigned long long t0 = 0;
  for (unsigned spins = 1; spins < kTablePollLimit; ++spins) {
    v = ld_relaxed_quad(p);
    if (has_tag(v, tag)) return true;
    if ((spins & 255u) == 1u) {
      const unsigned long long now = global_ns();
      if (spins == 1u) t0 = now;
      else if (now - t0 > table_time_limit_ns()) return false;
    }
    if (spins > 64u) __nanosleep(32);
  }
  return false;
}

// Thread 0 of each block reads this call's gen, and stores it and the table
// extent `hi` (loaded at the block's start) to shared memory.  Acquire: pairs
// with block 0's release of the next value, which comes after it has read
// this block's row (so this read sees the old value).  Called after the
// block's first id loads are issued, so neither round trip delays them
// (measured on GB300 against reading gen first and the extent in the block's
// last step: metadata-only permute 0.2-0.55 us faster, permute unchanged to
// 0.3 us faster).
__device__ __forceinline__ void read_gen(const WsHeader* hdr, unsigned hi, unsigned* s_gen,
                                         unsigned* s_hi) {
  if (threadIdx.x != 0) return;
  unsigned g;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(g) : "l"(&hdr->gen) : "memory");
  *s_gen = g;
  *s_hi = hi;
}

// Block 0's last step of a call, once it has read every block's row (so every
// block has read gen): zero the entries [ext, hi) an earlier call left (this
// call reads only entries below ext; hi = table_hi, which block 0 read at its
// start, since only this step of a completed grid writes it), record ext, and
// advance gen for the next call.  The release orders the gen store after the
// row reads; it comes last because it waits for the block's earlier stores,
// which the grid's completion waits for anyway.
__device__ __forceinline__ void retire_table(WsHeader* hdr, unsigned* table, unsigned ext,
                                             unsigned hi, unsigned gen) {
  if (blockIdx.x != 0) return;
  for (unsigned i = ext + threadIdx.x; i < hi; i += blockDim.x) st_relaxed(table + i, 0u);
  __syncthreads();
  if (threadIdx.x == 0) {
    st_relaxed(&hdr->table_hi, ext);
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(&hdr->gen), "r"(gen + 1u) : "memory");
  }
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
template <typename IdT, int J>
__global__ void __launch_bounds__(kRouteThreads, 2)
k_route_coop(const IdT* __restrict__ ids, const int32_t* __restrict__ emap,
             int64_t T, int K, int E, int E_local,
             int64_t* __restrict__ offsets, int32_t* __restrict__ permuted_idx,
             int32_t* __restrict__ inv_permuted_idx, WsHeader* __restrict__ hdr,
             unsigned* __restrict__ table, int64_t M, int32_t* __restrict__ expert_num_tokens) {
  extern __shared__ int smem[];
  __shared__ int s_warp[32];
  int* s_base = smem;                 // [E_local + 1]
  int* s_run = s_base + E_local + 1;  // [E_local]
  int* s_tot = s_run + E_local;       // [E_local] all blocks' rows per expert
  int* s_bef = s_tot + E_local;       // [E_local] rows per expert in blocks before b
  int* cnt = s_bef + E_local;         // [kRouteWarps][E_local]
  __shared__ unsigned s_gen, s_hi;
  const int B = gridDim.x;
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t R = T * K;
  const int64_t tpb = (T + B - 1) / B;
  const int64_t t0 = min(T, static_cast<int64_t>(b) * tpb);
  const int64_t t1 = min(T, t0 + tpb);
  const int64_t r0 = t0 * K, r1 = t1 * K;
  constexpr int kRoundRows = kRouteThreads * J;
  const bool one_round = r1 - r0 <= kRoundRows;

  pdl_wait();
  pdl_launch_dependents();
  // The table extent the last call left, for block 0's retire_table: loaded
  // now, stored to shared memory by read_gen.
  unsigned hi = 0;
  if (b == 0 && threadIdx.x == 0)
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(hi) : "l"(&hdr->table_hi) : "memory");
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
    read_gen(hdr, hi, &s_gen, &s_hi);
    rank_warp_slice<J>(key, cnt + warp * E_local, rank);
    __syncthreads();
    scan_counts_over_warps(cnt, E_local, kRouteWarps, s_run);  // s_run = block totals
  } else {
    read_gen(hdr, hi, &s_gen, &s_hi);
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
  const int e_pad = (E_local + 3) & ~3;  // table rows padded to whole 16-byte quads
  const unsigned tag = call_tag(s_gen);
  const unsigned tag_bits = tag << kTagShift;
  for (int e = threadIdx.x; e < e_pad; e += blockDim.x)
    st_relaxed(table + static_cast<int64_t>(b) * e_pad + e,
               tag_bits | (e < E_local ? static_cast<unsigned>(s_run[e]) : 0u));

  // Phase 2: totals, offsets and this block's bases from the whole table.
  // Thread i reads 4 experts (quad i % n_quads) of the table rows
  // bb = i / n_quads, i / n_quads + n_groups, ..., kPollBatch rows at a time
  // with 16-byte loads; a quad that does not carry this call's tag yet is
  // re-read until it does.
  bool timed_out = false;
  {
    const int B_read = B + debug_extra_rows();  // B outside debug builds
    const int n_quads = e_pad / 4;
    const int n_groups = max(1, static_cast<int>(blockDim.x) / n_quads);
    for (int i = threadIdx.x; i < n_quads * n_groups && !timed_out; i += blockDim.x) {
      const int q = i % n_quads;
      const int g = i / n_quads;
      unsigned tot[4] = {0u, 0u, 0u, 0u}, bef[4] = {0u, 0u, 0u, 0u};
      for (int bb0 = g; bb0 < B_read && !timed_out; bb0 += kPollBatch * n_groups) {
        uint4 c[kPollBatch];
#pragma unroll
        for (int u = 0; u < kPollBatch; ++u) {
          const int bb = bb0 + u * n_groups;
          c[u] = bb < B_read ? ld_relaxed_quad(table + static_cast<int64_t>(bb) * e_pad + 4 * q)
                        : make_uint4(tag_bits, tag_bits, tag_bits, tag_bits);
        }
#pragma unroll
        for (int u = 0; u < kPollBatch; ++u) {
          const int bb = bb0 + u * n_groups;
          if (!has_tag(c[u], tag) &&
              !poll_quad(table + static_cast<int64_t>(bb) * e_pad + 4 * q, tag, c[u])) {
            timed_out = true;
            break;
          }
          const unsigned v[4] = {c[u].x & kCountMask, c[u].y & kCountMask, c[u].z & kCountMask,
                                 c[u].w & kCountMask};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            tot[k] += v[k];
            if (bb < b) bef[k] += v[k];
          }
        }
      }
      const int e0 = q * 4;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (e0 + u < E_local) {
          atomicAdd(&s_tot[e0 + u], static_cast<int>(tot[u]));
          atomicAdd(&s_bef[e0 + u], static_cast<int>(bef[u]));
        }
      }
    }
  }
  const unsigned ext = static_cast<unsigned>(B) * static_cast<unsigned>(e_pad);
  if (__syncthreads_or(timed_out)) {
    if (threadIdx.x == 0) atomicOr(&hdr->status, MOE_FLAG_BARRIER_TIMEOUT);
    retire_table(hdr, table, ext, s_hi, s_gen);
    return;
  }
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

  // Phase 3: positions.
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
    retire_table(hdr, table, ext, s_hi, s_gen);
    return;
  }
  // More rows than one round: rank round by round; s_run[e] = this block's
  // rows of expert e placed so far.
  for (int e = threadIdx.x; e < E_local; e += blockDim.x) s_run[e] = 0;
  for (int64_t q0 = r0; q0 < r1; q0 += kRoundRows) {
    const int64_t q1 = min(r1, q0 + kRoundRows);
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
  retire_table(hdr, table, ext, s_hi, s_gen);
}

}  // namespace moe
