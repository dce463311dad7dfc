// onepass.cuh -- moe_permute with an expert map, for large batches, in ONE
// launch: the routing metadata and the row gather of a contiguous block of
// tokens are done by the same thread block, so the gather needs no second
// kernel and no source row is read unless its token keeps at least one row.
//
// vLLM PR #14568 ("permute/unpermute kernel for moe optimization",
// description): expand each token into its K rows, order the rows by expert
// (stable by r = t*K + k), and gather each row's token into the permuted
// buffer for the grouped GEMM; with an expert map only the rows of local
// experts are kept, which on one GPU is index filtering only.
//
// Why only with a map: with a map most rows are dropped (three quarters for
// the DeepSeek-V2-Lite shape, 16 of 64 experts local), and a sixth of the
// tokens keep none; this kernel reads exactly the kept tokens, where the
// two-kernel path (routing grid, then a gather that starts loading rows while
// routing runs) reads every token.  Measured on GB300 against the two-kernel
// path: equal from 3000 to 8192 tokens, 3.5% faster at 16384, with 1.0x the
// algorithmic source reads instead of 1.2x.  Without a map every token is
// read anyway, and the single launch measured slower (Mixtral T = 4096
// 19.9 us against 18.4): it loads all of a block's rows while routing runs,
// so after routing only writes remain, and a write-only stream runs at about
// 4.0 TB/s on GB300 against 6.7 TB/s for a copy.
//
// Grid: B <= #SM blocks of kOpThreads threads, one per SM (cooperative
// launch: every block must be resident, since each waits for the others'
// histogram rows).  Block b owns the tokens [t0, t1) = rows [r0, r1), at most
// kOpRouteThreads * J rows, so the ranks stay in registers.
//
// Warp roles:
//  - warps 0..15 (routing, then consumers): the routing of k_route_coop's
//    single-round path -- keys (the map staged in shared memory), stable
//    in-block ranks, the block's histogram row in the tagged table, the
//    whole table read back for the offsets and the block's bases, positions
//    -> inv_permuted_idx / permuted_idx and a shared-memory copy of the
//    block's positions -- plus the list of the block's tokens that keep a
//    row.  Then each consumes row chunks from a ring of shared-memory stages:
//    once a stage's chunk has landed, the warp reads it into registers
//    (16-byte vectors), hands the stage back, and stores the chunk to each
//    kept destination row.
//  - warp 16 (producer, all lanes): once the token list exists, fills the
//    ring with cp.async.bulk loads of the listed tokens' row chunks and
//    refills each stage as soon as its consumer releases it.  The loads go
//    out from all 32 lanes: one thread's bulk copies are issued one after
//    another (measured: 54 loads of 4 KB took 18 us to issue from a single
//    thread).
// The producer's loads overlap the rest of the routing.
//
// Ring: N = n_stages full/empty mbarrier pairs, N a multiple of 16; item i
// (a (token, chunk) pair of the block's item list) goes to stage s = i % N,
// round i / N.  Each stage has exactly one producer thread (lane s % 32 of
// the producer warp) and one consumer warp (s % 16), and each takes the
// stage's rounds in order: the consumer waits for phase i / N of full[s], the
// producer for phase i / N - 1 of empty[s] before it reuses the stage, and
// neither can find the stage more than one phase behind, which the parity
// test of an mbarrier wait requires.
//
// Synchronisation: the routing warps use named barrier 1 (512 threads), never
// __syncthreads after the prologue, since the producer warp does not take
// part; barrier 2 (544 threads) releases the producer once the token list
// exists.  Every wait is bounded: a table wait that gives up sets
// MOE_FLAG_BARRIER_TIMEOUT and makes the block abort (the producer lets its
// loads in flight land before it returns); the producer's and consumers'
// mbarrier waits give up likewise.
// Requirements (checked on the host): an expert map; 16-byte aligned rows,
// pitch and base pointers (the bulk copies); T*K beyond the single-block
// kernel's range.
#pragma once

#include "common.cuh"
#include "routing.cuh"
#include "route_coop.cuh"
#include "gather_tma.cuh"

namespace moe {

constexpr int kOpRouteWarps = 16;
constexpr int kOpRouteThreads = kOpRouteWarps * kWarpSize;  // 512
constexpr int kOpThreads = kOpRouteThreads + kWarpSize;     // + the producer warp
constexpr int kOpProducerWarp = kOpRouteWarps;
constexpr int64_t kOpChunkBytes = 4096;  // largest row chunk one stage holds
constexpr int kOpVec = 8;                // 16-byte vectors per lane in one consumer pass

__device__ __forceinline__ void op_route_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kOpRouteThreads) : "memory");
}

// Barrier 1 over the routing warps, returning whether any thread's p is true.
__device__ __forceinline__ bool op_route_sync_or(bool p) {
  int r;
  asm volatile(
      "{\n .reg .pred a, b;\n setp.ne.s32 a, %1, 0;\n"
      " bar.red.or.pred b, 1, %2, a;\n selp.s32 %0, 1, 0, b;\n}\n"
      : "=r"(r)
      : "r"(static_cast<int>(p)), "n"(kOpRouteThreads)
      : "memory");
  return r != 0;
}

// Barrier 2: the routing warps arrive once the token list is written, the
// producer warp waits for it.
__device__ __forceinline__ void op_list_arrive() {
  asm volatile("bar.arrive 2, %0;" ::"n"(kOpThreads) : "memory");
}
__device__ __forceinline__ void op_list_wait() {
  asm volatile("bar.sync 2, %0;" ::"n"(kOpThreads) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Exclusive prefix sum over the 512 routing threads (named barrier 1).
__device__ __forceinline__ int op_exclusive_sum(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(kFullMask, x, d);
    if (lane >= d) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  op_route_sync();
  if (warp == 0) {
    int w = lane < kOpRouteWarps ? s_warp[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(kFullMask, w, d);
      if (lane >= d) w += y;
    }
    s_warp[lane] = w;
  }
  op_route_sync();
  const int before = warp ? s_warp[warp - 1] : 0;
  *total = s_warp[kOpRouteWarps - 1];
  op_route_sync();
  return before + x - v;
}

// Wait (bounded) for phase `parity` of an mbarrier, giving up early when the
// block has been told to abort.
__device__ __forceinline__ bool op_wait_or_abort(uint64_t* bar, uint32_t parity,
                                                 const volatile int* abort) {
  unsigned long long t0 = 0;
  for (unsigned spins = 0; spins < kTmaSpinLimit; ++spins) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if ((spins & 255u) == 0u) {
      const unsigned long long now = global_ns();
      if (spins == 0u) t0 = now;
      else if (now - t0 > kTmaTimeLimitNs) return false;
    }
  }
  return false;
}

// Shared memory (dynamic): ring [n_stages][pitch] | full [n_stages] |
// empty [n_stages] | s_last [n_stages] | s_base [E_local + 1] |
// s_tot, s_bef, s_run [E_local] | cnt [16][E_local] | s_pos [rows_max] |
// s_flag, s_list [tok_max] | s_map [E] (with an expert map).
template <typename IdT, int J>
__global__ void __launch_bounds__(kOpThreads, 1)
k_permute_onepass(const IdT* __restrict__ ids, const int32_t* __restrict__ emap,
                  int64_t T, int K, int E, int E_local,
                  const char* __restrict__ hidden, int64_t row_bytes, int64_t chunk_bytes,
                  int n_chunks, int n_stages, int64_t pitch,
                  const float* __restrict__ scales, int64_t scale_cols,
                  char* __restrict__ out, float* __restrict__ out_scales, int64_t num_out_rows,
                  int64_t* __restrict__ offsets, int32_t* __restrict__ permuted_idx,
                  int32_t* __restrict__ inv_permuted_idx, WsHeader* __restrict__ hdr,
                  unsigned* __restrict__ table, int64_t M,
                  int32_t* __restrict__ expert_num_tokens) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ int s_warp[32];
  __shared__ unsigned s_gen, s_hi;
  __shared__ int s_nlist;
  __shared__ volatile int s_abort;

  const int B = gridDim.x;
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t tpb = (T + B - 1) / B;
  const int64_t t0 = min(T, static_cast<int64_t>(b) * tpb);
  const int64_t t1 = min(T, t0 + tpb);
  const int nt = static_cast<int>(t1 - t0);
  const int64_t r0 = t0 * K, r1 = t1 * K;

  unsigned char* ring = smem_raw;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + static_cast<int64_t>(n_stages) * pitch);
  uint64_t* empty = full + n_stages;
  int* s_last = reinterpret_cast<int*>(empty + n_stages);  // [n_stages] last item loaded there
  int* s_base = s_last + n_stages;                           // [E_local + 1]
  int* s_tot = s_base + E_local + 1;                         // [E_local]
  int* s_bef = s_tot + E_local;                              // [E_local]
  int* s_run = s_bef + E_local;                              // [E_local]
  int* cnt = s_run + E_local;                                // [16][E_local]
  int* s_pos = cnt + kOpRouteWarps * E_local;                // [tpb * K]
  int* s_flag = s_pos + tpb * K;                             // [tpb]
  int* s_list = s_flag + tpb;                                // [tpb]
  int* s_map = s_list + tpb;                                 // [E] (with an expert map)

  pdl_wait();
  // The next kernel's launch may start now: its blocks cannot share an SM
  // with this block's shared memory, so they only take over as blocks exit.
  pdl_launch_dependents();
  for (int s = threadIdx.x; s < n_stages; s += kOpThreads) {
    mbar_init(&full[s]);
    mbar_init(&empty[s]);
  }
  if (threadIdx.x < n_stages)
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if (threadIdx.x == 0) {
    s_abort = 0;
    s_nlist = 0;
  }
  for (int i = threadIdx.x; i < kOpRouteWarps * E_local; i += kOpThreads) cnt[i] = 0;
  for (int i = threadIdx.x; i < E_local; i += kOpThreads) {
    s_tot[i] = 0;
    s_bef[i] = 0;
  }
  for (int i = threadIdx.x; i < nt; i += kOpThreads) s_flag[i] = 0;
  for (int i = threadIdx.x; i < n_stages; i += kOpThreads) s_last[i] = -1;
  // The routing threads' ids and the expert map are loaded together, before
  // the barrier, so the map lookup that follows is a shared-memory read
  // rather than a second dependent trip to global memory.
  const int64_t slice0 = r0 + static_cast<int64_t>(warp) * 32 * J;
  IdT raw[J];
  if (warp < kOpRouteWarps) {
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int64_t r = slice0 + j * 32 + lane;
      raw[j] = r < r1 ? __ldg(ids + r) : IdT(-1);
    }
  }
  for (int e = threadIdx.x; e < E; e += kOpThreads) s_map[e] = __ldg(emap + e);
  // The call's gen (its table tag) is read by the producer warp's lane 0,
  // which loads no ids, so the acquire overlaps the id loads instead of
  // following them on a routing warp (measured on GB300: DeepSeek-V2-Lite
  // permute 0.2 us faster per call from T = 700 to 8192).  Acquire: pairs with
  // block 0's release of the next value, which comes after it has read every
  // block's row.
  if (threadIdx.x == kOpProducerWarp * kWarpSize) {
    unsigned g;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(g) : "l"(&hdr->gen) : "memory");
    s_gen = g;
  }
  __syncthreads();  // the only whole-block barrier

  // ---------------------------------------------------------- producer ---
  if (warp == kOpProducerWarp) {
    op_list_wait();
    // All 32 lanes issue loads: one thread's bulk copies go out one after
    // another, so a single issuing thread per SM left the ring filling at a
    // fraction of the HBM rate (measured on GB300: 54 loads of 4 KB took 18 us
    // to issue from one thread).  Lane l owns stages l, l + 32, ... and fills
    // each with its items i = round * N + s in round order, so a stage's
    // rounds are issued by one thread, one after another: the empty-phase wait
    // before round r can only find the stage in phase r - 1 (not yet released)
    // or r (released), never further behind, and its parity test cannot alias.
    const int n_items = s_nlist * n_chunks;
    bool stop = false;
    for (int round = 0; !stop; ++round) {
      bool any = false;
      for (int s = lane; s < n_stages && !stop; s += 32) {
        const int i = round * n_stages + s;
        if (i >= n_items) continue;
        any = true;
        if (round > 0 &&
            !op_wait_or_abort(&empty[s], static_cast<uint32_t>(round - 1) & 1u, &s_abort)) {
          if (!s_abort) atomicOr(&hdr->status, MOE_FLAG_BARRIER_TIMEOUT);
          stop = true;
          break;
        }
        const int tok = s_list[i / n_chunks];
        const int c = i % n_chunks;
        const int64_t c0 = static_cast<int64_t>(c) * chunk_bytes;
        const uint32_t bytes = static_cast<uint32_t>(min(chunk_bytes, row_bytes - c0));
        s_last[s] = i;  // only this lane writes stage s's entry
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_load(ring + static_cast<int64_t>(s) * pitch, hidden + (t0 + tok) * row_bytes + c0,
                  bytes, &full[s]);
      }
      if (!any) stop = true;
    }
    // Stay until the last load issued to each stage has landed, so that no
    // bulk copy still writes the block's shared memory after the block is
    // gone, even if a consumer gave up or the block aborted.  Only a stage's
    // last load is waited for: its phase is the stage's final one, so its
    // parity cannot alias a phase that never starts.
    __syncwarp();
    for (int st = lane; st < n_stages; st += 32) {
      const int j = s_last[st];
      if (j >= 0)
        (void)mbar_wait_bounded(&full[st], static_cast<uint32_t>(j / n_stages) & 1u);
    }
    return;
  }

  // ----------------------------------------------------------- routing ---
  int key[J], rank[J];
  unsigned flags = 0;
  unsigned hi = 0;
  if (b == 0 && threadIdx.x == 0)
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(hi) : "l"(&hdr->table_hi) : "memory");
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int64_t r = slice0 + j * 32 + lane;
    key[j] = r < r1 ? local_expert(raw[j], s_map, E, E_local, flags) : -1;
  }
  if (threadIdx.x == 0) s_hi = hi;  // block 0's retire step reads it
  rank_warp_slice<J>(key, cnt + warp * E_local, rank);
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int64_t r = slice0 + j * 32 + lane;
    if (r < r1 && key[j] >= 0) s_flag[(r - r0) / K] = 1;
  }
  flags = __reduce_or_sync(kFullMask, flags);
  if (flags != 0 && lane == 0) atomicOr(&hdr->status, flags);
  op_route_sync();
  // per-warp counts -> exclusive prefixes over the warps; s_run = block totals
  for (int e = threadIdx.x; e < E_local; e += kOpRouteThreads) {
    int run = 0;
    for (int w = 0; w < kOpRouteWarps; ++w) {
      const int c = cnt[w * E_local + e];
      cnt[w * E_local + e] = run;
      run += c;
    }
    s_run[e] = run;
  }
  // The block's tokens that keep at least one row, one shared-memory atomic
  // each: the list's order is free (the producer and the consumers read the
  // same list), and no block-wide scan stands between the ranking and the
  // histogram row the other blocks wait for.
  for (int i = threadIdx.x; i < nt; i += kOpRouteThreads)
    if (s_flag[i]) s_list[atomicAdd(&s_nlist, 1)] = i;
  op_route_sync();   // s_run and the token list are complete
  op_list_arrive();  // the producer can start on the list
  // the block's histogram row, tagged with this call's tag
  const int e_pad = (E_local + 3) & ~3;
  const unsigned tag = call_tag(s_gen);
  const unsigned tag_bits = tag << kTagShift;
  for (int e = threadIdx.x; e < e_pad; e += kOpRouteThreads)
    st_relaxed(table + static_cast<int64_t>(b) * e_pad + e,
               tag_bits | (e < E_local ? static_cast<unsigned>(s_run[e]) : 0u));

  // totals and this block's bases from the whole table (as k_route_coop)
  bool timed_out = false;
  {
    const int B_read = B + debug_extra_rows();  // B outside debug builds
    const int n_quads = e_pad / 4;
    const int n_groups = max(1, kOpRouteThreads / n_quads);
    for (int i = threadIdx.x; i < n_quads * n_groups && !timed_out; i += kOpRouteThreads) {
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
  if (op_route_sync_or(timed_out)) {
    if (threadIdx.x == 0) {
      atomicOr(&hdr->status, MOE_FLAG_BARRIER_TIMEOUT);
      s_abort = 1;
    }
    if (b == 0) {
      for (unsigned i = ext + threadIdx.x; i < s_hi; i += kOpRouteThreads) st_relaxed(table + i, 0u);
      op_route_sync();
      if (threadIdx.x == 0) {
        st_relaxed(&hdr->table_hi, ext);
        asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(&hdr->gen), "r"(s_gen + 1u)
                     : "memory");
      }
    }
    return;
  }
  // exclusive scan of the totals -> offsets (block 0) and this block's bases
  {
    constexpr int kPer = MOE_MAX_LOCAL_EXPERTS / kOpRouteThreads;
    int tot[kPer], sum = 0;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = threadIdx.x * kPer + u;
      tot[u] = e < E_local ? s_tot[e] : 0;
      sum += tot[u];
    }
    int n_valid;
    int run = op_exclusive_sum(sum, s_warp, &n_valid);
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
  op_route_sync();
  if (M == 0) {
    const int64_t R = T * K;
    for (int64_t p = s_base[E_local] + static_cast<int64_t>(b) * kOpRouteThreads + threadIdx.x;
         p < R; p += static_cast<int64_t>(B) * kOpRouteThreads)
      permuted_idx[p] = -1;
  }
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
      s_pos[r - r0] = p;
    }
  }
  op_route_sync();  // s_pos complete; block 0's reads of the table are done
  if (b == 0) {
    for (unsigned i = ext + threadIdx.x; i < s_hi; i += kOpRouteThreads) st_relaxed(table + i, 0u);
    op_route_sync();
    if (threadIdx.x == 0) {
      st_relaxed(&hdr->table_hi, ext);
      asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(&hdr->gen), "r"(s_gen + 1u)
                   : "memory");
    }
  }

  // ---------------------------------------------------------- consumers ---
  // n_stages is a multiple of 16, so every item of stage s belongs to warp
  // s % 16: each stage has one consumer, which takes its rounds in order.
  // When it waits for round r, round r - 1 is consumed (by itself) and round
  // r + 1 cannot have been loaded (the producer waits for this warp's release
  // of round r first), so the stage is in phase r and the parity test is exact.
  const int n_items = s_nlist * n_chunks;
  for (int i = warp; i < n_items; i += kOpRouteWarps) {
    const int s = i % n_stages;
    const uint32_t parity = static_cast<uint32_t>(i / n_stages) & 1u;
    const int tok = s_list[i / n_chunks];
    const int c = i % n_chunks;
    const int64_t c0 = static_cast<int64_t>(c) * chunk_bytes;
    const uint32_t bytes = static_cast<uint32_t>(min(chunk_bytes, row_bytes - c0));
    const int64_t t = t0 + tok;
    int p = lane < K ? s_pos[tok * K + lane] : -1;
    if (p >= num_out_rows) p = -1;
    const unsigned valid = __ballot_sync(kFullMask, p >= 0);
    const bool with_scales = out_scales != nullptr && c == 0 && valid != 0u;
    float sc[kPreScaleChunks];
    if (with_scales) load_token_scales(scales + t * scale_cols, scale_cols, sc);
    int ok = 1;
    if (lane == 0) ok = op_wait_or_abort(&full[s], parity, &s_abort) ? 1 : 0;
    ok = __shfl_sync(kFullMask, ok, 0);
    if (!ok) {
      if (lane == 0) {
        atomicOr(&hdr->status, MOE_FLAG_BARRIER_TIMEOUT);
        s_abort = 1;
      }
      break;
    }
    // The chunk goes from the stage to registers in 16-byte vectors (kOpVec
    // per lane per pass) and from there to each kept destination row; the
    // stage is handed back as soon as it has been read.
    const uint4* src = reinterpret_cast<const uint4*>(ring + static_cast<int64_t>(s) * pitch);
    const int n_vec = static_cast<int>(bytes >> 4);
    for (int v0 = 0; v0 < n_vec; v0 += 32 * kOpVec) {
      uint4 x[kOpVec];
#pragma unroll
      for (int u = 0; u < kOpVec; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < n_vec) x[u] = src[v];
      }
      if (v0 + 32 * kOpVec >= n_vec) {
        // every lane's reads of the stage are done: order them before the
        // producer's next bulk load into it, then release the stage
        __syncwarp();
        if (lane == 0) {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_arrive(&empty[s]);
        }
      }
      unsigned m = valid;
      while (m != 0u) {
        const int k = __ffs(m) - 1;
        m &= m - 1u;
        const int pk = __shfl_sync(kFullMask, p, k);
        uint4* dst = reinterpret_cast<uint4*>(out + static_cast<int64_t>(pk) * row_bytes + c0);
#pragma unroll
        for (int u = 0; u < kOpVec; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < n_vec) dst[v] = x[u];
        }
      }
    }
    if (with_scales)
      store_token_scales(scales + t * scale_cols, scale_cols, sc, out_scales, p, valid);
  }
}

}  // namespace moe
