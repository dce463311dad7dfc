// gather_tma.cuh -- the large-batch row gather with bulk asynchronous copies.
//
// vLLM PR #14568 ("permute/unpermute kernel for moe optimization",
// description): permute gathers each expert's tokens into contiguous rows for
// the grouped GEMM.  This kernel moves the rows with the Blackwell bulk-copy
// engine instead of registers: lane 0 of each warp copies a row chunk (up to
// kTmaChunkBytes) from HBM into a shared-memory stage with
// cp.async.bulk (completion counted on an mbarrier), then lanes 0..K-1 write
// it to the token's K destinations with one cp.async.bulk store each.  No registers hold
// data in flight, so shared memory bounds the bytes in flight (~190 KB per
// SM) rather than the register file.
//
// Each warp owns the items gw, gw + n_warps, ... of the (token, chunk) list
// and keeps kTmaStages of them in flight.  Its first kTmaStages loads are
// issued before it waits for the routing grid (the caller's rows are complete
// by then: this grid only starts once the routing grid has passed its own
// dependency wait), so they overlap the routing.  They go out one at a time,
// each after the previous one has landed: with every warp's stages requested
// at once (tens of MB) the memory system's queues fill, and the routing
// grid's few small reads of its histogram table wait behind them for the
// whole drain (measured: 4-5 us instead of 1 us; the chained prefetch is
// 5-10% faster end to end on batches of about the prefetch capacity).
//
// Requirements (checked on the host): row pitch, chunk offsets and both base
// pointers are multiples of 16 bytes.
// Every mbarrier wait is bounded (2^22 polls or 2 s): on timeout the status
// word gets MOE_FLAG_BARRIER_TIMEOUT, the warp waits (again bounded) for its
// own loads still in flight, drains its stores, and returns.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kTmaWarps = 4;
constexpr int kTmaThreads = kTmaWarps * kWarpSize;
constexpr int kTmaStages = 3;
constexpr int64_t kTmaChunkBytes = 8192;
constexpr unsigned kTmaSpinLimit = 1u << 22;
constexpr unsigned long long kTmaTimeLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait for the phase `parity` of an mbarrier to complete.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  unsigned long long t0 = 0;
  for (unsigned spins = 0; spins < kTmaSpinLimit; ++spins) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((spins & 255u) == 0u) {
      unsigned long long now;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
      if (spins == 0u) t0 = now;
      else if (now - t0 > kTmaTimeLimitNs) return false;
    }
  }
  return false;
}

__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_store(void* dst, const void* src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_addr(src_smem)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N committed store groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Shared memory: kTmaWarps * kTmaStages stages of `pitch` bytes (a multiple of
// 128), then kTmaWarps * kTmaStages mbarriers.
__global__ void __launch_bounds__(kTmaThreads)
k_gather_rows_tma(const char* __restrict__ hidden, int64_t row_bytes, int64_t chunk_bytes,
                  int64_t pitch, const float* __restrict__ scales, int64_t scale_cols,
                  const int32_t* __restrict__ inv_permuted_idx, int64_t T, int K,
                  char* __restrict__ out, float* __restrict__ out_scales,
                  int64_t num_out_rows, unsigned* __restrict__ status) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  unsigned char* stages = smem_raw + static_cast<int64_t>(warp) * kTmaStages * pitch;
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(smem_raw + static_cast<int64_t>(kTmaWarps) * kTmaStages * pitch) +
      warp * kTmaStages;
  const int64_t n_chunks = (row_bytes + chunk_bytes - 1) / chunk_bytes;
  const int64_t n_items = T * n_chunks;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kTmaWarps + warp;
  const int64_t n_gw = static_cast<int64_t>(gridDim.x) * kTmaWarps;

  auto issue_load = [&](int64_t item, int s) {
    const int64_t t = item / n_chunks;
    const int64_t c0 = (item - t * n_chunks) * chunk_bytes;
    const uint32_t bytes = static_cast<uint32_t>(min(chunk_bytes, row_bytes - c0));
    mbar_arrive_expect_tx(&bars[s], bytes);
    bulk_load(stages + s * pitch, hidden + t * row_bytes + c0, bytes, &bars[s]);
  };

  if (lane == 0) {
    for (int s = 0; s < kTmaStages; ++s) mbar_init(&bars[s]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int s = 0; s < kTmaStages; ++s) {
      const int64_t item = gw + s * n_gw;
      if (item >= n_items) break;
      // A wait that gives up here is not acted on: the main loop's bounded
      // wait for the same stage flags it.
      if (s > 0) (void)mbar_wait_bounded(&bars[s - 1], 0u);
      issue_load(item, s);
    }
  }
  __syncwarp();
  pdl_wait();

  int i = 0;
  for (int64_t item = gw; item < n_items; item += n_gw, ++i) {
    const int s = i % kTmaStages;
    const uint32_t parity = static_cast<uint32_t>(i / kTmaStages) & 1u;
    const int64_t t = item / n_chunks;
    const int64_t c0 = (item - t * n_chunks) * chunk_bytes;
    const uint32_t bytes = static_cast<uint32_t>(min(chunk_bytes, row_bytes - c0));
    // The token's scales are loaded before the wait for its row, so the load
    // is not a second round trip after the stores.
    const bool with_scales = out_scales != nullptr && c0 == 0;
    float sc[kPreScaleChunks];
    if (with_scales) load_token_scales(scales + t * scale_cols, scale_cols, sc);
    int p = lane < K ? __ldcg(inv_permuted_idx + t * K + lane) : -1;
    if (p >= num_out_rows) p = -1;  // only a routing grid that gave up leaves such values
    const unsigned valid = __ballot_sync(kFullMask, p >= 0);
    int ok = 1;
    if (lane == 0) ok = mbar_wait_bounded(&bars[s], parity) ? 1 : 0;
    ok = __shfl_sync(kFullMask, ok, 0);
    if (!ok) {
      // Give up: flag it, let every load this warp still has in flight land
      // (bounded), drain the stores, return.
      if (lane == 0) {
        atomicOr(status, MOE_FLAG_BARRIER_TIMEOUT);
        int j = i;
        for (int64_t it = item; it < n_items && j < i + kTmaStages; it += n_gw, ++j)
          (void)mbar_wait_bounded(&bars[j % kTmaStages], static_cast<uint32_t>(j / kTmaStages) & 1u);
      }
      bulk_wait_all();
      __syncwarp();
      return;
    }
    // Lane k stores the chunk to destination k: one thread's bulk copies go
    // out one after another, so K stores from one lane took K times as long
    // to issue.
    if ((valid >> lane) & 1u) {
      bulk_store(out + static_cast<int64_t>(p) * row_bytes + c0, stages + s * pitch, bytes);
      bulk_commit();
    }
    if (with_scales && valid != 0u)
      store_token_scales(scales + t * scale_cols, scale_cols, sc, out_scales, p, valid);
    // Refill this stage with the item kTmaStages steps ahead once the stores
    // just issued (by any lane) have read it.
    const int64_t next = item + kTmaStages * n_gw;
    if (next < n_items) {
      bulk_wait_read<0>();
      __syncwarp();
      if (lane == 0) issue_load(next, s);
    }
    __syncwarp();
  }
  bulk_wait_all();
}

}  // namespace moe
