// common.cuh -- small device helpers shared by the routing and row kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "moe_permute.h"

namespace moe {

constexpr int kWarpSize = 32;
constexpr unsigned kFullMask = 0xffffffffu;

// Workspace control block: first 256 bytes of every workspace.
struct WsHeader {
  unsigned reserved0;
  unsigned status;  // OR of MOE_FLAG_* bits
  unsigned table_hi;  // histogram-table entries the last routing grid wrote or left
  unsigned gen;       // routing calls so far (mod 2^32): the source of each call's table tag
  unsigned reserved[60];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");
constexpr size_t kWsHeaderBytes = sizeof(WsHeader);

// Programmatic dependent launch.  wait: block until every grid this launch
// depends on has completed and its writes are visible; a no-op when the
// launch carries no programmatic dependency.  launch_dependents: allow the
// next grid in the stream to be scheduled once every block of this grid has
// issued it (or exited).
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Read-only, read-once global load (non-coherent path, no L1 allocation).
template <typename T>
__device__ __forceinline__ T ld_stream(const T* p) {
  return __ldg(p);
}
template <>
__device__ __forceinline__ uint4 ld_stream<uint4>(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// A token's first 64 scale columns, loaded ahead of its row stores so that the
// load is not a second round trip after them (lane l holds columns l and
// l + 32).  store_token_scales writes them, and loads and writes any further
// columns itself.
constexpr int kPreScaleChunks = 2;

__device__ __forceinline__ void load_token_scales(const float* __restrict__ src,
                                                  int64_t scale_cols,
                                                  float (&s)[kPreScaleChunks]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < kPreScaleChunks; ++i) {
    const int64_t c = i * 32 + lane;
    s[i] = c < scale_cols ? __ldg(src + c) : 0.f;
  }
}

__device__ __forceinline__ void store_token_scales(const float* __restrict__ src,
                                                   int64_t scale_cols,
                                                   const float (&s)[kPreScaleChunks],
                                                   float* __restrict__ out, int p_lane,
                                                   unsigned valid) {
  static_assert(kPreScaleChunks == 2, "the selection below names both preloaded chunks");
  const int lane = threadIdx.x & 31;
  for (int64_t c0 = 0; c0 < scale_cols; c0 += 32) {
    const int64_t c = c0 + lane;
    float v;
    if (c0 == 0) v = s[0];
    else if (c0 == 32) v = s[1];
    else v = c < scale_cols ? __ldg(src + c) : 0.f;
    unsigned m = valid;
    while (m != 0u) {
      const int k = __ffs(m) - 1;
      m &= m - 1u;
      const int pk = __shfl_sync(kFullMask, p_lane, k);
      if (c < scale_cols) out[static_cast<int64_t>(pk) * scale_cols + c] = v;
    }
  }
}

// Exclusive prefix sum of one int per thread across the block (blockDim.x a
// multiple of 32, at most 1024).  s_warp: 32 ints of shared memory.  Returns
// the thread's exclusive prefix; *total receives the block total.  Ends with
// a barrier, so s_warp may be reused right after.
__device__ __forceinline__ int block_exclusive_sum(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int n_warps = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(kFullMask, x, d);
    if (lane >= d) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < n_warps ? s_warp[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(kFullMask, w, d);
      if (lane >= d) w += y;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  const int before = warp ? s_warp[warp - 1] : 0;
  *total = s_warp[n_warps - 1];
  __syncthreads();
  return before + x - v;
}

}  // namespace moe
