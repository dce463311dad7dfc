// quant.cuh -- quantise-on-permute: bf16 rows in, fp8 e4m3 rows plus fp32
// per-token, per-128-column scales out, written straight to each row's K
// destinations.
//
// The fp8 grouped GEMM after the permute reads per-token, per-column-group
// quantised activations ("[Kernels] MoE refactor" (vLLM PR #19636), bot
// summary: quant_dtype, per_act_token_quant, block_shape).  Quantising inside
// the gather saves a separate pass over the activations:
//   scale = amax(|x| over the group) / 448   (1 when the group is all zero),
//   code  = e4m3(x / scale), round to nearest even, saturating at +-448.
// Both divisions are IEEE-rounded fp32 divisions (x / scale through
// div_by_scale, which returns the same value).
//
// Layout: a warp owns one (token, chunk) item of 32 lanes x V vectors of 8
// bf16 values.  Vector c of a row belongs to column group c / 16, so for each
// vector slot i the lanes 0-15 hold one 128-column group and lanes 16-31 the
// next: the group's amax is a 4-step max-shuffle inside a half warp.
#pragma once

#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {

constexpr int kQuantGroup = 128;  // columns per scale
constexpr float kE4m3Max = 448.0f;

// x / s rounded to nearest in fp32, for an element x of a group whose scale is
// s = amax / 448 (so |x| <= 448 s), by the correction step of division with a
// fused multiply-add (P. Markstein, "Computation of elementary functions on the
// IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990; also Muller
// et al., "Handbook of Floating-Point Arithmetic", division by iteration):
// with y = RN(1/s), q0 = RN(x y), r = x - q0 s (exact in one fma),
// q = RN(q0 + r y).  The sign is copied from x so that -0 stays -0 (the
// correction would return +0).  Valid when s lies in [2^-100, 2^100]: there
// r neither underflows nor overflows for any such x, and an exhaustive GPU
// comparison with IEEE division over every pair of finite bf16 values
// (x, amax), |x| <= amax, gave the same e4m3 code for all of them and the
// same fp32 quotient wherever |q| >= 2^-12 (tests/test_quant_division_gpu.py
// repeats it through the debug build).  scale_in_range says whether s is in
// that range; outside it the caller divides with __fdiv_rn.
__device__ __forceinline__ bool scale_in_range(float s) {
  return s >= 0x1p-100f && s <= 0x1p+100f;
}
__device__ __forceinline__ float div_by_scale(float x, float s, float y) {
  const float q0 = __fmul_rn(x, y);
  const float r = __fmaf_rn(-q0, s, x);
  return copysignf(__fmaf_rn(r, y, q0), x);
}

// Quantise one (token, chunk) item held in registers (V vectors of 8 bf16
// values per lane; lanes 0-15 and 16-31 of vector slot i cover one 128-column
// group each): codes[i] holds the lane's 8 e4m3 codes of vector i, scales[i]
// its group's scale.  Every lane of the warp must call it (the group maxima
// are half-warp shuffles).  It needs no destination, so the kernels run it
// before they wait for the routing positions.
template <int V>
__device__ __forceinline__ void quant_chunk(const uint4 (&v)[V], uint2 (&codes)[V],
                                            float (&scales)[V]) {
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v[i]);
    float x[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(h2[j]);
      x[2 * j] = f.x;
      x[2 * j + 1] = f.y;
    }
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(x[j]));
#pragma unroll
    for (int d = 8; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, d));
    const float scale = amax > 0.0f ? __fdiv_rn(amax, kE4m3Max) : 1.0f;
    unsigned short* q2 = reinterpret_cast<unsigned short*>(&codes[i]);
    if (scale_in_range(scale)) {
      const float y = __frcp_rn(scale);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = make_float2(div_by_scale(x[2 * j], scale, y),
                                     div_by_scale(x[2 * j + 1], scale, y));
        q2[j] = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = make_float2(__fdiv_rn(x[2 * j], scale), __fdiv_rn(x[2 * j + 1], scale));
        q2[j] = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
      }
    }
    scales[i] = scale;
  }
}

// Store an item quantised by quant_chunk to every destination row p_k whose
// bit k is set in `valid` (lane k < K holds p_k in `p`): 8 bytes of codes per
// lane and one scale per half-warp.  Vectors at or beyond row_vecs are not
// stored.
template <int V>
__device__ __forceinline__ void store_quant_chunk(const uint2 (&codes)[V], const float (&scales)[V],
                                                  int64_t c0, int64_t row_vecs, int p,
                                                  unsigned valid, uint2* __restrict__ out_codes,
                                                  float* __restrict__ out_scales) {
  const int lane = threadIdx.x & 31;
  const int64_t n_groups = row_vecs / (kQuantGroup / 8);
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int64_t c = c0 + i * 32 + lane;
    const int64_t g = c / (kQuantGroup / 8);
    unsigned m = valid;
    while (m != 0u) {
      const int k = __ffs(m) - 1;
      m &= m - 1u;
      const int pk = __shfl_sync(kFullMask, p, k);
      if (c < row_vecs) {
        out_codes[static_cast<int64_t>(pk) * row_vecs + c] = codes[i];
        if ((lane & 15) == 0) out_scales[static_cast<int64_t>(pk) * n_groups + g] = scales[i];
      }
    }
  }
}

// quant_chunk / store_quant_chunk for items of 64 vectors (V = 2, four 128-column groups)
// with 16-byte code stores, in two steps: quant_chunk_wide quantises (it needs
// no destination, so the gather runs it before it waits for the routing grid:
// measured on GB300, DeepSeek-V3 quantise-on-permute 1-5% faster from T = 512
// to 32768) and store_quant_wide writes to the destinations.  The codes are
// quantised in the load layout above, then shuffled so that lane L holds the
// 16 codes of vectors c0 + 2L and c0 + 2L + 1 (one uint4), and the item's four
// group scales are gathered into lane 0 as one float4.  Per destination row that is one 512-byte warp store
// of codes and one 16-byte store of scales, instead of two 256-byte code
// stores and four 4-byte scale stores.  Requires 16-byte aligned code rows
// (H a multiple of 16 bytes of codes and a 16-byte aligned base) and, for the
// float4 scale store, a number of groups per row that is a multiple of 4 and
// a 16-byte aligned scale base; otherwise the scales go out one per group.
struct QuantWide {
  uint4 packed;   // this lane's 16 codes
  float s[4];     // the item's four group scales (valid in every lane)
};

__device__ __forceinline__ QuantWide quant_chunk_wide(const uint4 (&v)[2]) {
  const int lane = threadIdx.x & 31;
  uint2 code[2];
  float scale[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v[i]);
    float x[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(h2[j]);
      x[2 * j] = f.x;
      x[2 * j + 1] = f.y;
    }
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(x[j]));
#pragma unroll
    for (int d = 8; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, d));
    scale[i] = amax > 0.0f ? __fdiv_rn(amax, kE4m3Max) : 1.0f;
    unsigned short* q2 = reinterpret_cast<unsigned short*>(&code[i]);
    if (scale_in_range(scale[i])) {
      const float y = __frcp_rn(scale[i]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = make_float2(div_by_scale(x[2 * j], scale[i], y),
                                     div_by_scale(x[2 * j + 1], scale[i], y));
        q2[j] = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f =
            make_float2(__fdiv_rn(x[2 * j], scale[i]), __fdiv_rn(x[2 * j + 1], scale[i]));
        q2[j] = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
      }
    }
  }
  // Vectors 2L and 2L + 1 sit in slot L / 16 of lanes (2L) % 32 and (2L + 1) % 32.
  const int src0 = (2 * lane) & 31, src1 = src0 + 1;
  uint2 a[2], b[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    a[i].x = __shfl_sync(kFullMask, code[i].x, src0);
    a[i].y = __shfl_sync(kFullMask, code[i].y, src0);
    b[i].x = __shfl_sync(kFullMask, code[i].x, src1);
    b[i].y = __shfl_sync(kFullMask, code[i].y, src1);
  }
  const int slot = lane >> 4;
  const uint4 packed = slot == 0 ? make_uint4(a[0].x, a[0].y, b[0].x, b[0].y)
                                 : make_uint4(a[1].x, a[1].y, b[1].x, b[1].y);
  QuantWide q;
  q.packed = packed;
  q.s[0] = scale[0];
  q.s[1] = __shfl_sync(kFullMask, scale[0], 16);
  q.s[2] = scale[1];
  q.s[3] = __shfl_sync(kFullMask, scale[1], 16);
  return q;
}

template <bool kScales16>
__device__ __forceinline__ void store_quant_wide(const QuantWide& q, int64_t c0,
                                                 int64_t row_vecs, int p, unsigned valid,
                                                 uint4* __restrict__ out_codes,
                                                 float* __restrict__ out_scales) {
  const int lane = threadIdx.x & 31;
  const int64_t n_groups = row_vecs / (kQuantGroup / 8);
  const int64_t pair = (c0 >> 1) + lane;             // this lane's uint4 in the row
  const bool in_row = c0 + 2 * lane < row_vecs;      // whole groups: pairs never straddle
  // The item's groups: g0 (slot 0, lanes 0-15), g0 + 1 (slot 0, lanes 16-31),
  // g0 + 2 and g0 + 3 (slot 1).
  const int64_t g0 = c0 / (kQuantGroup / 8);
  const bool whole = g0 + 4 <= n_groups;
  unsigned m = valid;
  while (m != 0u) {
    const int k = __ffs(m) - 1;
    m &= m - 1u;
    const int pk = __shfl_sync(kFullMask, p, k);
    if (in_row) out_codes[static_cast<int64_t>(pk) * (row_vecs >> 1) + pair] = q.packed;
    float* srow = out_scales + static_cast<int64_t>(pk) * n_groups + g0;
    if (kScales16 && whole) {
      if (lane == 0)
        *reinterpret_cast<float4*>(srow) = make_float4(q.s[0], q.s[1], q.s[2], q.s[3]);
    } else if (lane == 0) {
      const float sv[4] = {q.s[0], q.s[1], q.s[2], q.s[3]};
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (g0 + u < n_groups) srow[u] = sv[u];
    }
  }
}

template <int V>
__global__ void __launch_bounds__(256)
k_gather_quant_fp8(const uint4* __restrict__ hidden, int64_t row_vecs,
                   const int32_t* __restrict__ inv_permuted_idx, int64_t T, int K,
                   uint2* __restrict__ out_codes, float* __restrict__ out_scales,
                   int64_t num_out_rows) {
  constexpr int64_t kChunk = 32 * V;  // vectors of 8 values per item
  const int lane = threadIdx.x & 31;
  const int64_t n_chunks = (row_vecs + kChunk - 1) / kChunk;
  const int64_t item = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (item >= T * n_chunks) return;
  const int64_t t = item / n_chunks;
  const int64_t c0 = (item - t * n_chunks) * kChunk;

  uint4 v[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int64_t c = c0 + i * 32 + lane;
    v[i] = c < row_vecs ? ld_stream(hidden + t * row_vecs + c) : make_uint4(0, 0, 0, 0);
  }
  // The rows are the caller's input (complete: the routing grid has passed its
  // own dependency wait); the positions come from the routing grid.
  uint2 codes[V];
  float qs[V];
  quant_chunk<V>(v, codes, qs);  // before the wait: it needs no position
  pdl_wait();
  int p = lane < K ? __ldcg(inv_permuted_idx + t * K + lane) : -1;
  if (p >= num_out_rows) p = -1;  // only a routing grid that gave up leaves such values
  const unsigned valid = __ballot_sync(kFullMask, p >= 0);
  if (valid == 0u) return;
  store_quant_chunk<V>(codes, qs, c0, row_vecs, p, valid, out_codes, out_scales);
}

// k_gather_quant_fp8 with the 16-byte stores of quant_chunk_wide /
// store_quant_wide (items of 64 vectors).
template <bool kScales16>
__global__ void __launch_bounds__(256)
k_gather_quant_fp8_wide(const uint4* __restrict__ hidden, int64_t row_vecs,
                        const int32_t* __restrict__ inv_permuted_idx, int64_t T, int K,
                        uint4* __restrict__ out_codes, float* __restrict__ out_scales,
                        int64_t num_out_rows) {
  constexpr int64_t kChunk = 64;
  const int lane = threadIdx.x & 31;
  const int64_t n_chunks = (row_vecs + kChunk - 1) / kChunk;
  const int64_t item = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (item >= T * n_chunks) return;
  const int64_t t = item / n_chunks;
  const int64_t c0 = (item - t * n_chunks) * kChunk;

  uint4 v[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int64_t c = c0 + i * 32 + lane;
    v[i] = c < row_vecs ? ld_stream(hidden + t * row_vecs + c) : make_uint4(0, 0, 0, 0);
  }
  const QuantWide q = quant_chunk_wide(v);  // before the wait: it needs no position
  pdl_wait();
  int p = lane < K ? __ldcg(inv_permuted_idx + t * K + lane) : -1;
  if (p >= num_out_rows) p = -1;  // only a routing grid that gave up leaves such values
  const unsigned valid = __ballot_sync(kFullMask, p >= 0);
  if (valid == 0u) return;
  store_quant_wide<kScales16>(q, c0, row_vecs, p, valid, out_codes, out_scales);
}

}  // namespace moe
