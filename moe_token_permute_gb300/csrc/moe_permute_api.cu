// moe_permute_api.cu -- host side of the C ABI declared in include/moe_permute.h.
//
// Argument checks mirror MoEPermuteScratch.validate of the vLLM PR #43014
// digest ("key source excerpts": token count within the pre-allocated maximum,
// matching top-k, matching hidden size / dtype), returned as error codes.
// Nothing here allocates: the caller owns every buffer, including the
// workspace (same digest, "implementation breakdown" items 1-3).
//
// Dispatch:
//   R = T*K up to 3072 rows (4096 with an expert map; 2048 for the
//     metadata-only and the quantising permute): one launch of
//     k_permute_fused; every block redundantly ranks all rows and the blocks
//     share the row copy (no inter-block communication);
//   with an expert map and 16-byte aligned rows: k_permute_onepass, one
//     cooperative launch that routes a block of tokens and copies the rows of
//     the tokens that keep one;
//   otherwise: k_route_coop (cooperative grid; its blocks exchange their
//     histograms through a tagged table in the workspace) writes the
//     metadata, and the row gather (k_gather_rows_tma or k_gather_rows),
//     launched as its programmatic dependent, loads rows while the routing
//     runs and stores them once it has finished.
//   moe_permute_quant_fp8 splits the same way: k_permute_fused with its
//   quantising copy, or k_route_coop + k_gather_quant_fp8.
// Every launch carries programmatic stream serialization, so its launch
// latency overlaps the previous kernel's tail.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "moe_permute.h"
#ifdef MOE_DEBUG_HOOKS
#include "moe_permute_debug.h"
#endif
#include "common.cuh"
#include "routing.cuh"
#include "rows.cuh"
#include "route_coop.cuh"
#include "quant.cuh"
#include "gather_tma.cuh"
#include "onepass.cuh"

namespace moe {
namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int cc_major = 0;
  int cc_minor = 0;
  int sm_count = 0;
  int max_smem_optin = 0;
  int max_smem_per_sm = 0;
};

std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];

// Cached properties of the current device; nullptr if it cannot be queried.
const DeviceInfo* current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&d.max_smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                               dev) != cudaSuccess)
      return nullptr;
    d.ready = true;
  }
  return &d;
}

bool is_supported(const DeviceInfo* d) { return d != nullptr && d->cc_major == 10 && d->cc_minor == 3; }

// Raise a kernel's dynamic shared memory limit once per device.
template <typename Kern>
cudaError_t allow_smem(Kern kern, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(reinterpret_cast<const void*>(kern),
                              cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

// Launch with programmatic stream serialization: the grid may be scheduled as
// soon as the previous grid in the stream allows it; every kernel here calls
// griddepcontrol.wait before it touches memory a previous grid may write.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem,
                   cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Widest vector (16/8/4/2/1 bytes) that divides the row pitch and both bases.
size_t vec_bytes(int64_t row_bytes, const void* a, const void* b) {
  for (size_t w = 16; w > 1; w >>= 1)
    if (row_bytes % static_cast<int64_t>(w) == 0 && aligned(a, w) && (b == nullptr || aligned(b, w)))
      return w;
  return 1;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

constexpr int64_t kCoopMaxBlocks = 1024;  // table rows reserved for the cooperative grid
constexpr int64_t kLargeTable = 32768;     // [B][E_pad] entries from which routing halves B

#ifdef MOE_DEBUG_HOOKS
int g_debug_extra_rows_host = 0;  // host copy of the routing grid's g_debug_extra_rows
#endif

// Header plus the cooperative kernel's per-block histogram table
// [min(max_tokens, kCoopMaxBlocks)][num_experts rounded up to 4].
size_t workspace_bytes_for(int64_t max_tokens, int32_t topk, int32_t num_experts) {
  (void)topk;
  const int64_t e_pad = (static_cast<int64_t>(num_experts) + 3) / 4 * 4;
  const int64_t blocks = std::max<int64_t>(1, std::min(kCoopMaxBlocks, max_tokens));
  const size_t bytes = kWsHeaderBytes + static_cast<size_t>(e_pad * blocks * 4);
  return (bytes + 255) / 256 * 256;
}

constexpr int kFusedV = 4;   // vectors per lane in one gather chunk (fused kernel)
// Same, fused kernel with its quantising copy: one vector of 8 values per
// lane (two 128-column groups per item).  The arithmetic per item is long, so
// more, smaller items spread it over more warps: at DeepSeek-V3 shapes on
// GB300, T=1 4.0 us instead of 7.0 with 4 vectors, T=128 7.2 instead of 9.9.
constexpr int kFusedQuantV = 1;
constexpr int kGatherV = 8;  // same, gather kernel of the large-batch path
constexpr int64_t kFusedMaxRows = 2048;  // quantise-on-permute: R above this -> routing grid + gather
static_assert(kFusedMaxRows <= kMetaChunkRows, "one block must be able to rank every row");
// moe_permute takes the single launch a little further, ranking 4 rows per
// lane above 2048 rows.  Measured on GB300 against the two-kernel path:
// without a map 7-24% faster from 2080 to 3072 rows (Mixtral, Qwen3 and
// DeepSeek-V3 shapes; DeepSeek-V3 equal at 3072) and 4-18% slower at 3584-4096;
// with an expert map (DeepSeek-V2-Lite shape, a quarter of the rows kept)
// 10-25% faster than the single-launch expert-map kernel up to 4096.  The
// quantising copy measured no faster above 2048 rows and keeps kFusedMaxRows,
// and so does the metadata-only permute, which runs as one block there (from
// 2600 to 3072 rows 7-27% slower than the routing grid for the 128- and
// 256-expert shapes).
constexpr int64_t kFusedWideMaxRows = 3072;
constexpr int64_t kFusedWideMaxRowsMap = 4096;
static_assert(kFusedWideMaxRowsMap <= kMetaChunkRowsWide, "one block must be able to rank every row");

int64_t fused_max_rows(const int32_t* emap) {
  return emap != nullptr ? kFusedWideMaxRowsMap : kFusedWideMaxRows;
}

// (token, chunk) work items of a row kernel.
int64_t row_items(int64_t T, int64_t row_vecs, int V) {
  return T * std::max<int64_t>(1, ceil_div(row_vecs, 32 * static_cast<int64_t>(V)));
}

// Resident blocks per SM of a kernel, queried once per (device, kernel,
// block size, shared memory).  The key is the kernel's address: template
// instantiations with the same signature are different kernels.
int blocks_per_sm(const void* kern, int threads, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, const void*, int, size_t>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  const auto key = std::make_tuple(dev, kern, threads, smem);
  std::lock_guard<std::mutex> lock(mu);
  const auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess ||
      n < 1) {
    cudaGetLastError();
    n = 1;
  }
  cache[key] = n;
  return n;
}

// Grid for a warp-per-item kernel: one warp per item, capped at one wave of
// resident blocks (the kernels loop over items).
unsigned item_grid(int64_t items, int warps_per_block, const DeviceInfo* d, int per_sm) {
  const int64_t need = ceil_div(items, warps_per_block);
  const int64_t cap = static_cast<int64_t>(d->sm_count) * per_sm;
  return static_cast<unsigned>(std::max<int64_t>(1, std::min(need, cap)));
}

// From this many tokens the quantising single launch loads each warp's first
// row chunk before the ranking (k_permute_fused, kEarly).
constexpr int64_t kFusedEarlyMinTokens = 32;

template <typename IdT, typename VecT, int V, bool kQuant = false>
cudaError_t launch_fused(const IdT* ids, const int32_t* emap, int64_t T, int K, int E, int E_local,
                         const void* hidden, int64_t row_bytes, const float* scales,
                         int64_t scale_cols, void* out, float* out_scales, int64_t* offsets,
                         int32_t* pidx, int32_t* inv, WsHeader* hdr, const DeviceInfo* d,
                         cudaStream_t s) {
  const int64_t R = T * K;
  if (R > (kQuant ? kMetaChunkRows : kMetaChunkRowsWide)) return cudaErrorInvalidConfiguration;
  const int J = R <= kMetaChunkRows ? kMetaRowsPerLane : kMetaRowsPerLaneWide;
  const int64_t rank_warps = ceil_div(R, 32 * J);
  const size_t smem = (static_cast<size_t>(rank_warps) * E_local + E_local + 1 + R) * sizeof(int);
  auto kern = k_permute_fused<IdT, VecT, V, kQuant, false>;
  if constexpr (kQuant) {
    if (T >= kFusedEarlyMinTokens) kern = k_permute_fused<IdT, VecT, V, kQuant, true>;
  } else {
    if (J == kMetaRowsPerLaneWide)
      kern = k_permute_fused<IdT, VecT, V, false, false, kMetaRowsPerLaneWide>;
  }
  cudaError_t err = allow_smem(kern, smem);
  if (err != cudaSuccess) return err;
  const int64_t row_vecs = row_bytes / static_cast<int64_t>(sizeof(VecT));
  // One block per SM at most (each block redoes the routing), at least one
  // item per block.
  const unsigned grid = out == nullptr ? 1u : item_grid(row_items(T, row_vecs, V), 1, d, 1);
  return launch(kern, grid, kMetaThreads, smem, s, ids, emap, T, K, E, E_local,
                static_cast<const VecT*>(hidden), row_bytes / static_cast<int64_t>(sizeof(VecT)),
                scales, scale_cols, static_cast<VecT*>(out), out_scales, offsets, pidx, inv, hdr);
}

template <typename IdT>
cudaError_t launch_route(const IdT* ids, const int32_t* emap, int64_t T, int K, int E, int E_local,
                         int64_t* offsets, int32_t* pidx, int32_t* inv, WsHeader* hdr,
                         const DeviceInfo* d, cudaStream_t s, int64_t batch_capacity = 0,
                         int32_t* expert_num_tokens = nullptr) {
  // As few blocks as give each block at most one round of rows (so the ranks
  // stay in registers), and at most one per SM: the histogram table every
  // block reads is [B][E_pad], and the rest of each SM stays free for the
  // gather blocks that start while routing runs.  When that table reaches
  // kLargeTable entries (e.g. 152 blocks x 256 experts), reading it dominates:
  // rounds of twice the rows per lane halve the blocks (measured on GB300:
  // DeepSeek-V3 T = 32768 permute 2.2% faster; smaller tables were up to 6%
  // slower).
  const int64_t e_pad = (E_local + 3) / 4 * 4;
  int J = kRouteRowsPerLane;
  int64_t B = std::min<int64_t>(ceil_div(T, std::max<int64_t>(1, kRouteThreads * J / K)),
                                d->sm_count);
  if (B * e_pad >= kLargeTable) {
    J = kRouteRowsPerLaneLargeTable;
    B = std::min<int64_t>(ceil_div(T, std::max<int64_t>(1, kRouteThreads * J / K)), d->sm_count);
  }
  auto kern = J == kRouteRowsPerLane ? k_route_coop<IdT, kRouteRowsPerLane>
                                     : k_route_coop<IdT, kRouteRowsPerLaneLargeTable>;
  const size_t smem = (static_cast<size_t>(kRouteWarps) * E_local + 4 * E_local + 1) * sizeof(int);
  cudaError_t err = allow_smem(kern, smem);
  if (err != cudaSuccess) return err;
  // A table entry holds a block's rows of one expert in 24 bits.
  B = std::max(B, ceil_div(T, static_cast<int64_t>(kCountMask) / K));
  B = std::max<int64_t>(1, std::min(B, kCoopMaxBlocks));
  if (ceil_div(T, B) * K > static_cast<int64_t>(kCountMask)) return cudaErrorInvalidConfiguration;
#ifdef MOE_DEBUG_HOOKS
  // The extra rows the blocks wait for must lie inside the workspace's table,
  // which holds min(T, kCoopMaxBlocks) rows.
  if (B + g_debug_extra_rows_host > std::min(T, kCoopMaxBlocks)) return cudaErrorInvalidValue;
#endif
  unsigned* table = reinterpret_cast<unsigned*>(reinterpret_cast<char*>(hdr) + kWsHeaderBytes);
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(static_cast<unsigned>(B));
  cfg.blockDim = dim3(kRouteThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;  // all blocks co-resident (each waits for the others' table rows)
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, ids, emap, T, K, E, E_local, offsets, pidx, inv, hdr,
                            table, batch_capacity, expert_num_tokens);
}

template <typename VecT, int V>
cudaError_t launch_gather(const void* hidden, int64_t row_bytes, const float* scales,
                          int64_t scale_cols, const int32_t* inv, int64_t T, int K, void* out,
                          float* out_scales, int64_t num_out_rows, cudaStream_t s) {
  const int64_t row_vecs = row_bytes / static_cast<int64_t>(sizeof(VecT));
  const int64_t blocks = ceil_div(row_items(T, row_vecs, V), kRowWarps);
  if (blocks > INT32_MAX) return cudaErrorInvalidConfiguration;
  return launch(k_gather_rows<VecT, V>, static_cast<unsigned>(blocks), kRowThreads, 0, s,
                static_cast<const VecT*>(hidden), row_vecs, scales, scale_cols, inv, T, K,
                static_cast<VecT*>(out), out_scales, num_out_rows);
}

// Geometry of the bulk-copy gather for one row size.
struct TmaGeometry {
  int64_t chunk, pitch, grid;
  size_t smem;
  int64_t prefetch_bytes;  // source bytes the whole grid loads before routing ends
};

TmaGeometry tma_geometry(int64_t row_bytes, int64_t T, const DeviceInfo* d) {
  TmaGeometry g;
  g.chunk = std::min<int64_t>(row_bytes, kTmaChunkBytes);
  g.pitch = (g.chunk + 127) / 128 * 128;
  g.smem = static_cast<size_t>(kTmaWarps) * kTmaStages * (g.pitch + sizeof(uint64_t));
  const int64_t items = T * ceil_div(row_bytes, g.chunk);
  const int64_t per_sm = std::max<int64_t>(
      1, std::min<int64_t>(16, d->max_smem_per_sm / static_cast<int64_t>(g.smem + 1024)));
  g.grid = std::max<int64_t>(1, std::min(ceil_div(items, kTmaWarps), per_sm * d->sm_count));
  g.prefetch_bytes = g.grid * kTmaWarps * kTmaStages * g.chunk;
  return g;
}

// Bulk-copy gather (16-byte aligned rows): a persistent grid of warps, each
// with kTmaStages shared-memory stages of up to kTmaChunkBytes.  When a
// source row is written to 4 or more rows, the store phase dominates and the
// grid is trimmed so that every warp gets the same whole number of items:
// with one wave of warps at about 3.4 items each, the last round ran 40%
// full (measured on GB300: DeepSeek-V3 T = 4096 permute 50.5 -> 48.4 us).
// With fewer writes the full grid's larger early-load capacity matters more
// (Mixtral T = 4096: 18.3 us with it, 18.9 us trimmed).
cudaError_t launch_gather_tma(const void* hidden, int64_t row_bytes, const float* scales,
                              int64_t scale_cols, const int32_t* inv, int64_t T, int K,
                              double writes_per_row, void* out, float* out_scales,
                              int64_t num_out_rows, unsigned* status, const DeviceInfo* d,
                              cudaStream_t s) {
  TmaGeometry g = tma_geometry(row_bytes, T, d);
  if (writes_per_row >= 4.0) {
    const int64_t items = T * ceil_div(row_bytes, g.chunk);
    const int64_t per_warp = ceil_div(items, g.grid * kTmaWarps);
    g.grid = std::max<int64_t>(1, ceil_div(ceil_div(items, per_warp), kTmaWarps));
  }
  cudaError_t err = allow_smem(k_gather_rows_tma, g.smem);
  if (err != cudaSuccess) return err;
  return launch(k_gather_rows_tma, static_cast<unsigned>(g.grid), kTmaThreads, g.smem, s,
                static_cast<const char*>(hidden), row_bytes, g.chunk, g.pitch, scales, scale_cols,
                inv, T, K, static_cast<char*>(out), out_scales, num_out_rows, status);
}

// Expected rows written per source row: K, scaled by the kept share of the
// experts when an expert map drops some.
double writes_per_row(int K, int E, int E_local, const int32_t* emap) {
  return emap == nullptr ? static_cast<double>(K)
                         : static_cast<double>(K) * static_cast<double>(E_local) / E;
}

// Source bytes, as a multiple of the bulk-copy gather's prefetch, up to which
// it beats the register gather.  The bulk-copy gather loads most rows while
// routing runs, but its stores of each chunk come from one warp; the register
// gather keeps more stores in flight.  So the crossover falls as the rows
// written per source row grow: measured on GB300, about 2x at 1-2 writes per
// row, and at 8 about 1.05x for rows the register gather moves in whole
// 16-byte-vector chunks (a multiple of 32 * kGatherV vectors, e.g. 4 KB), but
// 1.25x for rows it splits raggedly (e.g. 7168 bytes: a 4 KB and a 3 KB
// chunk).  writes_per_row: K, or K * E_local / E with an expert map (uniform
// routing).
double tma_max_ratio(double writes_per_row, int64_t row_bytes) {
  const bool whole_chunks = row_bytes % (32 * kGatherV * 16) == 0;
  const double at8 = whole_chunks ? 1.05 : 1.25;
  return std::min(2.0, std::max(at8, 2.0 - (writes_per_row - 2.0) * (2.0 - at8) / 6.0));
}

// The row gather for any vector width: out rows are indexed by inv values in
// [0, num_out_rows).  16-byte aligned rows go through the bulk-copy engine
// when the source rows fit its prefetch well enough (tma_max_ratio); larger
// batches keep more loads in flight with the register gather.
cudaError_t launch_gather_any(size_t vb, const void* hidden, int64_t row_bytes,
                              const float* scales, int64_t scale_cols, const int32_t* inv,
                              int64_t T, int K, double writes_per_row, void* out,
                              float* out_scales, int64_t num_out_rows, unsigned* status,
                              const DeviceInfo* d, cudaStream_t s) {
  if (vb == 16 && static_cast<double>(T * row_bytes) <=
                      tma_max_ratio(writes_per_row, row_bytes) *
                          static_cast<double>(tma_geometry(row_bytes, T, d).prefetch_bytes))
    return launch_gather_tma(hidden, row_bytes, scales, scale_cols, inv, T, K, writes_per_row,
                             out, out_scales, num_out_rows, status, d, s);
  switch (vb) {
    case 16: return launch_gather<uint4, kGatherV>(hidden, row_bytes, scales, scale_cols, inv, T, K, out, out_scales, num_out_rows, s);
    case 8: return launch_gather<uint2, kGatherV>(hidden, row_bytes, scales, scale_cols, inv, T, K, out, out_scales, num_out_rows, s);
    case 4: return launch_gather<uint32_t, kGatherV>(hidden, row_bytes, scales, scale_cols, inv, T, K, out, out_scales, num_out_rows, s);
    case 2: return launch_gather<uint16_t, kGatherV>(hidden, row_bytes, scales, scale_cols, inv, T, K, out, out_scales, num_out_rows, s);
    default: return launch_gather<uint8_t, kGatherV>(hidden, row_bytes, scales, scale_cols, inv, T, K, out, out_scales, num_out_rows, s);
  }
}

// Stages in the single-launch permute's ring, at most.
constexpr int64_t kOpMaxStages = 1024;
static_assert(kOpMaxStages % kOpRouteWarps == 0, "stages come in multiples of the consumer warps");

// Geometry of the single-launch large-batch permute (k_permute_onepass).
struct OnepassPlan {
  bool ok = false;
  int64_t blocks = 0, tpb = 0, chunk = 0, pitch = 0;
  int J = 0, n_chunks = 0, n_stages = 0;
  size_t smem = 0;
};

OnepassPlan onepass_plan(int64_t T, int K, int E, int E_local, bool with_map, int64_t row_bytes,
                         const DeviceInfo* d) {
  OnepassPlan p;
  // One block per SM (or one per token when there are fewer tokens); each
  // block's rows must fit one ranking round of its 512 routing threads.
  int64_t B = std::min<int64_t>(d->sm_count, T);
  p.tpb = ceil_div(T, B);
  B = ceil_div(T, p.tpb);
  const int64_t rows = p.tpb * K;
  if (rows > static_cast<int64_t>(kOpRouteThreads) * 4) return p;
  p.J = rows <= static_cast<int64_t>(kOpRouteThreads) * 2 ? 2 : 4;
  p.blocks = B;
  p.n_chunks = static_cast<int>(ceil_div(row_bytes, kOpChunkBytes));
  p.chunk = ceil_div(ceil_div(row_bytes, p.n_chunks), 16) * 16;
  p.n_chunks = static_cast<int>(ceil_div(row_bytes, p.chunk));
  p.pitch = ceil_div(p.chunk, 128) * 128;
  const int64_t ints = (E_local + 1) + 3 * static_cast<int64_t>(E_local) +
                       static_cast<int64_t>(kOpRouteWarps) * E_local + rows + 2 * p.tpb +
                       (with_map ? E : 0);
  const int64_t int_bytes = ints * 4;
  const int64_t static_bytes = 1024;  // the kernel's static shared memory, rounded up
  const int64_t avail = static_cast<int64_t>(d->max_smem_optin) - int_bytes - static_bytes;
  const int64_t per_stage = p.pitch + 2 * static_cast<int64_t>(sizeof(uint64_t)) + 4;
  // A multiple of the 16 consumer warps (one consumer per stage), enough for
  // the block's items or as many as fit.
  const int64_t items = p.tpb * p.n_chunks;
  int64_t n = std::min<int64_t>(avail / per_stage, std::max<int64_t>(16, ceil_div(items, 16) * 16));
  n = std::min<int64_t>(n, kOpMaxStages) / kOpRouteWarps * kOpRouteWarps;
  if (n < kOpRouteWarps) return p;
  p.n_stages = static_cast<int>(n);
  p.smem = static_cast<size_t>(n * per_stage + int_bytes);
  p.ok = true;
  return p;
}

template <typename IdT>
cudaError_t launch_onepass(const OnepassPlan& g, const IdT* ids, const int32_t* emap, int64_t T,
                           int K, int E, int E_local, const void* hidden, int64_t row_bytes,
                           const float* scales, int64_t scale_cols, void* out, float* out_scales,
                           int64_t num_out_rows, int64_t* offsets, int32_t* pidx, int32_t* inv,
                           WsHeader* hdr, cudaStream_t s, int64_t M = 0,
                           int32_t* expert_num_tokens = nullptr) {
  auto kern = g.J == 2 ? k_permute_onepass<IdT, 2> : k_permute_onepass<IdT, 4>;
  cudaError_t err = allow_smem(kern, g.smem);
  if (err != cudaSuccess) return err;
#ifdef MOE_DEBUG_HOOKS
  if (g.blocks + g_debug_extra_rows_host > std::min(T, kCoopMaxBlocks)) return cudaErrorInvalidValue;
#endif
  unsigned* table = reinterpret_cast<unsigned*>(reinterpret_cast<char*>(hdr) + kWsHeaderBytes);
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(static_cast<unsigned>(g.blocks));
  cfg.blockDim = dim3(kOpThreads);
  cfg.dynamicSmemBytes = g.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;  // every block waits for the others' table rows
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, ids, emap, T, K, E, E_local,
                            static_cast<const char*>(hidden), row_bytes, g.chunk, g.n_chunks,
                            g.n_stages, g.pitch, scales, scale_cols, static_cast<char*>(out),
                            out_scales, num_out_rows, offsets, pidx, inv, hdr, table, M,
                            expert_num_tokens);
}

// Whether the single-launch large-batch permute serves this call: an expert
// map (it reads only the tokens that keep a row, which pays when the map
// drops most rows; without a map the two-kernel path measured faster),
// 16-byte aligned rows (bulk copies) and a plan that fits.
bool use_onepass(const int32_t* emap, size_t vb, const void* out, const OnepassPlan& g) {
  return emap != nullptr && out != nullptr && vb == 16 && g.ok;
}

template <typename IdT>
cudaError_t permute_typed(const IdT* ids, const int32_t* emap, int64_t T, int K, int E,
                          int E_local, const void* hidden, int64_t row_bytes, const float* scales,
                          int64_t scale_cols, void* out, float* out_scales, int64_t* offsets,
                          int32_t* pidx, int32_t* inv, void* ws, const DeviceInfo* d,
                          cudaStream_t s) {
  WsHeader* hdr = static_cast<WsHeader*>(ws);
  const int64_t R = T * K;
  const size_t vb = out == nullptr ? 16 : vec_bytes(row_bytes, hidden, out);
  if (R <= (out == nullptr ? kFusedMaxRows : fused_max_rows(emap))) {
    switch (vb) {
      case 16: return launch_fused<IdT, uint4, kFusedV>(ids, emap, T, K, E, E_local, hidden, row_bytes, scales, scale_cols, out, out_scales, offsets, pidx, inv, hdr, d, s);
      case 8: return launch_fused<IdT, uint2, kFusedV>(ids, emap, T, K, E, E_local, hidden, row_bytes, scales, scale_cols, out, out_scales, offsets, pidx, inv, hdr, d, s);
      case 4: return launch_fused<IdT, uint32_t, kFusedV>(ids, emap, T, K, E, E_local, hidden, row_bytes, scales, scale_cols, out, out_scales, offsets, pidx, inv, hdr, d, s);
      case 2: return launch_fused<IdT, uint16_t, kFusedV>(ids, emap, T, K, E, E_local, hidden, row_bytes, scales, scale_cols, out, out_scales, offsets, pidx, inv, hdr, d, s);
      default: return launch_fused<IdT, uint8_t, kFusedV>(ids, emap, T, K, E, E_local, hidden, row_bytes, scales, scale_cols, out, out_scales, offsets, pidx, inv, hdr, d, s);
    }
  }
  const OnepassPlan g = onepass_plan(T, K, E, E_local, emap != nullptr, row_bytes, d);
  if (use_onepass(emap, vb, out, g))
    return launch_onepass<IdT>(g, ids, emap, T, K, E, E_local, hidden, row_bytes, scales,
                               scale_cols, out, out_scales, R, offsets, pidx, inv, hdr, s);
  cudaError_t err = launch_route<IdT>(ids, emap, T, K, E, E_local, offsets, pidx, inv, hdr, d, s);
  if (err != cudaSuccess || out == nullptr) return err;
  return launch_gather_any(vb, hidden, row_bytes, scales, scale_cols, inv, T, K,
                           writes_per_row(K, E, E_local, emap), out, out_scales, R, &hdr->status,
                           d, s);
}

template <typename IdT>
cudaError_t permute_batched_typed(const IdT* ids, const int32_t* emap, int64_t T, int K, int E,
                                  int E_local, int64_t M, const void* hidden, int64_t row_bytes,
                                  const float* scales, int64_t scale_cols, void* out,
                                  float* out_scales, int32_t* counts, int32_t* inv, void* ws,
                                  const DeviceInfo* d, cudaStream_t s) {
  cudaError_t err = launch_route<IdT>(ids, emap, T, K, E, E_local, nullptr, nullptr, inv,
                                      static_cast<WsHeader*>(ws), d, s, M, counts);
  if (err != cudaSuccess || out == nullptr) return err;
  const size_t vb = vec_bytes(row_bytes, hidden, out);
  return launch_gather_any(vb, hidden, row_bytes, scales, scale_cols, inv, T, K,
                           writes_per_row(K, E, E_local, emap), out, out_scales,
                           static_cast<int64_t>(E_local) * M,
                           &static_cast<WsHeader*>(ws)->status, d, s);
}

constexpr int kQuantV = 2;  // vectors of 8 bf16 per lane in one quantise item (4 groups);
                            // measured 0.3-6% faster than 4 on GB300, 1 is 3-10% slower

template <typename IdT>
cudaError_t permute_quant_typed(const IdT* ids, const int32_t* emap, int64_t T, int K, int E,
                                int E_local, const void* hidden, int64_t H, void* codes,
                                float* scales, int64_t* offsets, int32_t* pidx, int32_t* inv,
                                void* ws, const DeviceInfo* d, cudaStream_t s) {
  if (T * K <= kFusedMaxRows)
    return launch_fused<IdT, uint4, kFusedQuantV, true>(ids, emap, T, K, E, E_local, hidden,
                                                        H * 2, nullptr, 0, codes, scales,
                                                        offsets, pidx, inv,
                                                        static_cast<WsHeader*>(ws), d, s);
  cudaError_t err = launch_route<IdT>(ids, emap, T, K, E, E_local, offsets, pidx, inv,
                                      static_cast<WsHeader*>(ws), d, s);
  if (err != cudaSuccess) return err;
  const int64_t row_vecs = H / 8;
  const int64_t blocks = ceil_div(row_items(T, row_vecs, kQuantV), kRowWarps);
  if (blocks > INT32_MAX) return cudaErrorInvalidConfiguration;
  if (aligned(codes, 16)) {
    // 16-byte code stores; float4 scale stores when every row's scales are
    // whole 16-byte groups of four
    if ((H / MOE_QUANT_GROUP) % 4 == 0 && aligned(scales, 16))
      return launch(k_gather_quant_fp8_wide<true>, static_cast<unsigned>(blocks), kRowThreads, 0,
                    s, static_cast<const uint4*>(hidden), row_vecs,
                    static_cast<const int32_t*>(inv), T, K, static_cast<uint4*>(codes), scales,
                    T * K);
    return launch(k_gather_quant_fp8_wide<false>, static_cast<unsigned>(blocks), kRowThreads, 0,
                  s, static_cast<const uint4*>(hidden), row_vecs, static_cast<const int32_t*>(inv),
                  T, K, static_cast<uint4*>(codes), scales, T * K);
  }
  return launch(k_gather_quant_fp8<kQuantV>, static_cast<unsigned>(blocks), kRowThreads, 0, s,
                static_cast<const uint4*>(hidden), row_vecs, static_cast<const int32_t*>(inv), T,
                K, static_cast<uint2*>(codes), scales, T * K);
}

template <typename VecT, int KG, int V>
cudaError_t launch_unpermute_kv(const void* rows, int64_t num_rows, int64_t H, const float* w,
                                const int32_t* inv, int64_t T, int K, void* out,
                                unsigned* status, const DeviceInfo* d, cudaStream_t s) {
  const int64_t row_vecs = H * 2 / static_cast<int64_t>(sizeof(VecT));
  auto kern = k_unpermute<VecT, KG, V>;
  const int64_t items = row_items(T, row_vecs, V);
  int per_sm = blocks_per_sm(reinterpret_cast<const void*>(kern), kRowThreads, 0);
  // A fourth block per SM adds loads in flight, which pays when a warp's
  // kept rows do not fill its KG * V vectors (K < 8: fewer rows per token,
  // or rows dropped by an expert map) or when there are few items per warp.
  // With K >= 8 dense rows and many items per warp it measured 1-3% slower
  // on GB300 (more streams competing for DRAM), so those keep three.
  if (per_sm > 3 && K >= 8 && items > 6 * static_cast<int64_t>(d->sm_count) * 3 * kRowWarps)
    per_sm = 3;
  unsigned grid = item_grid(items, kRowWarps, d, per_sm);
  // With 8 or more rows per token, one item per warp over as many blocks as
  // the items need: the block scheduler then balances the last wave, and every
  // SM holds as many blocks as fit.  Measured on GB300: DeepSeek-V3 T = 4096
  // 81.3 -> 79.7 us, T = 32768 616 -> 605 us, Qwen3 T = 8192 46.9 -> 46.4 us;
  // for K = 2 and 6 the persistent grid stays ahead (Mixtral T = 16384 60.8 us
  // against 64.6, DeepSeek-V2-Lite T = 8192 15.6 against 16.8).
  if (K >= 8 && ceil_div(items, kRowWarps) <= INT32_MAX)
    grid = static_cast<unsigned>(std::max<int64_t>(1, ceil_div(items, kRowWarps)));
  return launch(kern, grid, kRowThreads, 0, s, static_cast<const VecT*>(rows), num_rows, row_vecs,
                w, inv, T, K, static_cast<VecT*>(out), status);
}

// Rows whose loads are in flight together (KG) times vectors per lane (V):
// about 8 vectors per lane for any K.
template <typename VecT>
cudaError_t launch_unpermute(const void* rows, int64_t num_rows, int64_t H, const float* w,
                             const int32_t* inv, int64_t T, int K, void* out, unsigned* status,
                             const DeviceInfo* d, cudaStream_t s) {
  if (K == 1)
    return launch_unpermute_kv<VecT, 1, 8>(rows, num_rows, H, w, inv, T, K, out, status, d, s);
  if (K == 2)
    return launch_unpermute_kv<VecT, 2, 4>(rows, num_rows, H, w, inv, T, K, out, status, d, s);
  return launch_unpermute_kv<VecT, 4, 2>(rows, num_rows, H, w, inv, T, K, out, status, d, s);
}

int elem_bytes(moe_dtype_t dt) {
  switch (dt) {
    case MOE_DTYPE_BF16:
    case MOE_DTYPE_FP16: return 2;
    case MOE_DTYPE_FP8_E4M3:
    case MOE_DTYPE_FP8_E5M2: return 1;
    case MOE_DTYPE_FP32: return 4;
    default: return 0;
  }
}

// Host checks of moe_permute's arguments, before anything touches a device.
// check_workspace_ptr: false when the caller supplies the scratch itself
// (moe_permute_noalloc); workspace_bytes is then the scratch's size.
int permute_args_status(const void* hidden_states, moe_dtype_t hidden_dtype,
                        const float* hidden_scales, int64_t scale_cols, const void* topk_ids,
                        moe_index_t topk_ids_dtype, const int32_t* expert_map, int64_t T,
                        int64_t H, int32_t topk, int32_t num_experts, int32_t num_local_experts,
                        const void* permuted_hidden_states, const float* permuted_scales,
                        const int64_t* expert_first_token_offset, const int32_t* permuted_idx,
                        const int32_t* inv_permuted_idx, bool check_workspace_ptr,
                        const void* workspace, size_t workspace_bytes) {
  const int eb = elem_bytes(hidden_dtype);
  if (eb == 0 || T < 0 || H < 1 || topk < 1 || topk > MOE_MAX_TOPK || num_experts < 1 ||
      num_local_experts < 1 || num_local_experts > num_experts ||
      num_local_experts > MOE_MAX_LOCAL_EXPERTS)
    return MOE_ERR_INVALID_ARG;
  if (expert_map == nullptr && num_local_experts != num_experts) return MOE_ERR_INVALID_ARG;
  if (topk_ids_dtype != MOE_INDEX_INT32 && topk_ids_dtype != MOE_INDEX_INT64)
    return MOE_ERR_INVALID_ARG;
  if (T > INT32_MAX / topk) return MOE_ERR_INVALID_ARG;
  if (H > INT64_MAX / 16 / eb) return MOE_ERR_INVALID_ARG;
  if (expert_first_token_offset == nullptr || !aligned(expert_first_token_offset, 8))
    return MOE_ERR_INVALID_ARG;
  if (scale_cols < 0) return MOE_ERR_INVALID_ARG;
  // With T = 0 only the offsets are written; empty tensors may come as NULL.
  if (T == 0) return MOE_OK;
  const size_t id_bytes = topk_ids_dtype == MOE_INDEX_INT64 ? 8 : 4;
  if (topk_ids == nullptr || !aligned(topk_ids, id_bytes)) return MOE_ERR_INVALID_ARG;
  if (expert_map != nullptr && !aligned(expert_map, 4)) return MOE_ERR_INVALID_ARG;
  if (permuted_idx == nullptr || inv_permuted_idx == nullptr || !aligned(permuted_idx, 4) ||
      !aligned(inv_permuted_idx, 4))
    return MOE_ERR_INVALID_ARG;
  if (permuted_hidden_states != nullptr && hidden_states == nullptr) return MOE_ERR_INVALID_ARG;
  const bool with_scales = hidden_scales != nullptr || permuted_scales != nullptr;
  if (with_scales) {
    if (hidden_scales == nullptr || permuted_scales == nullptr || scale_cols < 1 ||
        permuted_hidden_states == nullptr || !aligned(hidden_scales, 4) ||
        !aligned(permuted_scales, 4))
      return MOE_ERR_INVALID_ARG;
  } else if (scale_cols != 0) {
    return MOE_ERR_INVALID_ARG;
  }
  if (check_workspace_ptr && (workspace == nullptr || !aligned(workspace, 256)))
    return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < workspace_bytes_for(T, topk, num_experts))
    return MOE_ERR_WORKSPACE_TOO_SMALL;
  return MOE_OK;
}

// Copy of the status word for moe_permute_read_status: one thread, so that
// the destination may be device memory or pinned host memory, and the read
// (and the optional clear) stay ordered in the stream like any kernel.
__global__ void k_copy_status(unsigned* __restrict__ status, uint32_t* __restrict__ dst,
                              int clear) {
  pdl_wait();
  if (threadIdx.x == 0) {
    *dst = *status;
    if (clear) *status = 0u;
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_permute_supported(int device) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return (major == 10 && minor == 3) ? 1 : 0;
}

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs sm_103)";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
  }
}

size_t moe_permute_workspace_size(int64_t max_tokens, int32_t topk, int32_t num_experts) {
  if (max_tokens < 0 || topk < 1 || topk > MOE_MAX_TOPK || num_experts < 1) return 0;
  if (max_tokens > INT32_MAX / topk) return 0;
  return workspace_bytes_for(max_tokens, topk, num_experts);
}

int moe_permute_workspace_init(void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < kWsHeaderBytes)
    return MOE_ERR_INVALID_ARG;
  if (!is_supported(current_device())) return MOE_ERR_UNSUPPORTED_DEVICE;
  if (cudaMemsetAsync(workspace, 0, workspace_bytes, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_permute(const void* hidden_states, moe_dtype_t hidden_dtype, const float* hidden_scales,
                int64_t scale_cols, const void* topk_ids, moe_index_t topk_ids_dtype,
                const int32_t* expert_map, int64_t num_tokens, int64_t hidden_size, int32_t topk,
                int32_t num_experts, int32_t num_local_experts, void* permuted_hidden_states,
                float* permuted_scales, int64_t* expert_first_token_offset, int32_t* permuted_idx,
                int32_t* inv_permuted_idx, void* workspace, size_t workspace_bytes,
                moe_stream_t stream) {
  const int rc = permute_args_status(hidden_states, hidden_dtype, hidden_scales, scale_cols,
                                     topk_ids, topk_ids_dtype, expert_map, num_tokens,
                                     hidden_size, topk, num_experts, num_local_experts,
                                     permuted_hidden_states, permuted_scales,
                                     expert_first_token_offset, permuted_idx, inv_permuted_idx,
                                     /*check_workspace_ptr=*/true, workspace, workspace_bytes);
  if (rc != MOE_OK) return rc;
  const DeviceInfo* d = current_device();
  if (!is_supported(d)) return MOE_ERR_UNSUPPORTED_DEVICE;

  const int64_t T = num_tokens, H = hidden_size;
  const int eb = elem_bytes(hidden_dtype);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (T == 0) {
    err = launch(k_zero_offsets, 1, 256, 0, s, expert_first_token_offset, num_local_experts + 1);
  } else if (topk_ids_dtype == MOE_INDEX_INT32) {
    err = permute_typed<int32_t>(static_cast<const int32_t*>(topk_ids), expert_map, T, topk,
                                 num_experts, num_local_experts, hidden_states, H * eb,
                                 hidden_scales, scale_cols, permuted_hidden_states,
                                 permuted_scales, expert_first_token_offset, permuted_idx,
                                 inv_permuted_idx, workspace, d, s);
  } else {
    err = permute_typed<int64_t>(static_cast<const int64_t*>(topk_ids), expert_map, T, topk,
                                 num_experts, num_local_experts, hidden_states, H * eb,
                                 hidden_scales, scale_cols, permuted_hidden_states,
                                 permuted_scales, expert_first_token_offset, permuted_idx,
                                 inv_permuted_idx, workspace, d, s);
  }
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_permute_quant_fp8(const void* hidden_states, const void* topk_ids,
                          moe_index_t topk_ids_dtype, const int32_t* expert_map,
                          int64_t num_tokens, int64_t hidden_size, int32_t topk,
                          int32_t num_experts, int32_t num_local_experts, void* permuted_codes,
                          float* permuted_scales, int64_t* expert_first_token_offset,
                          int32_t* permuted_idx, int32_t* inv_permuted_idx, void* workspace,
                          size_t workspace_bytes, moe_stream_t stream) {
  const int64_t T = num_tokens, H = hidden_size;
  if (T < 0 || H < MOE_QUANT_GROUP || H % MOE_QUANT_GROUP != 0 || topk < 1 ||
      topk > MOE_MAX_TOPK || num_experts < 1 || num_local_experts < 1 ||
      num_local_experts > num_experts || num_local_experts > MOE_MAX_LOCAL_EXPERTS)
    return MOE_ERR_INVALID_ARG;
  if (expert_map == nullptr && num_local_experts != num_experts) return MOE_ERR_INVALID_ARG;
  if (topk_ids_dtype != MOE_INDEX_INT32 && topk_ids_dtype != MOE_INDEX_INT64)
    return MOE_ERR_INVALID_ARG;
  if (T > INT32_MAX / topk || H > INT64_MAX / 64) return MOE_ERR_INVALID_ARG;
  if (expert_first_token_offset == nullptr || !aligned(expert_first_token_offset, 8))
    return MOE_ERR_INVALID_ARG;
  if (T > 0) {
    const size_t id_bytes = topk_ids_dtype == MOE_INDEX_INT64 ? 8 : 4;
    if (topk_ids == nullptr || !aligned(topk_ids, id_bytes)) return MOE_ERR_INVALID_ARG;
    if (expert_map != nullptr && !aligned(expert_map, 4)) return MOE_ERR_INVALID_ARG;
    if (permuted_idx == nullptr || inv_permuted_idx == nullptr || !aligned(permuted_idx, 4) ||
        !aligned(inv_permuted_idx, 4))
      return MOE_ERR_INVALID_ARG;
    if (hidden_states == nullptr || !aligned(hidden_states, 16) || permuted_codes == nullptr ||
        !aligned(permuted_codes, 8) || permuted_scales == nullptr || !aligned(permuted_scales, 4))
      return MOE_ERR_INVALID_ARG;
    if (workspace == nullptr || !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < workspace_bytes_for(T, topk, num_experts))
      return MOE_ERR_WORKSPACE_TOO_SMALL;
  }
  const DeviceInfo* d = current_device();
  if (!is_supported(d)) return MOE_ERR_UNSUPPORTED_DEVICE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (T == 0) {
    err = launch(k_zero_offsets, 1, 256, 0, s, expert_first_token_offset, num_local_experts + 1);
  } else if (topk_ids_dtype == MOE_INDEX_INT32) {
    err = permute_quant_typed<int32_t>(static_cast<const int32_t*>(topk_ids), expert_map, T, topk,
                                       num_experts, num_local_experts, hidden_states, H,
                                       permuted_codes, permuted_scales, expert_first_token_offset,
                                       permuted_idx, inv_permuted_idx, workspace, d, s);
  } else {
    err = permute_quant_typed<int64_t>(static_cast<const int64_t*>(topk_ids), expert_map, T, topk,
                                       num_experts, num_local_experts, hidden_states, H,
                                       permuted_codes, permuted_scales, expert_first_token_offset,
                                       permuted_idx, inv_permuted_idx, workspace, d, s);
  }
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_permute_batched(const void* hidden_states, moe_dtype_t hidden_dtype,
                        const float* hidden_scales, int64_t scale_cols, const void* topk_ids,
                        moe_index_t topk_ids_dtype, const int32_t* expert_map,
                        int64_t num_tokens, int64_t hidden_size, int32_t topk,
                        int32_t num_experts, int32_t num_local_experts,
                        int64_t max_rows_per_expert, void* batched_hidden_states,
                        float* batched_scales, int32_t* expert_num_tokens,
                        int32_t* inv_permuted_idx, void* workspace, size_t workspace_bytes,
                        moe_stream_t stream) {
  const int eb = elem_bytes(hidden_dtype);
  const int64_t T = num_tokens, H = hidden_size, M = max_rows_per_expert;
  if (eb == 0 || T < 0 || H < 1 || topk < 1 || topk > MOE_MAX_TOPK || num_experts < 1 ||
      num_local_experts < 1 || num_local_experts > num_experts ||
      num_local_experts > MOE_MAX_LOCAL_EXPERTS || M < 1 || M > INT32_MAX / num_local_experts)
    return MOE_ERR_INVALID_ARG;
  if (expert_map == nullptr && num_local_experts != num_experts) return MOE_ERR_INVALID_ARG;
  if (topk_ids_dtype != MOE_INDEX_INT32 && topk_ids_dtype != MOE_INDEX_INT64)
    return MOE_ERR_INVALID_ARG;
  if (T > INT32_MAX / topk || H > INT64_MAX / 16 / eb || scale_cols < 0) return MOE_ERR_INVALID_ARG;
  if (expert_num_tokens == nullptr || !aligned(expert_num_tokens, 4)) return MOE_ERR_INVALID_ARG;
  if (T > 0) {
    const size_t id_bytes = topk_ids_dtype == MOE_INDEX_INT64 ? 8 : 4;
    if (topk_ids == nullptr || !aligned(topk_ids, id_bytes)) return MOE_ERR_INVALID_ARG;
    if (expert_map != nullptr && !aligned(expert_map, 4)) return MOE_ERR_INVALID_ARG;
    if (inv_permuted_idx == nullptr || !aligned(inv_permuted_idx, 4)) return MOE_ERR_INVALID_ARG;
    if (batched_hidden_states != nullptr && hidden_states == nullptr) return MOE_ERR_INVALID_ARG;
    const bool with_scales = hidden_scales != nullptr || batched_scales != nullptr;
    if (with_scales) {
      if (hidden_scales == nullptr || batched_scales == nullptr || scale_cols < 1 ||
          batched_hidden_states == nullptr || !aligned(hidden_scales, 4) ||
          !aligned(batched_scales, 4))
        return MOE_ERR_INVALID_ARG;
    } else if (scale_cols != 0) {
      return MOE_ERR_INVALID_ARG;
    }
    if (workspace == nullptr || !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < workspace_bytes_for(T, topk, num_experts))
      return MOE_ERR_WORKSPACE_TOO_SMALL;
  }
  const DeviceInfo* d = current_device();
  if (!is_supported(d)) return MOE_ERR_UNSUPPORTED_DEVICE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (T == 0) {
    err = cudaMemsetAsync(expert_num_tokens, 0, sizeof(int32_t) * num_local_experts, s);
  } else if (topk_ids_dtype == MOE_INDEX_INT32) {
    err = permute_batched_typed<int32_t>(static_cast<const int32_t*>(topk_ids), expert_map, T,
                                         topk, num_experts, num_local_experts, M, hidden_states,
                                         H * eb, hidden_scales, scale_cols, batched_hidden_states,
                                         batched_scales, expert_num_tokens, inv_permuted_idx,
                                         workspace, d, s);
  } else {
    err = permute_batched_typed<int64_t>(static_cast<const int64_t*>(topk_ids), expert_map, T,
                                         topk, num_experts, num_local_experts, M, hidden_states,
                                         H * eb, hidden_scales, scale_cols, batched_hidden_states,
                                         batched_scales, expert_num_tokens, inv_permuted_idx,
                                         workspace, d, s);
  }
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_unpermute(const void* permuted_rows, int64_t num_rows, const float* topk_weights,
                  const int32_t* inv_permuted_idx, int64_t num_tokens, int64_t hidden_size,
                  int32_t topk, void* out, void* workspace, moe_stream_t stream) {
  const int64_t T = num_tokens, H = hidden_size;
  if (T < 0 || H < 1 || topk < 1 || topk > MOE_MAX_TOPK || num_rows < 0) return MOE_ERR_INVALID_ARG;
  if (T > INT32_MAX / topk || num_rows > INT32_MAX || H > INT64_MAX / 32)
    return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (permuted_rows == nullptr && num_rows > 0) return MOE_ERR_INVALID_ARG;
  if (topk_weights == nullptr || inv_permuted_idx == nullptr || out == nullptr ||
      !aligned(topk_weights, 4) || !aligned(inv_permuted_idx, 4) || !aligned(out, 2) ||
      (permuted_rows != nullptr && !aligned(permuted_rows, 2)))
    return MOE_ERR_INVALID_ARG;
  if (workspace != nullptr && !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
  const DeviceInfo* d = current_device();
  if (!is_supported(d)) return MOE_ERR_UNSUPPORTED_DEVICE;
  unsigned* status = workspace != nullptr ? &static_cast<WsHeader*>(workspace)->status : nullptr;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t vb = vec_bytes(H * 2, permuted_rows != nullptr ? permuted_rows : out, out);
  cudaError_t err;
  switch (vb) {
    case 16: err = launch_unpermute<uint4>(permuted_rows, num_rows, H, topk_weights, inv_permuted_idx, T, topk, out, status, d, s); break;
    case 8: err = launch_unpermute<uint2>(permuted_rows, num_rows, H, topk_weights, inv_permuted_idx, T, topk, out, status, d, s); break;
    case 4: err = launch_unpermute<uint32_t>(permuted_rows, num_rows, H, topk_weights, inv_permuted_idx, T, topk, out, status, d, s); break;
    default: err = launch_unpermute<uint16_t>(permuted_rows, num_rows, H, topk_weights, inv_permuted_idx, T, topk, out, status, d, s); break;
  }
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_read_status(const void* workspace, uint32_t* host_status, moe_stream_t stream) {
  if (workspace == nullptr || host_status == nullptr || !aligned(workspace, 256))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const void* src = &static_cast<const WsHeader*>(workspace)->status;
  if (cudaMemcpyAsync(host_status, src, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_clear_status(void* workspace, moe_stream_t stream) {
  if (workspace == nullptr || !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
  void* dst = &static_cast<WsHeader*>(workspace)->status;
  if (cudaMemsetAsync(dst, 0, sizeof(uint32_t), reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_permute_read_status(void* workspace, uint32_t* dst, int clear_after_read,
                            moe_stream_t stream) {
  if (workspace == nullptr || dst == nullptr || !aligned(workspace, 256) || !aligned(dst, 4))
    return MOE_ERR_INVALID_ARG;
  // The kernel writes through dst, so it must be memory the device can
  // reach: device (or managed) memory, or page-locked host memory.
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, dst) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_INVALID_ARG;
  }
  if (a.type == cudaMemoryTypeUnregistered) return MOE_ERR_INVALID_ARG;
  if (!is_supported(current_device())) return MOE_ERR_UNSUPPORTED_DEVICE;
  unsigned* status = &static_cast<WsHeader*>(workspace)->status;
  const cudaError_t err = launch(k_copy_status, 1, 32, 0, reinterpret_cast<cudaStream_t>(stream),
                                 status, dst, clear_after_read != 0 ? 1 : 0);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"

// ---- allocation-free variant of moe_permute ------------------------------
// The scratch of moe_permute_noalloc: a file-scope device array, one per GPU
// that loads this library.  Host code must never use its name as an address
// (on the host it names a stand-in, not device memory): the device address
// is looked up once per device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {nullptr};
}  // namespace

extern "C" int moe_permute_noalloc(const void* hidden_states, moe_dtype_t hidden_dtype,
                                   const float* hidden_scales, int64_t scale_cols,
                                   const void* topk_ids, moe_index_t topk_ids_dtype,
                                   const int32_t* expert_map, int64_t num_tokens,
                                   int64_t hidden_size, int32_t topk, int32_t num_experts,
                                   int32_t num_local_experts, void* permuted_hidden_states,
                                   float* permuted_scales, int64_t* expert_first_token_offset,
                                   int32_t* permuted_idx, int32_t* inv_permuted_idx,
                                   moe_stream_t stream) {
  // moe_permute's own argument checks first, with the static array standing
  // in for the workspace: a request it cannot hold is
  // MOE_ERR_WORKSPACE_TOO_SMALL, decided before any device is touched.
  const int rc = permute_args_status(hidden_states, hidden_dtype, hidden_scales, scale_cols,
                                     topk_ids, topk_ids_dtype, expert_map, num_tokens,
                                     hidden_size, topk, num_experts, num_local_experts,
                                     permuted_hidden_states, permuted_scales,
                                     expert_first_token_offset, permuted_idx, inv_permuted_idx,
                                     /*check_workspace_ptr=*/false, nullptr,
                                     MOE_NOALLOC_SCRATCH_BYTES);
  if (rc != MOE_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
      // set-up, once per device, with that device current
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
      }
      if (cudaMemsetAsync(ptr, 0, MOE_NOALLOC_SCRATCH_BYTES,
                          reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
      }
      g_noalloc_ptr[dev] = ptr;
    }
    scratch = g_noalloc_ptr[dev];
  }
  return moe_permute(hidden_states, hidden_dtype, hidden_scales, scale_cols, topk_ids,
                     topk_ids_dtype, expert_map, num_tokens, hidden_size, topk, num_experts,
                     num_local_experts, permuted_hidden_states, permuted_scales,
                     expert_first_token_offset, permuted_idx, inv_permuted_idx, scratch,
                     MOE_NOALLOC_SCRATCH_BYTES, stream);
}

#ifdef MOE_DEBUG_HOOKS
namespace moe {
namespace {
// Every pair (x, amax) of finite bf16 bit patterns, amax > 0, |x| <= amax:
// div_by_scale against __fdiv_rn (moe_debug_check_quant_division).
__device__ unsigned long long g_div_counts[4];

__global__ void k_check_quant_division() {
  unsigned long long checked = 0, code_diff = 0, quot_diff = 0, outside = 0;
  const uint64_t n = 1ull << 32;
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
    const uint32_t ab = static_cast<uint32_t>(i >> 16), xb = static_cast<uint32_t>(i & 0xffffu);
    if ((ab & 0x8000u) != 0u || (ab & 0x7f80u) == 0x7f80u || (xb & 0x7f80u) == 0x7f80u) continue;
    const float amax = __uint_as_float(ab << 16), x = __uint_as_float(xb << 16);
    if (!(amax > 0.0f) || !(fabsf(x) <= amax)) continue;
    ++checked;
    const float s = __fdiv_rn(amax, kE4m3Max);
    const float qa = __fdiv_rn(x, s);
    float qb = qa;
    if (scale_in_range(s)) qb = div_by_scale(x, s, __frcp_rn(s));
    else ++outside;
    const unsigned short ca = __nv_cvt_float2_to_fp8x2(make_float2(qa, 0.f), __NV_SATFINITE, __NV_E4M3);
    const unsigned short cb = __nv_cvt_float2_to_fp8x2(make_float2(qb, 0.f), __NV_SATFINITE, __NV_E4M3);
    code_diff += ca != cb;
    quot_diff += __float_as_uint(qa) != __float_as_uint(qb) && fabsf(qa) >= 0x1p-12f;
  }
  atomicAdd(&g_div_counts[0], checked);
  atomicAdd(&g_div_counts[1], code_diff);
  atomicAdd(&g_div_counts[2], quot_diff);
  atomicAdd(&g_div_counts[3], outside);
}
}  // namespace
}  // namespace moe

extern "C" int moe_debug_check_quant_division(unsigned long long* counts) {
  if (counts == nullptr) return MOE_ERR_INVALID_ARG;
  const unsigned long long zero[4] = {0, 0, 0, 0};
  if (cudaMemcpyToSymbol(moe::g_div_counts, zero, sizeof zero) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  moe::k_check_quant_division<<<1216, 256>>>();
  if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpyFromSymbol(counts, moe::g_div_counts, sizeof zero) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

extern "C" int moe_debug_set_table_wait(int extra_rows, unsigned long long wait_ns) {
  if (extra_rows < 0 || extra_rows > MOE_DEBUG_MAX_EXTRA_ROWS || wait_ns == 0)
    return MOE_ERR_INVALID_ARG;
  if (cudaMemcpyToSymbol(moe::g_debug_extra_rows, &extra_rows, sizeof(extra_rows)) !=
          cudaSuccess ||
      cudaMemcpyToSymbol(moe::g_debug_table_wait_ns, &wait_ns, sizeof(wait_ns)) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  moe::g_debug_extra_rows_host = extra_rows;
  return MOE_OK;
}
#endif
