// Shared device/host definitions of the int8 paged-KV verify-attention library.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <mutex>

#include "splash_kv.h"

namespace splash {

constexpr int kPageSize = 16;
constexpr int kClassTensor = 0;   // sequences whose T*G rows go to the tensor-core kernel
constexpr int kClassSimt = 1;     // sequences whose rows go to the CUDA-core kernel
constexpr int kNumClasses = 2;
constexpr int kMaxRows = 128;     // T*G limit per sequence and KV head
// Automatic routing: units with at least this many query rows go to the
// tensor-core kernel. Its cost per key tile does not depend on the row count
// (rows are padded to 128), and measured on a ragged batch (T in {1,4,8,16},
// G = 6) it beats the CUDA-core kernel even at T*G = 6, so every unit goes
// there when a tensor-core kernel exists for the head size.
constexpr int kTensorMinRows = 1;

// Split of a class's tile stream over its CTAs by estimated cost, not by tile
// count (a CTA's range is [cta_start[c], cta_start[c+1])). Cost of one tile of
// a unit with R query rows: tile_cost + R * row_cost; every unit adds
// segment_cost for the pipeline fill / drain of a segment. Measured on the
// tensor-core kernel (64-key tiles, ragged T in {1, 4, 8, 16}, G = 6): a tile
// costs 1.22 us at R = 6 and 1.37 us at R = 96, a segment start ~7.5 us.
constexpr int kMaxCtas = 1023;                 // per class (starts fit one 1024-thread scan)
__host__ __device__ constexpr long long tile_cost(int cls) { return cls == kClassTensor ? 4096 : 1024; }
__host__ __device__ constexpr long long row_cost(int cls) { return cls == kClassTensor ? 6 : 256; }
__host__ __device__ constexpr long long segment_cost(int cls) { return cls == kClassTensor ? 6 * 4096 : 4096; }

// Plan written by the planner kernel at the start of the workspace.
struct PlanHeader {
  int total_tiles[kNumClasses];   // key tiles of all (seq, KV head) units of a class
  int ncta[kNumClasses];          // CTAs of the class's kernel that own tiles: min(launched, tiles);
                                  // CTAs with blockIdx.x >= ncta exit at once
  int tile_keys[kNumClasses];     // keys per tile
  int num_seqs;
  int num_kv_heads;
  int group;                      // G = Hq / Hkv
  int total_part_rows;            // partial rows the split units use
  int rows_bound;                 // capacity of the partial buffers (rows)
  int window;                     // sliding window W (0: none)
  int pad_[4];
};
static_assert(sizeof(PlanHeader) == 64, "header size");

// Code pool layout: one allocation [num_pages][Hkv][2][kPageSize][D] int8;
// the (page, KV head) block holds the K codes of its 16 slots followed by
// the V codes, so v_pages = k_pages + kPageSize * D and consecutive blocks are
// 2 * kPageSize * D bytes apart (one 8 KB bulk copy stages both at D = 256).
// Byte offset of slot `slot` of block (page, h) from k_pages (or v_pages):
__host__ __device__ inline size_t code_offset(int page, int h, int num_kv_heads, int slot, int D) {
  return (((size_t)page * num_kv_heads + h) * 2 * kPageSize + slot) * D;
}

// First key a unit (context ctx) needs: with a sliding window W > 0, verify
// token t sees keys ctx + t - W < j <= ctx + t, so no row sees a key below
// ctx - W + 1; tiles wholly below it are skipped and their pages never read.
__host__ __device__ inline int unit_first_key(int ctx, int window) {
  return window > 0 ? (ctx - window + 1 > 0 ? ctx - window + 1 : 0) : 0;
}
// Key tiles of a unit: [first, first + count) of tile_keys keys each.
__host__ __device__ inline int unit_first_tile(int ctx, int window, int tile_keys) {
  return unit_first_key(ctx, window) / tile_keys;
}
__host__ __device__ inline int unit_tiles(int ctx, int T, int window, int tile_keys) {
  return (ctx + T + tile_keys - 1) / tile_keys - unit_first_tile(ctx, window, tile_keys);
}

// Byte offsets of the workspace regions (all 256-aligned).
struct WorkspaceLayout {
  size_t q_off;        // int32 [B+1]   first token row of each sequence
  size_t seq_T;        // int32 [B]     validated block length (0 if skipped)
  size_t seq_ctx;      // int32 [B]
  size_t seq_class;    // int32 [B]     kClassTensor / kClassSimt / -1
  size_t stp;          // int32 [2][B+1] per-class exclusive prefix of tiles per sequence
  size_t nseg;         // int32 [B*Hkv] CTAs (segments) that cover the unit
  size_t cfirst;       // int32 [B*Hkv] first CTA of the unit
  size_t part_base;    // int32 [B*Hkv] first partial row of the unit
  size_t wcost;        // int64 [2][B+1] per-class exclusive prefix of sequence costs
  size_t cta_start;    // int32 [2][kMaxCtas+1] first tile of each CTA, per class
  size_t o_part;       // fp32  [rows_bound, D]
  size_t lse_part;     // fp32  [rows_bound]
  size_t total;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ inline WorkspaceLayout make_layout(int B, int Hkv, int D, long long rows_bound) {
  WorkspaceLayout L;
  size_t o = align256(sizeof(PlanHeader));
  L.q_off = o;      o = align256(o + sizeof(int) * (size_t)(B + 1));
  L.seq_T = o;      o = align256(o + sizeof(int) * (size_t)B);
  L.seq_ctx = o;    o = align256(o + sizeof(int) * (size_t)B);
  L.seq_class = o;  o = align256(o + sizeof(int) * (size_t)B);
  L.stp = o;        o = align256(o + sizeof(int) * (size_t)kNumClasses * (B + 1));
  L.nseg = o;       o = align256(o + sizeof(int) * (size_t)B * Hkv);
  L.cfirst = o;     o = align256(o + sizeof(int) * (size_t)B * Hkv);
  L.part_base = o;  o = align256(o + sizeof(int) * (size_t)B * Hkv);
  L.wcost = o;      o = align256(o + sizeof(long long) * (size_t)kNumClasses * (B + 1));
  L.cta_start = o;  o = align256(o + sizeof(int) * (size_t)kNumClasses * (kMaxCtas + 1));
  L.o_part = o;     o = align256(o + sizeof(float) * (size_t)rows_bound * D);
  L.lse_part = o;   o = align256(o + sizeof(float) * (size_t)rows_bound);
  L.total = o;
  return L;
}


struct AttnParams {
  const __nv_bfloat16* q;
  const int8_t* k_pages;
  const int8_t* v_pages;
  const float* k_scales;
  const float* v_scales;
  const int32_t* page_table;
  int max_pages_per_seq;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int group;
  int head_dim;
  int num_pages;
  float sm_scale_log2;            // sm_scale * log2(e)
  int window;                     // sliding window W (0: none); the planner has the same value
  unsigned long long wait_ns;     // limit of each pipeline wait of the tensor-core kernel
  __nv_bfloat16* out;
  float* lse;
  unsigned char* ws;
  int* device_status;
};

// Programmatic dependent launch: a kernel launched with launch_dependent()
// may start while the kernel before it on the stream is still running; it
// calls grid_dependency_wait() before it reads anything that kernel wrote
// (a no-op for a kernel launched the ordinary way). allow_dependent_launch()
// lets the next such kernel be scheduled early.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Raises kernel K's dynamic shared-memory limit to `bytes` on the current
// device, calling the driver only the first time (and when a larger size is
// asked for): the attribute is per device and persists, and one driver call
// per launch would be host time on every call.
template <auto K>
inline cudaError_t ensure_dynamic_smem(int bytes) {
  static std::mutex mu;
  static int set_to[64] = {0};        // largest size set so far, per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64)
    return cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  std::lock_guard<std::mutex> lock(mu);
  if (set_to[dev] >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) set_to[dev] = bytes;
  return e;
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

__device__ inline void report(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ inline float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ inline float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Largest index i in [0, n] with a[i] <= x, for a non-decreasing array a[0..n].
template <typename V>
__device__ inline int upper_index(const V* a, int n, V x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (a[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace splash
