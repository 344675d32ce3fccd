// Tensor-core verify attention for sm_103a (tcgen05 + TMEM).
//
// One persistent CTA per SM walks its share of the tensor-core class's tile
// stream (64 keys per tile). For a unit (sequence b, KV head h) the R = T*G
// query rows (row r = t*G + g, padded to M = 128) sit in tensor memory as the
// A operand; each int8 K/V tile is read from its pages once and serves all R
// rows (the reuse across query heads and verify tokens):
//
//   S  = Q' . C_K^T            tcgen05.mma kind::f16, A = Q' (TMEM), B = K tile (SMEM)
//   s' = S * sK_j  ;  p = exp2(f_r * (s' - m_r))   (f_r = sm_scale*log2e / 2^e_r)
//   O += (p * sV_j) . C_V      tcgen05.mma kind::f16, A = P (TMEM), B = V tile (SMEM)
//
// Q' = Q * 2^e_r per row, e_r chosen so max|Q'| is in [2^14, 2^15): an exact
// power-of-two rescale that lets bf16 Q enter the fp16 MMA exactly (int8 codes
// are exact in fp16). The K scale multiplies score columns, the V scale is
// folded into P before P is rounded to fp16.
//
// Warp roles (512 threads):
//   warps 0-7   softmax + epilogue: warp w owns TMEM lanes 32(w%4) + 16(w/4)
//               .. +15; with the 16x256b load shape each lane's row is spread
//               over 4 threads (2 rows per thread, row reductions = 2
//               shuffles). A unit's R rows are spread evenly over the four
//               lane quarters (row q*ceil(R/4) + i in lane 32q + i), so each
//               SM sub-partition's softmax warps carry a quarter of them.
//   warps 8-11  converters: int8 codes from the staging ring -> fp16 in
//               registers -> 128B-swizzled SMEM tiles (K: K-major, V: MN-major)
//   warp  12    TMEM allocation; one thread issues the QK MMAs of even tiles
//   warp  13    one thread issues the QK MMAs of odd tiles
//   warp  14    one thread issues the PV MMAs
//               (one thread issues a tcgen05.mma about every 45 cycles at
//               N <= 128, while an N = 64 MMA needs 32 cycles of the tensor
//               pipe: the QK issue is split over two threads)
//   warp  15    producer: one bulk async copy (TMA, untiled) per (page, KV
//               head) block, K and V codes together (8 KB at D = 256; the
//               pool keeps them adjacent because a copy's issue cost is
//               mostly per copy), into a 3-stage int8 staging ring ahead of
//               the converters; scales straight into the 3-stage scale arrays
//               the softmax reads. It also prefetches the codes of the tile
//               a ring's depth ahead into L2 (cp.async.bulk.prefetch).
// Buffers (shared memory): int8 staging ring x3, fp16 K tiles x2 (free once
// QK of the tile is done), fp16 V tiles x2 (free once PV is done), scales x3.
// A third staging stage bought with a V tile measured 5% faster: the copies'
// latency, not the PV chain, limited the loop.
// Handshakes are mbarriers, one arrival per warp, with warp-uniform wait
// results. Every wait gives up after AttnParams::wait_ns (1 s by default),
// sets SPLASH_DEVICE_TIMEOUT and an abort flag; the CTA then lets the copies
// and MMAs it issued complete and frees its TMEM.
// The CTA's share of the tile stream (a contiguous range, cut by estimated
// cost) and the units' segment layout come from the split planner; barriers
// and TMEM are set up before the kernel waits for the plan (programmatic
// dependent launch).
// With prefix groups (kItems) a unit is (work item, KV head) instead: a row
// block of several sequences' stacked rows against their common prefix keys,
// or one sequence's rows against its keys after the prefix. The item table
// gives each segment its page-table row, first query token, row offset and
// key range; the pipeline above is the same.
#include <type_traits>

#include "splash_groups.cuh"
#include "tcgen05_ptx.cuh"

namespace splash {
namespace tc {
using namespace dev;

constexpr int kTileKeys = 64;
constexpr int kPagesPerTile = kTileKeys / kPageSize;
constexpr int kStages = 2;                    // S/P buffers in TMEM, fp16 K tiles
constexpr int kVStages = 2;                   // fp16 V tiles
constexpr int kScStages = 3;                  // K/V scale arrays
constexpr int kRing = 3;                      // int8 staging stages
constexpr int kSoftmaxWarps = 8;              // 2 per TMEM lane quarter, 16 rows each
constexpr int kLoadWarps = 4;
constexpr int kLoadThreads = 32 * kLoadWarps;
constexpr int kMmaWarp = kSoftmaxWarps + kLoadWarps;   // TMEM allocation, QK issue (even tiles)
constexpr int kQkOddWarp = kMmaWarp + 1;                // QK issue (odd tiles)
constexpr int kPvWarp = kQkOddWarp + 1;                 // PV issue
constexpr int kProducerWarp = kPvWarp + 1;
// 16 warps = 4 per SM sub-partition, so each thread may hold 128 registers
constexpr int kThreads = 32 * (kProducerWarp + 1);
static_assert(kThreads == 512, "warp roles");
static_assert(kStages == 2, "one QK-issuing warp per S/P buffer");
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;          // lazy rescale threshold (factor 256)

template <int D>
struct Cfg {
  static constexpr int kTileBytes = kTileKeys * D * 2;          // fp16 tile
  static constexpr int kQCol = 0;                                // Q': D/2 columns
  static constexpr int kSCol = D / 2;                            // S[2]: 64 columns each
  static constexpr int kOCol = D / 2 + 2 * kTileKeys;            // O: D columns
  static_assert(kOCol + D <= (int)kTmemCols, "TMEM budget");
  // staging ring stage: 4 (page, KV head) blocks of [K codes 16 x D][V codes 16 x D]
  static constexpr int kRingStage = 2 * kTileKeys * D;
  // dynamic shared memory (offsets from a 1024-byte aligned base)
  static constexpr int kOffK = 0;                                        // fp16 K [kStages]
  static constexpr int kOffV = kOffK + kStages * kTileBytes;             // fp16 V [kVStages]
  static constexpr int kOffRing = kOffV + kVStages * kTileBytes;         // int8 [kRing]
  static constexpr int kOffScales = kOffRing + kRing * kRingStage;       // fp32 [kScStages][2][64]
  static constexpr int kOffBars = kOffScales + kScStages * 2 * kTileKeys * 4;
  static constexpr int kBarBytes = 512;
  static constexpr int kSmemUsed = kOffBars + kBarBytes;
  // + up to 1 KB to align the base (the kernel checks the room it got); at
  // least 120 KB so that one CTA (and its 512 TMEM columns) owns the SM
  static constexpr int kSmemMax = 227 * 1024;
  static constexpr int kSmemAligned = kSmemUsed + 1024 < kSmemMax ? kSmemUsed + 1024 : kSmemMax;
  static constexpr int kSmemBytes = kSmemAligned > 120 * 1024 ? kSmemAligned : 120 * 1024;
  static_assert(kSmemUsed <= kSmemMax, "shared memory budget");
};

// ------------------------------------------------------------- work iteration
struct Seg {
  int b, h, i0, i1, T, ctx, Lk, R, u;
  int klo;                        // first key any row of the unit sees
  int qbase, r0;                  // items only: row r is query token qbase + (r0 + r) / G,
                                  // head h * G + (r0 + r) % G
};

// The CTA's tiles [t, t_end) of the stream of all units, one segment (a run
// of tiles of one unit) at a time. One item per sequence: units are
// (sequence, KV head).
struct SegIter {
  const int* stp;
  const int* seq_T;
  const int* seq_ctx;
  int B, G, Hkv, window;
  int t, t_end;
  __device__ bool next(Seg& s) {
    if (t >= t_end) return false;
    s.b = upper_index(stp, B - 1, t);
    s.T = seq_T[s.b];
    s.ctx = seq_ctx[s.b];
    s.Lk = s.ctx + s.T;
    s.klo = unit_first_key(s.ctx, window);
    const int first = unit_first_tile(s.ctx, window, kTileKeys);
    const int tiles = unit_tiles(s.ctx, s.T, window, kTileKeys);
    const int local = t - stp[s.b];
    s.h = local / tiles;
    s.i0 = first + local % tiles;
    s.i1 = min(first + tiles, s.i0 + (t_end - t));
    s.R = s.T * G;
    s.u = s.b * Hkv + s.h;
    t += s.i1 - s.i0;
    return true;
  }
};

// The same over the item table of a plan with prefix groups: units are
// (item, KV head), and an item's rows and keys come from its descriptor.
struct ItemSegIter {
  const int* stp;                 // item prefix sums; entries past the items are INT_MAX
  const ItemDesc* items;
  int NB, G, Hkv;                 // NB: entries searched
  int t, t_end;
  __device__ bool next(Seg& s) {
    if (t >= t_end) return false;
    const int item = upper_index(stp, NB - 1, t);
    const int4* dp = reinterpret_cast<const int4*>(items + item);
    const int4 d0 = dp[0], d1 = dp[1];           // b, qbase, r0, R | ctx, Lk, klo, grouped
    s.b = d0.x;
    s.qbase = d0.y;
    s.r0 = d0.z;
    s.R = d0.w;
    s.ctx = d1.x;
    s.Lk = d1.y;
    s.T = s.Lk - s.ctx;
    s.klo = d1.z;
    const int first = s.klo / kTileKeys;
    const int tiles = (s.Lk + kTileKeys - 1) / kTileKeys - first;
    const int local = t - stp[item];
    s.h = local / tiles;
    s.i0 = first + local % tiles;
    s.i1 = min(first + tiles, s.i0 + (t_end - t));
    s.u = item * Hkv + s.h;
    t += s.i1 - s.i0;
    return true;
  }
};

// The plan's workspace layout: the plain one, or the one of a plan with
// prefix groups (the same names for the regions the kernel reads).
template <bool kItems>
__device__ __forceinline__ typename std::conditional<kItems, GroupLayout, WorkspaceLayout>::type
layout_for(int B, int Hkv, int D, long long rows_bound) {
  if constexpr (kItems)
    return make_group_layout(B, Hkv, D, rows_bound);
  else
    return make_layout(B, Hkv, D, rows_bound);
}

template <bool kItems>
__device__ __forceinline__ typename std::conditional<kItems, ItemSegIter, SegIter>::type
make_iter(const int* stp, const int* seq_T, const int* seq_ctx, const ItemDesc* items, int B,
          int G, int Hkv, int window, int t, int t_end) {
  if constexpr (kItems)
    return ItemSegIter{stp, items, max_items(B), G, Hkv, t, t_end};
  else
    return SegIter{stp, seq_T, seq_ctx, B, G, Hkv, window, t, t_end};
}

struct Smem {
  uint64_t ring_full[kRing];      // producer tx (K and V codes) -> converters
  uint64_t ring_empty[2][kRing];  // converters done with a stage's [0] K / [1] V codes -> producer
  uint64_t sc_full[kScStages];    // producer cp.async (scales) -> softmax
  uint64_t sc_free[kScStages];    // softmax done with the scales -> producer
  uint64_t k_full[kStages];       // converters -> QK issuer (fp16 K of the tile ready)
  uint64_t v_full[kVStages];      // converters -> PV issuer (fp16 V of the tile ready)
  uint64_t k_free[kStages];       // QK done -> converters
  uint64_t v_free[kVStages];      // PV done -> converters, producer (scales)
  uint64_t s_full[kStages];       // QK done -> softmax
  uint64_t p_full[kStages];       // softmax -> MMA
  uint64_t p_free[kStages];       // PV of the buffer's tile done -> MMA (QK may
                                  // overwrite the S/P buffer), softmax (O rescale, epilogue)
  uint64_t q_full;                // softmax (Q' in TMEM) -> QK issuers
  uint64_t q_ack;                 // both QK issuers saw q_full -> softmax (the next
                                  // segment's Q' may complete q_full's next phase)
  uint64_t drain[3];              // QK even / QK odd / PV issuer: its MMAs complete
  uint32_t tmem_base;
  int abort_flag;
};


// Page ids of a sequence, 32 at a time: lane l holds entry base + l of the
// sequence's page-table row (-1 past the pages the sequence needs). The next
// window is fetched when the current one is first used, so the table read
// latency is paid once per 8 tiles and mostly hidden.
struct PageWindow {
  int b = -1, base = 0, cur = -1;
  int nb = -1, nbase = 0, nxt = -1;
  __device__ __forceinline__ static int fetch(const AttnParams& p, int b, int base, int npages,
                                              int lane) {
    const int i = base + lane;
    return i < npages ? p.page_table[(size_t)b * p.max_pages_per_seq + i] : -1;
  }
  // make entries [first, first + 4) of sequence b available; returns the id of
  // page `first + (lane & 3)` in every lane
  __device__ __forceinline__ int get(const AttnParams& p, int sb, int first, int npages,
                                     int lane) {
    const int want = first & ~31;
    if (sb != b || want != base) {
      if (sb == nb && want == nbase) {
        cur = nxt;
      } else {
        cur = fetch(p, sb, want, npages, lane);
      }
      b = sb;
      base = want;
      nb = sb;
      nbase = want + 32;
      nxt = fetch(p, sb, nbase, npages, lane);      // prefetch the next window
    }
    return __shfl_sync(0xffffffffu, cur, (first - base) + (lane & 3));
  }
  // id of page idx of sequence sb when the current or the prefetched window
  // holds it, else -1 (called by the whole warp; idx may differ per lane)
  __device__ __forceinline__ int peek(int sb, int idx) const {
    const int a = __shfl_sync(0xffffffffu, cur, (idx - base) & 31);
    const int c = __shfl_sync(0xffffffffu, nxt, (idx - nbase) & 31);
    if (sb == b && idx >= base && idx < base + 32) return a;
    if (sb == nb && idx >= nbase && idx < nbase + 32) return c;
    return -1;
  }
};

// Producer (one warp): the K and V codes of tile `it` of segment s into a
// ring stage. The tile's 4 page ids come from the page window; lanes 0..3
// each issue one bulk copy of a (page, KV head) block (K codes then V codes,
// 2 x 16 x D bytes). Pages past the sequence end, below a sliding window or
// with an invalid id are skipped: their stale codes are finite and the
// softmax gives their keys probability 0 without reading their scales.
// Returns the page id of page (lane & 3), -1 if skipped.
template <int D>
__device__ __forceinline__ int stage_codes(const AttnParams& p, const Seg& s, int it,
                                           uint8_t* dst, uint32_t bar, int lane,
                                           PageWindow& win) {
  const int k0 = it * kTileKeys;
  const int npages = (s.Lk + kPageSize - 1) / kPageSize;
  int page = win.get(p, s.b, k0 / kPageSize, npages, lane);
  const bool needed = k0 + kPageSize * (lane & 3) < s.Lk &&
                      k0 + kPageSize * ((lane & 3) + 1) > s.klo;
  if (!needed || page >= p.num_pages) page = -1;
  if (needed && page < 0 && lane < kPagesPerTile) report(p.device_status, SPLASH_DEVICE_BAD_PAGE);
  const int mask = (int)(__ballot_sync(0xffffffffu, page >= 0 && lane < kPagesPerTile) &
                         ((1u << kPagesPerTile) - 1));
  constexpr uint32_t kBlock = 2 * kPageSize * D;      // K and V codes of one (page, head)
  if (lane == 0) mbar_expect_tx(bar, (uint32_t)__popc(mask) * kBlock);
  __syncwarp();
  if (lane < kPagesPerTile && page >= 0)
    bulk_g2s(smem_u32(dst) + lane * kBlock,
             p.k_pages + code_offset(page, s.h, p.num_kv_heads, 0, D), kBlock, bar);
  return page;
}

// Producer: the tile's K and V scales, 16 bytes per lane by cp.async (lanes
// 0..15 K, 16..31 V; page (lane & 15) / 4, slots 4 * (lane & 3) ..); each
// lane's arrival on the scale barrier fires when its copy has landed.
__device__ __forceinline__ void stage_scales(const AttnParams& p, const Seg& s, int page,
                                             float* scales, uint32_t scale_bar, int lane) {
  const int sj = (lane & 15) >> 2;
  const int ps = __shfl_sync(0xffffffffu, page, sj);
  if (ps >= 0) {
    const float* src = (lane < 16 ? p.k_scales : p.v_scales) +
                       ((size_t)ps * p.num_kv_heads + s.h) * kPageSize + 4 * (lane & 3);
    // page sj's 16-byte chunk c sits at chunk c ^ sj of the page's 64 bytes, so
    // the softmax's four lanes reading chunk c of pages 0..3 hit distinct banks
    const uint32_t dst = smem_u32(scales) + (lane < 16 ? 0 : kTileKeys * 4) +
                         (sj * kPageSize + 4 * ((lane & 3) ^ sj)) * 4;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
  }
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(scale_bar)
               : "memory");
}

// Tile row of key n: keys are permuted inside a tile (K and V alike, so the
// contraction over keys is unchanged) so that S/P column 8i + 2q + b, which the
// 16x256b TMEM load hands to the thread with q = lane % 4, holds key
// 16q + 2i + b: each softmax thread then owns 16 consecutive keys.
__host__ __device__ constexpr int tile_row_of_key(int n) {
  return 8 * ((n % 16) / 2) + 2 * (n / 16) + (n % 2);
}

// src: the K (or V) codes of page 0 of a ring stage, pages 2 x 16 x D bytes apart.
// Units of 16 codes: one 16-byte shared load, two 16-byte fp16 stores into the
// 128B-swizzled tile (row tile_row_of_key(key), 16-byte chunks 2c and 2c + 1
// of the row's 64-column atom c / 4). 16-byte accesses are served per quarter
// warp, so each quarter takes 4 chunks of an even key row and 4 of the next
// key's row (tile rows n, n + 1): its 8 loads and each of its two stores fall
// in 8 distinct bank groups.
template <int D>
__device__ __forceinline__ void convert_codes(const uint8_t* src, uint8_t* dst, int lt) {
  constexpr int kPageStride = 2 * kPageSize * D;
  constexpr int kChunks = D / 16;                     // 16-code chunks per key row
  constexpr int kQuartersPerPair = kChunks / 4;       // quarter warps per two key rows
  constexpr int kKeysPerPass = kLoadThreads * 16 / D;
  constexpr int kPer = kTileKeys / kKeysPerPass;
  static_assert(kChunks % 4 == 0 && kTileKeys % kKeysPerPass == 0, "converter units");
  const int w = lt >> 5, l = lt & 31, qtr = l >> 3, rsel = (l >> 2) & 1, j = l & 3;
  const int pair = qtr / kQuartersPerPair, qq = qtr % kQuartersPerPair;
  const int c16 = 8 * (qq >> 1) + 4 * (rsel ^ (qq & 1)) + j;
  const int key_in_pass = w * (32 * 16 / D) + 2 * pair + rsel;
  uint4 wv[kPer];
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int key = q * kKeysPerPass + key_in_pass;
    wv[q] = *reinterpret_cast<const uint4*>(src + (key / kPageSize) * kPageStride +
                                            (key % kPageSize) * D + c16 * 16);
  }
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int key = q * kKeysPerPass + key_in_pass;
    const int n = tile_row_of_key(key), c8 = 2 * c16;
    uint4 h0, h1;
    i8x4_to_h2x2(wv[q].x, h0.x, h0.y);
    i8x4_to_h2x2(wv[q].y, h0.z, h0.w);
    i8x4_to_h2x2(wv[q].z, h1.x, h1.y);
    i8x4_to_h2x2(wv[q].w, h1.z, h1.w);
    const uint32_t row = (c8 / 8) * (kTileKeys * 128) + n * 128;
    *reinterpret_cast<uint4*>(dst + row + (((c8 & 7) ^ (n & 7)) << 4)) = h0;
    *reinterpret_cast<uint4*>(dst + row + ((((c8 + 1) & 7) ^ (n & 7)) << 4)) = h1;
  }
}

// ------------------------------------------------------------------- kernel
// kSwa: sliding-window instantiation (window read from the parameters); the
// plain one compiles the window bounds out. kItems: the plan holds prefix
// groups, and the kernel walks its item table (never with a window).
template <int D, bool kSwa, bool kItems>
__global__ void __launch_bounds__(kThreads, 1) verify_tc_kernel(AttnParams p) {
  static_assert(!(kSwa && kItems), "prefix groups are planned without a window");
  using C = Cfg<D>;
  static_assert(sizeof(Smem) <= C::kBarBytes, "barrier area");
  extern __shared__ uint8_t smem_raw[];
  allow_dependent_launch();
  // 128-byte swizzled operand tiles need a 1024-byte aligned base
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  if (smem - smem_raw + C::kSmemUsed > C::kSmemBytes) {
    if (threadIdx.x == 0) report(p.device_status, SPLASH_DEVICE_INTERNAL);
    return;
  }
  uint8_t* kbuf = smem + C::kOffK;
  uint8_t* vbuf = smem + C::kOffV;
  uint8_t* ring = smem + C::kOffRing;
  float* scales = reinterpret_cast<float*>(smem + C::kOffScales);   // [3][K 64, V 64]
  Smem* sh = reinterpret_cast<Smem*>(smem + C::kOffBars);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kRing; ++s) {
      mbar_init(smem_u32(&sh->ring_full[s]), 1);
      for (int kv = 0; kv < 2; ++kv) mbar_init(smem_u32(&sh->ring_empty[kv][s]), kLoadWarps);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sh->k_full[s]), kLoadWarps);
      mbar_init(smem_u32(&sh->k_free[s]), 1);
      mbar_init(smem_u32(&sh->s_full[s]), 1);
      mbar_init(smem_u32(&sh->p_full[s]), kSoftmaxWarps);
      mbar_init(smem_u32(&sh->p_free[s]), 1);
    }
    for (int s = 0; s < kScStages; ++s) {
      mbar_init(smem_u32(&sh->sc_full[s]), 32);     // one cp.async arrival per producer lane
      mbar_init(smem_u32(&sh->sc_free[s]), kSoftmaxWarps);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(smem_u32(&sh->v_free[s]), 1);
      mbar_init(smem_u32(&sh->v_full[s]), kLoadWarps);
    }
    mbar_init(smem_u32(&sh->q_full), kSoftmaxWarps);
    mbar_init(smem_u32(&sh->q_ack), 2);
    for (int i = 0; i < 3; ++i) mbar_init(smem_u32(&sh->drain[i]), 1);
    sh->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(&sh->tmem_base)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = sh->tmem_base;
  const Sync sync{&sh->abort_flag, p.device_status, p.wait_ns};

  // the set-up above overlaps the planner; from here on the plan is read
  grid_dependency_wait();
  const PlanHeader* hd = reinterpret_cast<const PlanHeader*>(p.ws);
  if ((int)blockIdx.x >= hd->ncta[kClassTensor]) {         // no tiles for this CTA
    if (warp == kMmaWarp)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                   "r"(kTmemCols) : "memory");
    return;
  }
  const int B = p.num_seqs, Hkv = p.num_kv_heads, G = p.group;
  const auto L = layout_for<kItems>(B, Hkv, D, hd->rows_bound);
  const int* q_off = reinterpret_cast<const int*>(p.ws + L.q_off);
  const int* seq_T = reinterpret_cast<const int*>(p.ws + L.seq_T);
  const int* seq_ctx = reinterpret_cast<const int*>(p.ws + L.seq_ctx);
  const ItemDesc* items = static_cast<const ItemDesc*>(nullptr);
  if constexpr (kItems) items = reinterpret_cast<const ItemDesc*>(p.ws + L.items);
  const int* stp = reinterpret_cast<const int*>(p.ws + L.stp) + kClassTensor * (B + 1);
  const int* nseg = reinterpret_cast<const int*>(p.ws + L.nseg);
  const int* cfirst = reinterpret_cast<const int*>(p.ws + L.cfirst);
  const int* part_base = reinterpret_cast<const int*>(p.ws + L.part_base);
  float* o_part = reinterpret_cast<float*>(p.ws + L.o_part);
  float* lse_part = reinterpret_cast<float*>(p.ws + L.lse_part);

  const int window = kSwa ? p.window : 0;
  const int* cst = reinterpret_cast<const int*>(p.ws + L.cta_start) + kClassTensor * (kMaxCtas + 1);
  typename std::conditional<kItems, ItemSegIter, SegIter>::type iter =
      make_iter<kItems>(stp, seq_T, seq_ctx, items, B, G, Hkv, window, cst[blockIdx.x],
                        cst[blockIdx.x + 1]);

  if (warp < kSoftmaxWarps) {
    // ===================================================== softmax + epilogue
    const int lb = 32 * (warp % 4) + 16 * (warp / 4);     // first TMEM lane of the warp
    const uint32_t lane_base = (uint32_t)lb << 16;
    const int quad = lane & 3;                            // column pair within 8 columns
    // TMEM lanes of this thread's two rows
    const int ln[2] = {lb + (lane >> 2), lb + 8 + (lane >> 2)};
    int g = 0, nsegs = 0;
    Seg s;
    bool ok = true;
    while (ok && iter.next(s)) {
      // Q' of this segment overwrites the previous one: both QK issuers must
      // have seen the previous q_full phase (so neither lags it by two phases)
      if (nsegs > 0) {
        ok = __all_sync(0xffffffffu, sync.wait(smem_u32(&sh->q_ack), (nsegs - 1) & 1));
        if (!ok) break;
      }
      ++nsegs;
      // The unit's rows are spread evenly over the four TMEM lane quarters
      // (each served by the softmax warps of one SM sub-partition): row
      // q * rpq + i sits in lane 32q + i, i < rpq = ceil(R / 4). Lanes past
      // rpq in a quarter hold no row.
      const int rpq = (s.R + 3) >> 2;
      int rr[2];                                          // row of each of this thread's lanes, -1: none
      bool live[2];
      int lim[2], lo[2];
      size_t qrow_off[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int i = ln[k] & 31, r = (ln[k] >> 5) * rpq + i;
        live[k] = i < rpq && r < s.R;
        rr[k] = live[k] ? r : -1;
        if constexpr (kItems) {
          const int j = s.r0 + (live[k] ? r : 0);
          const int tt = j / G, gg = j - tt * G;
          lim[k] = s.ctx + tt;                            // last visible key of the row
          lo[k] = 0;
          qrow_off[k] = (size_t)(s.qbase + tt) * p.num_q_heads + s.h * G + gg;
        } else {
          const int tt = live[k] ? r / G : 0, gg = live[k] ? r - tt * G : 0;
          lim[k] = s.ctx + tt;                            // last visible key of the row
          lo[k] = kSwa ? lim[k] - window + 1 : 0;         // first visible key (with a window)
          qrow_off[k] = (size_t)(q_off[s.b] + tt) * p.num_q_heads + s.h * G + gg;
        }
      }
      const bool warp_live = __any_sync(0xffffffffu, live[0]);
      const bool k1_live = __any_sync(0xffffffffu, live[1]);   // second row set of the warp
      float rowfac[2] = {0.f, 0.f};
      // Q rows -> TMEM as fp16 after an exact per-row power-of-two rescale.
      // Thread covers d = 8i + 2*quad + {0,1} (i < D/8) of both rows; all of
      // its Q words are loaded in one batch (one memory latency per segment).
      if (warp_live) {
        uint32_t qw[2][D / 8];                             // bf16 pairs
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint32_t* qr = reinterpret_cast<const uint32_t*>(p.q + qrow_off[k] * D) + quad;
#pragma unroll
          for (int i = 0; i < D / 8; ++i) {
            qw[k][i] = 0u;
            if (live[k]) qw[k][i] = __ldg(qr + 4 * i);
          }
        }
        float up[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          uint32_t amax_bits = 0;                          // max |q| as bf16 magnitude bits
#pragma unroll
          for (int i = 0; i < D / 8; ++i)
            amax_bits = max(amax_bits, max(qw[k][i] & 0x7fffu, (qw[k][i] >> 16) & 0x7fffu));
          float amax = __uint_as_float(amax_bits << 16);
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
          // 2^e with max|q| * 2^e in [2^14, 2^15)
          int e = 0;
          const int ex = (int)((__float_as_uint(amax) >> 23) & 0xff);
          if (amax > 0.f) e = ex == 0 ? 14 + 126 : 14 - ex + 127;
          e = max(-126, min(127, e));
          up[k] = __uint_as_float((uint32_t)(e + 127) << 23);
          rowfac[k] = p.sm_scale_log2 / up[k];
        }
        static_assert((D / 2) % 64 == 0, "Q' stores of 64 packed columns");
#pragma unroll
        for (int c0 = 0; c0 < D / 2; c0 += 64) {          // 64 packed columns per store
          uint32_t v[32];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            // packed column c0 + 4i + quad holds d pair 8j + 2*quad, j = c0/4 + i
            const int j = c0 / 4 + i;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const float2 f =
                  __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qw[k][j]));
              __half2 hv = __floats2half2_rn(f.x * up[k], f.y * up[k]);
              v[2 * i + k] = *reinterpret_cast<uint32_t*>(&hv);
            }
          }
          tmem_st16x128_x16(tmem + lane_base + C::kQCol + c0, v);
        }
        tmem_wait_st();
      }
      fence_before();
      warp_arrive(smem_u32(&sh->q_full), lane);

      float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};   // l: this thread's columns
      for (int it = s.i0; it < s.i1 && ok; ++it, ++g) {
        const int st = g % kStages, sst = g % kScStages;
        ok = sync.wait(smem_u32(&sh->sc_full[sst]), (g / kScStages) & 1) &&
             sync.wait(smem_u32(&sh->s_full[st]), (g / kStages) & 1);
        ok = __all_sync(0xffffffffu, ok);       // a timeout seen by some lanes stops the warp
        if (!ok) break;
        fence_after();
        uint32_t pw[16];                                   // P: 32 packed columns
        float alpha[2] = {1.f, 1.f};
        if (warp_live) {
          const int k0 = it * kTileKeys;
          const float* ks = scales + sst * 2 * kTileKeys;
          const float* vs = ks + kTileKeys;
          uint32_t sv[32];
          tmem_ld16x256_x8(tmem + lane_base + C::kSCol + st * kTileKeys, sv);
          // the K scales load while the TMEM load is in flight
          float2 ks2[8], x[2][8];
#pragma unroll
          for (int i4 = 0; i4 < 4; ++i4) {
            const float4 kq = *reinterpret_cast<const float4*>(ks + 16 * quad + 4 * (i4 ^ quad));
            ks2[2 * i4] = make_float2(kq.x, kq.y);
            ks2[2 * i4 + 1] = make_float2(kq.z, kq.w);
          }
          tmem_wait_ld(sv);         // sv is read only after the wait
          // x = S * sK (packed fp32x2); masked columns -> -inf (their scales
          // are not read: pages past the end may hold anything)
          // this thread's keys: 16*quad + 2i + {0,1} (see tile_row_of_key)
#pragma unroll
          for (int i = 0; i < 8; ++i) {
#pragma unroll
            for (int k = 0; k < 2; ++k)
              x[k][i] = (k == 0 || k1_live)
                            ? __fmul2_rn(make_float2(__uint_as_float(sv[4 * i + 2 * k]),
                                                     __uint_as_float(sv[4 * i + 2 * k + 1])), ks2[i])
                            : make_float2(-INFINITY, -INFINITY);
          }
          // tile keys jj with nlo <= jj < nvis are visible to the row
          int nvis[2] = {kTileKeys, kTileKeys}, nlo[2] = {-1, -1};
          bool full = true;
          // a tile below the block's keys (and, with a window, above every
          // row's lower bound) is visible to every row: no per-row bounds
          const bool tile_inside = k0 + kTileKeys <= s.ctx &&
                                   (!kSwa || s.ctx + s.T - window <= k0);
          if (!tile_inside) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              nvis[k] = live[k] ? min(kTileKeys, lim[k] - k0 + 1) : 0;
              nlo[k] = kSwa ? max(lo[k] - k0, -1) : -1;       // compile-time -1 without a window
              // rows that hold no query row need no mask (their P only reaches
              // output rows that are never read)
              full = full && (!live[k] || (nvis[k] == kTileKeys && (!kSwa || nlo[k] <= 0)));
            }
          }
          if (!full) {
#pragma unroll
            for (int k = 0; k < 2; ++k)
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int j = 16 * quad + 2 * i;
                if (j >= nvis[k] || j < nlo[k]) x[k][i].x = -INFINITY;
                if (j + 1 >= nvis[k] || j + 1 < nlo[k]) x[k][i].y = -INFINITY;
              }
          }
          float base[2] = {0.f, 0.f};
          // both row sets' maxima at once (independent chains); the second is
          // unused when the warp's second row set holds no row
          float mts[2];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            mts[k] = -INFINITY;
#pragma unroll
            for (int i = 0; i < 8; ++i) mts[k] = fmax3(mts[k], x[k][i].x, x[k][i].y);
          }
#pragma unroll
          for (int k = 0; k < 2; ++k) mts[k] = fmaxf(mts[k], __shfl_xor_sync(0xffffffffu, mts[k], 1));
#pragma unroll
          for (int k = 0; k < 2; ++k) mts[k] = fmaxf(mts[k], __shfl_xor_sync(0xffffffffu, mts[k], 2));
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            if (k == 1 && !k1_live) break;                // no row in the warp's second set
            const float mt = mts[k];
            const float m_new = fmaxf(m[k], mt);
            float m_use = m[k];
            if (m[k] == -INFINITY) {
              m_use = m_new;
            } else if (rowfac[k] * (m_new - m[k]) > kRescaleLog2) {
              alpha[k] = ex2(rowfac[k] * (m[k] - m_new));
              m_use = m_new;
            }
            m[k] = m_use;
            base[k] = (m_use == -INFINITY) ? 0.f : rowfac[k] * m_use;
          }
          float2 vs2[8];
#pragma unroll
          for (int i4 = 0; i4 < 4; ++i4) {
            const float4 vq4 = *reinterpret_cast<const float4*>(vs + 16 * quad + 4 * (i4 ^ quad));
            vs2[2 * i4] = make_float2(vq4.x, vq4.y);
            vs2[2 * i4 + 1] = make_float2(vq4.z, vq4.w);
          }
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            if (k == 1 && !k1_live) {
#pragma unroll
              for (int i = 0; i < 8; ++i) pw[2 * i + 1] = 0u;
              break;
            }
            const float2 rf2 = make_float2(rowfac[k], rowfac[k]);
            const float2 nb2 = make_float2(-base[k], -base[k]);
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              float2 vq = vs2[i];
              if (!full) {      // scales of masked keys are not trusted
                const int j = 16 * quad + 2 * i;
                if (j >= nvis[k] || j < nlo[k]) vq.x = 0.f;
                if (j + 1 >= nvis[k] || j + 1 < nlo[k]) vq.y = 0.f;
              }
              const float2 e0 = __ffma2_rn(x[k][i], rf2, nb2);
              const float2 p0 = make_float2(ex2(e0.x), ex2(e0.y));
              acc = __fadd2_rn(acc, p0);
              __half2 h0 = __float22half2_rn(__fmul2_rn(p0, vq));
              pw[2 * i + k] = *reinterpret_cast<uint32_t*>(&h0);   // packed column 4i + quad
            }
            l[k] = l[k] * alpha[k] + (acc.x + acc.y);
          }
        }
        // a rescale of O waits for the previous tile's PV (rare: the running
        // max is only moved when it grows by more than 2^8). p_free of that
        // tile's buffer: its previous phase (PV three tiles back) is complete,
        // so a parity wait cannot be satisfied by an older phase.
        if (it > s.i0 && warp_live &&
            __any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
          ok = __all_sync(0xffffffffu,
                          sync.wait(smem_u32(&sh->p_free[(g - 1) % kStages]), ((g - 1) / kStages) & 1));
          if (!ok) break;
          fence_after();
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 64) {
            uint32_t v[32];
            tmem_ld16x256_x8(tmem + lane_base + C::kOCol + c0, v);
            tmem_wait_ld(v);
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
              for (int k = 0; k < 2; ++k) {
                v[4 * i + 2 * k] = __float_as_uint(__uint_as_float(v[4 * i + 2 * k]) * alpha[k]);
                v[4 * i + 2 * k + 1] =
                    __float_as_uint(__uint_as_float(v[4 * i + 2 * k + 1]) * alpha[k]);
              }
            tmem_st16x256_x8(tmem + lane_base + C::kOCol + c0, v);
          }
        }
        warp_arrive(smem_u32(&sh->sc_free[sst]), lane);    // scales of this tile are read
        if (warp_live) {
          tmem_st16x128_x8(tmem + lane_base + C::kSCol + st * kTileKeys, pw);
          tmem_wait_st();
        }
        fence_before();
        warp_arrive(smem_u32(&sh->p_full[st]), lane);
      }
      if (!ok) break;
      // epilogue: last PV of the segment complete -> normalise, write out
      ok = __all_sync(0xffffffffu,
                      sync.wait(smem_u32(&sh->p_free[(g - 1) % kStages]), ((g - 1) / kStages) & 1));
      if (!ok) break;
      fence_after();
      if (warp_live) {
        // rows go to the output when one CTA covers the unit (and, with
        // prefix groups, the unit is in none: part_base < 0 says both)
        const int ns = kItems ? (part_base[s.u] < 0 ? 1 : 2) : nseg[s.u];
        float inv[2];
        long long prow[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          float lt = l[k];
          lt += __shfl_xor_sync(0xffffffffu, lt, 1);
          lt += __shfl_xor_sync(0xffffffffu, lt, 2);
          l[k] = lt;
          inv[k] = lt > 0.f ? 1.f / lt : 0.f;
          prow[k] = (long long)part_base[s.u] + (long long)(blockIdx.x - cfirst[s.u]) * s.R + rr[k];
        }
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 64) {
          uint32_t v[32];
          tmem_ld16x256_x8(tmem + lane_base + C::kOCol + c0, v);
          tmem_wait_ld(v);
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            if (!live[k]) continue;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int d = c0 + 8 * i + 2 * quad;
              const float o0 = __uint_as_float(v[4 * i + 2 * k]) * inv[k];
              const float o1 = __uint_as_float(v[4 * i + 2 * k + 1]) * inv[k];
              if (ns == 1)
                *reinterpret_cast<__nv_bfloat162*>(p.out + qrow_off[k] * D + d) =
                    __floats2bfloat162_rn(o0, o1);
              else
                *reinterpret_cast<float2*>(o_part + prow[k] * D + d) = make_float2(o0, o1);
            }
          }
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          if (live[k] && quad == 0) {
            const float lse =
                l[k] > 0.f ? (rowfac[k] * m[k] + __log2f(l[k])) * 0.69314718055994531f : -INFINITY;
            if (ns == 1) p.lse[qrow_off[k]] = lse;
            else lse_part[prow[k]] = lse;
          }
        }
      }
      fence_before();
    }
  } else if (warp < kSoftmaxWarps + kLoadWarps) {
    // =========================================================== converters
    const int lt = tid - 32 * kSoftmaxWarps;
    int g = 0;
    Seg s;
    bool ok = true;
    while (ok && iter.next(s)) {
      for (int it = s.i0; it < s.i1; ++it, ++g) {
        const int r = g % kRing, st = g % kStages, vst = g % kVStages;
        const uint32_t ph = (g / kRing) & 1;
        const uint8_t* stage = ring + r * C::kRingStage;
        // K codes -> fp16 K tile; the QK of the tile may start at once
        ok = sync.wait(smem_u32(&sh->ring_full[r]), ph) &&
             sync.wait(smem_u32(&sh->k_free[st]), ((g / kStages) & 1) ^ 1);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        convert_codes<D>(stage, kbuf + st * C::kTileBytes, lt);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&sh->ring_empty[0][r]));
          mbar_arrive(smem_u32(&sh->k_full[st]));
        }
        // V codes -> fp16 V tile
        ok = __all_sync(0xffffffffu, sync.wait(smem_u32(&sh->v_free[vst]), ((g / kVStages) & 1) ^ 1));
        if (!ok) break;
        convert_codes<D>(stage + kPageSize * D, vbuf + vst * C::kTileBytes, lt);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&sh->ring_empty[1][r]));
          mbar_arrive(smem_u32(&sh->v_full[vst]));
        }
      }
    }
  } else if (warp >= kProducerWarp) {
    // ============================================================ producer
    int g = 0, armed = 0;                                   // armed: tiles staged so far
    Seg s;
    bool ok = true;
    PageWindow win;
    while (ok && iter.next(s)) {
      for (int it = s.i0; it < s.i1; ++it, ++g) {
        const int r = g % kRing, sst = g % kScStages;
        const uint32_t ph = ((g / kRing) & 1) ^ 1;
        uint8_t* stage = ring + r * C::kRingStage;
        // codes once the converters are done with the K and V codes of tile
        // g - kRing, scales once the softmax is done with those of g - kScStages
        if (lane == 0)
          ok = sync.wait(smem_u32(&sh->ring_empty[0][r]), ph) &&
               sync.wait(smem_u32(&sh->ring_empty[1][r]), ph) &&
               sync.wait(smem_u32(&sh->sc_free[sst]), ((g / kScStages) & 1) ^ 1);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const int page = stage_codes<D>(p, s, it, stage, smem_u32(&sh->ring_full[r]), lane, win);
        stage_scales(p, s, page, scales + sst * 2 * kTileKeys, smem_u32(&sh->sc_full[sst]), lane);
        ++armed;
        {
          // the codes of the tile kRing ahead into L2 only (no shared
          // memory): its staging copy, issued when this ring stage frees
          // again, then hits L2. Measured 5-6% faster on 16 x 32K and the
          // ragged batch; 2 to 4 tiles ahead do the same, 6 less. The scale
          // rows take plain L2 prefetches (bulk prefetches of 64 bytes each
          // measured slower).
          const int ahead = it + kRing;
          const int k0a = ahead * kTileKeys;
          const int pg = win.peek(s.b, k0a / kPageSize + (lane & 3));
          // the pages stage_codes will copy: inside the sequence and not
          // wholly below a sliding window
          const bool want = ahead < s.i1 && k0a + kPageSize * (lane & 3) < s.Lk &&
                            k0a + kPageSize * ((lane & 3) + 1) > s.klo;
          if (want && lane < kPagesPerTile && pg >= 0 && pg < p.num_pages)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                         ::"l"(p.k_pages + code_offset(pg, s.h, p.num_kv_heads, 0, D)),
                         "r"((uint32_t)(2 * kPageSize * D)) : "memory");
          // and its K / V scale rows (64 bytes each) with plain L2 prefetches
          const int pgs = __shfl_sync(0xffffffffu, pg, lane & 3);
          if (want && lane >= 4 && lane < 12 && pgs >= 0 && pgs < p.num_pages) {
            const size_t sc = ((size_t)pgs * p.num_kv_heads + s.h) * kPageSize;
            const float* src = (lane < 8 ? p.k_scales : p.v_scales) + sc;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(src) : "memory");
          }
        }
      }
    }
    // copies still in flight (only after an abort: on the normal path the
    // converters consumed every staged tile) land before the CTA exits. A stage
    // is re-armed only after its previous tile was consumed, so the last tile
    // armed on it is its only one outstanding.
    if (lane == 0) {
      for (int r = 0; r < kRing && r < armed; ++r) {
        const int last = r + ((armed - 1 - r) / kRing) * kRing;
        sync.drain(smem_u32(&sh->ring_full[r]), (last / kRing) & 1);
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else {
    // ============================================================ MMA issue
    // warps kMmaWarp / kQkOddWarp: QK(i) (i even / odd) into S[i % 2] once its
    // K tile is converted and the PV that last read that S/P buffer (tile
    // i - 2) has completed (issue order alone does not order a later TMEM
    // write after an earlier MMA's read).
    // warp kPvWarp: PV(i) into O once the softmax has written P(i).
    const bool is_qk = warp != kPvWarp;
    const int qk_par = warp - kMmaWarp;          // tiles of this parity (QK issuers)
    const int role = is_qk ? qk_par : 2;
    if (lane == 0) {
      constexpr uint32_t kIdescQK = idesc_f16(128, kTileKeys, 0, 0);
      constexpr uint32_t kIdescPV = idesc_f16(128, D, 0, 1);
      // descriptors of k-step 0 of buffer 0; buffers and k-steps add byte offsets >> 4
      const uint64_t kdesc0 = sdesc(smem_u32(kbuf), 16, 1024);
      const uint64_t vdesc0 = sdesc(smem_u32(vbuf), kTileKeys * 128, 1024);
      int g = 0, nsegs = 0;
      Seg s;
      bool ok = true;
      while (ok && iter.next(s)) {
        if (is_qk) {
          ok = sync.wait(smem_u32(&sh->q_full), nsegs & 1);
          if (!ok) break;
          fence_after();
          mbar_arrive(smem_u32(&sh->q_ack));
        }
        for (int it = s.i0; it < s.i1 && ok; ++it, ++g) {
          const int st = g % kStages, vst = g % kVStages;
          if (is_qk) {
            if (st != qk_par) continue;
            ok = sync.wait(smem_u32(&sh->p_free[st]), ((g / kStages) & 1) ^ 1) &&
                 sync.wait(smem_u32(&sh->k_full[st]), (g / kStages) & 1);
            if (!ok) break;
            fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_ts(tmem + C::kSCol + st * kTileKeys, tmem + C::kQCol + kk * 8,
                     kdesc0 + (uint64_t)((st * C::kTileBytes + (kk / 4) * (kTileKeys * 128) +
                                          (kk % 4) * 32) >> 4),
                     kIdescQK, kk > 0);
            mma_commit(smem_u32(&sh->s_full[st]));
            mma_commit(smem_u32(&sh->k_free[st]));
          } else {
            ok = sync.wait(smem_u32(&sh->p_full[st]), (g / kStages) & 1) &&
                 sync.wait(smem_u32(&sh->v_full[vst]), (g / kVStages) & 1);
            if (!ok) break;
            fence_after();
#pragma unroll
            for (int kk = 0; kk < kTileKeys / 16; ++kk)
              mma_ts(tmem + C::kOCol, tmem + C::kSCol + st * kTileKeys + kk * 8,
                     vdesc0 + (uint64_t)((vst * C::kTileBytes + kk * 16 * 128) >> 4), kIdescPV,
                     (it == s.i0 && kk == 0) ? 0u : 1u);
            mma_commit(smem_u32(&sh->v_free[vst]));
            mma_commit(smem_u32(&sh->p_free[st]));
          }
        }
        ++nsegs;
      }
      // every MMA this thread issued is complete before TMEM is released and
      // the shared-memory operands go away; the drain wait ignores the abort
      // flag (after an abort the MMAs already issued still run to completion)
      mma_commit(smem_u32(&sh->drain[role]));
      sync.drain(smem_u32(&sh->drain[role]), 0);
    }
    __syncwarp();
  }

  fence_before();
  __syncthreads();
  fence_after();
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols) : "memory");
  }
}

}  // namespace tc

bool tc_supported(int head_dim) { return head_dim == 128 || head_dim == 256; }

cudaError_t launch_verify_tc(const AttnParams& p, int rows_cap, int ncta, bool items,
                             cudaStream_t stream) {
  (void)rows_cap;
#define SPLASH_TC(DD, SWA, IT)                                                                 \
  do {                                                                                         \
    constexpr int smem = tc::Cfg<DD>::kSmemBytes;                                              \
    cudaError_t e = ensure_dynamic_smem<tc::verify_tc_kernel<DD, SWA, IT>>(smem);             \
    if (e != cudaSuccess) return e;                                                            \
    e = launch_dependent(tc::verify_tc_kernel<DD, SWA, IT>, dim3(ncta), dim3(tc::kThreads),    \
                         smem, stream, p);                                                     \
    if (e != cudaSuccess) return e;                                                            \
  } while (0)
  const bool swa = p.window > 0;
  if (swa && items) return cudaErrorInvalidValue;
  switch (p.head_dim) {
    case 128:
      if (swa) SPLASH_TC(128, true, false);
      else if (items) SPLASH_TC(128, false, true);
      else SPLASH_TC(128, false, false);
      break;
    case 256:
      if (swa) SPLASH_TC(256, true, false);
      else if (items) SPLASH_TC(256, false, true);
      else SPLASH_TC(256, false, false);
      break;
    default: return cudaErrorNotSupported;
  }
#undef SPLASH_TC
  return cudaGetLastError();
}

}  // namespace splash
