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
// Warp roles (448 threads):
//   warps 0-3   softmax + epilogue: thread = TMEM lane = query row
//   warps 4-11  converters: int8 codes from the staging ring -> fp16 in
//               registers -> 128B-swizzled SMEM tiles (K: K-major, V: MN-major)
//   warp  12    TMEM allocation and the single MMA-issuing thread
//   warp  13    producer: bulk async copies (TMA, untiled) of whole
//               (page, KV head) blocks: codes into a 2-stage int8 staging
//               ring ahead of the converters, scales straight into the
//               3-stage scale arrays the softmax reads
// Buffers: fp16 K tiles x2 (free once QK of the tile is done), fp16 V tiles x3
// (free once PV is done), so a slow stage does not stall the two behind it.
// Handshakes are mbarriers; every wait gives up after ~1 s, sets
// SPLASH_DEVICE_TIMEOUT and lets the CTA drain and free its TMEM.
#include "splash_common.cuh"

namespace splash {
namespace tc {

constexpr int kTileKeys = 64;
constexpr int kPagesPerTile = kTileKeys / kPageSize;
constexpr int kStages = 2;                    // S/P buffers in TMEM, fp16 K tiles
constexpr int kVStages = 3;                   // fp16 V tiles and the scale arrays
constexpr int kRing = 2;                      // int8 staging stages
constexpr int kSoftmaxWarps = 4;
constexpr int kLoadWarps = 8;
constexpr int kLoadThreads = 32 * kLoadWarps;
constexpr int kMmaWarp = kSoftmaxWarps + kLoadWarps;
constexpr int kProducerWarp = kMmaWarp + 1;
constexpr int kThreads = 32 * (kProducerWarp + 1);
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;          // lazy rescale threshold (factor 256)
constexpr unsigned long long kWaitNs = 1000000000ull;

template <int D>
struct Cfg {
  static constexpr int kTileBytes = kTileKeys * D * 2;          // fp16 tile
  static constexpr int kQCol = 0;                                // Q': D/2 columns
  static constexpr int kSCol = D / 2;                            // S[2]: 64 columns each
  static constexpr int kOCol = D / 2 + 2 * kTileKeys;            // O: D columns
  static_assert(kOCol + D <= (int)kTmemCols, "TMEM budget");
  // staging ring stage: K codes [64][D], V codes [64][D]
  static constexpr int kRingCodes = kTileKeys * D;
  static constexpr int kRingStage = 2 * kRingCodes;
  // dynamic shared memory (offsets from a 1024-byte aligned base)
  static constexpr int kOffK = 0;                                        // fp16 K [2]
  static constexpr int kOffV = kOffK + kStages * kTileBytes;             // fp16 V [3]
  static constexpr int kOffRing = kOffV + kVStages * kTileBytes;         // int8 [2]
  static constexpr int kOffScales = kOffRing + kRing * kRingStage;       // fp32 [3][2][64]
  static constexpr int kOffBars = kOffScales + kVStages * 2 * kTileKeys * 4;
  static constexpr int kBarBytes = 512;
  static constexpr int kSmemUsed = kOffBars + kBarBytes;
  // + up to 1 KB to align the base (the kernel checks the room it got); at
  // least 120 KB so that one CTA (and its 512 TMEM columns) owns the SM
  static constexpr int kSmemMax = 227 * 1024;
  static constexpr int kSmemAligned = kSmemUsed + 1024 < kSmemMax ? kSmemUsed + 1024 : kSmemMax;
  static constexpr int kSmemBytes = kSmemAligned > 120 * 1024 ? kSmemAligned : 120 * 1024;
  static_assert(kSmemUsed <= kSmemMax, "shared memory budget");
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

struct Sync {
  volatile int* abort_flag;
  int* status;
  // Bounded wait for the phase of `parity` to complete. false = gave up.
  __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
      if (mbar_try_wait(bar, parity)) return true;
      if (*abort_flag) return false;
      if (global_ns() - t0 > kWaitNs) {
        *abort_flag = 1;
        report(status, SPLASH_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
};

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// smem matrix descriptor, 128-byte swizzle (sm_100 encoding, version 1)
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// instruction descriptor: kind::f16, fp16 A and B, fp32 D, A K-major
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int b_mn_major) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (0u << 15) | ((uint32_t)b_mn_major << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

#define SPLASH_R8(i) "=r"(v[i]), "=r"(v[i + 1]), "=r"(v[i + 2]), "=r"(v[i + 3]), \
                     "=r"(v[i + 4]), "=r"(v[i + 5]), "=r"(v[i + 6]), "=r"(v[i + 7])
#define SPLASH_W8(i) "r"(v[i]), "r"(v[i + 1]), "r"(v[i + 2]), "r"(v[i + 3]), \
                     "r"(v[i + 4]), "r"(v[i + 5]), "r"(v[i + 6]), "r"(v[i + 7])

// 32 consecutive columns of this thread's lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : SPLASH_R8(0), SPLASH_R8(8), SPLASH_R8(16), SPLASH_R8(24)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};"
      ::"r"(taddr), SPLASH_W8(0), SPLASH_W8(8), SPLASH_W8(16), SPLASH_W8(24)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 4 int8 codes -> 2 x half2 (exact): 1024 + (c + 128) built by byte permute, minus 1152
__device__ __forceinline__ void i8x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));
  const __half2 bias = __floats2half2_rn(1152.f, 1152.f);
  __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
  lo = *reinterpret_cast<uint32_t*>(&ha);
  hi = *reinterpret_cast<uint32_t*>(&hb);
}

// ------------------------------------------------------------- work iteration
struct Seg {
  int b, h, i0, i1, T, ctx, Lk, R, u;
};

struct SegIter {
  const int* stp;
  const int* seq_T;
  const int* seq_ctx;
  int B, G, Hkv;
  int t, t_end;
  __device__ bool next(Seg& s) {
    if (t >= t_end) return false;
    s.b = upper_index(stp, B - 1, t);
    s.T = seq_T[s.b];
    s.ctx = seq_ctx[s.b];
    s.Lk = s.ctx + s.T;
    const int tiles = (s.Lk + kTileKeys - 1) / kTileKeys;
    const int local = t - stp[s.b];
    s.h = local / tiles;
    s.i0 = local % tiles;
    s.i1 = min(tiles, s.i0 + (t_end - t));
    s.R = s.T * G;
    s.u = s.b * Hkv + s.h;
    t += s.i1 - s.i0;
    return true;
  }
};

struct Smem {
  uint64_t ring_full[kRing];      // producer tx -> converters
  uint64_t ring_empty[kRing];     // converters -> producer
  uint64_t sc_full[kVStages];     // producer tx (scales) -> softmax
  uint64_t kv_full[kStages];      // converters -> MMA (fp16 K and V of the tile ready)
  uint64_t k_free[kStages];       // QK done -> converters
  uint64_t v_free[kVStages];      // PV done -> converters, producer (scales)
  uint64_t s_full[kStages];       // QK done -> softmax
  uint64_t p_full[kStages];       // softmax -> MMA
  uint64_t p_free[kStages];       // PV of the buffer's tile done -> MMA (QK may
                                  // overwrite the S/P buffer), softmax (O rescale, epilogue)
  uint64_t q_full;                // softmax (Q' in TMEM) -> MMA
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Producer (one warp): stage tile `it` of segment s. Lanes 0..3 look up the
// tile's page ids in parallel; lanes 0..15 issue one bulk copy each (page
// j = lane/4: K codes, V codes into the ring stage; K scales, V scales into the
// scale arrays). Pages past the sequence end or with an invalid id are
// skipped: their stale codes are finite and the softmax gives their keys
// probability 0 without reading their scales.
template <int D>
__device__ __forceinline__ void stage_tile(const AttnParams& p, const Seg& s, int it,
                                           uint8_t* stage, float* scales, uint32_t ring_bar,
                                           uint32_t scale_bar, int lane) {
  using C = Cfg<D>;
  const int k0 = it * kTileKeys;
  const int32_t* ptab = p.page_table + (size_t)s.b * p.max_pages_per_seq;
  int page = -1;
  if (lane < kPagesPerTile && k0 + kPageSize * lane < s.Lk) {
    page = ptab[(k0 / kPageSize) + lane];
    if (page < 0 || page >= p.num_pages) {
      report(p.device_status, SPLASH_DEVICE_BAD_PAGE);
      page = -1;
    }
  }
  const int mask = (int)(__ballot_sync(0xffffffffu, page >= 0) & ((1u << kPagesPerTile) - 1));
  constexpr uint32_t kBlock = kPageSize * D;          // codes of one (page, head)
  constexpr uint32_t kScaleBlock = kPageSize * 4;
  if (lane == 0) {
    mbar_expect_tx(ring_bar, (uint32_t)__popc(mask) * (2 * kBlock));
    mbar_expect_tx(scale_bar, (uint32_t)__popc(mask) * (2 * kScaleBlock));
  }
  __syncwarp();
  const int j = lane >> 2, kind = lane & 3;
  const int pj = __shfl_sync(0xffffffffu, page, j & (kPagesPerTile - 1));
  if (lane < 4 * kPagesPerTile && pj >= 0) {
    const size_t blk = (size_t)pj * p.num_kv_heads + s.h;
    if (kind == 0)
      bulk_g2s(smem_u32(stage) + j * kBlock, p.k_pages + blk * kBlock, kBlock, ring_bar);
    else if (kind == 1)
      bulk_g2s(smem_u32(stage) + C::kRingCodes + j * kBlock, p.v_pages + blk * kBlock, kBlock,
               ring_bar);
    else if (kind == 2)
      bulk_g2s(smem_u32(scales) + j * kScaleBlock, p.k_scales + blk * kPageSize, kScaleBlock,
               scale_bar);
    else
      bulk_g2s(smem_u32(scales) + kTileKeys * 4 + j * kScaleBlock, p.v_scales + blk * kPageSize,
               kScaleBlock, scale_bar);
  }
}

// Converters: 8 consecutive codes (one key, channels d0..d0+7) per unit; the
// 8 threads of a quarter warp cover one 128-byte swizzled row, so the 16-byte
// stores are free of bank conflicts. fp16 element (key n, d) lives at block
// d/64, row n, 16-byte chunk ((d%64)/8) ^ (n%8) (SWIZZLE_128B, 1024-byte atoms).
template <int D>
__device__ __forceinline__ void convert_codes(const uint8_t* src, uint8_t* dst, int lt) {
  constexpr int kUnits = kTileKeys * D / 8;
  constexpr int kPer = kUnits / kLoadThreads;
  uint2 w[kPer];
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int u = q * kLoadThreads + lt;
    w[q] = *reinterpret_cast<const uint2*>(src + (u / (D / 8)) * D + (u % (D / 8)) * 8);
  }
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int u = q * kLoadThreads + lt;
    const int n = u / (D / 8), c8 = u % (D / 8);
    uint4 h;
    i8x4_to_h2x2(w[q].x, h.x, h.y);
    i8x4_to_h2x2(w[q].y, h.z, h.w);
    const uint32_t a = (c8 / 8) * (kTileKeys * 128) + n * 128 + (((c8 & 7) ^ (n & 7)) << 4);
    *reinterpret_cast<uint4*>(dst + a) = h;
  }
}

// ------------------------------------------------------------------- kernel
template <int D>
__global__ void __launch_bounds__(kThreads, 1) verify_tc_kernel(AttnParams p) {
  using C = Cfg<D>;
  static_assert(sizeof(Smem) <= C::kBarBytes, "barrier area");
  extern __shared__ uint8_t smem_raw[];
  const PlanHeader* hd = reinterpret_cast<const PlanHeader*>(p.ws);
  const int total = hd->total_tiles[kClassTensor];
  const int ncta = hd->ncta[kClassTensor];
  if ((int)blockIdx.x >= ncta) return;
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
  const int B = p.num_seqs, Hkv = p.num_kv_heads, G = p.group;
  const WorkspaceLayout L = make_layout(B, Hkv, D, hd->rows_bound);
  const int* q_off = reinterpret_cast<const int*>(p.ws + L.q_off);
  const int* seq_T = reinterpret_cast<const int*>(p.ws + L.seq_T);
  const int* seq_ctx = reinterpret_cast<const int*>(p.ws + L.seq_ctx);
  const int* stp = reinterpret_cast<const int*>(p.ws + L.stp) + kClassTensor * (B + 1);
  const int* nseg = reinterpret_cast<const int*>(p.ws + L.nseg);
  const int* cfirst = reinterpret_cast<const int*>(p.ws + L.cfirst);
  const int* part_base = reinterpret_cast<const int*>(p.ws + L.part_base);
  float* o_part = reinterpret_cast<float*>(p.ws + L.o_part);
  float* lse_part = reinterpret_cast<float*>(p.ws + L.lse_part);

  if (tid == 0) {
    for (int s = 0; s < kRing; ++s) {
      mbar_init(smem_u32(&sh->ring_full[s]), 1);
      mbar_init(smem_u32(&sh->ring_empty[s]), kLoadThreads);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sh->kv_full[s]), kLoadThreads);
      mbar_init(smem_u32(&sh->k_free[s]), 1);
      mbar_init(smem_u32(&sh->s_full[s]), 1);
      mbar_init(smem_u32(&sh->p_full[s]), 32 * kSoftmaxWarps);
      mbar_init(smem_u32(&sh->p_free[s]), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(smem_u32(&sh->sc_full[s]), 1);
      mbar_init(smem_u32(&sh->v_free[s]), 1);
    }
    mbar_init(smem_u32(&sh->q_full), 32 * kSoftmaxWarps);
    mbar_init(smem_u32(&sh->drain), 1);
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
  const Sync sync{&sh->abort_flag, p.device_status};

  SegIter iter{stp, seq_T, seq_ctx, B, G, Hkv, tile_begin(blockIdx.x, total, ncta),
               tile_begin(blockIdx.x + 1, total, ncta)};

  if (warp < kSoftmaxWarps) {
    // ===================================================== softmax + epilogue
    const int r = tid;                                    // query row = TMEM lane
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    int g = 0;
    Seg s;
    bool ok = true;
    while (ok && iter.next(s)) {
      const bool warp_live = warp * 32 < s.R;
      const bool row_live = r < s.R;
      const int tt = r / G, gg = r % G;
      const int lim = s.ctx + tt;                         // last visible key
      float rowfac = 0.f;
      // Q row -> TMEM (fp16 after an exact power-of-two rescale)
      if (warp_live) {
        const __nv_bfloat16* qrow =
            p.q + ((size_t)(q_off[s.b] + tt) * p.num_q_heads + s.h * G + gg) * D;
        float amax = 0.f;
        if (row_live) {
          for (int d = 0; d < D; d += 8) {
            const uint4 w = *reinterpret_cast<const uint4*>(qrow + d);
            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __bfloat1622float2(h2[e]);
              amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
          }
        }
        // 2^e with max|q| * 2^e in [2^14, 2^15)
        int e = 0;
        if (amax > 0.f) e = 14 - (int)((__float_as_uint(amax) >> 23) & 0xff) + 127;
        if (amax > 0.f && ((__float_as_uint(amax) >> 23) & 0xff) == 0) e = 14 + 126;
        e = max(-126, min(127, e));
        const float up = __uint_as_float((uint32_t)(e + 127) << 23);
        rowfac = p.sm_scale_log2 / up;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 64) {
          uint32_t v[32];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            uint4 w = make_uint4(0, 0, 0, 0);
            if (row_live) w = *reinterpret_cast<const uint4*>(qrow + c0 + 8 * k);
            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const float2 f = __bfloat1622float2(h2[e2]);
              __half2 hv = __floats2half2_rn(f.x * up, f.y * up);
              v[4 * k + e2] = *reinterpret_cast<uint32_t*>(&hv);
            }
          }
          tmem_st32(tmem + lane_base + C::kQCol + c0 / 2, v);
        }
        tmem_wait_st();
      }
      fence_before();
      mbar_arrive(smem_u32(&sh->q_full));

      float m = -INFINITY, l = 0.f;
      for (int it = s.i0; it < s.i1 && ok; ++it, ++g) {
        const int st = g % kStages, vst = g % kVStages;
        ok = sync.wait(smem_u32(&sh->sc_full[vst]), (g / kVStages) & 1) &&
             sync.wait(smem_u32(&sh->s_full[st]), (g / kStages) & 1);
        if (!ok) break;
        fence_after();
        uint32_t pw[32];
        float alpha = 1.f;
        if (warp_live) {
          const int k0 = it * kTileKeys;
          const float4* ks4 = reinterpret_cast<const float4*>(scales + vst * 2 * kTileKeys);
          const float4* vs4 = ks4 + kTileKeys / 4;
          uint32_t s0[32], s1[32];
          tmem_ld32(tmem + lane_base + C::kSCol + st * kTileKeys, s0);
          tmem_ld32(tmem + lane_base + C::kSCol + st * kTileKeys + 32, s1);
          tmem_wait_ld();
          const int nvis = row_live ? min(kTileKeys, lim - k0 + 1) : 0;   // visible keys
          const bool full = nvis == kTileKeys;
          // x = S * sK (packed fp32x2); masked columns -> -inf (their scales
          // are not read: pages past the end may hold anything)
          float2 x[32];
#pragma unroll
          for (int j4 = 0; j4 < 16; ++j4) {
            const float4 kq = ks4[j4];
            const uint32_t* src = j4 < 8 ? &s0[4 * j4] : &s1[4 * j4 - 32];
            x[2 * j4] = __fmul2_rn(make_float2(__uint_as_float(src[0]), __uint_as_float(src[1])),
                                   make_float2(kq.x, kq.y));
            x[2 * j4 + 1] = __fmul2_rn(make_float2(__uint_as_float(src[2]), __uint_as_float(src[3])),
                                       make_float2(kq.z, kq.w));
          }
          if (!full) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (2 * j >= nvis) x[j].x = -INFINITY;
              if (2 * j + 1 >= nvis) x[j].y = -INFINITY;
            }
          }
          float mt = -INFINITY;
#pragma unroll
          for (int j = 0; j < 32; ++j) mt = fmax3(mt, x[j].x, x[j].y);
          const float m_new = fmaxf(m, mt);
          float m_use = m;
          if (m == -INFINITY) {
            m_use = m_new;
          } else if (rowfac * (m_new - m) > kRescaleLog2) {
            alpha = ex2(rowfac * (m - m_new));
            m_use = m_new;
          }
          m = m_use;
          const float base = (m_use == -INFINITY) ? 0.f : rowfac * m_use;
          const float2 rf2 = make_float2(rowfac, rowfac), nb2 = make_float2(-base, -base);
          float2 acc = make_float2(0.f, 0.f);
#pragma unroll
          for (int j4 = 0; j4 < 16; ++j4) {
            float4 vq = vs4[j4];
            if (!full) {      // scales of masked keys are not trusted
              const int j = 4 * j4;
              if (j >= nvis) vq.x = 0.f;
              if (j + 1 >= nvis) vq.y = 0.f;
              if (j + 2 >= nvis) vq.z = 0.f;
              if (j + 3 >= nvis) vq.w = 0.f;
            }
            const float2 e0 = __ffma2_rn(x[2 * j4], rf2, nb2);
            const float2 e1 = __ffma2_rn(x[2 * j4 + 1], rf2, nb2);
            const float2 p0 = make_float2(ex2(e0.x), ex2(e0.y));
            const float2 p1 = make_float2(ex2(e1.x), ex2(e1.y));
            acc = __fadd2_rn(acc, __fadd2_rn(p0, p1));
            const float2 q0 = __fmul2_rn(p0, make_float2(vq.x, vq.y));
            const float2 q1 = __fmul2_rn(p1, make_float2(vq.z, vq.w));
            __half2 h0 = __float22half2_rn(q0), h1 = __float22half2_rn(q1);
            pw[2 * j4] = *reinterpret_cast<uint32_t*>(&h0);
            pw[2 * j4 + 1] = *reinterpret_cast<uint32_t*>(&h1);
          }
          l = l * alpha + (acc.x + acc.y);
        }
        // a rescale of O waits for the previous tile's PV (rare: the running
        // max is only moved when it grows by more than 2^8). p_free of that
        // tile's buffer: its previous phase (PV three tiles back) is complete,
        // so a parity wait cannot be satisfied by an older phase.
        if (it > s.i0 && warp_live && __any_sync(0xffffffffu, alpha != 1.f)) {
          ok = sync.wait(smem_u32(&sh->p_free[(g - 1) % kStages]), ((g - 1) / kStages) & 1);
          if (!ok) break;
          fence_after();
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + C::kOCol + c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
            tmem_st32(tmem + lane_base + C::kOCol + c0, v);
          }
        }
        if (warp_live) {
          tmem_st32(tmem + lane_base + C::kSCol + st * kTileKeys, pw);
          tmem_wait_st();
        }
        fence_before();
        mbar_arrive(smem_u32(&sh->p_full[st]));
      }
      if (!ok) break;
      // epilogue: last PV of the segment complete -> normalise, write out
      ok = sync.wait(smem_u32(&sh->p_free[(g - 1) % kStages]), ((g - 1) / kStages) & 1);
      if (!ok) break;
      fence_after();
      if (warp_live) {
        const int ns = nseg[s.u];
        const long long prow = (long long)part_base[s.u] +
                               (long long)(blockIdx.x - cfirst[s.u]) * s.R + r;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const size_t orow = ((size_t)(q_off[s.b] + tt) * p.num_q_heads + s.h * G + gg);
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + C::kOCol + c0, v);
          tmem_wait_ld();
          if (row_live) {
            if (ns == 1) {
              __nv_bfloat16* dst = p.out + orow * D + c0;
#pragma unroll
              for (int k = 0; k < 32; k += 8) {
                uint4 w;
                __nv_bfloat162 b0 = __floats2bfloat162_rn(__uint_as_float(v[k]) * inv, __uint_as_float(v[k + 1]) * inv);
                __nv_bfloat162 b1 = __floats2bfloat162_rn(__uint_as_float(v[k + 2]) * inv, __uint_as_float(v[k + 3]) * inv);
                __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[k + 4]) * inv, __uint_as_float(v[k + 5]) * inv);
                __nv_bfloat162 b3 = __floats2bfloat162_rn(__uint_as_float(v[k + 6]) * inv, __uint_as_float(v[k + 7]) * inv);
                w.x = *reinterpret_cast<uint32_t*>(&b0);
                w.y = *reinterpret_cast<uint32_t*>(&b1);
                w.z = *reinterpret_cast<uint32_t*>(&b2);
                w.w = *reinterpret_cast<uint32_t*>(&b3);
                *reinterpret_cast<uint4*>(dst + k) = w;
              }
            } else {
              float* dst = o_part + prow * D + c0;
#pragma unroll
              for (int k = 0; k < 32; k += 4)
                *reinterpret_cast<float4*>(dst + k) =
                    make_float4(__uint_as_float(v[k]) * inv, __uint_as_float(v[k + 1]) * inv,
                                __uint_as_float(v[k + 2]) * inv, __uint_as_float(v[k + 3]) * inv);
            }
          }
        }
        if (row_live) {
          const float lse = l > 0.f ? (rowfac * m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
          if (ns == 1) p.lse[orow] = lse;
          else lse_part[prow] = lse;
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
        ok = sync.wait(smem_u32(&sh->ring_full[r]), (g / kRing) & 1);
        if (!ok) break;
        const uint8_t* stage = ring + r * C::kRingStage;
        ok = sync.wait(smem_u32(&sh->k_free[st]), ((g / kStages) & 1) ^ 1);
        if (!ok) break;
        convert_codes<D>(stage, kbuf + st * C::kTileBytes, lt);
        ok = sync.wait(smem_u32(&sh->v_free[vst]), ((g / kVStages) & 1) ^ 1);
        if (!ok) break;
        convert_codes<D>(stage + C::kRingCodes, vbuf + vst * C::kTileBytes, lt);
        mbar_arrive(smem_u32(&sh->ring_empty[r]));
        fence_async_smem();
        mbar_arrive(smem_u32(&sh->kv_full[st]));
      }
    }
  } else if (warp == kProducerWarp) {
    // ============================================================ producer
    int g = 0;
    Seg s;
    bool ok = true;
    while (ok && iter.next(s)) {
      for (int it = s.i0; it < s.i1; ++it, ++g) {
        const int r = g % kRing, vst = g % kVStages;
        if (lane == 0) {
          // ring stage free (converted), scale stage free (PV three tiles back done)
          ok = sync.wait(smem_u32(&sh->ring_empty[r]), ((g / kRing) & 1) ^ 1) &&
               sync.wait(smem_u32(&sh->v_free[vst]), ((g / kVStages) & 1) ^ 1);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        stage_tile<D>(p, s, it, ring + r * C::kRingStage, scales + vst * 2 * kTileKeys,
                      smem_u32(&sh->ring_full[r]), smem_u32(&sh->sc_full[vst]), lane);
      }
    }
  } else {
    // ================================================================= MMA
    if (lane == 0) {
      constexpr uint32_t kIdescQK = idesc_f16(128, kTileKeys, 0);
      constexpr uint32_t kIdescPV = idesc_f16(128, D, 1);
      // descriptors of k-step 0 of every buffer; k-steps add byte offsets >> 4
      uint64_t kdesc[kStages], vdesc[kVStages];
#pragma unroll
      for (int i = 0; i < kStages; ++i) kdesc[i] = sdesc(smem_u32(kbuf + i * C::kTileBytes), 16, 1024);
#pragma unroll
      for (int i = 0; i < kVStages; ++i)
        vdesc[i] = sdesc(smem_u32(vbuf + i * C::kTileBytes), kTileKeys * 128, 1024);
      int g = 0, nsegs = 0;
      Seg s;
      bool ok = true;
      while (ok && iter.next(s)) {
        ok = sync.wait(smem_u32(&sh->q_full), nsegs & 1);
        if (!ok) break;
        fence_after();
        const int n = s.i1 - s.i0;
        // PV(i) and QK(i) are issued in their own orders, each as soon as its
        // inputs are ready (PV first: it frees V buffers). QK(i) overwrites the
        // S/P buffer that PV(i-2) reads as its A operand: issue order does not
        // order that write after the read, so QK(i) waits for PV(i-2) to
        // complete (p_free).
        int nq = 0, np = 0;
        unsigned long long t_idle = 0;
        while (np < n) {
          bool progressed = false;
          if (np < nq) {
            const int gi = g + np, st = gi % kStages, vst = gi % kVStages;
            if (mbar_test_wait(smem_u32(&sh->p_full[st]), (gi / kStages) & 1)) {
              fence_after();
#pragma unroll
              for (int kk = 0; kk < kTileKeys / 16; ++kk)
                mma_ts(tmem + C::kOCol, tmem + C::kSCol + st * kTileKeys + kk * 8,
                       vdesc[vst] + (uint64_t)((kk * 16 * 128) >> 4), kIdescPV,
                       (np == 0 && kk == 0) ? 0u : 1u);
              mma_commit(smem_u32(&sh->v_free[vst]));
              mma_commit(smem_u32(&sh->p_free[st]));
              ++np;
              progressed = true;
            }
          }
          if (nq < n && nq <= np + 1) {
            const int gi = g + nq, st = gi % kStages;
            if (mbar_test_wait(smem_u32(&sh->p_free[st]), ((gi / kStages) & 1) ^ 1) &&
                mbar_test_wait(smem_u32(&sh->kv_full[st]), (gi / kStages) & 1)) {
              fence_after();
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk)
                mma_ts(tmem + C::kSCol + st * kTileKeys, tmem + C::kQCol + kk * 8,
                       kdesc[st] + (uint64_t)(((kk / 4) * (kTileKeys * 128) + (kk % 4) * 32) >> 4),
                       kIdescQK, kk > 0);
              mma_commit(smem_u32(&sh->s_full[st]));
              mma_commit(smem_u32(&sh->k_free[st]));
              ++nq;
              progressed = true;
            }
          }
          if (progressed) {
            t_idle = 0;
          } else {
            if (sh->abort_flag) { ok = false; break; }
            const unsigned long long now = global_ns();
            if (t_idle == 0) {
              t_idle = now;
            } else if (now - t_idle > kWaitNs) {
              sh->abort_flag = 1;
              report(p.device_status, SPLASH_DEVICE_TIMEOUT);
              ok = false;
              break;
            }
          }
        }
        g += n;
        ++nsegs;
      }
      // every MMA issued so far is complete before TMEM is released
      mma_commit(smem_u32(&sh->drain));
      sync.wait(smem_u32(&sh->drain), 0);
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

cudaError_t launch_verify_tc(const AttnParams& p, int rows_cap, int ncta, cudaStream_t stream) {
  (void)rows_cap;
#define SPLASH_TC(DD)                                                                          \
  do {                                                                                         \
    constexpr int smem = tc::Cfg<DD>::kSmemBytes;                                              \
    cudaError_t e = cudaFuncSetAttribute(tc::verify_tc_kernel<DD>,                             \
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);   \
    if (e != cudaSuccess) return e;                                                            \
    tc::verify_tc_kernel<DD><<<ncta, tc::kThreads, smem, stream>>>(p);                        \
  } while (0)
  switch (p.head_dim) {
    case 128: SPLASH_TC(128); break;
    case 256: SPLASH_TC(256); break;
    default: return cudaErrorNotSupported;
  }
#undef SPLASH_TC
  return cudaGetLastError();
}

}  // namespace splash
