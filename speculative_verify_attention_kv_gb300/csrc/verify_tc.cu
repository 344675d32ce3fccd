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
// Warp roles (416 threads):
//   warps 0-3   softmax + epilogue: thread = TMEM lane = query row
//   warps 4-11  loaders: 16-byte loads of int8 pages -> fp16 in registers ->
//               128B-swizzled SMEM tiles (K: K-major, V: MN-major), scales
//   warp  12    TMEM allocation and the single MMA-issuing thread
// Handshakes are mbarriers; every wait gives up after ~1 s, sets
// SPLASH_DEVICE_TIMEOUT and lets the CTA drain and free its TMEM.
#include "splash_common.cuh"

namespace splash {
namespace tc {

constexpr int kTileKeys = 64;
constexpr int kStages = 2;
constexpr int kSoftmaxWarps = 4;
constexpr int kLoadWarps = 8;
constexpr int kLoadThreads = 32 * kLoadWarps;
constexpr int kThreads = 32 * (kSoftmaxWarps + kLoadWarps + 1);
constexpr int kMmaWarp = kSoftmaxWarps + kLoadWarps;
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
  // dynamic shared memory: K[2], V[2] tiles, scales, barriers (+1 KB for alignment)
  static constexpr int kSmemTiles = 2 * kStages * kTileBytes;
  static constexpr int kSmemScales = 2 * kStages * kTileKeys * 4;
  // at least 120 KB so that one CTA (and its 512 TMEM columns) owns the SM
  static constexpr int kSmemUsed = 1024 + kSmemTiles + kSmemScales + 256;
  static constexpr int kSmemBytes = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;
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
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[kStages];
  uint64_t p_full[kStages];
  uint64_t o_done;
  uint64_t q_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

// loader registers for one tile: 4*D/256 chunks of 16 B of K and of V, scales
template <int D>
struct LoadRegs {
  uint4 k[4 * D / kLoadThreads];
  uint4 v[4 * D / kLoadThreads];
  float sk, sv;
  int key0;
};

template <int D>
__device__ __forceinline__ void load_tile(const AttnParams& p, const Seg& s, int it, int lt,
                                          LoadRegs<D>& r) {
  constexpr int kPer = 4 * D / kLoadThreads;
  const int k0 = it * kTileKeys;
  const int32_t* ptab = p.page_table + (size_t)s.b * p.max_pages_per_seq;
  r.key0 = k0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int c = q * kLoadThreads + lt;          // 16-byte chunk of the tile
    const int j = c / D;                          // page of the tile
    const int off = (c % D) * 16;                 // byte in the (page, head) block
    uint4 kk = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
    if (k0 + 16 * j < s.Lk) {
      const int page = ptab[(k0 >> 4) + j];
      if (page >= 0 && page < p.num_pages) {
        const size_t base = ((size_t)page * p.num_kv_heads + s.h) * (kPageSize * D) + off;
        kk = __ldg(reinterpret_cast<const uint4*>(p.k_pages + base));
        vv = __ldg(reinterpret_cast<const uint4*>(p.v_pages + base));
      }
    }
    r.k[q] = kk;
    r.v[q] = vv;
  }
  r.sk = 0.f;
  r.sv = 0.f;
  if (lt < kTileKeys) {
    const int key = k0 + lt;
    if (key < s.Lk) {
      const int page = ptab[key >> 4];
      if (page >= 0 && page < p.num_pages) {
        const size_t si = ((size_t)page * p.num_kv_heads + s.h) * kPageSize + (key & 15);
        r.sk = __ldg(p.k_scales + si);
        r.sv = __ldg(p.v_scales + si);
      } else {
        report(p.device_status, SPLASH_DEVICE_BAD_PAGE);
      }
    }
  }
}

// fp16 tile element (key n, d) lives at block d/64, row n, 16-byte chunk
// ((d%64)/8) ^ (n%8) of that 128-byte row (SWIZZLE_128B, 1024-byte atoms)
template <int D>
__device__ __forceinline__ void store_tile(const LoadRegs<D>& r, int lt, uint8_t* kbuf,
                                           uint8_t* vbuf, float* ks, float* vs) {
  constexpr int kPer = 4 * D / kLoadThreads;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int c = q * kLoadThreads + lt;
    const int j = c / D;
    const int off = (c % D) * 16;
    const int n = 16 * j + off / D;               // key within the tile
    const int d0 = off % D;                       // first of 16 channels
    const int blk = d0 / 64;
    const int c16 = (d0 % 64) / 8;
    const uint32_t row = blk * (kTileKeys * 128) + n * 128;
    const uint32_t a0 = row + (((c16) ^ (n & 7)) << 4);
    const uint32_t a1 = row + (((c16 + 1) ^ (n & 7)) << 4);
    uint4 h0, h1;
    i8x4_to_h2x2(r.k[q].x, h0.x, h0.y);
    i8x4_to_h2x2(r.k[q].y, h0.z, h0.w);
    i8x4_to_h2x2(r.k[q].z, h1.x, h1.y);
    i8x4_to_h2x2(r.k[q].w, h1.z, h1.w);
    *reinterpret_cast<uint4*>(kbuf + a0) = h0;
    *reinterpret_cast<uint4*>(kbuf + a1) = h1;
    i8x4_to_h2x2(r.v[q].x, h0.x, h0.y);
    i8x4_to_h2x2(r.v[q].y, h0.z, h0.w);
    i8x4_to_h2x2(r.v[q].z, h1.x, h1.y);
    i8x4_to_h2x2(r.v[q].w, h1.z, h1.w);
    *reinterpret_cast<uint4*>(vbuf + a0) = h0;
    *reinterpret_cast<uint4*>(vbuf + a1) = h1;
  }
  if (lt < kTileKeys) {
    ks[lt] = r.sk;
    vs[lt] = r.sv;
  }
}

// ------------------------------------------------------------------- kernel
template <int D>
__global__ void __launch_bounds__(kThreads, 1) verify_tc_kernel(AttnParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* kbuf = smem;                                   // [kStages][tile]
  uint8_t* vbuf = smem + kStages * C::kTileBytes;         // [kStages][tile]
  float* kscale = reinterpret_cast<float*>(smem + C::kSmemTiles);   // [kStages][64]
  float* vscale = kscale + kStages * kTileKeys;                     // [kStages][64]
  Smem* sh = reinterpret_cast<Smem*>(smem + C::kSmemTiles + C::kSmemScales);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = p.num_seqs, Hkv = p.num_kv_heads, G = p.group;
  const PlanHeader* hd = reinterpret_cast<const PlanHeader*>(p.ws);
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

  const int total = hd->total_tiles[kClassTensor];
  const int ncta = hd->ncta[kClassTensor];
  if ((int)blockIdx.x >= ncta) return;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sh->kv_full[s]), kLoadThreads);
      mbar_init(smem_u32(&sh->kv_empty[s]), 1);
      mbar_init(smem_u32(&sh->s_full[s]), 1);
      mbar_init(smem_u32(&sh->p_full[s]), 32 * kSoftmaxWarps);
    }
    mbar_init(smem_u32(&sh->o_done), 1);
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
    int g = 0, nsegs = 0;
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
        if (amax > 0.f && ((__float_as_uint(amax) >> 23) & 0xff) == 0) e = 14 + 126;  // subnormal max
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
        const int st = g % kStages;
        const uint32_t ph = (g / kStages) & 1;
        ok = sync.wait(smem_u32(&sh->kv_full[st]), ph) && sync.wait(smem_u32(&sh->s_full[st]), ph);
        if (!ok) break;
        fence_after();
        uint32_t pw[32];
        float alpha = 1.f;
        if (warp_live) {
          const int k0 = it * kTileKeys;
          const float* ks = kscale + st * kTileKeys;
          const float* vs = vscale + st * kTileKeys;
          uint32_t s0[32], s1[32];
          tmem_ld32(tmem + lane_base + C::kSCol + st * kTileKeys, s0);
          tmem_ld32(tmem + lane_base + C::kSCol + st * kTileKeys + 32, s1);
          tmem_wait_ld();
          float x[64];
          float mt = -INFINITY;
          const int nvis = row_live ? min(kTileKeys, lim - k0 + 1) : 0;   // visible keys in tile
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const float sj = __uint_as_float(j < 32 ? s0[j] : s1[j - 32]);
            x[j] = (j < nvis) ? sj * ks[j] : -INFINITY;
            mt = fmaxf(mt, x[j]);
          }
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
          float sum = 0.f;
#pragma unroll
          for (int j = 0; j < 64; j += 2) {
            const float p0 = (j < nvis) ? ex2(fmaf(rowfac, x[j], -base)) : 0.f;
            const float p1 = (j + 1 < nvis) ? ex2(fmaf(rowfac, x[j + 1], -base)) : 0.f;
            sum += p0 + p1;
            __half2 hv = __floats2half2_rn(p0 * vs[j], p1 * vs[j + 1]);
            pw[j / 2] = *reinterpret_cast<uint32_t*>(&hv);
          }
          l = l * alpha + sum;
        }
        // PV of the previous tile has to be complete before O is rescaled
        if (it > s.i0) {
          ok = sync.wait(smem_u32(&sh->o_done), (g - 1) & 1);
          if (!ok) break;
          fence_after();
          if (warp_live && __any_sync(0xffffffffu, alpha != 1.f)) {
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
      ok = sync.wait(smem_u32(&sh->o_done), (g - 1) & 1);
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
      ++nsegs;
    }
  } else if (warp < kSoftmaxWarps + kLoadWarps) {
    // ============================================================== loaders
    const int lt = tid - 32 * kSoftmaxWarps;
    int g = 0;
    Seg s;
    bool have = iter.next(s);
    int it = have ? s.i0 : 0;
    LoadRegs<D> ra, rb;
    if (have) load_tile<D>(p, s, it, lt, ra);
    bool ok = true;
    auto step = [&](LoadRegs<D>& cur, LoadRegs<D>& nxt) -> bool {
      // advance to the next tile and prefetch it
      Seg s2 = s;
      int it2 = it + 1;
      bool have2 = true;
      if (it2 >= s.i1) {
        have2 = iter.next(s2);
        it2 = have2 ? s2.i0 : 0;
      }
      if (have2) load_tile<D>(p, s2, it2, lt, nxt);
      const int st = g % kStages;
      if (!sync.wait(smem_u32(&sh->kv_empty[st]), ((g / kStages) & 1) ^ 1)) return false;
      store_tile<D>(cur, lt, kbuf + st * C::kTileBytes, vbuf + st * C::kTileBytes,
                    kscale + st * kTileKeys, vscale + st * kTileKeys);
      fence_async_smem();
      mbar_arrive(smem_u32(&sh->kv_full[st]));
      ++g;
      s = s2;
      it = it2;
      have = have2;
      return true;
    };
    while (have && ok) {
      ok = step(ra, rb);
      if (!have || !ok) break;
      ok = step(rb, ra);
    }
  } else {
    // ================================================================= MMA
    if (lane == 0) {
      constexpr uint32_t kIdescQK = idesc_f16(128, kTileKeys, 0);
      constexpr uint32_t kIdescPV = idesc_f16(128, D, 1);
      int g = 0, nsegs = 0;
      Seg s;
      bool ok = true;
      while (ok && iter.next(s)) {
        ok = sync.wait(smem_u32(&sh->q_full), nsegs & 1);
        if (!ok) break;
        fence_after();
        const int n = s.i1 - s.i0;
        auto issue_qk = [&](int gi) -> bool {
          const int st = gi % kStages;
          if (!sync.wait(smem_u32(&sh->kv_full[st]), (gi / kStages) & 1)) return false;
          fence_after();
          const uint32_t kaddr = smem_u32(kbuf + st * C::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t bd = sdesc(kaddr + (kk / 4) * (kTileKeys * 128) + (kk % 4) * 32, 16, 1024);
            mma_ts(tmem + C::kSCol + st * kTileKeys, tmem + C::kQCol + kk * 8, bd, kIdescQK,
                   kk > 0);
          }
          mma_commit(smem_u32(&sh->s_full[st]));
          return true;
        };
        auto issue_pv = [&](int gi, bool first) -> bool {
          const int st = gi % kStages;
          if (!sync.wait(smem_u32(&sh->p_full[st]), (gi / kStages) & 1)) return false;
          fence_after();
          const uint32_t vaddr = smem_u32(vbuf + st * C::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < kTileKeys / 16; ++kk) {
            const uint64_t bd = sdesc(vaddr + kk * 16 * 128, kTileKeys * 128, 1024);
            mma_ts(tmem + C::kOCol, tmem + C::kSCol + st * kTileKeys + kk * 8, bd, kIdescPV,
                   (first && kk == 0) ? 0u : 1u);
          }
          mma_commit(smem_u32(&sh->kv_empty[st]));
          mma_commit(smem_u32(&sh->o_done));
          return true;
        };
        ok = issue_qk(g);
        for (int i = 1; i < n && ok; ++i) {
          ok = issue_qk(g + i);
          if (ok) ok = issue_pv(g + i - 1, i == 1);
        }
        if (ok) ok = issue_pv(g + n - 1, n == 1);
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
