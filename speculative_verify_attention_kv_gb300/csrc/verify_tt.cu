// Tensor-core verify attention, transposed orientation (sm_103a, tcgen05 +
// TMEM), for head_dim 256 and at most 96 query rows per (sequence, KV head).
//
// One persistent CTA per SM walks its share of the stream of 128-key tiles.
// For a unit (sequence b, KV head h) with R = T*G query rows (row r = t*G + g)
// the key tile is the 128-row M side of both products and the query rows are
// the N side, N = R rounded up to 16, so no row is padded to 128:
//
//   S^T[key, r] = K^ . Q'^T      A = K^ (TMEM, lane = key), B = Q'^T (smem, K-major)
//   x = S^T * sK_key * f         f = sm_scale*log2(e) / 2^e_u   (log2 units)
//   w = 2^(x - m_r)              m_r: the row's reference point (below)
//   O^T[d, r] += V^T . P^T       A = V^T (smem, MN-major), B = P^T = w*sV (smem, MN-major)
//   l_r += w;   O = O^T / l,  LSE = (m_r + log2 l) * ln 2
//
// Q' = Q * 2^e_u with one power of two per unit, chosen so max|Q'| lies in
// [2^14, 2^15): the bf16 query enters the fp16 MMA exactly (int8 codes are
// exact in fp16). The K scale multiplies the score of its key (one scalar per
// softmax thread); the V scale is folded into P before P is rounded to fp16.
// Each KV tile is read from its pages once and serves every query head of
// the GQA group and every verify token of the block.
//
// Reference points. Any m_r gives the same O and LSE as long as O^T and l
// use it alike; it is chosen so that the fp16 operand P = 2^(x - m_r) * sV
// stays in range for any magnitude of V: m_r is the running maximum over the
// keys row r sees of max(x + log2 sV - 7, x - 100), moved only when a tile
// breaks the bound (then O^T and l are rescaled by 2^(m_old - m_new)). Only
// keys visible to a row move its reference point. Each tile is first checked
// (x - m_r + log2 sV <= 15 and x - m_r <= 100 for every visible key); the
// common case needs no row reduction at all. When the check fails (the first
// tile of every segment, and rare jumps), all softmax warps take the slow
// path: the tile's row candidates by a cross-lane reduction, then the O^T
// rescale.
//
// Warp roles (512 threads):
//   warps 0-7   softmax + epilogue: warp w reads TMEM lane quarter w%4 (keys
//               32(w%4)..+31 of the tile), columns (rows) 48(w/4)..+47
//   warps 8-11  K converters: warp 8+q issues the tensor-map loads of its two
//               pages of each tile and their K / V scales (cp.async), two
//               tiles ahead (swizzled staging), then turns its 32 keys' int8
//               K codes into the fp16 A operand in TMEM lanes 32q..+31
//   warps 12,13,15  V converters: int8 V codes -> fp16 V^T, 16 keys at a
//               time into a ring of 4 buffers (conversion runs up to half a
//               tile ahead of PV); warp 12 also issues the V-code tensor-map
//               loads (4 pages = 64 keys per stage)
//   warp  14    lane 0 issues every MMA: QK^T (16 per tile) and PV (16 per
//               tile, 2 per 16 keys), whichever is ready first
// TMEM (512 columns): K^ 128 | S^T x2 (96 each) | O^T d-halves x2 (96 each).
// Every cross-warp handshake is an mbarrier with a bounded wait.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "tcgen05_ptx.cuh"

namespace splash {
namespace tt {
using namespace dev;

constexpr int D = 256;
constexpr int kTileKeys = 128;
constexpr int kNMax = 96;                  // query rows per unit this kernel takes
constexpr int kSubKeys = 64;               // keys per V stage
constexpr int kVtKeys = 16;                // keys per V^T buffer (one PV step)
constexpr int kVtBufs = 4;
constexpr int kSoftmaxWarps = 8;
constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
constexpr int kKConvWarp0 = 8;
constexpr int kVConvWarp0 = 12;            // warps 12, 13 and 15
constexpr int kVConvThreads = 96;
constexpr int kMmaWarp = 14;
constexpr int kThreads = 512;
constexpr int kKDepth = 2;                 // tiles of K staging per K converter
constexpr int kVRing = 2;                  // V stages (64 keys each)
constexpr int kScSlots = 4;                // scale slots (one tile each)
constexpr float kPTop = 7.0f;              // a slow path puts the tile's largest P at 2^7
constexpr float kPLimit = 15.0f;           // fast path while P <= 2^15 (fp16 max ~2^16)
constexpr float kWLimit = 100.0f;          // and the weights w stay <= 2^100 (fp32 sums)
constexpr float kMInit = -1.0e30f;         // "no key seen yet" (finite: no inf - inf)

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColK = 0;              // K^: 128 columns (256 d as fp16 pairs)
constexpr uint32_t kColS = 128;            // S^T buffers: + buf * kNMax
constexpr uint32_t kColO = 128 + 2 * kNMax;  // O^T: + d_half * kNMax
static_assert(kColO + 2 * kNMax == kTmemCols, "TMEM budget");

// Shared memory (offsets from a 1024-byte aligned base). Staged code pages
// keep the pool's row order, [128-byte half of the row][slot][128 B], with
// 16-byte chunk c of a row stored at chunk c ^ (slot & 7) (the tensor map's
// 128-byte swizzle), so the converters' reads are free of bank conflicts.
constexpr int kPageHalf = 16 * 128;                    // one half of 16 rows: 2 KB
constexpr int kPageBytes = 2 * kPageHalf;              // 16 rows x 256 B: 4 KB
constexpr int kKStage = 2 * kPageBytes;                // a K converter's 2 pages: 8 KB
constexpr int kVStage = 4 * kPageBytes;                // 4 pages: 16 KB
constexpr int kVtBytes = D * kVtKeys * 2;              // V^T [d-atom 4][key 16][128 B]: 8 KB
constexpr int kVtAtom = kVtKeys * 128;                 // 2 KB
constexpr int kPHalfBytes = 2 * kSubKeys * 128;        // P^T [row-atom 2][key 64][128 B]: 16 KB
constexpr int kPAtom = kSubKeys * 128;                 // 8 KB
constexpr int kQAtom = kNMax * 128;                    // Q'^T [d-atom 4][row 96][128 B]: 12 KB
constexpr int kOffKst = 0;
constexpr int kOffVst = kOffKst + 4 * kKDepth * kKStage;
constexpr int kOffVt = kOffVst + kVRing * kVStage;
constexpr int kOffP = kOffVt + kVtBufs * kVtBytes;
constexpr int kOffQ = kOffP + 2 * kPHalfBytes;
constexpr int kOffSc = kOffQ + 4 * kQAtom;             // [slot][K 128 | V 128] fp32
constexpr int kOffRed = kOffSc + kScSlots * 2 * kTileKeys * 4;
constexpr int kRedBytes = (4 * 128 + 3 * 128 + 64) * 4;
constexpr int kOffBars = kOffRed + kRedBytes;
constexpr int kBarBytes = 512;
constexpr int kSmemUsed = kOffBars + kBarBytes;
constexpr int kSmemBytes = kSmemUsed + 1024;           // + room to align the base
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kOffQ % 1024 == 0 && kQAtom % 1024 == 0 && kOffP % 1024 == 0 &&
              kOffVt % 1024 == 0 && kOffVst % 1024 == 0, "swizzled operands are 1 KB aligned");

struct Red {                    // softmax scratch
  float part[4][128];           // per lane quarter: column candidates / sums
  float m[128];                 // row reference points (log2 units)
  float alpha[128];             // O^T / l rescale of the slow path
  float osc[128];               // epilogue: 1 / l
  float wmax[8];                // per softmax warp: max |q|
  volatile int slow_tile[2];    // by tile parity: the tile whose check failed. Two
                                // slots: a warp may vote on tile g + 1 before a
                                // slower one has read the decision for tile g
};
static_assert(sizeof(Red) <= kRedBytes, "scratch");

struct Bars {
  uint64_t kst_full[4][kKDepth];  // K converter q's copies of a tile landed (tx)
  uint64_t kt_full;               // K^ of the tile in TMEM (one arrival per warp)
  uint64_t kt_free;               // QK^T done reading K^ (MMA commit)
  uint64_t vst_full[kVRing];      // V stage landed (tx)
  uint64_t vst_empty[kVRing];     // V converters done with a stage (3 warps)
  uint64_t sc_full[kScSlots];     // scales of a tile landed (128 cp.async arrivals)
  uint64_t sc_free[kScSlots];     // softmax done with the scales (8 warps)
  uint64_t s_full[2];             // QK^T done (commit)
  uint64_t s_free[2];             // softmax done reading S^T (8 warps)
  uint64_t p_full[2];             // P^T half written (4 warps)
  uint64_t p_free[2];             // PV of that half done (commit)
  uint64_t vt_full[kVtBufs];      // V^T buffer written (3 warps)
  uint64_t vt_free[kVtBufs];      // PV of that buffer done (commit)
  uint64_t o_done[2];             // all PVs of a tile done (commit), by tile parity
  uint64_t o_free;                // epilogue done reading O^T (8 warps)
  uint64_t q_full;                // Q'^T of the segment in smem (8 warps)
  uint64_t smx;                   // barrier of the softmax warps (8 warps)
  uint64_t drain;                 // the MMA issuer's MMAs complete
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= kBarBytes, "barrier area");

// ---------------------------------------------------------- tile stream
struct Seg {
  int b, h, i0, i1, T, ctx, Lk, R, u;
  int klo;                        // first key any row of the unit sees
};

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

// Page ids of a sequence, 32 at a time (lane l holds entry base + l; -1 past
// the pages the sequence needs); the next window is fetched ahead.
struct PageWindow {
  int b = -1, base = 0, cur = -1;
  int nb = -1, nbase = 0, nxt = -1;
  __device__ __forceinline__ static int fetch(const AttnParams& p, int b, int base, int npages,
                                              int lane) {
    const int i = base + lane;
    return i < npages ? p.page_table[(size_t)b * p.max_pages_per_seq + i] : -1;
  }
  // entries [first, first + 4) of sequence b; returns entry first + (lane & 3)
  __device__ __forceinline__ int get(const AttnParams& p, int sb, int first, int npages,
                                     int lane) {
    const int want = first & ~31;
    if (sb != b || want != base) {
      cur = (sb == nb && want == nbase) ? nxt : fetch(p, sb, want, npages, lane);
      b = sb;
      base = want;
      nb = sb;
      nbase = want + 32;
      nxt = fetch(p, sb, nbase, npages, lane);
    }
    return __shfl_sync(0xffffffffu, cur, (first - base) + (lane & 3));
  }
};

// Page id of page `pg` (lane & 3 selects among first..first+3) if the page
// holds a key in [klo, Lk) and its id is valid, else -1 (a needed page with
// an invalid id is reported).
__device__ __forceinline__ int needed_page(const AttnParams& p, const Seg& s, int first_page,
                                           int lane_sel_ok, int id, int lane) {
  const int k0 = (first_page + (lane & 3)) * kPageSize;
  const bool needed = lane_sel_ok && k0 < s.Lk && k0 + kPageSize > s.klo;
  if (needed && (id < 0 || id >= p.num_pages)) {
    report(p.device_status, SPLASH_DEVICE_BAD_PAGE);
    return -1;
  }
  return needed ? id : -1;
}

// Cross-lane reduction of 16 values per lane (one column each) over the 32
// lanes: afterwards lanes 2i and 2i+1 hold the reduction of column
// 8*b4 + 4*b3 + 2*b2 + b1 (b_k = bit k of the lane). 16 shuffles.
template <bool kMax>
__device__ __forceinline__ float reduce_scatter16(const float (&v)[16], int lane) {
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
  float a8[8], a4[4], a2[2];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float send = b4 ? v[i] : v[8 + i], keep = b4 ? v[8 + i] : v[i];
    a8[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = b3 ? a8[i] : a8[4 + i], keep = b3 ? a8[4 + i] : a8[i];
    a4[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = b2 ? a4[i] : a4[2 + i], keep = b2 ? a4[2 + i] : a4[i];
    a2[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
  }
  const float send = b1 ? a2[0] : a2[1], keep = b1 ? a2[1] : a2[0];
  const float a1 = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
  return op(a1, __shfl_xor_sync(0xffffffffu, a1, 1));
}
__device__ __forceinline__ int scatter_col(int lane) {
  return 8 * ((lane >> 4) & 1) + 4 * ((lane >> 3) & 1) + 2 * ((lane >> 2) & 1) + ((lane >> 1) & 1);
}

// ------------------------------------------------------------------- kernel
template <bool kSwa>
__global__ void __launch_bounds__(kThreads, 1)
verify_tt_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmap) {
  extern __shared__ uint8_t smem_raw[];
  grid_dependency_wait();          // the split plan is complete
  allow_dependent_launch();
  const PlanHeader* hd = reinterpret_cast<const PlanHeader*>(p.ws);
  const int ncta = hd->ncta[kClassTensor];
  if ((int)blockIdx.x >= ncta) return;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  if (smem - smem_raw + kSmemUsed > kSmemBytes) {
    if (threadIdx.x == 0) report(p.device_status, SPLASH_DEVICE_INTERNAL);
    return;
  }
  uint8_t* kst = smem + kOffKst;
  uint8_t* vst = smem + kOffVst;
  uint8_t* vtb = smem + kOffVt;
  uint8_t* pbuf = smem + kOffP;
  uint8_t* qbuf = smem + kOffQ;
  float* scales = reinterpret_cast<float*>(smem + kOffSc);
  Red* rd = reinterpret_cast<Red*>(smem + kOffRed);
  Bars* sh = reinterpret_cast<Bars*>(smem + kOffBars);

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
    for (int q = 0; q < 4; ++q)
      for (int d = 0; d < kKDepth; ++d) mbar_init(smem_u32(&sh->kst_full[q][d]), 1);
    mbar_init(smem_u32(&sh->kt_full), 4);
    mbar_init(smem_u32(&sh->kt_free), 1);
    for (int i = 0; i < kVRing; ++i) {
      mbar_init(smem_u32(&sh->vst_full[i]), 1);
      mbar_init(smem_u32(&sh->vst_empty[i]), kVConvThreads / 32);
    }
    for (int i = 0; i < kScSlots; ++i) {
      mbar_init(smem_u32(&sh->sc_full[i]), 128);
      mbar_init(smem_u32(&sh->sc_free[i]), kSoftmaxWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sh->s_full[i]), 1);
      mbar_init(smem_u32(&sh->s_free[i]), kSoftmaxWarps);
      mbar_init(smem_u32(&sh->p_full[i]), kSoftmaxWarps / 2);
      mbar_init(smem_u32(&sh->p_free[i]), 1);
      mbar_init(smem_u32(&sh->o_done[i]), 1);
    }
    for (int i = 0; i < kVtBufs; ++i) {
      mbar_init(smem_u32(&sh->vt_full[i]), kVConvThreads / 32);
      mbar_init(smem_u32(&sh->vt_free[i]), 1);
    }
    mbar_init(smem_u32(&sh->o_free), kSoftmaxWarps);
    mbar_init(smem_u32(&sh->q_full), kSoftmaxWarps);
    mbar_init(smem_u32(&sh->smx), kSoftmaxWarps);
    mbar_init(smem_u32(&sh->drain), 1);
    sh->abort_flag = 0;
    rd->slow_tile[0] = rd->slow_tile[1] = -1;
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
  const int window = kSwa ? p.window : 0;
  const int* cst = reinterpret_cast<const int*>(p.ws + L.cta_start) + kClassTensor * (kMaxCtas + 1);
  SegIter iter{stp, seq_T, seq_ctx, B, G, Hkv, window, cst[blockIdx.x], cst[blockIdx.x + 1]};

  // Register split: the softmax warpgroups (warps 0-7) take 160 registers a
  // thread, the converter / MMA warpgroups 96: 256 x 160 + 256 x 96 = 65536,
  // the launch's 512 x 128. Each warpgroup changes its share uniformly.
  if (warp < kSoftmaxWarps) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 160;" ::: "memory");
    // ===================================================== softmax + epilogue
    const int q = warp & 3, part = warp >> 2, st = tid;
    const int cb = 48 * part;                             // first column (row) of this thread
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    const int kl = 32 * (q & 1) + lane;                   // key within its 64-key half
    const uint32_t smx = smem_u32(&sh->smx);
    int g = 0, sbp = 0, nsg = 0;
    Seg s;
    bool ok = true;
    auto smx_sync = [&]() -> bool {
      warp_arrive(smx, lane);
      const bool r = __all_sync(0xffffffffu, sync.wait(smx, sbp & 1));
      ++sbp;
      return r;
    };
    while (ok && iter.next(s)) {
      const int R = s.R;
      const int N = (R + 15) & ~15;
      // ---- Q' = Q * 2^e (one exponent for the unit) -> Q'^T, K-major fp16
      float rowfac;
      {
        uint4 qv[12];
        uint32_t amax_bits = 0;
        const int nch = R * 32;                           // 16-byte chunks of the unit's Q rows
#pragma unroll
        for (int k = 0; k < 12; ++k) {
          const int ch = st + kSoftmaxThreads * k;
          qv[k] = make_uint4(0u, 0u, 0u, 0u);
          if (ch < nch) {
            const int r = ch >> 5, c = ch & 31;
            const int t = r / G, gg = r - t * G;
            const uint4* src = reinterpret_cast<const uint4*>(
                p.q + ((size_t)(q_off[s.b] + t) * p.num_q_heads + s.h * G + gg) * D) + c;
            qv[k] = __ldg(src);
            const uint32_t w[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
              amax_bits = max(amax_bits, max(w[i] & 0x7fffu, (w[i] >> 16) & 0x7fffu));
          }
        }
        float amax = __uint_as_float(amax_bits << 16);
        amax = warp_max(amax);
        if (lane == 0) rd->wmax[warp] = amax;
        ok = smx_sync();                                  // previous segment fully done too
        if (!ok) break;
#pragma unroll
        for (int w = 0; w < kSoftmaxWarps; ++w) amax = fmaxf(amax, rd->wmax[w]);
        int e = 0;
        const int ex = (int)((__float_as_uint(amax) >> 23) & 0xff);
        if (amax > 0.f) e = ex == 0 ? 14 + 126 : 14 - ex + 127;
        e = max(-126, min(127, e));
        const float up = __uint_as_float((uint32_t)(e + 127) << 23);
        rowfac = p.sm_scale_log2 / up;
#pragma unroll
        for (int k = 0; k < 12; ++k) {
          const int ch = st + kSoftmaxThreads * k;
          if (ch < N * 32) {
            const int r = ch >> 5, c = ch & 31;
            uint32_t w[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
              __half2 hv = __floats2half2_rn(f.x * up, f.y * up);
              w[i] = *reinterpret_cast<uint32_t*>(&hv);
            }
            *reinterpret_cast<uint4*>(qbuf + (c >> 3) * kQAtom + r * 128 + (((c & 7) ^ (r & 7)) << 4)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        if (st < 128) rd->m[st] = kMInit;
        fence_async_smem();
        warp_arrive(smem_u32(&sh->q_full), lane);
        ok = smx_sync();
        if (!ok) break;
      }
      ++nsg;
      const bool live = cb < R;                           // this warp's columns hold rows
      float lsum[48];
#pragma unroll
      for (int i = 0; i < 48; ++i) lsum[i] = 0.f;

      for (int it = s.i0; it < s.i1 && ok; ++it, ++g) {
        const int ssl = g % kScSlots;
        ok = sync.wait(smem_u32(&sh->sc_full[ssl]), (g / kScSlots) & 1) &&
             sync.wait(smem_u32(&sh->s_full[g & 1]), (g >> 1) & 1);
        ok = __all_sync(0xffffffffu, ok);       // a timeout seen by some lanes stops the warp
        if (!ok) break;
        fence_after();
        const int j = it * kTileKeys + 32 * q + lane;     // this thread's key
        const bool kvalid = j < s.Lk && j >= (s.klo & ~(kPageSize - 1));
        const float* sc = scales + ssl * 2 * kTileKeys;
        const float ksc = kvalid ? sc[32 * q + lane] : 0.f;
        const float vsc = kvalid ? sc[kTileKeys + 32 * q + lane] : 0.f;
        warp_arrive(smem_u32(&sh->sc_free[ssl]), lane);
        // rows that see key j: t >= j - ctx (and t < j - ctx + W with a window)
        int c_lo = R, c_hi = 0;
        if (kvalid) {
          c_lo = max(0, j - s.ctx) * G;
          c_hi = R;
          if (kSwa) c_hi = min(R, max(0, j - s.ctx + window) * G);
        }
        const bool all_vis = __all_sync(0xffffffffu, c_lo <= cb && c_hi >= cb + 48);
        const float kf = ksc * rowfac;
        const float lv = __log2f(vsc);                    // -inf for a zero (or untrusted) scale
        const uint32_t s_addr = tmem + lane_off + kColS + (uint32_t)((g & 1) * kNMax + cb);

        // ---- pass 1: does any visible key break its row's bounds? (the
        // TMEM load of the next 16 columns is in flight while one is checked)
        float tmx = -INFINITY;
        if (live) {
          auto check = [&](const uint32_t (&sv)[16], int k) {
            const float4* mp = reinterpret_cast<const float4*>(rd->m + cb + 16 * k);
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
              const float4 m4 = mp[i4];
              const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int c = cb + 16 * k + 4 * i4 + i;
                float x = __uint_as_float(sv[4 * i4 + i]) * kf - mm[i];
                if (!all_vis && (c < c_lo || c >= c_hi)) x = -INFINITY;
                tmx = fmaxf(tmx, x);
              }
            }
          };
          uint32_t sa[16], sb[16];
          tmem_ld32x32b_x16(s_addr, sa);
          tmem_wait_ld(sa);
          tmem_ld32x32b_x16(s_addr + 16, sb);
          check(sa, 0);
          tmem_wait_ld(sb);
          tmem_ld32x32b_x16(s_addr + 32, sa);
          check(sb, 1);
          tmem_wait_ld(sa);
          check(sa, 2);
        }
        const bool need = tmx + lv > kPLimit || tmx > kWLimit;
        if (__any_sync(0xffffffffu, need) && lane == 0) rd->slow_tile[g & 1] = g;
        ok = smx_sync();
        if (!ok) break;

        if (rd->slow_tile[g & 1] == g) {
          // ---- slow path: the tile's row candidates, new reference points, O^T / l rescale
#pragma unroll
          for (int k = 0; k < 3; ++k) {
            float xv[16];
            if (live) {
              uint32_t sv[16];
              tmem_ld32x32b_x16(s_addr + 16 * k, sv);
              tmem_wait_ld(sv);
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int c = cb + 16 * k + i;
                const float x = __uint_as_float(sv[i]) * kf;
                xv[i] = (c < c_lo || c >= c_hi) ? -INFINITY : fmaxf(x + lv - kPTop, x - kWLimit);
              }
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) xv[i] = -INFINITY;
            }
            const float cm = reduce_scatter16<true>(xv, lane);
            if (!(lane & 1)) rd->part[q][cb + 16 * k + scatter_col(lane)] = cm;
          }
          ok = smx_sync();
          if (!ok) break;
          if (st < 128) {
            const int c = st;
            const float mt = fmaxf(fmaxf(rd->part[0][c], rd->part[1][c]),
                                   fmaxf(rd->part[2][c], rd->part[3][c]));
            const float mo = rd->m[c];
            const float mn = fmaxf(mo, mt);
            rd->alpha[c] = ex2(mo - mn);                  // 0 while nothing was seen
            rd->m[c] = mn;
          }
          ok = smx_sync();
          if (!ok) break;
          if (it > s.i0) {
            // O^T holds the tiles before this one: rescale once their PVs are done
            ok = __all_sync(0xffffffffu, sync.wait(smem_u32(&sh->o_done[(g - 1) & 1]), ((g - 1) >> 1) & 1));
            if (!ok) break;
            fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < kNMax; c0 += 32) {
              uint32_t v[32];
              const uint32_t oa = tmem + lane_off + kColO + (uint32_t)(part * kNMax + c0);
              tmem_ld32x32b_x32(oa, v);
              tmem_wait_ld(v);
#pragma unroll
              for (int i = 0; i < 32; ++i)
                v[i] = __float_as_uint(__uint_as_float(v[i]) * rd->alpha[c0 + i]);
              tmem_st32x32b_x32(oa, v);
            }
            tmem_wait_st();
#pragma unroll
            for (int i = 0; i < 48; ++i) lsum[i] *= rd->alpha[cb + i];
          }
        }

        // ---- pass 2: w = 2^(x - m), row sums, P^T = w * sV (fp16).
        // P^T half q/2 is free once the PVs of the previous tile that read it
        // are done (normally long before: they were issued a tile ago).
        if (g > 0) {
          ok = __all_sync(0xffffffffu, sync.wait(smem_u32(&sh->p_free[q >> 1]), (g - 1) & 1));
          if (!ok) break;
        }
        const float vsv = vsc;                            // 0 for keys outside the pages
        if (live) {
          uint8_t* pd = pbuf + (q >> 1) * kPHalfBytes + kl * 128;
          auto emit = [&](const uint32_t (&sv)[16], int k) {
            uint32_t pk[8];
            const float4* mp = reinterpret_cast<const float4*>(rd->m + cb + 16 * k);
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
              const float4 m4 = mp[i4];
              const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
              float pp[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int c = cb + 16 * k + 4 * i4 + i;
                float x = __uint_as_float(sv[4 * i4 + i]) * kf - mm[i];
                if (!all_vis && (c < c_lo || c >= c_hi)) x = -INFINITY;
                pp[i] = ex2(x);
                lsum[16 * k + 4 * i4 + i] += pp[i];
              }
              __half2 h0 = __floats2half2_rn(pp[0] * vsv, pp[1] * vsv);
              __half2 h1 = __floats2half2_rn(pp[2] * vsv, pp[3] * vsv);
              pk[2 * i4] = *reinterpret_cast<uint32_t*>(&h0);
              pk[2 * i4 + 1] = *reinterpret_cast<uint32_t*>(&h1);
            }
            // rows r0..r0+7 and r0+8..r0+15 of this key: 16-byte chunks of P^T
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int r0 = cb + 16 * k + 8 * hh;
              *reinterpret_cast<uint4*>(pd + (r0 >> 6) * kPAtom + ((((r0 & 63) >> 3) ^ (kl & 7)) << 4)) =
                  make_uint4(pk[4 * hh], pk[4 * hh + 1], pk[4 * hh + 2], pk[4 * hh + 3]);
            }
          };
          uint32_t sa[16], sb[16];
          tmem_ld32x32b_x16(s_addr, sa);
          tmem_wait_ld(sa);
          tmem_ld32x32b_x16(s_addr + 16, sb);
          emit(sa, 0);
          tmem_wait_ld(sb);
          tmem_ld32x32b_x16(s_addr + 32, sa);
          emit(sb, 1);
          tmem_wait_ld(sa);
          emit(sa, 2);
        }
        fence_before();
        warp_arrive(smem_u32(&sh->s_free[g & 1]), lane);
        fence_async_smem();
        warp_arrive(smem_u32(&sh->p_full[q >> 1]), lane);
      }
      if (!ok) break;

      // ---- epilogue: row sums, O = O^T / l, LSE
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        float lv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) lv[i] = lsum[16 * k + i];
        const float cs = reduce_scatter16<false>(lv, lane);
        if (!(lane & 1)) rd->part[q][cb + 16 * k + scatter_col(lane)] = cs;
      }
      ok = smx_sync();
      if (!ok) break;
      const int ns = nseg[s.u];
      const long long prow0 = (long long)part_base[s.u] + (long long)(blockIdx.x - cfirst[s.u]) * R;
      if (st < R) {
        const int c = st;
        const float l = rd->part[0][c] + rd->part[1][c] + rd->part[2][c] + rd->part[3][c];
        rd->osc[c] = l > 0.f ? 1.f / l : 0.f;
        const float lse = l > 0.f ? (rd->m[c] + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        const int t = c / G, gg = c - t * G;
        if (ns == 1) p.lse[(size_t)(q_off[s.b] + t) * p.num_q_heads + s.h * G + gg] = lse;
        else lse_part[prow0 + c] = lse;
      }
      ok = smx_sync() &&
           __all_sync(0xffffffffu, sync.wait(smem_u32(&sh->o_done[(g - 1) & 1]), ((g - 1) >> 1) & 1));
      if (!ok) break;
      fence_after();
      {
        const int d = 128 * part + 32 * q + lane;
        int t = 0, gg = 0;
#pragma unroll 1
        for (int c0 = 0; c0 < R; c0 += 16) {
          uint32_t v[16];
          tmem_ld32x32b_x16(tmem + lane_off + kColO + (uint32_t)(part * kNMax + c0), v);
          tmem_wait_ld(v);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = c0 + i;
            if (c < R) {
              const float o = __uint_as_float(v[i]) * rd->osc[c];
              if (ns == 1)
                p.out[((size_t)(q_off[s.b] + t) * p.num_q_heads + s.h * G + gg) * D + d] =
                    __float2bfloat16_rn(o);
              else
                o_part[(prow0 + c) * D + d] = o;
              if (++gg == G) {
                gg = 0;
                ++t;
              }
            }
          }
        }
      }
      fence_before();
      warp_arrive(smem_u32(&sh->o_free), lane);
    }
  } else if (warp < kVConvWarp0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 96;" ::: "memory");
    // ============================================================ K converters
    const int q = warp - kKConvWarp0;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    uint8_t* mystage = kst + q * kKDepth * kKStage;
    // copies run kKDepth tiles ahead of the conversion, on their own iterator
    SegIter cit = iter;
    Seg cs;
    int c_it = 0, c_end = 0, issued = 0;
    PageWindow win;
    auto issue_next = [&]() -> bool {
      if (c_it >= c_end) {
        if (!cit.next(cs)) return true;
        c_it = cs.i0;
        c_end = cs.i1;
      }
      const int slot = issued % kKDepth, ssl = issued % kScSlots;
      // the scale slot is free once the softmax is done with tile issued - kScSlots
      bool okk = true;
      if (lane == 0) okk = sync.wait(smem_u32(&sh->sc_free[ssl]), ((issued / kScSlots) & 1) ^ 1);
      if (!__shfl_sync(0xffffffffu, okk, 0)) return false;
      const uint32_t bar = smem_u32(&sh->kst_full[q][slot]);
      const int first = (c_it * kTileKeys + 32 * q) / kPageSize;       // this warp's 2 pages
      const int npages = (cs.Lk + kPageSize - 1) / kPageSize;
      const int id = win.get(p, cs.b, first, npages, lane);
      const int page = needed_page(p, cs, first, lane < 2, id, lane);
      const unsigned mask = __ballot_sync(0xffffffffu, page >= 0) & 3u;
      if (lane == 0) mbar_expect_tx(bar, (uint32_t)__popc(mask) * kPageBytes);
      __syncwarp();
      if (page >= 0)
        tensor_g2s_3d(smem_u32(mystage + slot * kKStage + lane * kPageBytes), &tmap, 0,
                      (page * Hkv + cs.h) * 2 * kPageSize, 0, bar);
      // K / V scales of the two pages: lanes 0-7 K, 8-15 V; page (lane >> 2) & 1
      const int which = (lane >> 3) & 1, pg = (lane >> 2) & 1, ch = lane & 3;
      const int ps = __shfl_sync(0xffffffffu, page, pg);
      if (lane < 16 && ps >= 0)
        cp_async16(smem_u32(scales + ssl * 2 * kTileKeys + which * kTileKeys + 32 * q + 16 * pg + 4 * ch),
                   (which ? p.v_scales : p.k_scales) + ((size_t)ps * Hkv + cs.h) * kPageSize + 4 * ch);
      cp_async_arrive_noinc(smem_u32(&sh->sc_full[ssl]));
      ++c_it;
      ++issued;
      return true;
    };
    bool ok = true;
    for (int d = 0; d < kKDepth && ok; ++d) ok = issue_next();
    int g = 0;
    Seg s;
    const int slot_row = lane & 15;
    while (ok && iter.next(s)) {
      for (int it = s.i0; it < s.i1 && ok; ++it, ++g) {
        const int slot = g % kKDepth;
        ok = sync.wait(smem_u32(&sh->kst_full[q][slot]), (g / kKDepth) & 1) &&
             (g == 0 || sync.wait(smem_u32(&sh->kt_free), (g - 1) & 1));
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        fence_after();
        const uint8_t* row = mystage + slot * kKStage + (lane >> 4) * kPageBytes + slot_row * 128;
#pragma unroll
        for (int cg = 0; cg < 4; ++cg) {                  // 64 d = 32 TMEM columns each
          uint32_t v[32];
          const int hh = cg >> 1;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int c = 4 * (cg & 1) + k;
            const uint4 w = *reinterpret_cast<const uint4*>(row + hh * kPageHalf +
                                                            ((c ^ (slot_row & 7)) << 4));
            i8x4_to_h2x2(w.x, v[8 * k], v[8 * k + 1]);
            i8x4_to_h2x2(w.y, v[8 * k + 2], v[8 * k + 3]);
            i8x4_to_h2x2(w.z, v[8 * k + 4], v[8 * k + 5]);
            i8x4_to_h2x2(w.w, v[8 * k + 6], v[8 * k + 7]);
          }
          tmem_st32x32b_x32(tmem + lane_off + kColK + (uint32_t)(32 * cg), v);
        }
        tmem_wait_st();
        fence_before();
        warp_arrive(smem_u32(&sh->kt_full), lane);
        __syncwarp();                                     // the stage is read: refill it
        ok = issue_next();
      }
    }
    // copies still in flight (only after an abort) land before the CTA exits
    if (lane == 0)
      for (int t = g; t < issued; ++t)
        sync.drain(smem_u32(&sh->kst_full[q][t % kKDepth]), (t / kKDepth) & 1);
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 96;" ::: "memory");
    if (warp != kMmaWarp) {
    // ============================================================ V converters
    const int tv = (warp == 15 ? 64 : 32 * (warp - kVConvWarp0)) + lane;
    const bool issuer = warp == kVConvWarp0;            // also issues the V copies
    SegIter vit = iter;
    Seg cs;
    int v_it = 0, v_end = 0, v_hh = 0, vissued = 0;
    PageWindow win;
    // V codes of the next 64-key stage into slot vissued % kVRing
    auto issue_v = [&]() {
      if (v_hh == 0 && v_it >= v_end) {
        if (!vit.next(cs)) return;
        v_it = cs.i0;
        v_end = cs.i1;
      }
      const int slot = vissued % kVRing;
      const uint32_t bar = smem_u32(&sh->vst_full[slot]);
      const int first = (v_it * kTileKeys + v_hh * kSubKeys) / kPageSize;
      const int npages = (cs.Lk + kPageSize - 1) / kPageSize;
      const int id = win.get(p, cs.b, first, npages, lane);
      const int page = needed_page(p, cs, first, lane < 4, id, lane);
      const unsigned mask = __ballot_sync(0xffffffffu, page >= 0) & 15u;
      if (lane == 0) mbar_expect_tx(bar, (uint32_t)__popc(mask) * kPageBytes);
      __syncwarp();
      if (page >= 0)
        tensor_g2s_3d(smem_u32(vst + slot * kVStage + lane * kPageBytes), &tmap, 0,
                      (page * Hkv + cs.h) * 2 * kPageSize + kPageSize, 0, bar);
      if (++v_hh == 2) {
        v_hh = 0;
        ++v_it;
      }
      ++vissued;
    };
    if (issuer)
      for (int i = 0; i < kVRing; ++i) issue_v();
    int g = 0;
    Seg s;
    bool ok = true;
    while (ok && iter.next(s)) {
      for (int it = s.i0; it < s.i1 && ok; ++it, ++g) {
        for (int c = 0; c < kTileKeys / kVtKeys; ++c) {
          const int gc = 8 * g + c, sub = 2 * g + (c >> 2), vs = sub % kVRing, vb = gc % kVtBufs;
          ok = ((c & 3) || sync.wait(smem_u32(&sh->vst_full[vs]), (sub / kVRing) & 1)) &&
               sync.wait(smem_u32(&sh->vt_free[vb]), ((gc / kVtBufs) & 1) ^ 1);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          uint8_t* dstb = vtb + vb * kVtBytes;
          const uint8_t* srcb = vst + vs * kVStage + (c & 3) * kPageBytes;   // page c & 3 of the stage
          // job j: key (slot) j & 15, 16-byte chunk j >> 4 of its row; a
          // quarter warp takes 8 consecutive keys of one chunk: its loads and
          // stores fall in 8 distinct bank groups (both layouts swizzle by key & 7)
#pragma unroll
          for (int i = 0; i < 3; ++i) {
            const int jb = tv + kVConvThreads * i;
            if (jb < kVtKeys * 16) {
              const int kloc = jb & 15, hc = jb >> 4, hh = hc >> 3, cc = hc & 7;
              const uint4 w = *reinterpret_cast<const uint4*>(
                  srcb + hh * kPageHalf + kloc * 128 + ((cc ^ (kloc & 7)) << 4));
              uint4 h0, h1;
              i8x4_to_h2x2(w.x, h0.x, h0.y);
              i8x4_to_h2x2(w.y, h0.z, h0.w);
              i8x4_to_h2x2(w.z, h1.x, h1.y);
              i8x4_to_h2x2(w.w, h1.z, h1.w);
              uint8_t* da = dstb + (2 * hh + (cc >> 2)) * kVtAtom + kloc * 128;
              const int e0 = 2 * (cc & 3);
              *reinterpret_cast<uint4*>(da + ((e0 ^ (kloc & 7)) << 4)) = h0;
              *reinterpret_cast<uint4*>(da + (((e0 + 1) ^ (kloc & 7)) << 4)) = h1;
            }
          }
          fence_async_smem();
          warp_arrive(smem_u32(&sh->vt_full[vb]), lane);
          if ((c & 3) == 3) {
            warp_arrive(smem_u32(&sh->vst_empty[vs]), lane);
            if (issuer) {                               // refill the stage once all have read it
              bool okk = true;
              if (lane == 0) okk = sync.wait(smem_u32(&sh->vst_empty[vs]), (sub / kVRing) & 1);
              ok = __shfl_sync(0xffffffffu, okk, 0);
              if (!ok) break;
              issue_v();
            }
          }
        }
      }
    }
    // V copies in flight after an abort land before the CTA exits (a stage is
    // re-armed only after its previous copies were consumed)
    if (issuer && lane == 0)
      for (int r = 0; r < kVRing && r < vissued; ++r) {
        const int last = r + ((vissued - 1 - r) / kVRing) * kVRing;
        sync.drain(smem_u32(&sh->vst_full[r]), (last / kVRing) & 1);
      }
    } else {
    // ============================================================ MMA issue (warp 14)
    if (lane == 0) {
      const uint64_t qdesc0 = sdesc(smem_u32(qbuf), 16, 1024);
      const uint64_t vtdesc0 = sdesc(smem_u32(vtb), kVtAtom, 1024);
      const uint64_t pdesc0 = sdesc(smem_u32(pbuf), kPAtom, 1024);
      SegIter qi = iter, pi = iter;
      Seg qs, ps;
      bool qk_more = qi.next(qs), pv_more = pi.next(ps);
      int qk_tile = qk_more ? qs.i0 : 0, g_qk = 0, seg_qk = 0;
      int pv_tile = pv_more ? ps.i0 : 0, g_pv = 0, ck = 0, seg_pv = 0;
      bool q_ready = false, pv_first = true;
      uint32_t idq = idesc_f16(128, (qs.R + 15) & ~15, 0, 0);
      uint32_t idp = idesc_f16(128, (ps.R + 15) & ~15, 1, 1);
      unsigned long long t_last = global_ns();
      while (qk_more || pv_more) {
        bool prog = false;
        if (qk_more) {
          if (!q_ready) q_ready = mbar_test_wait(smem_u32(&sh->q_full), seg_qk & 1);
          if (q_ready && mbar_test_wait(smem_u32(&sh->kt_full), g_qk & 1) &&
              (g_qk < 2 ||
               mbar_test_wait(smem_u32(&sh->s_free[g_qk & 1]), ((g_qk >> 1) - 1) & 1))) {
            fence_after();
            const uint32_t dcol = tmem + kColS + (uint32_t)((g_qk & 1) * kNMax);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_ts(dcol, tmem + kColK + (uint32_t)(8 * kk),
                     qdesc0 + (uint64_t)(((kk >> 2) * kQAtom + (kk & 3) * 32) >> 4), idq, kk > 0);
            mma_commit(smem_u32(&sh->s_full[g_qk & 1]));
            mma_commit(smem_u32(&sh->kt_free));
            ++g_qk;
            if (++qk_tile == qs.i1) {
              qk_more = qi.next(qs);
              if (qk_more) {
                qk_tile = qs.i0;
                ++seg_qk;
                q_ready = false;
                idq = idesc_f16(128, (qs.R + 15) & ~15, 0, 0);
              }
            }
            prog = true;
          }
        }
        if (pv_more && g_pv < g_qk) {
          const int gc = 8 * g_pv + ck, vb = gc % kVtBufs;
          bool rdy = mbar_test_wait(smem_u32(&sh->p_full[ck >> 2]), g_pv & 1) &&
                     mbar_test_wait(smem_u32(&sh->vt_full[vb]), (gc / kVtBufs) & 1);
          if (rdy && pv_first && ck == 0 && seg_pv > 0)
            rdy = mbar_test_wait(smem_u32(&sh->o_free), (seg_pv - 1) & 1);
          if (rdy) {
            fence_after();
            const uint64_t pdesc = pdesc0 + (uint64_t)(((ck >> 2) * kPHalfBytes + (ck & 3) * 2048) >> 4);
            const uint64_t vdesc = vtdesc0 + (uint64_t)((vb * kVtBytes) >> 4);
            const uint32_t acc = (pv_first && ck == 0) ? 0u : 1u;
            mma_ss(tmem + kColO, vdesc, pdesc, idp, acc);
            mma_ss(tmem + kColO + kNMax, vdesc + (uint64_t)((2 * kVtAtom) >> 4), pdesc, idp, acc);
            mma_commit(smem_u32(&sh->vt_free[vb]));
            if ((ck & 3) == 3) mma_commit(smem_u32(&sh->p_free[ck >> 2]));
            if (ck == 7) mma_commit(smem_u32(&sh->o_done[g_pv & 1]));
            if (++ck == kTileKeys / kVtKeys) {
              ck = 0;
              pv_first = false;
              ++g_pv;
              if (++pv_tile == ps.i1) {
                pv_more = pi.next(ps);
                if (pv_more) {
                  pv_tile = ps.i0;
                  ++seg_pv;
                  pv_first = true;
                  idp = idesc_f16(128, (ps.R + 15) & ~15, 1, 1);
                }
              }
            }
            prog = true;
          }
        }
        if (prog) {
          t_last = global_ns();
        } else {
          if (sh->abort_flag) break;
          if (global_ns() - t_last > sync.limit_ns) {
            sync.give_up();
            break;
          }
        }
      }
      // every MMA issued is complete before TMEM and the operands go away
      mma_commit(smem_u32(&sh->drain));
      sync.drain(smem_u32(&sh->drain), 0);
    }
    __syncwarp();
    }
  }

  fence_before();
  __syncthreads();
  fence_after();
  if (warp == kMmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols) : "memory");
}

}  // namespace tt

// Units this kernel takes: head_dim 256, at most 96 query rows each.
bool tt_supported(int head_dim, int rows_cap) {
  return head_dim == tt::D && rows_cap >= 1 && rows_cap <= tt::kNMax;
}
int tt_tile_keys() { return tt::kTileKeys; }

// Tensor map over the code pool viewed as [half of a row (128 B)][row][2
// halves]: a row is the D = 256 codes of one (page, KV head, K|V, slot); the
// box {128 B, 16 rows, 2 halves} is the K (or V) codes of one (page, KV
// head), 4 KB, stored in shared memory with the 128-byte swizzle.
namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}
}  // namespace

bool tt_encode_map(CUtensorMap* map, const int8_t* k_pages, int num_pages, int num_kv_heads) {
  auto fn = encode_fn();
  if (fn == nullptr || num_pages <= 0) return false;
  const unsigned long long rows = (unsigned long long)num_pages * num_kv_heads * 2 * kPageSize;
  if (rows >= (1ull << 31)) return false;
  cuuint64_t gdim[3] = {128, (cuuint64_t)rows, 2};
  cuuint64_t gstride[2] = {(cuuint64_t)tt::D, 128};
  cuuint32_t box[3] = {128, (cuuint32_t)kPageSize, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<int8_t*>(k_pages), gdim, gstride,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_verify_tt(const AttnParams& p, const CUtensorMap& map, int ncta,
                             cudaStream_t stream) {
  constexpr int smem = tt::kSmemBytes;
  cudaError_t e;
  if (p.window > 0) {
    e = ensure_dynamic_smem<tt::verify_tt_kernel<true>>(smem);
    if (e != cudaSuccess) return e;
    e = launch_dependent(tt::verify_tt_kernel<true>, dim3(ncta), dim3(tt::kThreads), smem, stream, p,
                         map);
    if (e != cudaSuccess) return e;
  } else {
    e = ensure_dynamic_smem<tt::verify_tt_kernel<false>>(smem);
    if (e != cudaSuccess) return e;
    e = launch_dependent(tt::verify_tt_kernel<false>, dim3(ncta), dim3(tt::kThreads), smem, stream, p,
                         map);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace splash
