// Split plan and log-sum-exp combine of split-KV verify attention.
//
// Work unit = (sequence b, KV head h): its T_b*G query rows against keys
// 0 .. ctx_b + T_b - 1 (with a sliding window W, from the tile holding key
// ctx_b - W + 1 on). Each unit is cut into key tiles; the tiles of all units
// of one class (tensor-core or CUDA-core kernel) form one stream that is split
// over that kernel's persistent CTAs into ranges of about equal estimated cost
// (per-tile cost grows with the unit's rows; each unit start adds a fill cost). A unit touched by one CTA is
// finished by it; a unit touched by n > 1 CTAs leaves n partials (o_i
// normalised by its own sum, lse_i) that lse_combine merges:
//   lse = ln sum_i exp(lse_i),  O = sum_i exp(lse_i - lse) o_i
// (an empty partial has lse_i = -inf and weight 0).
#include <climits>
#include <type_traits>

#include "splash_common.cuh"

namespace splash {

// The planner runs as one CTA of kPlanThreadsLarge threads, or of
// kPlanThreadsSmall for batches of at most kPlanSmallSeqs sequences (fewer
// warps make its many block-wide barriers cheaper; every pass loops over its
// items in chunks of the block size).
constexpr int kPlanThreadsLarge = 1024;
constexpr int kPlanThreadsSmall = 128;
constexpr int kPlanSmallSeqs = 128;
// Batches up to this many sequences keep the planner's per-sequence arrays in
// shared memory as well (the later passes read them back many times; from
// global memory each read would cost an L2 round trip).
constexpr int kPlanSmemSeqs = 1024;

struct PlanSmem {
  int T[kPlanSmemSeqs], ctx[kPlanSmemSeqs], cls[kPlanSmemSeqs];
  int stp[kNumClasses][kPlanSmemSeqs + 1];
  long long wcost[kNumClasses][kPlanSmemSeqs + 1];
};

// Inclusive max-scans of two values over the CTA (any multiple of 32 threads).
__device__ inline int2 block_inclusive_max2(int2 v, int2* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int2 incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y0 = __shfl_up_sync(0xffffffffu, incl.x, o);
    const int y1 = __shfl_up_sync(0xffffffffu, incl.y, o);
    if (lane >= o) incl = make_int2(max(incl.x, y0), max(incl.y, y1));
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int2 x = lane < nw ? s_warp[lane] : make_int2(INT_MIN, INT_MIN);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y0 = __shfl_up_sync(0xffffffffu, x.x, o);
      const int y1 = __shfl_up_sync(0xffffffffu, x.y, o);
      if (lane >= o) x = make_int2(max(x.x, y0), max(x.y, y1));
    }
    s_warp[lane] = x;
  }
  __syncthreads();
  int2 res = incl;
  if (warp) res = make_int2(max(s_warp[warp - 1].x, incl.x), max(s_warp[warp - 1].y, incl.y));
  __syncthreads();
  return res;
}

// The per-sequence quantities pass 1 sums: Q/O rows laid out, key tiles and
// estimated cost per class.
struct PlanSums {
  long long q, w0, w1;
  int t0, t1;
  __device__ PlanSums operator+(const PlanSums& o) const {
    return PlanSums{q + o.q, w0 + o.w0, w1 + o.w1, t0 + o.t0, t1 + o.t1};
  }
};
__device__ inline PlanSums shfl_up(const PlanSums& v, int o) {
  return PlanSums{__shfl_up_sync(0xffffffffu, v.q, o), __shfl_up_sync(0xffffffffu, v.w0, o),
                  __shfl_up_sync(0xffffffffu, v.w1, o), __shfl_up_sync(0xffffffffu, v.t0, o),
                  __shfl_up_sync(0xffffffffu, v.t1, o)};
}

// Exclusive scan of PlanSums over the CTA (one set of barriers for all five).
__device__ inline PlanSums block_exclusive_scan_sums(PlanSums v, PlanSums* s_warp, PlanSums* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const PlanSums zero{0, 0, 0, 0, 0};
  PlanSums incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const PlanSums y = shfl_up(incl, o);
    if (lane >= o) incl = incl + y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    PlanSums x = lane < nw ? s_warp[lane] : zero;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const PlanSums y = shfl_up(x, o);
      if (lane >= o) x = x + y;
    }
    s_warp[lane] = x;
  }
  __syncthreads();
  PlanSums res = (warp ? s_warp[warp - 1] : zero) + incl;
  res = PlanSums{res.q - v.q, res.w0 - v.w0, res.w1 - v.w1, res.t0 - v.t0, res.t1 - v.t1};
  *total = s_warp[nw - 1];
  __syncthreads();
  return res;
}

// Exclusive scan over the CTA (any multiple of 32 threads); *total receives the sum.
template <typename V>
__device__ inline V block_exclusive_scan(V v, V* s_warp, V* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  V incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    V y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    V x = lane < nw ? s_warp[lane] : V(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      V y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    s_warp[lane] = x;
  }
  __syncthreads();
  const V res = (warp ? s_warp[warp - 1] : V(0)) + incl - v;
  *total = s_warp[nw - 1];
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(kPlanThreadsLarge)
plan_kernel(const int32_t* __restrict__ context_lens, const int32_t* __restrict__ block_lens,
            int num_seqs, int num_kv_heads, int group, int max_pages, int max_block_len,
            int tile_tc, int tile_simt, int ncta_tc, int ncta_simt, int path, int rows_bound,
            int num_q_tokens, int window, unsigned char* ws, int* device_status) {
  __shared__ int s_warp[32];
  __shared__ int2 s_warp2[32];
  __shared__ PlanSums s_sums[32];
  __shared__ int s_start[kNumClasses][kMaxCtas + 1];
  extern __shared__ __align__(16) unsigned char s_dyn[];
  allow_dependent_launch();        // the attention kernel may get its SMs now
  const bool small = num_seqs <= kPlanSmemSeqs;     // launched with sizeof(PlanSmem) then
  PlanSmem* ps = reinterpret_cast<PlanSmem*>(s_dyn);
  const WorkspaceLayout L = make_layout(num_seqs, num_kv_heads, 0, rows_bound);
  int* q_off = reinterpret_cast<int*>(ws + L.q_off);
  int* seq_T = reinterpret_cast<int*>(ws + L.seq_T);
  int* seq_ctx = reinterpret_cast<int*>(ws + L.seq_ctx);
  int* seq_class = reinterpret_cast<int*>(ws + L.seq_class);
  int* stp = reinterpret_cast<int*>(ws + L.stp);
  int* nseg = reinterpret_cast<int*>(ws + L.nseg);
  int* cfirst = reinterpret_cast<int*>(ws + L.cfirst);
  int* part_base = reinterpret_cast<int*>(ws + L.part_base);
  long long* wcost = reinterpret_cast<long long*>(ws + L.wcost);
  int* cta_start = reinterpret_cast<int*>(ws + L.cta_start);
  const int tile[kNumClasses] = {tile_tc, tile_simt};
  const int ncta[kNumClasses] = {ncta_tc, ncta_simt};

  // pass 1: per sequence — validate, classify, prefix sums of rows and tiles.
  // The Q / O rows of sequence b start at the sum of the caller's block_lens
  // before it (negative lengths count as 0), whether or not b itself is valid:
  // a rejected sequence is idle, and the others keep their rows.
  long long run_q = 0, run_w[kNumClasses] = {0, 0};
  int run_t0 = 0, run_t1 = 0;
  for (int base = 0; base < num_seqs; base += (int)blockDim.x) {
    const int b = base + threadIdx.x;
    int T = 0, ctx = 0, cls = -1, tiles = 0;
    long long rows_laid_out = 0;
    if (b < num_seqs) {
      T = block_lens[b];
      rows_laid_out = T > 0 ? T : 0;
      ctx = context_lens[b];
      const bool ok = T >= 0 && ctx >= 0 && T <= max_block_len &&
                      (long long)ctx + T <= (long long)max_pages * kPageSize;
      if (!ok) {
        report(device_status, SPLASH_DEVICE_BAD_LENGTH);
        T = 0;
        ctx = 0;
      }
      if (T > 0) {
        const int rows = T * group;
        cls = path == 1 ? kClassSimt : path == 2 ? kClassTensor
                        : (rows >= kTensorMinRows ? kClassTensor : kClassSimt);
        tiles = unit_tiles(ctx, T, window, cls == 0 ? tile[0] : tile[1]);
      }
      seq_T[b] = T;
      seq_ctx[b] = ctx;
      seq_class[b] = cls;
      if (small) {
        ps->T[b] = T;
        ps->ctx[b] = ctx;
        ps->cls[b] = cls;
      }
    }
    // estimated cost of the sequence's units in its class (see tile_cost)
    long long cost = 0;
    if (cls >= 0)
      cost = (long long)num_kv_heads *
             ((long long)tiles * (tile_cost(cls) + row_cost(cls) * T * group) + segment_cost(cls));
    const PlanSums mine{rows_laid_out, cls == 0 ? cost : 0, cls == 1 ? cost : 0,
                        cls == 0 ? tiles * num_kv_heads : 0, cls == 1 ? tiles * num_kv_heads : 0};
    PlanSums tot;
    const PlanSums ex = block_exclusive_scan_sums(mine, s_sums, &tot);
    if (b < num_seqs) {
      // offsets past the caller's rows only occur when the plan is dropped below
      q_off[b] = (int)min(run_q + ex.q, (long long)num_q_tokens);
      stp[b] = run_t0 + ex.t0;
      stp[(num_seqs + 1) + b] = run_t1 + ex.t1;
      wcost[b] = run_w[0] + ex.w0;
      wcost[(num_seqs + 1) + b] = run_w[1] + ex.w1;
      if (small) {
        ps->stp[0][b] = run_t0 + ex.t0;
        ps->stp[1][b] = run_t1 + ex.t1;
        ps->wcost[0][b] = run_w[0] + ex.w0;
        ps->wcost[1][b] = run_w[1] + ex.w1;
      }
    }
    run_q += tot.q;
    run_t0 += tot.t0;
    run_t1 += tot.t1;
    run_w[0] += tot.w0;
    run_w[1] += tot.w1;
  }
  if (threadIdx.x == 0) {
    q_off[num_seqs] = (int)min(run_q, (long long)num_q_tokens);
    stp[num_seqs] = run_t0;
    stp[(num_seqs + 1) + num_seqs] = run_t1;
    for (int c = 0; c < kNumClasses; ++c) wcost[c * (num_seqs + 1) + num_seqs] = run_w[c];
    if (small) {
      ps->stp[0][num_seqs] = run_t0;
      ps->stp[1][num_seqs] = run_t1;
      for (int c = 0; c < kNumClasses; ++c) ps->wcost[c][num_seqs] = run_w[c];
    }
  }
  __syncthreads();
  // where the later passes read the per-sequence arrays
  const int* rT = small ? ps->T : seq_T;
  const int* rctx = small ? ps->ctx : seq_ctx;
  // block lengths that sum past the q / out rows the caller passed: do nothing
  const bool rows_ok = run_q <= num_q_tokens;
  if (!rows_ok) {
    if (threadIdx.x == 0) report(device_status, SPLASH_DEVICE_BAD_LENGTH);
    run_t0 = run_t1 = 0;
    for (int b = threadIdx.x; b < num_seqs; b += blockDim.x) {
      seq_class[b] = -1;
      if (small) ps->cls[b] = -1;
    }
    __syncthreads();
  }
  const int total[kNumClasses] = {run_t0, run_t1};
  // a class's kernel uses at most one CTA per tile, so that every CTA it uses
  // owns >= 1 tile and the CTAs covering a unit are consecutive, all non-empty
  int ncta_eff[kNumClasses];
  for (int c = 0; c < kNumClasses; ++c) ncta_eff[c] = min(min(ncta[c], total[c]), kMaxCtas);

  // CTA c of a class starts where the class's cumulative cost reaches
  // c / n of its total: find the sequence, then the unit (KV head), then the
  // tile (the first segment_cost of a unit maps to its first tile). Then the
  // starts are made strictly increasing (every CTA owns >= 1 tile) and the
  // last ones are pulled back so that CTA n - 1 still fits before `total`.
  // one CTA start per thread, in chunks of the block size; the prefix max
  // carries from chunk to chunk
  {
    int2 carry = make_int2(INT_MIN, INT_MIN);
    const int kmax = max(ncta_eff[0], ncta_eff[1]);
    for (int base = 0; base <= kmax; base += (int)blockDim.x) {
      const int k = base + threadIdx.x;
      int start[kNumClasses] = {0, 0};
#pragma unroll
      for (int c = 0; c < kNumClasses; ++c) {
        const int n = ncta_eff[c];
        const long long* wc = small ? ps->wcost[c] : wcost + c * (num_seqs + 1);
        const int* sp = small ? ps->stp[c] : stp + c * (num_seqs + 1);
        if (k <= n && n > 0 && rows_ok) {
          if (k == n) {
            start[c] = total[c];
          } else if (k > 0) {
            const long long target = run_w[c] * k / n;      // < 2^63 for any realistic batch
            const int b = upper_index(wc, num_seqs - 1, target);
            const long long off = target - wc[b];
            const int T = rT[b];
            const int tiles = unit_tiles(rctx[b], T, window, tile[c]);
            const long long w = tile_cost(c) + row_cost(c) * T * group;
            const long long uc = (long long)tiles * w + segment_cost(c);
            const int h = (int)min(off / uc, (long long)num_kv_heads - 1);
            const long long rem = off - h * uc;
            const int t = rem < segment_cost(c) ? 0 : (int)min((rem - segment_cost(c)) / w, (long long)tiles - 1);
            start[c] = sp[b] + h * tiles + t;
          }
        }
      }
      // strictly increasing: prefix max of start - k, plus k (both classes at once)
      int2 y = block_inclusive_max2(make_int2(k <= ncta_eff[0] ? start[0] - k : INT_MIN,
                                              k <= ncta_eff[1] ? start[1] - k : INT_MIN),
                                    s_warp2);
      y = make_int2(max(y.x, carry.x), max(y.y, carry.y));
      if (k <= ncta_eff[0]) s_start[0][k] = min(y.x + k, total[0] - (ncta_eff[0] - k));
      if (k <= ncta_eff[1]) s_start[1][k] = min(y.y + k, total[1] - (ncta_eff[1] - k));
      // this chunk's maximum (the last thread's inclusive value) carries on
      if (threadIdx.x == blockDim.x - 1) s_warp2[0] = y;
      __syncthreads();
      carry = s_warp2[0];
      __syncthreads();
    }
  }
  __syncthreads();
  for (int c = 0; c < kNumClasses; ++c)
    for (int k = threadIdx.x; k <= ncta_eff[c]; k += blockDim.x)
      cta_start[c * (kMaxCtas + 1) + k] = s_start[c][k];

  // pass 2: per unit (b, h) — segments and partial rows
  const int num_units = num_seqs * num_kv_heads;
  int run_rows = 0;
  for (int base = 0; base < num_units; base += (int)blockDim.x) {
    const int u = base + threadIdx.x;
    int rows = 0;
    if (u < num_units) {
      const int b = u / num_kv_heads, h = u % num_kv_heads;
      const int cls = small ? ps->cls[b] : seq_class[b];
      int ns = 0, cf = 0;
      if (cls >= 0) {
        const int T = rT[b], ctx = rctx[b];
        const int tk = cls == 0 ? tile[0] : tile[1];        // selects, not a local-memory index
        const int nce = cls == 0 ? ncta_eff[0] : ncta_eff[1];
        const int tiles = unit_tiles(ctx, T, window, tk);
        const int tp = (small ? ps->stp[cls][b] : stp[cls * (num_seqs + 1) + b]) + h * tiles;
        const int* cs = s_start[cls == 0 ? 0 : 1];
        cf = upper_index(cs, nce - 1, tp);
        const int cl = upper_index(cs, nce - 1, tp + tiles - 1);
        ns = cl - cf + 1;
        if (ns > 1) rows = ns * T * group;
      }
      nseg[u] = ns;
      cfirst[u] = cf;
    }
    int tot;
    const int pb = block_exclusive_scan(rows, s_warp, &tot);
    if (u < num_units) part_base[u] = run_rows + pb;
    run_rows += tot;
  }
  if (threadIdx.x == 0) {
    PlanHeader* hd = reinterpret_cast<PlanHeader*>(ws);
    hd->total_tiles[0] = run_t0;
    hd->total_tiles[1] = run_t1;
    hd->ncta[0] = ncta_eff[0];
    hd->ncta[1] = ncta_eff[1];
    hd->tile_keys[0] = tile_tc;
    hd->tile_keys[1] = tile_simt;
    hd->num_seqs = num_seqs;
    hd->num_kv_heads = num_kv_heads;
    hd->group = group;
    hd->total_part_rows = run_rows;
    hd->rows_bound = rows_bound;
    hd->window = window;
  }
}

// WPR warps per (token row, query head) of a split unit; warp `sub` of a row
// accumulates the partials j = sub, sub + WPR, ... (four or eight partial rows
// in flight), and the WPR sums meet in shared memory. Every warp of a row reads all
// lse_j in one pass (running max and rescaled sum per lane, then merged across
// the warp), so the weights exp(lse_j - lse) agree across the row's warps.
template <int D, int WPR>
__global__ void __launch_bounds__(256, 2)
lse_combine_kernel(int num_q_tokens, int num_q_heads, int num_seqs, int num_kv_heads, int group,
                   int rows_bound, const unsigned char* __restrict__ ws,
                   __nv_bfloat16* __restrict__ out, float* __restrict__ lse_out) {
  constexpr int EPL = D / 32;                     // output columns per lane
  constexpr int kRowsPerBlock = 8 / WPR;
  constexpr int kUnroll = WPR >= 4 ? 8 : 4;      // partial rows in flight per warp
  constexpr int VW = EPL >= 4 ? 4 : 2;           // floats per vector load
  using Vec = typename std::conditional<VW == 4, float4, float2>::type;
  static_assert(EPL % VW == 0, "vector loads of a lane's columns");
  __shared__ float s_acc[WPR > 1 ? 8 : 1][WPR > 1 ? D : 1];
  grid_dependency_wait();          // the attention kernel's partials are complete
  const WorkspaceLayout L = make_layout(num_seqs, num_kv_heads, D, rows_bound);
  const int* q_off = reinterpret_cast<const int*>(ws + L.q_off);
  const int* seq_T = reinterpret_cast<const int*>(ws + L.seq_T);
  const int* nseg = reinterpret_cast<const int*>(ws + L.nseg);
  const int* part_base = reinterpret_cast<const int*>(ws + L.part_base);
  const float* o_part = reinterpret_cast<const float*>(ws + L.o_part);
  const float* lse_part = reinterpret_cast<const float*>(ws + L.lse_part);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, sub = warp % WPR;
  const long long row = (long long)blockIdx.x * kRowsPerBlock + warp / WPR;
  // the warp's row, when it belongs to a unit with two or more partials
  bool active = row < (long long)num_q_tokens * num_q_heads;
  int i = 0, hq = 0, n = 0, R = 0, r = 0;
  long long base = 0;
  if (active) {
    i = (int)(row / num_q_heads);
    hq = (int)(row % num_q_heads);
    const int b = upper_index(q_off, num_seqs - 1, i);
    const int h = hq / group, g = hq % group;
    const int u = b * num_kv_heads + h;
    n = nseg[u];
    active = n > 1 && i - q_off[b] < seq_T[b];
    R = seq_T[b] * group;
    r = (i - q_off[b]) * group + g;
    base = part_base[u];
  }
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  float m = -INFINITY, wsum = 0.f;
  if (active) {
    // lse = m + ln(wsum) over all partials, one pass
    float sl = 0.f;
    for (int j = lane; j < n; j += 32) {
      const float lj = lse_part[base + (long long)j * R + r];
      if (lj > m) {
        sl = sl * __expf(m - lj) + 1.f;     // m = -inf: sl is 0 and stays finite
        m = lj;
      } else if (lj != -INFINITY) {
        sl += __expf(lj - m);
      }
    }
    const float mw = warp_max(m);
    wsum = warp_sum(m == -INFINITY ? 0.f : sl * __expf(m - mw));
    m = mw;
    for (int j0 = sub; j0 < n; j0 += kUnroll * WPR) {
      float w[kUnroll];
      Vec v[kUnroll][EPL / VW];
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        const int j = j0 + k * WPR;
        w[k] = 0.f;
        if (j < n) {
          const long long pr = base + (long long)j * R + r;
          const float lj = lse_part[pr];
          w[k] = (lj == -INFINITY) ? 0.f : __expf(lj - m);
          const Vec* src = reinterpret_cast<const Vec*>(o_part + pr * D + lane * EPL);
#pragma unroll
          for (int e = 0; e < EPL / VW; ++e) v[k][e] = src[e];
        }
      }
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        if (w[k] == 0.f) continue;
#pragma unroll
        for (int e = 0; e < EPL / VW; ++e) {
          const float* x = reinterpret_cast<const float*>(&v[k][e]);
#pragma unroll
          for (int c = 0; c < VW; ++c) acc[VW * e + c] = fmaf(w[k], x[c], acc[VW * e + c]);
        }
      }
    }
  }
  if (WPR > 1) {
    if (active) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) s_acc[warp][lane * EPL + e] = acc[e];
    }
    __syncthreads();
    if (active && sub == 0) {
#pragma unroll
      for (int o = 1; o < WPR; ++o)
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] += s_acc[warp + o][lane * EPL + e];
    }
  }
  if (!active || sub != 0) return;
  const float inv = 1.f / wsum;
  __nv_bfloat16* dst = out + ((long long)i * num_q_heads + hq) * D + lane * EPL;
#pragma unroll
  for (int e = 0; e < EPL; e += 2)
    *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
  if (lane == 0) lse_out[(long long)i * num_q_heads + hq] = m + logf(wsum);
}

cudaError_t launch_plan(const int32_t* context_lens, const int32_t* block_lens, int num_seqs,
                        int num_kv_heads, int group, int max_pages, int max_block_len, int tile_tc,
                        int tile_simt, int ncta_tc, int ncta_simt, int path, int rows_bound,
                        int num_q_tokens, int window, unsigned char* ws, int* device_status,
                        cudaStream_t stream) {
  const size_t dyn = num_seqs <= kPlanSmemSeqs ? sizeof(PlanSmem) : 0;
  const int threads = num_seqs <= kPlanSmallSeqs ? kPlanThreadsSmall : kPlanThreadsLarge;
  plan_kernel<<<1, threads, dyn, stream>>>(context_lens, block_lens, num_seqs, num_kv_heads,
                                              group, max_pages, max_block_len, tile_tc, tile_simt,
                                              ncta_tc, ncta_simt, path, rows_bound, num_q_tokens,
                                              window, ws, device_status);
  return cudaGetLastError();
}

cudaError_t launch_combine(int num_q_tokens, int num_q_heads, int num_seqs, int num_kv_heads,
                           int group, int head_dim, int rows_bound, int sms,
                           const unsigned char* ws, __nv_bfloat16* out, float* lse,
                           cudaStream_t stream) {
  const long long rows = (long long)num_q_tokens * num_q_heads;
  if (rows == 0) return cudaSuccess;
  // warps per row: enough to give every SM about 16 warps when there are few
  // rows (few rows means few units, each split over many CTAs)
  const long long want = 16LL * (sms > 0 ? sms : 1);
  const int wpr = rows * 4 <= want ? 8 : rows * 2 <= want ? 4 : rows <= want ? 2 : 1;
  const long long rows_per_block = 8 / wpr;
  const int grid = (int)((rows + rows_per_block - 1) / rows_per_block);
  cudaError_t e = cudaErrorInvalidValue;
#define SPLASH_COMBINE(DD, WW)                                                                  \
  e = launch_dependent(lse_combine_kernel<DD, WW>, dim3(grid), dim3(256), 0, stream,            \
                       num_q_tokens, num_q_heads, num_seqs, num_kv_heads, group, rows_bound, ws, \
                       out, lse)
#define SPLASH_COMBINE_D(DD)          \
  switch (wpr) {                      \
    case 1: SPLASH_COMBINE(DD, 1); break; \
    case 2: SPLASH_COMBINE(DD, 2); break; \
    case 4: SPLASH_COMBINE(DD, 4); break; \
    default: SPLASH_COMBINE(DD, 8); break; \
  }
  switch (head_dim) {
    case 64: SPLASH_COMBINE_D(64); break;
    case 128: SPLASH_COMBINE_D(128); break;
    case 256: SPLASH_COMBINE_D(256); break;
    default: return cudaErrorInvalidValue;
  }
#undef SPLASH_COMBINE_D
#undef SPLASH_COMBINE
  return e;
}

}  // namespace splash
