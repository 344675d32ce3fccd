// Split plan and log-sum-exp combine of verify attention with prefix groups
// (cross-sequence query stacking over shared prefix pages).
//
// shared_lens[b] keys at the start of sequence b's context sit in the same
// pages as sequence b - 1's. A run of consecutive sequences each linked to the
// one before it by at least one key tile is a prefix group. Its common prefix
// is the smallest link, cut to every member's context and down to a whole
// tile. The members' query rows, stacked in sequence order, are cut into row
// blocks of kMaxRows; each block is a work item that reads the common prefix
// (through the first member's page-table row) once for all of its rows, and
// each member's own item reads only its keys after the prefix. A group is
// stacked only when it needs fewer blocks than it has members.
//
// Every sequence is in the tensor-core class here. As in the plain plan, the
// tiles of all units (item, KV head) form one stream that is split over the
// attention kernel's persistent CTAs into ranges of about equal estimated
// cost. A grouped unit always leaves partials (o_i normalised by its own sum,
// lse_i), and the combine merges, for every grouped row, its block's partials
// and its own unit's:
//   lse = ln sum_i exp(lse_i),  O = sum_i exp(lse_i - lse) o_i
#include <climits>
#include <type_traits>

#include "splash_common.cuh"
#include "splash_groups.cuh"

namespace splash {
namespace {

constexpr int kGThreadsLarge = 1024;
constexpr int kGThreadsSmall = 128;
constexpr int kGSmallSeqs = 128;
constexpr int kGS = kPrefixGroupMaxSeqs;

struct GroupSmem {
  int T[kGS], ctx[kGS], qo[kGS];
  int sl[kGS];                      // keys shared with the previous sequence (0: none)
  int pg[kGS];                      // stacked prefix keys of the sequence's group (0: none)
  int iR[2 * kGS], itiles[2 * kGS];  // rows and tiles of each item
  int stp[2 * kGS + 1];
  long long wcost[2 * kGS + 1];
};

// Exclusive scan over the CTA (any multiple of 32 threads); *total receives the sum.
template <typename V>
__device__ inline V g_exclusive_scan(V v, V* s_warp, V* total) {
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

// Inclusive max-scan over the CTA.
__device__ inline int g_inclusive_max(int v, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl = max(incl, y);
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int x = lane < nw ? s_warp[lane] : INT_MIN;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x = max(x, y);
    }
    s_warp[lane] = x;
  }
  __syncthreads();
  const int res = warp ? max(s_warp[warp - 1], incl) : incl;
  __syncthreads();
  return res;
}

// Pair (tiles, cost) summed by one scan.
struct TileCost {
  long long w;
  int t;
  __device__ TileCost operator+(const TileCost& o) const { return TileCost{w + o.w, t + o.t}; }
  __device__ TileCost& operator+=(const TileCost& o) {
    w += o.w;
    t += o.t;
    return *this;
  }
  __device__ TileCost operator-(const TileCost& o) const { return TileCost{w - o.w, t - o.t}; }
};
__device__ inline TileCost shfl_up_tc(const TileCost& v, int o) {
  return TileCost{__shfl_up_sync(0xffffffffu, v.w, o), __shfl_up_sync(0xffffffffu, v.t, o)};
}
__device__ inline TileCost g_exclusive_scan_tc(TileCost v, TileCost* s_warp, TileCost* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const TileCost zero{0, 0};
  TileCost incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const TileCost y = shfl_up_tc(incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    TileCost x = lane < nw ? s_warp[lane] : zero;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const TileCost y = shfl_up_tc(x, o);
      if (lane >= o) x += y;
    }
    s_warp[lane] = x;
  }
  __syncthreads();
  const TileCost res = (warp ? s_warp[warp - 1] : zero) + incl - v;
  *total = s_warp[nw - 1];
  __syncthreads();
  return res;
}

}  // namespace

__global__ void __launch_bounds__(kGThreadsLarge)
plan_groups_kernel(const int32_t* __restrict__ context_lens, const int32_t* __restrict__ block_lens,
                   const int32_t* __restrict__ shared_lens, int num_seqs, int num_kv_heads,
                   int group, int max_pages, int max_block_len, int tile, int ncta,
                   int rows_bound, int num_q_tokens, unsigned char* ws, int* device_status) {
  __shared__ int s_warp[32];
  __shared__ long long s_warp_ll[32];
  __shared__ TileCost s_tc[32];
  __shared__ int s_start[kMaxCtas + 1];
  extern __shared__ __align__(16) unsigned char s_dyn[];
  allow_dependent_launch();        // the attention kernel may get its SMs now
  GroupSmem* ps = reinterpret_cast<GroupSmem*>(s_dyn);
  const GroupLayout L = make_group_layout(num_seqs, num_kv_heads, 0, rows_bound);
  int* q_off = reinterpret_cast<int*>(ws + L.q_off);
  int* seq_T = reinterpret_cast<int*>(ws + L.seq_T);
  int* seq_ctx = reinterpret_cast<int*>(ws + L.seq_ctx);
  int2* seq_grp = reinterpret_cast<int2*>(ws + L.seq_grp);
  ItemDesc* items = reinterpret_cast<ItemDesc*>(ws + L.items);
  int* stp = reinterpret_cast<int*>(ws + L.stp);
  int* nseg = reinterpret_cast<int*>(ws + L.nseg);
  int* cfirst = reinterpret_cast<int*>(ws + L.cfirst);
  int* part_base = reinterpret_cast<int*>(ws + L.part_base);
  long long* wcost = reinterpret_cast<long long*>(ws + L.wcost);
  int* cta_start = reinterpret_cast<int*>(ws + L.cta_start);

  // pass 1: per sequence — validate, lay out the Q / O rows (they start at the
  // sum of the caller's block_lens before the sequence, negative ones as 0),
  // and write the sequence's item (all its keys for now)
  long long run_q = 0;
  for (int base = 0; base < num_seqs; base += (int)blockDim.x) {
    const int b = base + threadIdx.x;
    int T = 0, ctx = 0;
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
    }
    long long tot;
    const long long ex = g_exclusive_scan(rows_laid_out, s_warp_ll, &tot);
    if (b < num_seqs) {
      const int qo = (int)min(run_q + ex, (long long)num_q_tokens);
      q_off[b] = qo;
      seq_T[b] = T;
      seq_ctx[b] = ctx;
      seq_grp[b] = make_int2(-1, 0);
      ps->T[b] = T;
      ps->ctx[b] = ctx;
      ps->qo[b] = qo;
      ps->pg[b] = 0;
    }
    run_q += tot;
  }
  if (threadIdx.x == 0) q_off[num_seqs] = (int)min(run_q, (long long)num_q_tokens);
  __syncthreads();
  // block lengths that sum past the q / out rows the caller passed: do nothing
  const bool rows_ok = run_q <= num_q_tokens;
  if (!rows_ok) {
    if (threadIdx.x == 0) report(device_status, SPLASH_DEVICE_BAD_LENGTH);
    for (int b = threadIdx.x; b < num_seqs; b += blockDim.x) ps->T[b] = 0;
    __syncthreads();
  }

  // links of b to b - 1: the shared keys, cut to both contexts; 0 below a tile
  for (int b = threadIdx.x; b < num_seqs; b += blockDim.x) {
    int sl = 0;
    if (b > 0 && ps->T[b] > 0 && ps->T[b - 1] > 0) {
      sl = min(shared_lens[b], min(ps->ctx[b], ps->ctx[b - 1]));
      if (sl < tile) sl = 0;
    }
    ps->sl[b] = sl;
  }
  __syncthreads();
  // the first sequence of each group walks its group and writes its blocks
  int num_blocks = 0;
  for (int base = 0; base < num_seqs; base += (int)blockDim.x) {
    const int b = base + threadIdx.x;
    int nblk = 0, m = 0, pg = 0, rows = 0;
    if (b < num_seqs && ps->T[b] > 0 && ps->sl[b] == 0 && b + 1 < num_seqs && ps->sl[b + 1] > 0) {
      pg = ps->ctx[b];
      rows = ps->T[b] * group;
      int e = b + 1;
      for (; e < num_seqs && ps->sl[e] > 0; ++e) {
        pg = min(pg, ps->sl[e]);
        rows += ps->T[e] * group;
      }
      m = e - b;
      pg = pg / tile * tile;
      nblk = (rows + kMaxRows - 1) / kMaxRows;
      if (pg < tile || nblk >= m) nblk = 0;          // stacking would not save a pass
    }
    int tot;
    const int ex = g_exclusive_scan(nblk, s_warp, &tot);
    if (nblk > 0) {
      const int first_item = num_seqs + num_blocks + ex;
      int so = 0;
      for (int e = b; e < b + m; ++e) {
        seq_grp[e] = make_int2(first_item, so);
        ps->pg[e] = pg;
        so += ps->T[e] * group;
      }
      for (int k = 0; k < nblk; ++k) {
        ItemDesc d;
        d.b = b;
        d.qbase = ps->qo[b];
        d.r0 = k * kMaxRows;
        d.R = min(kMaxRows, rows - k * kMaxRows);
        d.ctx = pg;
        d.Lk = pg;
        d.klo = 0;
        d.grouped = 1;
        items[first_item + k] = d;
        ps->iR[first_item + k] = d.R;
        ps->itiles[first_item + k] = pg / tile;
      }
    }
    num_blocks += tot;
  }
  __syncthreads();
  const int num_items = num_seqs + num_blocks;

  // the sequences' items (after the prefix when grouped), then the prefix
  // sums of tiles and cost over all items
  int run_t = 0;
  long long run_w = 0;
  for (int base = 0; base < num_items; base += (int)blockDim.x) {
    const int i = base + threadIdx.x;
    int R = 0, tiles = 0;
    if (i < num_seqs) {
      const int T = ps->T[i], ctx = ps->ctx[i], pg = ps->pg[i];
      ItemDesc d;
      d.b = i;
      d.qbase = ps->qo[i];
      d.r0 = 0;
      d.R = T * group;
      d.ctx = ctx;
      d.Lk = T > 0 ? ctx + T : 0;
      d.klo = T > 0 ? pg : 0;
      d.grouped = pg > 0 ? 1 : 0;
      items[i] = d;
      R = d.R;
      tiles = T > 0 ? (d.Lk + tile - 1) / tile - d.klo / tile : 0;
      ps->iR[i] = R;
      ps->itiles[i] = tiles;
    } else if (i < num_items) {
      R = ps->iR[i];
      tiles = ps->itiles[i];
    }
    long long cost = 0;
    if (tiles > 0)
      cost = (long long)num_kv_heads *
             ((long long)tiles * (tile_cost(0) + row_cost(0) * R) + segment_cost(0));
    TileCost tot;
    const TileCost ex = g_exclusive_scan_tc(TileCost{cost, tiles * num_kv_heads}, s_tc, &tot);
    if (i < num_items) {
      stp[i] = run_t + ex.t;
      wcost[i] = run_w + ex.w;
      ps->stp[i] = run_t + ex.t;
      ps->wcost[i] = run_w + ex.w;
    }
    run_t += tot.t;
    run_w += tot.w;
  }
  if (threadIdx.x == 0) {
    stp[num_items] = run_t;
    wcost[num_items] = run_w;
    ps->stp[num_items] = run_t;
    ps->wcost[num_items] = run_w;
  }
  // the attention kernel searches max_items(num_seqs) entries of stp: the ones
  // past the items must exceed every tile index
  for (int i = num_items + 1 + threadIdx.x; i <= max_items(num_seqs); i += blockDim.x)
    stp[i] = INT_MAX;
  __syncthreads();

  const int total = run_t;
  // at most one CTA per tile: every CTA owns >= 1 tile and the CTAs covering a
  // unit are consecutive, all non-empty
  const int n = min(min(ncta, total), kMaxCtas);

  // CTA k starts where the cumulative cost reaches k / n of the total: the
  // item, then the unit (KV head), then the tile (the first segment_cost of a
  // unit maps to its first tile); then the starts are made strictly
  // increasing and the last ones pulled back so that CTA n - 1 fits
  {
    int carry = INT_MIN;
    for (int base = 0; base <= n; base += (int)blockDim.x) {
      const int k = base + threadIdx.x;
      int start = 0;
      if (k <= n && n > 0) {
        if (k == n) {
          start = total;
        } else if (k > 0) {
          const long long target = run_w * k / n;
          const int i = upper_index(ps->wcost, num_items - 1, target);
          const long long off = target - ps->wcost[i];
          const int tiles = ps->itiles[i];
          const long long w = tile_cost(0) + row_cost(0) * ps->iR[i];
          const long long uc = (long long)tiles * w + segment_cost(0);
          const int h = (int)min(off / uc, (long long)num_kv_heads - 1);
          const long long rem = off - h * uc;
          const int t = rem < segment_cost(0) ? 0
                                              : (int)min((rem - segment_cost(0)) / w, (long long)tiles - 1);
          start = ps->stp[i] + h * tiles + t;
        }
      }
      int y = g_inclusive_max(k <= n ? start - k : INT_MIN, s_warp);
      y = max(y, carry);
      if (k <= n) s_start[k] = min(y + k, total - (n - k));
      if (threadIdx.x == blockDim.x - 1) s_warp[0] = y;
      __syncthreads();
      carry = s_warp[0];
      __syncthreads();
    }
  }
  __syncthreads();
  for (int k = threadIdx.x; k <= n; k += blockDim.x) cta_start[k] = s_start[k];

  // per unit (item i, KV head h): segments and partial rows
  const int num_units = num_items * num_kv_heads;
  int run_rows = 0;
  for (int base = 0; base < num_units; base += (int)blockDim.x) {
    const int u = base + threadIdx.x;
    int rows = 0, ns = 0, cf = 0;
    if (u < num_units) {
      const int i = u / num_kv_heads, h = u % num_kv_heads;
      const int tiles = ps->itiles[i], R = ps->iR[i];
      const bool grouped = i >= num_seqs || ps->pg[i] > 0;
      if (tiles > 0 && n > 0) {
        const int tp = ps->stp[i] + h * tiles;
        cf = upper_index(s_start, n - 1, tp);
        const int cl = upper_index(s_start, n - 1, tp + tiles - 1);
        ns = cl - cf + 1;
        if (ns > 1 || grouped) rows = ns * R;
      }
      nseg[u] = ns;
      cfirst[u] = cf;
    }
    int tot;
    const int pb = g_exclusive_scan(rows, s_warp, &tot);
    if (u < num_units) part_base[u] = rows > 0 ? run_rows + pb : -1;
    run_rows += tot;
  }
  if (threadIdx.x == 0) {
    PlanHeader* hd = reinterpret_cast<PlanHeader*>(ws);
    hd->total_tiles[0] = total;
    hd->total_tiles[1] = 0;
    hd->ncta[0] = n;
    hd->ncta[1] = 0;
    hd->tile_keys[0] = tile;
    hd->tile_keys[1] = 0;
    hd->num_seqs = num_seqs;
    hd->num_kv_heads = num_kv_heads;
    hd->group = group;
    hd->total_part_rows = run_rows;
    hd->rows_bound = rows_bound;
    hd->window = 0;
    hd->pad_[0] = num_items;
  }
}

// WPR warps per (token row, query head) whose result is in partials: rows of a
// split unit, and every row of a prefix group (its row block's partials, then
// its own unit's). As the plain combine: warp `sub` of a row accumulates the
// partials j = sub, sub + WPR, ..., every warp of the row reads all lse_j in
// one pass, and the WPR sums meet in shared memory.
template <int D, int WPR>
__global__ void __launch_bounds__(256, 2)
lse_combine_groups_kernel(int num_q_tokens, int num_q_heads, int num_seqs, int num_kv_heads,
                          int group, int rows_bound, const unsigned char* __restrict__ ws,
                          __nv_bfloat16* __restrict__ out, float* __restrict__ lse_out) {
  constexpr int EPL = D / 32;                     // output columns per lane
  constexpr int kRowsPerBlock = 8 / WPR;
  constexpr int kUnroll = WPR >= 4 ? 8 : 4;      // partial rows in flight per warp
  constexpr int VW = EPL >= 4 ? 4 : 2;           // floats per vector load
  using Vec = typename std::conditional<VW == 4, float4, float2>::type;
  static_assert(EPL % VW == 0, "vector loads of a lane's columns");
  __shared__ float s_acc[WPR > 1 ? 8 : 1][WPR > 1 ? D : 1];
  grid_dependency_wait();          // the attention kernel's partials are complete
  const GroupLayout L = make_group_layout(num_seqs, num_kv_heads, D, rows_bound);
  const int* q_off = reinterpret_cast<const int*>(ws + L.q_off);
  const int* seq_T = reinterpret_cast<const int*>(ws + L.seq_T);
  const int2* seq_grp = reinterpret_cast<const int2*>(ws + L.seq_grp);
  const ItemDesc* items = reinterpret_cast<const ItemDesc*>(ws + L.items);
  const int* nseg = reinterpret_cast<const int*>(ws + L.nseg);
  const int* part_base = reinterpret_cast<const int*>(ws + L.part_base);
  const float* o_part = reinterpret_cast<const float*>(ws + L.o_part);
  const float* lse_part = reinterpret_cast<const float*>(ws + L.lse_part);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, sub = warp % WPR;
  const long long row = (long long)blockIdx.x * kRowsPerBlock + warp / WPR;
  // the warp's row, when its result is in partials: n1 of its own unit's
  // (rows R1 apart from row r1 on), then the rest of its row block's (R2
  // apart from r2 on)
  bool active = row < (long long)num_q_tokens * num_q_heads;
  int i = 0, hq = 0, n1 = 0, n = 0, R1 = 0, r1 = 0, R2 = 0, r2 = 0;
  long long base1 = 0, base2 = 0;
  if (active) {
    i = (int)(row / num_q_heads);
    hq = (int)(row % num_q_heads);
    const int b = upper_index(q_off, num_seqs - 1, i);
    const int h = hq / group, g = hq % group;
    const int u = b * num_kv_heads + h;
    const int t = i - q_off[b];
    const int T = seq_T[b];
    const int2 gr = seq_grp[b];
    n1 = nseg[u];
    base1 = part_base[u];
    active = t < T;
    if (active) {
      R1 = T * group;
      r1 = t * group + g;
      n = n1 > 1 ? n1 : 0;
      if (gr.x >= 0) {                // a group row: its block's partials, and its own unit's always
        const int js = gr.y + r1;
        const int it = gr.x + js / kMaxRows;
        const int u2 = it * num_kv_heads + h;
        R2 = items[it].R;
        r2 = js % kMaxRows;
        base2 = part_base[u2];
        n = n1 + nseg[u2];
      }
      active = n > 0;
    }
  }
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  float m = -INFINITY, wsum = 0.f;
  if (active) {
    // lse = m + ln(wsum) over all partials, one pass
    float sl = 0.f;
    for (int j = lane; j < n; j += 32) {
      const float lj = lse_part[j < n1 ? base1 + (long long)j * R1 + r1
                                       : base2 + (long long)(j - n1) * R2 + r2];
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
          const long long pr = j < n1 ? base1 + (long long)j * R1 + r1
                                      : base2 + (long long)(j - n1) * R2 + r2;
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

cudaError_t launch_plan_groups(const int32_t* context_lens, const int32_t* block_lens,
                               const int32_t* shared_lens, int num_seqs, int num_kv_heads,
                               int group, int max_pages, int max_block_len, int tile, int ncta,
                               int rows_bound, int num_q_tokens, unsigned char* ws,
                               int* device_status, cudaStream_t stream) {
  if (num_seqs > kPrefixGroupMaxSeqs) return cudaErrorInvalidValue;
  const int dyn = (int)sizeof(GroupSmem);
  cudaError_t e = ensure_dynamic_smem<plan_groups_kernel>(dyn);
  if (e != cudaSuccess) return e;
  const int threads = num_seqs <= kGSmallSeqs ? kGThreadsSmall : kGThreadsLarge;
  plan_groups_kernel<<<1, threads, dyn, stream>>>(context_lens, block_lens, shared_lens,
                                                  num_seqs, num_kv_heads, group, max_pages,
                                                  max_block_len, tile, ncta, rows_bound,
                                                  num_q_tokens, ws, device_status);
  return cudaGetLastError();
}

cudaError_t launch_combine_groups(int num_q_tokens, int num_q_heads, int num_seqs,
                                  int num_kv_heads, int group, int head_dim, int rows_bound,
                                  int sms, const unsigned char* ws, __nv_bfloat16* out,
                                  float* lse, cudaStream_t stream) {
  const long long rows = (long long)num_q_tokens * num_q_heads;
  if (rows == 0) return cudaSuccess;
  // warps per row as in the plain combine
  const long long want = 16LL * (sms > 0 ? sms : 1);
  const int wpr = rows * 4 <= want ? 8 : rows * 2 <= want ? 4 : rows <= want ? 2 : 1;
  const long long rows_per_block = 8 / wpr;
  const int grid = (int)((rows + rows_per_block - 1) / rows_per_block);
  cudaError_t e = cudaErrorInvalidValue;
#define SPLASH_COMBINE_G(DD, WW)                                                               \
  e = launch_dependent(lse_combine_groups_kernel<DD, WW>, dim3(grid), dim3(256), 0, stream,    \
                       num_q_tokens, num_q_heads, num_seqs, num_kv_heads, group, rows_bound,  \
                       ws, out, lse)
#define SPLASH_COMBINE_GD(DD)                \
  switch (wpr) {                             \
    case 1: SPLASH_COMBINE_G(DD, 1); break;  \
    case 2: SPLASH_COMBINE_G(DD, 2); break;  \
    case 4: SPLASH_COMBINE_G(DD, 4); break;  \
    default: SPLASH_COMBINE_G(DD, 8); break; \
  }
  switch (head_dim) {
    case 128: SPLASH_COMBINE_GD(128); break;
    case 256: SPLASH_COMBINE_GD(256); break;
    default: return cudaErrorInvalidValue;
  }
#undef SPLASH_COMBINE_GD
#undef SPLASH_COMBINE_G
  return e;
}

}  // namespace splash
