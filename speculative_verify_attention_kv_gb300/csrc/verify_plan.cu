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
constexpr int kPlanSmemSeqs = kPrefixGroupMaxSeqs;

// The planner's shared-memory arrays for batches of up to kPlanSmemSeqs
// sequences: per sequence T, ctx, class and the prefix sums per class (the
// tensor-core ones per item); with prefix groups also the Q row offsets, the
// links and stacked prefixes, and the rows and tiles of every item.
struct PlanSmem {
  int T[kPlanSmemSeqs], ctx[kPlanSmemSeqs], cls[kPlanSmemSeqs], qo[kPlanSmemSeqs];
  int sl[kPlanSmemSeqs];                       // keys shared with the previous sequence (0: none)
  int pg[kPlanSmemSeqs];                       // stacked prefix keys of the sequence's group (0: none)
  int iR[2 * kPlanSmemSeqs], itiles[2 * kPlanSmemSeqs];   // rows and tiles of each item
  int stp0[2 * kPlanSmemSeqs + 1], stp1[kPlanSmemSeqs + 1];
  long long wcost0[2 * kPlanSmemSeqs + 1], wcost1[kPlanSmemSeqs + 1];
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

// Per-sequence sums of pass 1: Q/O rows laid out, key tiles and estimated
// cost per class; the item pass of a plan with prefix groups sums the
// tensor-core class's tiles and cost over items (in w0 / t0).
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

// shared_lens (may be null): shared_lens[b] keys at the start of sequence b's
// context sit in the same pages as sequence b - 1's. With it (and no window),
// a run of consecutive tensor-core sequences linked this way is a prefix
// group: its sequences' rows, stacked in order, are cut into row blocks of
// kMaxRows, and each block reads the group's common prefix (the smallest link,
// cut to the sequences' contexts and down to a whole tile) once for all of its
// rows; each sequence then reads only its keys after the prefix. A group is
// stacked only when it needs fewer blocks than it has sequences.
__global__ void __launch_bounds__(kPlanThreadsLarge)
plan_kernel(const int32_t* __restrict__ context_lens, const int32_t* __restrict__ block_lens,
            const int32_t* __restrict__ shared_lens, int num_seqs, int num_kv_heads, int group,
            int max_pages, int max_block_len, int tile_tc, int tile_simt, int ncta_tc,
            int ncta_simt, int path, int rows_bound, int num_q_tokens, int window,
            unsigned char* ws, int* device_status) {
  __shared__ int s_warp[32];
  __shared__ int2 s_warp2[32];
  __shared__ PlanSums s_sums[32];
  __shared__ int s_start[kNumClasses][kMaxCtas + 1];
  extern __shared__ __align__(16) unsigned char s_dyn[];
  allow_dependent_launch();        // the attention kernel may get its SMs now
  const bool small = num_seqs <= kPlanSmemSeqs;     // launched with sizeof(PlanSmem) then
  // prefix groups are possible: the plan then has an item table
  const bool grp = shared_lens != nullptr && small && window == 0;
  PlanSmem* ps = reinterpret_cast<PlanSmem*>(s_dyn);
  const WorkspaceLayout L = make_layout(num_seqs, num_kv_heads, 0, rows_bound);
  int* q_off = reinterpret_cast<int*>(ws + L.q_off);
  int* seq_T = reinterpret_cast<int*>(ws + L.seq_T);
  int* seq_ctx = reinterpret_cast<int*>(ws + L.seq_ctx);
  int* seq_class = reinterpret_cast<int*>(ws + L.seq_class);
  int2* seq_grp = reinterpret_cast<int2*>(ws + L.seq_grp);
  ItemDesc* items = reinterpret_cast<ItemDesc*>(ws + L.items);
  int* stp0 = reinterpret_cast<int*>(ws + L.stp0);
  int* stp1 = reinterpret_cast<int*>(ws + L.stp1);
  int* nseg = reinterpret_cast<int*>(ws + L.nseg);
  int* cfirst = reinterpret_cast<int*>(ws + L.cfirst);
  int* part_base = reinterpret_cast<int*>(ws + L.part_base);
  long long* wcost0 = reinterpret_cast<long long*>(ws + L.wcost0);
  long long* wcost1 = reinterpret_cast<long long*>(ws + L.wcost1);
  int* cta_start = reinterpret_cast<int*>(ws + L.cta_start);
  const int tile[kNumClasses] = {tile_tc, tile_simt};
  const int ncta[kNumClasses] = {ncta_tc, ncta_simt};

  // pass 1: per sequence — validate, classify, prefix sums of rows and of
  // tiles and cost per class; sequence b's tensor-core item is item b.
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
      if (shared_lens != nullptr) seq_grp[b] = make_int2(-1, 0);   // read by the combine then
      if (small) {
        ps->T[b] = T;
        ps->ctx[b] = ctx;
        ps->cls[b] = cls;
      }
      if (grp) ps->pg[b] = 0;
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
      const int qo = (int)min(run_q + ex.q, (long long)num_q_tokens);
      q_off[b] = qo;
      stp0[b] = run_t0 + ex.t0;
      stp1[b] = run_t1 + ex.t1;
      wcost0[b] = run_w[0] + ex.w0;
      wcost1[b] = run_w[1] + ex.w1;
      if (grp) {                   // the sequence's item (the item walk reads it)
        ItemDesc d;
        d.b = b;
        d.qbase = qo;
        d.r0 = 0;
        d.R = T * group;
        d.ctx = ctx;
        d.Lk = cls == kClassTensor ? ctx + T : 0;           // no tensor-core tiles otherwise
        d.klo = cls == kClassTensor ? unit_first_key(ctx, window) : 0;
        d.grouped = 0;
        items[b] = d;
        ps->qo[b] = qo;
        ps->iR[b] = d.R;
        ps->itiles[b] = cls == kClassTensor ? tiles : 0;
      }
      if (small) {
        ps->stp0[b] = run_t0 + ex.t0;
        ps->stp1[b] = run_t1 + ex.t1;
        ps->wcost0[b] = run_w[0] + ex.w0;
        ps->wcost1[b] = run_w[1] + ex.w1;
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
    stp0[num_seqs] = run_t0;
    stp1[num_seqs] = run_t1;
    wcost0[num_seqs] = run_w[0];
    wcost1[num_seqs] = run_w[1];
    if (small) {
      ps->stp0[num_seqs] = run_t0;
      ps->stp1[num_seqs] = run_t1;
      ps->wcost0[num_seqs] = run_w[0];
      ps->wcost1[num_seqs] = run_w[1];
    }
  }
  __syncthreads();
  // where the later passes read the per-sequence arrays
  const int* rT = small ? ps->T : seq_T;
  const int* rctx = small ? ps->ctx : seq_ctx;
  const int* rcls = small ? ps->cls : seq_class;
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

  // prefix groups (tensor-core class; items num_seqs.. are their row blocks)
  int num_blocks = 0;
  if (grp && rows_ok) {
    // link of b to b - 1: the shared keys, cut to both contexts; 0 below a tile
    for (int b = threadIdx.x; b < num_seqs; b += blockDim.x) {
      int sl = 0;
      if (b > 0 && ps->cls[b] == kClassTensor && ps->cls[b - 1] == kClassTensor) {
        sl = min(shared_lens[b], min(ps->ctx[b], ps->ctx[b - 1]));
        if (sl < tile_tc) sl = 0;
      }
      ps->sl[b] = sl;
    }
    __syncthreads();
    // the first sequence of each group walks its group
    for (int base = 0; base < num_seqs; base += (int)blockDim.x) {
      const int b = base + threadIdx.x;
      int nblk = 0, m = 0, pg = 0, rows = 0;
      if (b < num_seqs && ps->cls[b] == kClassTensor && ps->sl[b] == 0 && b + 1 < num_seqs &&
          ps->sl[b + 1] > 0) {
        pg = ps->ctx[b];
        rows = ps->T[b] * group;
        int e = b + 1;
        for (; e < num_seqs && ps->sl[e] > 0; ++e) {
          pg = min(pg, ps->sl[e]);
          rows += ps->T[e] * group;
        }
        m = e - b;
        pg = pg / tile_tc * tile_tc;
        nblk = (rows + kMaxRows - 1) / kMaxRows;
        if (pg < tile_tc || nblk >= m) nblk = 0;     // stacking would not save a pass
      }
      int tot;
      const int ex = block_exclusive_scan(nblk, s_warp, &tot);
      if (nblk > 0) {
        const int first_item = num_seqs + num_blocks + ex;
        int so = 0;
        for (int e = b; e < b + m; ++e) {
          // the member reads only its keys past the prefix
          seq_grp[e] = make_int2(first_item, so);
          ps->pg[e] = pg;
          items[e].klo = pg;
          items[e].grouped = 1;
          ps->itiles[e] = (ps->ctx[e] + ps->T[e] + tile_tc - 1) / tile_tc - pg / tile_tc;
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
          ps->itiles[first_item + k] = pg / tile_tc;
        }
      }
      num_blocks += tot;
    }
    __syncthreads();
    if (num_blocks > 0) {
      // the tensor-core class's prefix sums again, over all items
      run_t0 = 0;
      run_w[0] = 0;
      const int ni = num_seqs + num_blocks;
      for (int base = 0; base < ni; base += (int)blockDim.x) {
        const int i = base + threadIdx.x;
        const int tiles = i < ni ? ps->itiles[i] : 0;
        long long cost = 0;
        if (tiles > 0)
          cost = (long long)num_kv_heads *
                 ((long long)tiles * (tile_cost(0) + row_cost(0) * ps->iR[i]) + segment_cost(0));
        const PlanSums mine{0, cost, 0, tiles * num_kv_heads, 0};
        PlanSums tot;
        const PlanSums ex = block_exclusive_scan_sums(mine, s_sums, &tot);
        if (i < ni) {
          stp0[i] = run_t0 + ex.t0;
          wcost0[i] = run_w[0] + ex.w0;
          ps->stp0[i] = run_t0 + ex.t0;
          ps->wcost0[i] = run_w[0] + ex.w0;
        }
        run_t0 += tot.t0;
        run_w[0] += tot.w0;
      }
      if (threadIdx.x == 0) {
        stp0[ni] = run_t0;
        wcost0[ni] = run_w[0];
        ps->stp0[ni] = run_t0;
        ps->wcost0[ni] = run_w[0];
      }
      __syncthreads();
    }
  }
  const int num_items = num_seqs + num_blocks;
  // the attention kernel's item walk searches max_items(num_seqs) entries of
  // stp0: the ones past the items must exceed every tile index
  if (grp)
    for (int i = num_items + 1 + threadIdx.x; i <= max_items(num_seqs); i += blockDim.x)
      stp0[i] = INT_MAX;

  // rows and tensor-core tiles of item i
  auto item_shape = [&](int i, int& R, int& tiles) {
    if (grp) {
      R = ps->iR[i];
      tiles = ps->itiles[i];
    } else {                       // one item per sequence
      R = rT[i] * group;
      tiles = rcls[i] == kClassTensor ? unit_tiles(rctx[i], rT[i], window, tile_tc) : 0;
    }
  };
  const int total[kNumClasses] = {run_t0, run_t1};
  // a class's kernel uses at most one CTA per tile, so that every CTA it uses
  // owns >= 1 tile and the CTAs covering a unit are consecutive, all non-empty
  int ncta_eff[kNumClasses];
  for (int c = 0; c < kNumClasses; ++c) ncta_eff[c] = min(min(ncta[c], total[c]), kMaxCtas);

  // CTA c of a class starts where the class's cumulative cost reaches
  // c / n of its total: find the item (sequence), then the unit (KV head), then the
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
        if (k <= n && n > 0) {
          if (k == n) {
            start[c] = total[c];
          } else if (k > 0) {
            const long long target = run_w[c] * k / n;      // < 2^63 for any realistic batch
            int b, tiles, R, sp;
            long long off;
            if (c == 0) {
              const long long* wc = small ? ps->wcost0 : wcost0;
              b = upper_index(wc, num_items - 1, target);
              off = target - wc[b];
              item_shape(b, R, tiles);
              sp = small ? ps->stp0[b] : stp0[b];
            } else {
              const long long* wc = small ? ps->wcost1 : wcost1;
              b = upper_index(wc, num_seqs - 1, target);
              off = target - wc[b];
              tiles = unit_tiles(rctx[b], rT[b], window, tile[1]);
              R = rT[b] * group;
              sp = small ? ps->stp1[b] : stp1[b];
            }
            const long long w = tile_cost(c) + row_cost(c) * R;
            const long long uc = (long long)tiles * w + segment_cost(c);
            const int h = (int)min(off / uc, (long long)num_kv_heads - 1);
            const long long rem = off - h * uc;
            const int t = rem < segment_cost(c) ? 0 : (int)min((rem - segment_cost(c)) / w, (long long)tiles - 1);
            start[c] = sp + h * tiles + t;
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

  // pass 2: per unit (item or sequence i, KV head h) — segments and partial
  // rows. Units i * Hkv + h with i < num_seqs are sequence i's (the CUDA-core
  // kernel's when the sequence is in its class).
  const int num_units = num_items * num_kv_heads;
  int run_rows = 0;
  for (int base = 0; base < num_units; base += (int)blockDim.x) {
    const int u = base + threadIdx.x;
    int rows = 0, ns = 0, cf = 0;
    if (u < num_units) {
      const int i = u / num_kv_heads, h = u % num_kv_heads;
      const bool simt = i < num_seqs && rcls[i] == kClassSimt;
      int tiles, R, grouped, tp;
      if (simt) {
        tiles = unit_tiles(rctx[i], rT[i], window, tile[1]);
        R = rT[i] * group;
        grouped = 0;
        tp = (small ? ps->stp1[i] : stp1[i]) + h * tiles;
      } else {
        item_shape(i, R, tiles);
        grouped = grp && (i >= num_seqs || ps->pg[i] > 0);
        tp = (small ? ps->stp0[i] : stp0[i]) + h * tiles;
      }
      const int nce = simt ? ncta_eff[1] : ncta_eff[0];
      if (tiles > 0 && nce > 0) {
        const int* cs = s_start[simt ? 1 : 0];
        cf = upper_index(cs, nce - 1, tp);
        const int cl = upper_index(cs, nce - 1, tp + tiles - 1);
        ns = cl - cf + 1;
        if (ns > 1 || grouped) rows = ns * R;
      }
      nseg[u] = ns;
      cfirst[u] = cf;
    }
    int tot;
    const int pb = block_exclusive_scan(rows, s_warp, &tot);
    if (u < num_units) part_base[u] = rows > 0 ? run_rows + pb : -1;
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
    hd->num_items = num_items;
  }
}

// WPR warps per (token row, query head) whose result is in partials: rows of a
// unit split over several CTAs, and every row of a prefix group (its row
// block's partials, then its own unit's). Warp `sub` of a row
// accumulates the partials j = sub, sub + WPR, ... (four or eight partial rows
// in flight), and the WPR sums meet in shared memory. Every warp of a row reads all
// lse_j in one pass (running max and rescaled sum per lane, then merged across
// the warp), so the weights exp(lse_j - lse) agree across the row's warps->
// kGroups: the plan may hold prefix groups (else the second source is never
// looked up, and the kernel keeps the registers of the one-source loop).
template <int D, int WPR, bool kGroups>
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
  const int2* seq_grp = reinterpret_cast<const int2*>(ws + L.seq_grp);
  const ItemDesc* items = reinterpret_cast<const ItemDesc*>(ws + L.items);
  const int* nseg = reinterpret_cast<const int*>(ws + L.nseg);
  const int* part_base = reinterpret_cast<const int*>(ws + L.part_base);
  const float* o_part = reinterpret_cast<const float*>(ws + L.o_part);
  const float* lse_part = reinterpret_cast<const float*>(ws + L.lse_part);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, sub = warp % WPR;
  const long long row = (long long)blockIdx.x * kRowsPerBlock + warp / WPR;
  // the warp's row, when its result is in partials: n1 of its own unit's
  // (rows R1 apart from row r1 on), then n2 of its row block's (R2 apart from r2)
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
    n1 = nseg[u];
    base1 = part_base[u];
    active = t < T;
    if (active) {
      R1 = T * group;
      r1 = t * group + g;
      n = n1 > 1 ? n1 : 0;
      const int2 gr = kGroups ? seq_grp[b] : make_int2(-1, 0);
      if (kGroups && gr.x >= 0) {       // prefix group: its row block, and its own unit always
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
      const float lj = lse_part[(!kGroups || j < n1) ? base1 + (long long)j * R1 + r1
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
          const long long pr = (!kGroups || j < n1) ? base1 + (long long)j * R1 + r1
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

cudaError_t launch_plan(const int32_t* context_lens, const int32_t* block_lens,
                        const int32_t* shared_lens, int num_seqs, int num_kv_heads, int group,
                        int max_pages, int max_block_len, int tile_tc, int tile_simt, int ncta_tc,
                        int ncta_simt, int path, int rows_bound, int num_q_tokens, int window,
                        unsigned char* ws, int* device_status, cudaStream_t stream) {
  const size_t dyn = num_seqs <= kPlanSmemSeqs ? sizeof(PlanSmem) : 0;
  const int threads = num_seqs <= kPlanSmallSeqs ? kPlanThreadsSmall : kPlanThreadsLarge;
  if (dyn > 0) {
    const cudaError_t e = ensure_dynamic_smem<plan_kernel>((int)dyn);
    if (e != cudaSuccess) return e;
  }
  plan_kernel<<<1, threads, dyn, stream>>>(context_lens, block_lens, shared_lens, num_seqs,
                                              num_kv_heads, group, max_pages, max_block_len,
                                              tile_tc, tile_simt, ncta_tc, ncta_simt, path,
                                              rows_bound, num_q_tokens, window, ws, device_status);
  return cudaGetLastError();
}

cudaError_t launch_combine(int num_q_tokens, int num_q_heads, int num_seqs, int num_kv_heads,
                           int group, int head_dim, int rows_bound, int sms, bool prefix_groups,
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
  e = prefix_groups                                                                             \
          ? launch_dependent(lse_combine_kernel<DD, WW, true>, dim3(grid), dim3(256), 0, stream, \
                             num_q_tokens, num_q_heads, num_seqs, num_kv_heads, group,          \
                             rows_bound, ws, out, lse)                                          \
          : launch_dependent(lse_combine_kernel<DD, WW, false>, dim3(grid), dim3(256), 0,       \
                             stream, num_q_tokens, num_q_heads, num_seqs, num_kv_heads, group,  \
                             rows_bound, ws, out, lse)
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
