// CUDA-core verify attention (the kernel for units with few query rows).
//
// Persistent CTAs walk their share of the CUDA-core class's tile stream. For
// one unit (sequence b, KV head h) the T*G query rows (row r = t*G + g) stay in
// shared memory; each tile of kTileKeys keys is gathered through the page
// table into shared memory as int8 codes plus fp32 scales, then
//   scores  S[r][j] = (q_r . c_j) * sK_j * sm_scale      (masked: j > ctx + t)
//   online softmax over the tile (running max m_r, sum l_r, in log2 units)
//   O[r][:] = O[r][:] * alpha_r + sum_j p_rj * sV_j * c_j
// Keys past the sequence end, and keys on an invalid page, get scale 0 and
// probability 0, so whatever bytes sit there cannot reach the output.
#include "splash_common.cuh"

namespace splash {

constexpr int kSimtThreads = 256;
constexpr int kSimtTileKeys = 64;

template <int D>
struct SimtSmem {
  static constexpr int kQStride = D + 8;   // bf16 elements per Q row (16-byte pad)
  static constexpr int kKStride = D + 16;  // bytes per K/V row (16-byte pad)
  static size_t bytes(int R) {
    return sizeof(__nv_bfloat16) * (size_t)R * kQStride + sizeof(float) * (size_t)R * D +
           sizeof(float) * (size_t)R * kSimtTileKeys + 2 * (size_t)kSimtTileKeys * kKStride +
           2 * sizeof(float) * kSimtTileKeys + 3 * sizeof(float) * (size_t)R + 64;
  }
};

template <int D>
__global__ void __launch_bounds__(kSimtThreads)
verify_simt_kernel(AttnParams p, int rows_cap) {
  using SM = SimtSmem<D>;
  constexpr int TK = kSimtTileKeys;
  extern __shared__ __align__(16) unsigned char smem[];
  __nv_bfloat16* q_s = reinterpret_cast<__nv_bfloat16*>(smem);
  float* o_s = reinterpret_cast<float*>(q_s + (size_t)rows_cap * SM::kQStride);
  float* s_s = o_s + (size_t)rows_cap * D;
  int8_t* k_s = reinterpret_cast<int8_t*>(s_s + (size_t)rows_cap * TK);
  int8_t* v_s = k_s + TK * SM::kKStride;
  float* ks_s = reinterpret_cast<float*>(v_s + TK * SM::kKStride);
  float* vs_s = ks_s + TK;
  float* m_s = vs_s + TK;
  float* l_s = m_s + rows_cap;
  float* a_s = l_s + rows_cap;

  grid_dependency_wait();          // the split plan is complete
  allow_dependent_launch();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = p.num_seqs, Hkv = p.num_kv_heads, G = p.group;
  const WorkspaceLayout L = make_layout(B, Hkv, D, reinterpret_cast<const PlanHeader*>(p.ws)->rows_bound);
  const PlanHeader* hd = reinterpret_cast<const PlanHeader*>(p.ws);
  const int* q_off = reinterpret_cast<const int*>(p.ws + L.q_off);
  const int* seq_T = reinterpret_cast<const int*>(p.ws + L.seq_T);
  const int* seq_ctx = reinterpret_cast<const int*>(p.ws + L.seq_ctx);
  const int* stp = reinterpret_cast<const int*>(p.ws + L.stp) + kClassSimt * (B + 1);
  const int* nseg = reinterpret_cast<const int*>(p.ws + L.nseg);
  const int* cfirst = reinterpret_cast<const int*>(p.ws + L.cfirst);
  const int* part_base = reinterpret_cast<const int*>(p.ws + L.part_base);
  float* o_part = reinterpret_cast<float*>(p.ws + L.o_part);
  float* lse_part = reinterpret_cast<float*>(p.ws + L.lse_part);

  const int ncta = hd->ncta[kClassSimt];
  const int window = hd->window;
  if ((int)blockIdx.x >= ncta) return;
  const int* cst = reinterpret_cast<const int*>(p.ws + L.cta_start) + kClassSimt * (kMaxCtas + 1);
  int t = cst[blockIdx.x];
  const int t_end = cst[blockIdx.x + 1];

  while (t < t_end) {
    const int b = upper_index(stp, B - 1, t);
    const int T = seq_T[b], ctx = seq_ctx[b];
    const int Lk = ctx + T;
    const int klo = unit_first_key(ctx, window);           // keys below are never visible
    const int first = unit_first_tile(ctx, window, TK);
    const int tiles = unit_tiles(ctx, T, window, TK);
    const int local = t - stp[b];
    const int h = local / tiles;
    const int i0 = first + local % tiles;
    const int i1 = min(first + tiles, i0 + (t_end - t));
    const int R = T * G;
    const int u = b * Hkv + h;
    const int32_t* ptab = p.page_table + (size_t)b * p.max_pages_per_seq;

    // Q rows of this unit -> shared memory; reset running state
    for (int idx = tid; idx < R * (D / 8); idx += kSimtThreads) {
      const int r = idx / (D / 8), c = idx % (D / 8);
      const int tt = r / G, g = r % G;
      const __nv_bfloat16* src =
          p.q + ((size_t)(q_off[b] + tt) * p.num_q_heads + h * G + g) * D + c * 8;
      *reinterpret_cast<uint4*>(q_s + (size_t)r * SM::kQStride + c * 8) =
          *reinterpret_cast<const uint4*>(src);
    }
    for (int idx = tid; idx < R * D; idx += kSimtThreads) o_s[idx] = 0.f;
    for (int r = tid; r < R; r += kSimtThreads) {
      m_s[r] = -INFINITY;
      l_s[r] = 0.f;
    }
    __syncthreads();

    for (int it = i0; it < i1; ++it) {
      const int k0 = it * TK;
      // gather codes + scales of keys k0 .. k0+TK-1
      for (int idx = tid; idx < 2 * TK * (D / 16); idx += kSimtThreads) {
        const int which = idx / (TK * (D / 16));          // 0: K, 1: V
        const int rem = idx % (TK * (D / 16));
        const int jj = rem / (D / 16), c = rem % (D / 16);
        const int j = k0 + jj;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (j < Lk && j >= klo) {
          const int page = ptab[j / kPageSize];
          if (page >= 0 && page < p.num_pages) {
            const int8_t* base = (which ? p.v_pages : p.k_pages) +
                                 code_offset(page, h, Hkv, j % kPageSize, D);
            val = *reinterpret_cast<const uint4*>(base + c * 16);
          }
        }
        *reinterpret_cast<uint4*>((which ? v_s : k_s) + jj * SM::kKStride + c * 16) = val;
      }
      for (int jj = tid; jj < 2 * TK; jj += kSimtThreads) {
        const int which = jj / TK, j = k0 + jj % TK;
        float sc = 0.f;
        if (j < Lk && j >= klo) {
          const int page = ptab[j / kPageSize];
          if (page >= 0 && page < p.num_pages) {
            const float* sp = which ? p.v_scales : p.k_scales;
            sc = sp[((size_t)page * Hkv + h) * kPageSize + j % kPageSize];
          } else {
            report(p.device_status, SPLASH_DEVICE_BAD_PAGE);
          }
        }
        (which ? vs_s : ks_s)[jj % TK] = sc;
      }
      __syncthreads();

      // scores (log2 units); consecutive threads take consecutive rows of one key
      for (int idx = tid; idx < R * TK; idx += kSimtThreads) {
        const int jj = idx / R, r = idx % R;
        const int j = k0 + jj;
        const bool vis = (j < Lk) && (j <= ctx + r / G) && (window <= 0 || j > ctx + r / G - window);
        float dot = 0.f;
        const __nv_bfloat16* qr = q_s + (size_t)r * SM::kQStride;
        const int8_t* kr = k_s + jj * SM::kKStride;
#pragma unroll 4
        for (int d = 0; d < D; d += 16) {
          const uint4 kw = *reinterpret_cast<const uint4*>(kr + d);
          const int8_t* kb = reinterpret_cast<const int8_t*>(&kw);
          const uint4 q0 = *reinterpret_cast<const uint4*>(qr + d);
          const uint4 q1 = *reinterpret_cast<const uint4*>(qr + d + 8);
          const __nv_bfloat162* qa = reinterpret_cast<const __nv_bfloat162*>(&q0);
          const __nv_bfloat162* qb = reinterpret_cast<const __nv_bfloat162*>(&q1);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 fa = __bfloat1622float2(qa[e]);
            const float2 fb = __bfloat1622float2(qb[e]);
            dot = fmaf(fa.x, (float)kb[2 * e], dot);
            dot = fmaf(fa.y, (float)kb[2 * e + 1], dot);
            dot = fmaf(fb.x, (float)kb[8 + 2 * e], dot);
            dot = fmaf(fb.y, (float)kb[8 + 2 * e + 1], dot);
          }
        }
        s_s[r * TK + jj] = vis ? dot * ks_s[jj] * p.sm_scale_log2 : -INFINITY;
      }
      __syncthreads();

      // online softmax: one warp per row
      for (int r = warp; r < R; r += kSimtThreads / 32) {
        float mx = -INFINITY;
        for (int jj = lane; jj < TK; jj += 32) mx = fmaxf(mx, s_s[r * TK + jj]);
        mx = warp_max(mx);
        const float m_old = m_s[r];
        const float m_new = fmaxf(m_old, mx);
        float sum = 0.f;
        for (int jj = lane; jj < TK; jj += 32) {
          const float sv = s_s[r * TK + jj];
          const float pv = (sv == -INFINITY) ? 0.f : exp2f(sv - m_new);
          s_s[r * TK + jj] = pv;
          sum += pv;
        }
        sum = warp_sum(sum);
        if (lane == 0) {
          const float alpha = (m_old == -INFINITY) ? 0.f : exp2f(m_old - m_new);
          l_s[r] = l_s[r] * alpha + sum;
          m_s[r] = m_new;
          a_s[r] = alpha;
        }
      }
      __syncthreads();

      // O update: consecutive threads take consecutive d of one row
      for (int idx = tid; idx < R * D; idx += kSimtThreads) {
        const int r = idx / D, d = idx % D;
        float acc = o_s[idx] * a_s[r];
        const float* pr = s_s + r * TK;
#pragma unroll 8
        for (int jj = 0; jj < TK; ++jj) acc = fmaf(pr[jj] * vs_s[jj], (float)v_s[jj * SM::kKStride + d], acc);
        o_s[idx] = acc;
      }
      __syncthreads();
    }

    // finalize: final output when this CTA covers the whole unit, else a partial
    const int ns = nseg[u];
    const int jseg = blockIdx.x - cfirst[u];
    const long long prow0 = (long long)part_base[u] + (long long)jseg * R;
    for (int idx = tid; idx < R * D; idx += kSimtThreads) {
      const int r = idx / D, d = idx % D;
      const float l = l_s[r];
      const float o = l > 0.f ? o_s[idx] / l : 0.f;
      if (ns == 1) {
        const int tt = r / G, g = r % G;
        p.out[((size_t)(q_off[b] + tt) * p.num_q_heads + h * G + g) * D + d] = __float2bfloat16_rn(o);
      } else {
        o_part[(prow0 + r) * D + d] = o;
      }
    }
    for (int r = tid; r < R; r += kSimtThreads) {
      const float l = l_s[r];
      const float lse = l > 0.f ? (m_s[r] + log2f(l)) * 0.69314718055994531f : -INFINITY;
      if (ns == 1) {
        const int tt = r / G, g = r % G;
        p.lse[(size_t)(q_off[b] + tt) * p.num_q_heads + h * G + g] = lse;
      } else {
        lse_part[prow0 + r] = lse;
      }
    }
    __syncthreads();
    t += i1 - i0;
  }
}

size_t simt_smem_bytes(int head_dim, int rows_cap) {
  switch (head_dim) {
    case 64: return SimtSmem<64>::bytes(rows_cap);
    case 128: return SimtSmem<128>::bytes(rows_cap);
    case 256: return SimtSmem<256>::bytes(rows_cap);
  }
  return 0;
}

cudaError_t launch_verify_simt(const AttnParams& p, int rows_cap, int ncta, cudaStream_t stream) {
  const size_t smem = simt_smem_bytes(p.head_dim, rows_cap);
#define SPLASH_SIMT(DD)                                                                        \
  do {                                                                                         \
    cudaError_t e = ensure_dynamic_smem<verify_simt_kernel<DD>>((int)smem);                   \
    if (e != cudaSuccess) return e;                                                            \
    e = launch_dependent(verify_simt_kernel<DD>, dim3(ncta), dim3(kSimtThreads), smem, stream, \
                         p, rows_cap);                                                         \
    if (e != cudaSuccess) return e;                                                            \
  } while (0)
  switch (p.head_dim) {
    case 64: SPLASH_SIMT(64); break;
    case 128: SPLASH_SIMT(128); break;
    case 256: SPLASH_SIMT(256); break;
    default: return cudaErrorInvalidValue;
  }
#undef SPLASH_SIMT
  return cudaGetLastError();
}

}  // namespace splash
