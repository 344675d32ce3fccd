// kv_quantize_append: quantise a verify block's K/V rows to int8 and scatter
// them into the paged cache.
//
// One warp per (new token, KV head) row; a CTA of 8 warps covers 8 / Hkv
// tokens (one token when Hkv >= 8, its warps then loop over the heads). A row
// of D fp32 values is spread over the 32 lanes (D/32 consecutive values per
// lane, 16-byte loads), its absmax is a warp max, and each lane writes its D/32
// codes as one store. Scale and quotient use correctly rounded fp32 division (no fast-math
// in this translation unit), rounding is half-to-even (cvt.rni).
#include "splash_common.cuh"

namespace splash {

constexpr int kAppendWarps = 8;
constexpr int kAppendThreads = 32 * kAppendWarps;
constexpr int kAppendTokPerCta = kAppendWarps;   // upper bound (Hkv = 1)

template <int EPL>
__device__ inline void load_row(const __nv_bfloat16* p, float (&x)[EPL]) {
  // bf16 -> fp32 is exact
  if constexpr (EPL == 2) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
    x[0] = f.x; x[1] = f.y;
  } else if constexpr (EPL == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
  } else {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[i]));
      x[2 * i] = f.x; x[2 * i + 1] = f.y;
    }
  }
}

template <int EPL>
__device__ inline void load_row(const float* p, float (&x)[EPL]) {
  if constexpr (EPL == 2) {
    float2 a = *reinterpret_cast<const float2*>(p);
    x[0] = a.x; x[1] = a.y;
  } else {
#pragma unroll
    for (int i = 0; i < EPL / 4; ++i) {
      float4 a = *reinterpret_cast<const float4*>(p + 4 * i);
      x[4 * i] = a.x; x[4 * i + 1] = a.y; x[4 * i + 2] = a.z; x[4 * i + 3] = a.w;
    }
  }
}

template <int EPL>
__device__ inline void quantise_store(const float (&x)[EPL], int8_t* codes_dst, float* scale_dst,
                                      int lane) {
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) a = fmaxf(a, fabsf(x[i]));
  a = warp_max(a);
  const float s = __fdiv_rn(a, 127.0f);
  uint32_t packed[(EPL + 3) / 4] = {};
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    int c = 0;
    if (s != 0.f) {
      c = __float2int_rn(__fdiv_rn(x[i], s));
      c = max(-127, min(127, c));
    }
    packed[i / 4] |= (uint32_t)(c & 0xff) << (8 * (i % 4));
  }
  if constexpr (EPL == 2) {
    *reinterpret_cast<uint16_t*>(codes_dst) = (uint16_t)packed[0];
  } else if constexpr (EPL == 4) {
    *reinterpret_cast<uint32_t*>(codes_dst) = packed[0];
  } else {
    *reinterpret_cast<uint2*>(codes_dst) = make_uint2(packed[0], packed[1]);
  }
  if (lane == 0) *scale_dst = s;
}

template <int D, typename TIn>
__global__ void __launch_bounds__(kAppendThreads)
kv_append_kernel(const TIn* __restrict__ k_new, const TIn* __restrict__ v_new,
                 int num_new_tokens, int8_t* __restrict__ k_pages, int8_t* __restrict__ v_pages,
                 float* __restrict__ k_scales, float* __restrict__ v_scales,
                 const int32_t* __restrict__ page_table, int max_pages,
                 const int32_t* __restrict__ context_lens, const int32_t* __restrict__ block_lens,
                 int num_seqs, int num_kv_heads, int num_pages, int tok_per_cta,
                 int* device_status) {
  constexpr int EPL = D / 32;
  __shared__ int s_seq[kAppendTokPerCta];
  __shared__ int s_first[kAppendTokPerCta];
  __shared__ int s_warp_tot[kAppendThreads / 32];
  __shared__ int s_running;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tok0 = blockIdx.x * tok_per_cta;
  if (tid < kAppendTokPerCta) s_seq[tid] = -1;
  if (tid == 0) s_running = 0;
  __syncthreads();

  // Chunked exclusive scan of block_lens: find the sequence of each token of this CTA.
  for (int base = 0; base < num_seqs; base += kAppendThreads) {
    const int b = base + tid;
    int T = 0;
    if (b < num_seqs) {
      T = block_lens[b];
      const int ctx = context_lens[b];
      if (T < 0 || ctx < 0 || (long long)ctx + T > (long long)max_pages * kPageSize) {
        if (blockIdx.x == 0) report(device_status, SPLASH_DEVICE_BAD_LENGTH);
        T = max(T, 0);
      }
    }
    int incl = T;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp_tot[warp] = incl;
    __syncthreads();
    int warp_off = 0, chunk_tot = 0;
#pragma unroll
    for (int w = 0; w < kAppendThreads / 32; ++w) {
      if (w < warp) warp_off += s_warp_tot[w];
      chunk_tot += s_warp_tot[w];
    }
    const int running = s_running;
    const int first = running + warp_off + incl - T;
    const int lo = max(first, tok0), hi = min(first + T, tok0 + tok_per_cta);
    for (int i = lo; i < hi; ++i) {
      s_seq[i - tok0] = b;
      s_first[i - tok0] = first;
    }
    __syncthreads();
    if (tid == 0) s_running = running + chunk_tot;
    __syncthreads();
    if (s_running >= tok0 + tok_per_cta) break;
  }

  for (int item = warp; item < tok_per_cta * num_kv_heads; item += kAppendWarps) {
    const int ti = item / num_kv_heads, h = item % num_kv_heads;
    const int tok = tok0 + ti;
    if (tok >= num_new_tokens) break;
    const int b = s_seq[ti];
    if (b < 0) continue;  // row past sum(block_lens)
    const int T = block_lens[b], ctx = context_lens[b];
    if (T < 0 || ctx < 0 || (long long)ctx + T > (long long)max_pages * kPageSize) continue;
    const int pos = ctx + (tok - s_first[ti]);
    const int page = page_table[(size_t)b * max_pages + pos / kPageSize];
    if (page < 0 || page >= num_pages) {
      if (lane == 0) report(device_status, SPLASH_DEVICE_BAD_PAGE);
      continue;
    }
    const int slot = pos % kPageSize;
    const size_t src = ((size_t)tok * num_kv_heads + h) * D + lane * EPL;
    const size_t row = ((size_t)page * num_kv_heads + h) * kPageSize + slot;   // scale index
    const size_t code = code_offset(page, h, num_kv_heads, slot, D);
    float xk[EPL], xv[EPL];
    load_row<EPL>(k_new + src, xk);
    load_row<EPL>(v_new + src, xv);
    quantise_store<EPL>(xk, k_pages + code + lane * EPL, k_scales + row, lane);
    quantise_store<EPL>(xv, v_pages + code + lane * EPL, v_scales + row, lane);
  }
}

template <typename TIn>
cudaError_t launch_kv_append_t(const TIn* k_new, const TIn* v_new, int num_new_tokens,
                               int8_t* k_pages, int8_t* v_pages, float* k_scales, float* v_scales,
                               const int32_t* page_table, int max_pages,
                               const int32_t* context_lens, const int32_t* block_lens,
                               int num_seqs, int num_kv_heads, int head_dim, int num_pages,
                               int* device_status, cudaStream_t stream) {
  if (num_new_tokens == 0 || num_seqs == 0) return cudaSuccess;
  const int tok_per_cta = num_kv_heads >= kAppendWarps ? 1 : kAppendWarps / num_kv_heads;
  const int grid = (num_new_tokens + tok_per_cta - 1) / tok_per_cta;
#define SPLASH_APPEND(DD)                                                                   \
  kv_append_kernel<DD, TIn><<<grid, kAppendThreads, 0, stream>>>(                                \
      k_new, v_new, num_new_tokens, k_pages, v_pages, k_scales, v_scales, page_table,       \
      max_pages, context_lens, block_lens, num_seqs, num_kv_heads, num_pages, tok_per_cta,   \
      device_status)
  switch (head_dim) {
    case 64: SPLASH_APPEND(64); break;
    case 128: SPLASH_APPEND(128); break;
    case 256: SPLASH_APPEND(256); break;
    default: return cudaErrorInvalidValue;
  }
#undef SPLASH_APPEND
  return cudaGetLastError();
}

cudaError_t launch_kv_append(const float* k_new, const float* v_new, int num_new_tokens,
                             int8_t* k_pages, int8_t* v_pages, float* k_scales, float* v_scales,
                             const int32_t* page_table, int max_pages,
                             const int32_t* context_lens, const int32_t* block_lens, int num_seqs,
                             int num_kv_heads, int head_dim, int num_pages, int* device_status,
                             cudaStream_t stream) {
  return launch_kv_append_t<float>(k_new, v_new, num_new_tokens, k_pages, v_pages, k_scales,
                                   v_scales, page_table, max_pages, context_lens, block_lens,
                                   num_seqs, num_kv_heads, head_dim, num_pages, device_status,
                                   stream);
}

cudaError_t launch_kv_append_bf16(const __nv_bfloat16* k_new, const __nv_bfloat16* v_new,
                                  int num_new_tokens, int8_t* k_pages, int8_t* v_pages,
                                  float* k_scales, float* v_scales, const int32_t* page_table,
                                  int max_pages, const int32_t* context_lens,
                                  const int32_t* block_lens, int num_seqs, int num_kv_heads,
                                  int head_dim, int num_pages, int* device_status,
                                  cudaStream_t stream) {
  return launch_kv_append_t<__nv_bfloat16>(k_new, v_new, num_new_tokens, k_pages, v_pages,
                                           k_scales, v_scales, page_table, max_pages,
                                           context_lens, block_lens, num_seqs, num_kv_heads,
                                           head_dim, num_pages, device_status, stream);
}

}  // namespace splash
