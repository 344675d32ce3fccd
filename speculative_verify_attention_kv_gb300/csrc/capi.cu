// C ABI of the library: argument validation, split planning and launches.
// Nothing here allocates or synchronises; every launch goes to the caller's stream.
#include <atomic>
#include <mutex>

#include <cuda.h>

#include "splash_common.cuh"
#include "splash_groups.cuh"

namespace splash {
cudaError_t launch_kv_append(const float*, const float*, int, int8_t*, int8_t*, float*, float*,
                             const int32_t*, int, const int32_t*, const int32_t*, int, int, int,
                             int, int*, cudaStream_t);
cudaError_t launch_kv_append_bf16(const __nv_bfloat16*, const __nv_bfloat16*, int, int8_t*,
                                  int8_t*, float*, float*, const int32_t*, int, const int32_t*,
                                  const int32_t*, int, int, int, int, int*, cudaStream_t);
cudaError_t launch_accept_commit(const int32_t*, const int32_t*, int, const int32_t*, int32_t*,
                                 int32_t*, int32_t*, int, int*, cudaStream_t);
cudaError_t launch_plan(const int32_t*, const int32_t*, int, int, int, int, int, int, int, int,
                        int, int, int, int, int, unsigned char*, int*, cudaStream_t);
cudaError_t launch_combine(int, int, int, int, int, int, int, int, const unsigned char*,
                           __nv_bfloat16*, float*, cudaStream_t);
cudaError_t launch_verify_simt(const AttnParams&, int, int, cudaStream_t);
size_t simt_smem_bytes(int, int);
cudaError_t launch_verify_tc(const AttnParams&, int, int, bool, cudaStream_t);
cudaError_t launch_plan_groups(const int32_t*, const int32_t*, const int32_t*, int, int, int, int,
                               int, int, int, int, int, unsigned char*, int*, cudaStream_t);
cudaError_t launch_combine_groups(int, int, int, int, int, int, int, int, const unsigned char*,
                                  __nv_bfloat16*, float*, cudaStream_t);
bool tc_supported(int head_dim);
bool tt_supported(int head_dim, int rows_cap);
int tt_tile_keys();
bool tt_encode_map(CUtensorMap* map, const int8_t* k_pages, int num_pages, int num_kv_heads);
cudaError_t launch_verify_tt(const AttnParams&, const CUtensorMap&, int, cudaStream_t);
constexpr int kSimtTile = 64;
constexpr int kTcTile = 64;

namespace {

int device_sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

bool head_dim_ok(int d) { return d == 64 || d == 128 || d == 256; }

constexpr unsigned long long kDefaultWaitNs = 1000000000ull;   // 1 s
std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitNs};
std::atomic<unsigned long long> g_launches{0};               // kernels enqueued so far

cudaError_t counted(cudaError_t e) {
  if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
  return e;
}

// CTAs per class: the tensor-core kernel runs one CTA per SM, the CUDA-core
// kernel as many as fit.
void default_ctas(int sms, int head_dim, int rows_cap, int* ncta_tc, int* ncta_simt) {
  const size_t smem = simt_smem_bytes(head_dim, rows_cap);
  int per_sm = smem ? (int)((227 * 1024) / (smem + 1024)) : 1;
  per_sm = per_sm < 1 ? 1 : (per_sm > 4 ? 4 : per_sm);
  *ncta_tc = sms < kMaxCtas ? sms : kMaxCtas;
  *ncta_simt = sms * per_sm < kMaxCtas ? sms * per_sm : kMaxCtas;
}

long long rows_bound_for(int num_q_tokens, int num_q_heads, int rows_cap, int ncta_tc,
                         int ncta_simt) {
  (void)num_q_tokens;
  (void)num_q_heads;
  return 2LL * rows_cap * ((long long)ncta_tc + ncta_simt) + 1;
}

}  // namespace
}  // namespace splash

using namespace splash;

extern "C" {

const char* splash_status_string(int status) {
  switch (status) {
    case SPLASH_OK: return "SPLASH_OK";
    case SPLASH_ERR_INVALID_ARGUMENT: return "SPLASH_ERR_INVALID_ARGUMENT";
    case SPLASH_ERR_UNSUPPORTED: return "SPLASH_ERR_UNSUPPORTED";
    case SPLASH_ERR_WORKSPACE_TOO_SMALL: return "SPLASH_ERR_WORKSPACE_TOO_SMALL";
    case SPLASH_ERR_CUDA: return "SPLASH_ERR_CUDA";
  }
  return "SPLASH_UNKNOWN_STATUS";
}

// 2: one interleaved K/V code pool (v_pages = k_pages + P * D)
int splash_abi_version(void) { return 2; }

unsigned long long splash_launch_count(void) { return g_launches.load(); }

unsigned long long splash_set_wait_limit_ns(unsigned long long ns) {
  return g_wait_limit_ns.exchange(ns == 0 ? kDefaultWaitNs : ns);
}

int splash_tensor_path_supported(int head_dim) {
  return head_dim_ok(head_dim) && tc_supported(head_dim) ? 1 : 0;
}

int splash_kv_append(const float* k_new, const float* v_new, int num_new_tokens, int8_t* k_pages,
                     int8_t* v_pages, float* k_scales, float* v_scales, const int32_t* page_table,
                     int max_pages_per_seq, const int32_t* context_lens, const int32_t* block_lens,
                     int num_seqs, int num_kv_heads, int head_dim, int page_size, int num_pages,
                     int* device_status, struct CUstream_st* stream) {
  if (num_new_tokens < 0 || num_seqs < 0 || num_kv_heads <= 0 || num_pages < 0 ||
      max_pages_per_seq <= 0)
    return SPLASH_ERR_INVALID_ARGUMENT;
  if (page_size != kPageSize || !head_dim_ok(head_dim)) return SPLASH_ERR_UNSUPPORTED;
  if (num_new_tokens == 0 || num_seqs == 0) return SPLASH_OK;
  if (k_pages && v_pages && v_pages != k_pages + (size_t)page_size * head_dim)
    return SPLASH_ERR_INVALID_ARGUMENT;
  if (!k_new || !v_new || !k_pages || !v_pages || !k_scales || !v_scales || !page_table ||
      !context_lens || !block_lens)
    return SPLASH_ERR_INVALID_ARGUMENT;
  cudaError_t e = counted(launch_kv_append(k_new, v_new, num_new_tokens, k_pages, v_pages,
                                           k_scales, v_scales, page_table, max_pages_per_seq,
                                           context_lens, block_lens, num_seqs, num_kv_heads,
                                           head_dim, num_pages, device_status, stream));
  return e == cudaSuccess ? SPLASH_OK : SPLASH_ERR_CUDA;
}

int splash_kv_append_bf16(const uint16_t* k_new, const uint16_t* v_new, int num_new_tokens,
                          int8_t* k_pages, int8_t* v_pages, float* k_scales, float* v_scales,
                          const int32_t* page_table, int max_pages_per_seq,
                          const int32_t* context_lens, const int32_t* block_lens, int num_seqs,
                          int num_kv_heads, int head_dim, int page_size, int num_pages,
                          int* device_status, struct CUstream_st* stream) {
  if (num_new_tokens < 0 || num_seqs < 0 || num_kv_heads <= 0 || num_pages < 0 ||
      max_pages_per_seq <= 0)
    return SPLASH_ERR_INVALID_ARGUMENT;
  if (page_size != kPageSize || !head_dim_ok(head_dim)) return SPLASH_ERR_UNSUPPORTED;
  if (num_new_tokens == 0 || num_seqs == 0) return SPLASH_OK;
  if (k_pages && v_pages && v_pages != k_pages + (size_t)page_size * head_dim)
    return SPLASH_ERR_INVALID_ARGUMENT;
  if (!k_new || !v_new || !k_pages || !v_pages || !k_scales || !v_scales || !page_table ||
      !context_lens || !block_lens)
    return SPLASH_ERR_INVALID_ARGUMENT;
  cudaError_t e = counted(launch_kv_append_bf16(
      reinterpret_cast<const __nv_bfloat16*>(k_new), reinterpret_cast<const __nv_bfloat16*>(v_new),
      num_new_tokens, k_pages, v_pages, k_scales, v_scales, page_table, max_pages_per_seq,
      context_lens, block_lens, num_seqs, num_kv_heads, head_dim, num_pages, device_status,
      stream));
  return e == cudaSuccess ? SPLASH_OK : SPLASH_ERR_CUDA;
}

int splash_accept_commit(const int32_t* block_tokens, const int32_t* target_tokens,
                         int num_tokens, const int32_t* block_lens, int32_t* context_lens,
                         int32_t* accepted, int32_t* next_tokens, int num_seqs,
                         int* device_status, struct CUstream_st* stream) {
  if (num_tokens < 0 || num_seqs < 0) return SPLASH_ERR_INVALID_ARGUMENT;
  if (num_seqs == 0) return SPLASH_OK;
  if (!block_lens || !context_lens || !accepted || !next_tokens ||
      (num_tokens > 0 && (!block_tokens || !target_tokens)))
    return SPLASH_ERR_INVALID_ARGUMENT;
  cudaError_t e = counted(launch_accept_commit(block_tokens, target_tokens, num_tokens,
                                               block_lens, context_lens, accepted, next_tokens,
                                               num_seqs, device_status,
                                               reinterpret_cast<cudaStream_t>(stream)));
  return e == cudaSuccess ? SPLASH_OK : SPLASH_ERR_CUDA;
}

static int check_attn_shape(int num_q_tokens, int num_seqs, int num_q_heads, int num_kv_heads,
                            int head_dim, int page_size, int max_block_len, int max_pages) {
  if (num_q_tokens < 0 || num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      max_block_len < 0 || max_pages <= 0 || num_q_heads % num_kv_heads != 0)
    return SPLASH_ERR_INVALID_ARGUMENT;
  if (page_size != kPageSize || !head_dim_ok(head_dim)) return SPLASH_ERR_UNSUPPORTED;
  if ((long long)max_block_len * (num_q_heads / num_kv_heads) > kMaxRows)
    return SPLASH_ERR_UNSUPPORTED;
  return SPLASH_OK;
}

static size_t workspace_bytes_for(int num_seqs, int num_q_tokens, int num_q_heads,
                                  int num_kv_heads, int head_dim, int max_block_len, int ncta_tc,
                                  int ncta_simt) {
  const int G = num_q_heads / num_kv_heads;
  const int rows_cap = max_block_len * G;
  const long long rb = rows_bound_for(num_q_tokens, num_q_heads, rows_cap, ncta_tc, ncta_simt);
  return make_layout(num_seqs, num_kv_heads, head_dim, rb).total;
}

size_t splash_verify_attention_workspace_size(int num_seqs, int num_q_tokens, int num_q_heads,
                                              int num_kv_heads, int head_dim, int max_block_len) {
  if (check_attn_shape(num_q_tokens, num_seqs, num_q_heads, num_kv_heads, head_dim, kPageSize,
                       max_block_len, 1) != SPLASH_OK)
    return 0;
  const int sms = device_sm_count();
  if (sms <= 0) return 0;
  // the largest CTA counts any automatic choice can make
  return workspace_bytes_for(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim,
                             max_block_len, sms, 4 * sms);
}

size_t splash_verify_attention_shared_workspace_size(int num_seqs, int num_q_tokens,
                                                     int num_q_heads, int num_kv_heads,
                                                     int head_dim, int max_block_len) {
  if (check_attn_shape(num_q_tokens, num_seqs, num_q_heads, num_kv_heads, head_dim, kPageSize,
                       max_block_len, 1) != SPLASH_OK)
    return 0;
  const int sms = device_sm_count();
  if (sms <= 0) return 0;
  // without groups (a batch too large, a kernel without them) the plain plan runs
  const size_t plain = workspace_bytes_for(num_seqs, num_q_tokens, num_q_heads, num_kv_heads,
                                           head_dim, max_block_len, sms, 4 * sms);
  const long long rb = group_rows_bound(num_q_tokens, num_q_heads,
                                        max_block_len * (num_q_heads / num_kv_heads), sms);
  const size_t grouped = make_group_layout(num_seqs, num_kv_heads, head_dim, rb).total;
  return plain > grouped ? plain : grouped;
}

}  // extern "C"

// All attention entry points: window 0 is the full block-causal mask.
static int verify_impl(
    const uint16_t* q, int num_q_tokens, const int8_t* k_pages, const int8_t* v_pages,
    const float* k_scales, const float* v_scales, const int32_t* page_table,
    int max_pages_per_seq, const int32_t* context_lens, const int32_t* block_lens, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int page_size, int num_pages,
    int max_block_len, float sm_scale, int window, uint16_t* out, float* lse, void* workspace,
    size_t workspace_bytes, int* device_status, struct CUstream_st* stream, int path,
    int ctas_per_class, struct CUevent_st* attn_begin, struct CUevent_st* attn_end,
    const int32_t* shared_lens = nullptr) {
  int st = check_attn_shape(num_q_tokens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                            page_size, max_block_len, max_pages_per_seq);
  if (st != SPLASH_OK) return st;
  if (path < 0 || path > 3 || ctas_per_class < 0 || ctas_per_class > kMaxCtas || num_pages < 0 ||
      window < 0)
    return SPLASH_ERR_INVALID_ARGUMENT;
  if (num_q_tokens == 0 || num_seqs == 0) return SPLASH_OK;
  if (k_pages && v_pages && v_pages != k_pages + (size_t)page_size * head_dim)
    return SPLASH_ERR_INVALID_ARGUMENT;
  if (!q || !k_pages || !v_pages || !k_scales || !v_scales || !page_table || !context_lens ||
      !block_lens || !out || !lse || !workspace)
    return SPLASH_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return SPLASH_ERR_INVALID_ARGUMENT;
  const int G = num_q_heads / num_kv_heads;
  const int rows_cap = max_block_len * G;
  if (rows_cap == 0) return SPLASH_OK;
  if (!(sm_scale > 0.f) || sm_scale == INFINITY) return SPLASH_ERR_INVALID_ARGUMENT;
  const bool tc_ok = tc_supported(head_dim);
  if (path == 2 && !tc_ok) return SPLASH_ERR_UNSUPPORTED;
  if (path == 3 && !tt_supported(head_dim, rows_cap)) return SPLASH_ERR_UNSUPPORTED;
  // the transposed tensor-core kernel takes head_dim 256 with at most 96 rows
  // per unit (path 3); it reads the codes through a tensor map
  CUtensorMap tmap;
  bool use_tt = false;
  if (path == 3 && tt_supported(head_dim, rows_cap)) {
    use_tt = tt_encode_map(&tmap, k_pages, num_pages, num_kv_heads);
    if (!use_tt && path == 3) return SPLASH_ERR_INVALID_ARGUMENT;
  }
  if (path == 3) path = 2;
  if (!tc_ok) path = 1;
  // rows the CUDA-core kernel may see: all (path 1), none (path 2), fewer than
  // kTensorMinRows (automatic)
  const int rows_simt = path == 1 ? rows_cap : path == 2 ? 0
                        : (rows_cap < kTensorMinRows - 1 ? rows_cap : kTensorMinRows - 1);
  // the CUDA-core kernel holds every row of a unit in shared memory
  if (rows_simt > 0 && simt_smem_bytes(head_dim, rows_simt) > 227 * 1024)
    return SPLASH_ERR_UNSUPPORTED;

  const int sms = device_sm_count();
  if (sms <= 0) return SPLASH_ERR_CUDA;
  int nt, ns;
  default_ctas(sms, head_dim, rows_simt > 0 ? rows_simt : 1, &nt, &ns);
  if (ctas_per_class > 0) nt = ns = ctas_per_class;
  // prefix groups: on the tensor-core kernel of 64-key tiles, without a window,
  // for batches of up to kPrefixGroupMaxSeqs (elsewhere the same result is
  // computed without them)
  const bool groups = shared_lens != nullptr && window == 0 && path != 1 && tc_ok && !use_tt &&
                      num_seqs <= kPrefixGroupMaxSeqs;
  const long long rb = groups ? group_rows_bound(num_q_tokens, num_q_heads, rows_cap, nt)
                              : rows_bound_for(num_q_tokens, num_q_heads, rows_cap, nt, ns);
  const size_t need = groups ? make_group_layout(num_seqs, num_kv_heads, head_dim, rb).total
                             : workspace_bytes_for(num_seqs, num_q_tokens, num_q_heads,
                                                   num_kv_heads, head_dim, max_block_len, nt, ns);
  if (workspace_bytes < need) return SPLASH_ERR_WORKSPACE_TOO_SMALL;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  // in automatic mode, units too tall for the CUDA-core kernel's shared memory
  // go to the tensor-core kernel (the planner's row threshold already does so
  // for every unit with >= 16 rows).
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e =
      groups ? counted(launch_plan_groups(context_lens, block_lens, shared_lens, num_seqs,
                                          num_kv_heads, G, max_pages_per_seq, max_block_len,
                                          kTcTile, nt, (int)rb, num_q_tokens, ws, device_status,
                                          s))
             : counted(launch_plan(context_lens, block_lens, num_seqs, num_kv_heads, G,
                                   max_pages_per_seq, max_block_len,
                                   use_tt ? tt_tile_keys() : kTcTile, kSimtTile, nt, ns, path,
                                   (int)rb, num_q_tokens, window, ws, device_status, s));
  if (e != cudaSuccess) return SPLASH_ERR_CUDA;

  AttnParams p;
  p.q = reinterpret_cast<const __nv_bfloat16*>(q);
  p.k_pages = k_pages;
  p.v_pages = v_pages;
  p.k_scales = k_scales;
  p.v_scales = v_scales;
  p.page_table = page_table;
  p.max_pages_per_seq = max_pages_per_seq;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = G;
  p.head_dim = head_dim;
  p.num_pages = num_pages;
  p.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  p.window = window;
  p.wait_ns = g_wait_limit_ns.load();
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.ws = ws;
  p.device_status = device_status;
  if (attn_begin && cudaEventRecord(reinterpret_cast<cudaEvent_t>(attn_begin), s) != cudaSuccess)
    return SPLASH_ERR_CUDA;
  if (path != 1 && tc_ok) {
    e = counted(use_tt ? launch_verify_tt(p, tmap, nt, s) : launch_verify_tc(p, rows_cap, nt, groups, s));
    if (e != cudaSuccess) return SPLASH_ERR_CUDA;
  }
  if (path != 2 && rows_simt > 0 && !groups) {
    e = counted(launch_verify_simt(p, rows_simt, ns, s));
    if (e != cudaSuccess) return SPLASH_ERR_CUDA;
  }
  if (attn_end && cudaEventRecord(reinterpret_cast<cudaEvent_t>(attn_end), s) != cudaSuccess)
    return SPLASH_ERR_CUDA;
  e = groups ? counted(launch_combine_groups(num_q_tokens, num_q_heads, num_seqs, num_kv_heads, G,
                                             head_dim, (int)rb, sms, ws, p.out, lse, s))
             : counted(launch_combine(num_q_tokens, num_q_heads, num_seqs, num_kv_heads, G,
                                      head_dim, (int)rb, sms, ws, p.out, lse, s));
  return e == cudaSuccess ? SPLASH_OK : SPLASH_ERR_CUDA;
}

extern "C" {

int splash_verify_attention_profiled(
    const uint16_t* q, int num_q_tokens, const int8_t* k_pages, const int8_t* v_pages,
    const float* k_scales, const float* v_scales, const int32_t* page_table,
    int max_pages_per_seq, const int32_t* context_lens, const int32_t* block_lens, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int page_size, int num_pages,
    int max_block_len, float sm_scale, uint16_t* out, float* lse, void* workspace,
    size_t workspace_bytes, int* device_status, struct CUstream_st* stream, int path,
    int ctas_per_class, struct CUevent_st* attn_begin, struct CUevent_st* attn_end) {
  return verify_impl(q, num_q_tokens, k_pages, v_pages, k_scales, v_scales, page_table,
                     max_pages_per_seq, context_lens, block_lens, num_seqs, num_q_heads,
                     num_kv_heads, head_dim, page_size, num_pages, max_block_len, sm_scale, 0, out,
                     lse, workspace, workspace_bytes, device_status, stream, path, ctas_per_class,
                     attn_begin, attn_end);
}

int splash_verify_attention_shared_profiled(
    const uint16_t* q, int num_q_tokens, const int8_t* k_pages, const int8_t* v_pages,
    const float* k_scales, const float* v_scales, const int32_t* page_table,
    int max_pages_per_seq, const int32_t* context_lens, const int32_t* block_lens,
    const int32_t* shared_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int page_size, int num_pages, int max_block_len, float sm_scale, uint16_t* out, float* lse,
    void* workspace, size_t workspace_bytes, int* device_status, struct CUstream_st* stream,
    int path, int ctas_per_class, struct CUevent_st* attn_begin, struct CUevent_st* attn_end) {
  if (!shared_lens && num_seqs > 0 && num_q_tokens > 0) return SPLASH_ERR_INVALID_ARGUMENT;
  return verify_impl(q, num_q_tokens, k_pages, v_pages, k_scales, v_scales, page_table,
                     max_pages_per_seq, context_lens, block_lens, num_seqs, num_q_heads,
                     num_kv_heads, head_dim, page_size, num_pages, max_block_len, sm_scale, 0, out,
                     lse, workspace, workspace_bytes, device_status, stream, path, ctas_per_class,
                     attn_begin, attn_end, shared_lens);
}

int splash_verify_attention_shared(const uint16_t* q, int num_q_tokens, const int8_t* k_pages,
                                   const int8_t* v_pages, const float* k_scales,
                                   const float* v_scales, const int32_t* page_table,
                                   int max_pages_per_seq, const int32_t* context_lens,
                                   const int32_t* block_lens, const int32_t* shared_lens,
                                   int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                   int page_size, int num_pages, int max_block_len,
                                   float sm_scale, uint16_t* out, float* lse, void* workspace,
                                   size_t workspace_bytes, int* device_status,
                                   struct CUstream_st* stream) {
  return splash_verify_attention_shared_profiled(
      q, num_q_tokens, k_pages, v_pages, k_scales, v_scales, page_table, max_pages_per_seq,
      context_lens, block_lens, shared_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
      page_size, num_pages, max_block_len, sm_scale, out, lse, workspace, workspace_bytes,
      device_status, stream, 0, 0, nullptr, nullptr);
}

int splash_verify_attention_swa(const uint16_t* q, int num_q_tokens, const int8_t* k_pages,
                                const int8_t* v_pages, const float* k_scales,
                                const float* v_scales, const int32_t* page_table,
                                int max_pages_per_seq, const int32_t* context_lens,
                                const int32_t* block_lens, int num_seqs, int num_q_heads,
                                int num_kv_heads, int head_dim, int page_size, int num_pages,
                                int max_block_len, float sm_scale, int window, uint16_t* out,
                                float* lse, void* workspace, size_t workspace_bytes,
                                int* device_status, struct CUstream_st* stream, int path,
                                int ctas_per_class) {
  return verify_impl(q, num_q_tokens, k_pages, v_pages, k_scales, v_scales, page_table,
                     max_pages_per_seq, context_lens, block_lens, num_seqs, num_q_heads,
                     num_kv_heads, head_dim, page_size, num_pages, max_block_len, sm_scale, window,
                     out, lse, workspace, workspace_bytes, device_status, stream, path,
                     ctas_per_class, nullptr, nullptr);
}

int splash_verify_attention_tuned(const uint16_t* q, int num_q_tokens, const int8_t* k_pages,
                                  const int8_t* v_pages, const float* k_scales,
                                  const float* v_scales, const int32_t* page_table,
                                  int max_pages_per_seq, const int32_t* context_lens,
                                  const int32_t* block_lens, int num_seqs, int num_q_heads,
                                  int num_kv_heads, int head_dim, int page_size, int num_pages,
                                  int max_block_len, float sm_scale, uint16_t* out, float* lse,
                                  void* workspace, size_t workspace_bytes, int* device_status,
                                  struct CUstream_st* stream, int path, int ctas_per_class) {
  return splash_verify_attention_profiled(
      q, num_q_tokens, k_pages, v_pages, k_scales, v_scales, page_table, max_pages_per_seq,
      context_lens, block_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, page_size,
      num_pages, max_block_len, sm_scale, out, lse, workspace, workspace_bytes, device_status,
      stream, path, ctas_per_class, nullptr, nullptr);
}

int splash_verify_attention(const uint16_t* q, int num_q_tokens, const int8_t* k_pages,
                            const int8_t* v_pages, const float* k_scales, const float* v_scales,
                            const int32_t* page_table, int max_pages_per_seq,
                            const int32_t* context_lens, const int32_t* block_lens, int num_seqs,
                            int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                            int num_pages, int max_block_len, float sm_scale, uint16_t* out,
                            float* lse, void* workspace, size_t workspace_bytes,
                            int* device_status, struct CUstream_st* stream) {
  return splash_verify_attention_tuned(q, num_q_tokens, k_pages, v_pages, k_scales, v_scales,
                                       page_table, max_pages_per_seq, context_lens, block_lens,
                                       num_seqs, num_q_heads, num_kv_heads, head_dim, page_size,
                                       num_pages, max_block_len, sm_scale, out, lse, workspace,
                                       workspace_bytes, device_status, stream, 0, 0);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Entry point for callers that cannot allocate device memory: the workspace is
// a fixed array in the library's own device image instead of caller memory.
// ---------------------------------------------------------------------------
namespace {
constexpr size_t kFixedScratchBytes = size_t(64) << 20;   // 64 MiB per device
}  // namespace

// Lives in every device image that loads this library, until the process exits.
static __device__ __align__(256) unsigned char g_fixed_scratch[kFixedScratchBytes];

namespace {
std::mutex g_fixed_mu;
void* g_fixed_ptr[64] = {};

// Device address of g_fixed_scratch on the current device, looked up once per
// device (host code only sees a host-side stand-in under that name).
void* fixed_scratch_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_fixed_mu);
  if (g_fixed_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_fixed_scratch) != cudaSuccess) return nullptr;
    g_fixed_ptr[dev] = ptr;
  }
  return g_fixed_ptr[dev];
}
}  // namespace

extern "C" size_t splash_verify_attention_fixed_scratch_bytes(void) { return kFixedScratchBytes; }

extern "C" int splash_verify_attention_fixed_scratch(
    const uint16_t* q, int num_q_tokens, const int8_t* k_pages, const int8_t* v_pages,
    const float* k_scales, const float* v_scales, const int32_t* page_table,
    int max_pages_per_seq, const int32_t* context_lens, const int32_t* block_lens, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int page_size, int num_pages,
    int max_block_len, float sm_scale, uint16_t* out, float* lse, int* device_status,
    struct CUstream_st* stream) {
  const int st = check_attn_shape(num_q_tokens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                  page_size, max_block_len, max_pages_per_seq);
  if (st != SPLASH_OK) return st;
  if (num_q_tokens == 0 || num_seqs == 0 || max_block_len == 0) return SPLASH_OK;
  const int sms = device_sm_count();
  if (sms <= 0) return SPLASH_ERR_CUDA;
  // one CTA per SM for each kernel keeps the partial-row bound small
  const size_t need = workspace_bytes_for(num_seqs, num_q_tokens, num_q_heads, num_kv_heads,
                                          head_dim, max_block_len, sms, sms);
  if (need > kFixedScratchBytes) return SPLASH_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = fixed_scratch_current_device();
  if (scratch == nullptr) return SPLASH_ERR_CUDA;
  return splash_verify_attention_tuned(q, num_q_tokens, k_pages, v_pages, k_scales, v_scales,
                                       page_table, max_pages_per_seq, context_lens, block_lens,
                                       num_seqs, num_q_heads, num_kv_heads, head_dim, page_size,
                                       num_pages, max_block_len, sm_scale, out, lse, scratch,
                                       kFixedScratchBytes, device_status, stream, 0, sms);
}
