// Accept / commit of a verified block (the step after verify attention).
//
// Reading: sequence b's verify block holds tokens x_0 .. x_{T-1}, where x_0 is
// the token the target produced at the previous step and x_1 .. x_{T-1} are the
// draft's proposals; the target's next-token choices after each of them are
// y_0 .. y_{T-1}. Draft x_{i+1} is accepted while x_{i+1} == y_i for every
// earlier i. With a accepted drafts, x_0 .. x_a are committed (their K/V are
// already in the cache from the block append), context_lens[b] grows by a + 1,
// and y_a becomes the next step's x_0. Slots past the committed length are
// rewritten by the next append. A sequence with T = 0 is left as it is.
#include "splash_common.cuh"

namespace splash {

constexpr int kAcceptThreads = 1024;

__device__ inline int block_exclusive_scan_1024(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int x = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    s_warp[lane] = x;
  }
  __syncthreads();
  const int res = (warp ? s_warp[warp - 1] : 0) + incl - v;
  *total = s_warp[31];
  __syncthreads();
  return res;
}

// one CTA; sequences in chunks of 1024
__global__ void __launch_bounds__(kAcceptThreads)
accept_commit_kernel(const int32_t* __restrict__ block_tokens,
                     const int32_t* __restrict__ target_tokens, int num_tokens,
                     const int32_t* __restrict__ block_lens, int32_t* __restrict__ context_lens,
                     int32_t* __restrict__ accepted, int32_t* __restrict__ next_tokens,
                     int num_seqs, int* device_status) {
  __shared__ int s_warp[32];
  int run = 0;
  for (int base = 0; base < num_seqs; base += kAcceptThreads) {
    const int b = base + threadIdx.x;
    int T = 0;
    if (b < num_seqs) T = max(block_lens[b], 0);
    int tot;
    const int off = run + block_exclusive_scan_1024(T, s_warp, &tot);
    run += tot;
    if (b < num_seqs) {
      if (T == 0) {
        accepted[b] = 0;
        next_tokens[b] = -1;
      } else if (off + T > num_tokens) {
        report(device_status, SPLASH_DEVICE_BAD_LENGTH);
        accepted[b] = 0;
        next_tokens[b] = -1;
      } else {
        int a = 0;
        while (a + 1 < T && block_tokens[off + a + 1] == target_tokens[off + a]) ++a;
        accepted[b] = a;
        next_tokens[b] = target_tokens[off + a];
        context_lens[b] += a + 1;
      }
    }
  }
}

cudaError_t launch_accept_commit(const int32_t* block_tokens, const int32_t* target_tokens,
                                 int num_tokens, const int32_t* block_lens, int32_t* context_lens,
                                 int32_t* accepted, int32_t* next_tokens, int num_seqs,
                                 int* device_status, cudaStream_t stream) {
  accept_commit_kernel<<<1, kAcceptThreads, 0, stream>>>(block_tokens, target_tokens, num_tokens,
                                                         block_lens, context_lens, accepted,
                                                         next_tokens, num_seqs, device_status);
  return cudaGetLastError();
}

}  // namespace splash
