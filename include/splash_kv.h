/*
 * splash_kv.h — C ABI of the int8 paged-KV verify-attention library (GB300, sm_103a).
 *
 * The operation. In-batch speculative decoding as the Splash engine describes it
 * ("Splash: 범용 엔진 대신 모델마다 커널과 초안 모델을 새로 만드는 Apple Silicon 추론
 * 엔진", discuss.pytorch.kr; section "옵션이 아니라 기본 경로인 DFlash 2 추측
 * 디코딩"): every sequence submits a block of T draft tokens that the target
 * model verifies in one forward pass, each sequence with its own T. Attention
 * state lives in a paged KV cache indexed by prefix, so sequences that share a
 * prefix share its pages (section "배치 스케줄링과 시작 시점에 확정되는 메모리
 * 예산"). The decode kernel reads the 8-bit KV cache directly and reuses each
 * KV tile across the query heads of a GQA group and across the verify tokens
 * (section "형상에 맞춰 자동으로 생성하는 Metal 커널"). The bnskd.com article
 * ("Splash：把推理引擎「围着模型造」…", section "技术内核") states the same.
 * The pages fix no quantisation scheme, layout, mask or precision; the ones
 * below are this library's readings.
 *
 * Conventions for every entry point
 *   - Pointers named *_pages, *_scales, q, out, lse, page_table, *_lens,
 *     k_new, v_new, workspace and device_status are DEVICE pointers owned by
 *     the caller. The library never allocates, frees or synchronises; all work
 *     is enqueued on `stream` (NULL = legacy default stream) and is async.
 *   - Return value: SPLASH_OK or a negative SPLASH_ERR_* code. Argument errors
 *     are detected on the host BEFORE anything is launched. A CUDA launch error
 *     returns SPLASH_ERR_CUDA (the CUDA error is left for cudaGetLastError).
 *   - Errors only visible on the device (a page id out of range or -1 where a
 *     page is needed, a length out of range) never trap: the kernel skips the
 *     affected work and, when device_status is non-NULL, stores the first such
 *     SPLASH_DEVICE_* code there (atomic compare-and-swap from 0). The caller
 *     zeroes *device_status before the call and reads it after the stream syncs.
 *
 * Shapes and layouts (row-major, innermost last)
 *   Hq = num_q_heads, Hkv = num_kv_heads, G = Hq / Hkv (query head hq uses KV
 *   head hq / G), D = head_dim in {64, 128, 256}, P = page_size = 16.
 *   codes            : int8  one pool [num_pages, Hkv, 2, P, D]; index 0 of the
 *                      third axis holds K codes, 1 holds V codes, so the K and V
 *                      codes of a (page, KV head) are one contiguous 2*P*D-byte
 *                      block. k_pages points at the pool, v_pages must equal
 *                      k_pages + P*D (anything else is SPLASH_ERR_INVALID_ARGUMENT).
 *                      v_pages is therefore fixed by k_pages: it carries no
 *                      information of its own, and separate K and V pools (the
 *                      layout of a two-pool cache) cannot be passed. The
 *                      interleaving lets one bulk copy move a (page, KV head)'s
 *                      K and V codes together; a copy's issue cost is mostly
 *                      per copy, and the same attention ran 6.8% faster than
 *                      with two pools of 4 KB copies at D = 256.
 *                      Slot s of (page, h): k_pages[((page*Hkv + h)*2*P + s)*D + d],
 *                      and the same offset from v_pages.
 *   k_scales, v_scales: fp32 [num_pages, Hkv, P]      one scale per (token, KV head)
 *   page_table       : int32 [num_seqs, max_pages_per_seq]; logical position j of
 *                      sequence b lives in page page_table[b][j / P], slot j % P.
 *                      Entries past a sequence's needed pages are ignored (-1 is
 *                      the customary sentinel). Pages may be shared between
 *                      sequences (shared prefix); they are read-only to attention.
 *   context_lens     : int32 [num_seqs] tokens cached before the block (ctx_b >= 0)
 *   block_lens       : int32 [num_seqs] verify-block length T_b >= 0 (0 = idle)
 *   Tokens of all blocks are packed by sequence: sequence b owns rows
 *   sum(block_lens[0..b-1]) .. + T_b - 1 of q / k_new / v_new / out / lse.
 */
#ifndef SPLASH_KV_H
#define SPLASH_KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t */

enum {
  SPLASH_OK = 0,
  SPLASH_ERR_INVALID_ARGUMENT = -1,   /* null pointer, negative size, Hq % Hkv != 0 ... */
  SPLASH_ERR_UNSUPPORTED = -2,        /* D not in {64,128,256}, P != 16, T*G too large */
  SPLASH_ERR_WORKSPACE_TOO_SMALL = -3,
  SPLASH_ERR_CUDA = -4                /* a kernel launch failed */
};

enum {
  SPLASH_DEVICE_BAD_PAGE = 1,         /* page id < 0 or >= num_pages where a page is needed */
  SPLASH_DEVICE_BAD_LENGTH = 2,       /* ctx or T negative, T > max_block_len, or
                                         ctx + T > max_pages_per_seq * P, or
                                         sum(block_lens) > num_q_tokens */
  SPLASH_DEVICE_TIMEOUT = 3,          /* an internal wait of the tensor-core kernel gave
                                         up (after 1 s by default, see
                                         splash_set_wait_limit_ns); outputs of that
                                         call undefined */
  SPLASH_DEVICE_INTERNAL = 4          /* the tensor-core kernel found its shared memory
                                         misaligned and did nothing */
};

/* Human-readable name of a SPLASH_* status (static string, never NULL). */
const char* splash_status_string(int status);

/* Library ABI version (increments on any signature or layout change; 2 = the
 * interleaved K/V code pool). */
int splash_abi_version(void);

/* 1 if the tensor-core attention kernel is built for this head_dim, else 0
 * (units then run on the CUDA-core kernel). */
int splash_tensor_path_supported(int head_dim);

/* Number of kernels the library has enqueued since it was loaded (all entry
 * points, all threads; a host-side count of successful launches). Lets a
 * caller count the device work one call or one benchmark step issues. */
unsigned long long splash_launch_count(void);

/* Limit, in nanoseconds, of every internal pipeline wait of the tensor-core
 * attention kernel for the launches that follow (process-wide; 0 restores the
 * default of 1 s). When a wait runs out, the kernel stops the call's work,
 * lets the copies and MMAs it already issued complete, frees its tensor
 * memory, returns, and stores SPLASH_DEVICE_TIMEOUT in device_status; the
 * outputs of that call are undefined and later calls are unaffected. Meant
 * for tests of that path and for diagnosing a stalled GPU. Returns the
 * previous limit. */
unsigned long long splash_set_wait_limit_ns(unsigned long long ns);

/*
 * splash_kv_append — quantise a block of new K/V rows to int8 and write them
 * into the pages.
 *
 * For every sequence b and t < T_b, row r = sum(block_lens[0..b-1]) + t of
 * k_new / v_new (fp32 [num_new_tokens, Hkv, D]) is written at logical position
 * context_lens[b] + t, separately per KV head:
 *   a = max_d |x_d|;  s = fl32(a / 127);  c_d = clamp(rne(fl32(x_d / s)), -127, 127)
 *   (s == 0 gives all-zero codes), with correctly rounded fp32 division and
 *   round-half-to-even. Codes go to k_pages / v_pages, s to k_scales / v_scales.
 * num_new_tokens must equal sum(block_lens) (not checked on the host, which
 * cannot read device memory; rows past the sum are ignored). The target slots
 * must not be shared with another sequence (copy-on-write is the caller's).
 * Populating a cache uses the same call with context_lens = start positions.
 */
int splash_kv_append(const float* k_new, const float* v_new, int num_new_tokens,
                     int8_t* k_pages, int8_t* v_pages, float* k_scales, float* v_scales,
                     const int32_t* page_table, int max_pages_per_seq,
                     const int32_t* context_lens, const int32_t* block_lens, int num_seqs,
                     int num_kv_heads, int head_dim, int page_size, int num_pages,
                     int* device_status, struct CUstream_st* stream);

/*
 * splash_kv_append_bf16 — splash_kv_append for bf16 K/V rows (bit patterns,
 * [num_new_tokens, Hkv, D]), the dtype a projection usually produces. Each
 * value converts exactly to fp32, then the same quantiser applies; codes and
 * scales equal those of splash_kv_append on the fp32 copies of the same rows.
 */
int splash_kv_append_bf16(const uint16_t* k_new, const uint16_t* v_new, int num_new_tokens,
                          int8_t* k_pages, int8_t* v_pages, float* k_scales, float* v_scales,
                          const int32_t* page_table, int max_pages_per_seq,
                          const int32_t* context_lens, const int32_t* block_lens, int num_seqs,
                          int num_kv_heads, int head_dim, int page_size, int num_pages,
                          int* device_status, struct CUstream_st* stream);

/*
 * splash_accept_commit — the step after verification: each sequence advances
 * by the tokens it accepted (Splash article, section "옵션이 아니라 기본 경로인
 * DFlash 2 추측 디코딩": every request carries its own draft state and moves on
 * by its accepted tokens).
 *
 * block_tokens, target_tokens: int32 [num_tokens], packed by sequence like q.
 * Sequence b's block is x_0 .. x_{T_b-1} (x_0 = the token the target emitted at
 * the previous step, x_1.. = the draft's proposals); target_tokens holds the
 * target's next-token choice y_i after each x_i. Draft x_{i+1} is accepted
 * while x_{i+1} == y_i for all earlier i. With a accepted drafts:
 *   accepted[b] = a;  context_lens[b] += a + 1 (x_0 .. x_a are committed: their
 *   K/V were written by the block append);  next_tokens[b] = y_a.
 * Sequences with T_b = 0 get accepted = 0, next_tokens = -1 and keep their
 * length. Slots beyond the new length are overwritten by the next append.
 * context_lens is updated in place on the device; one small launch, no sync.
 */
int splash_accept_commit(const int32_t* block_tokens, const int32_t* target_tokens,
                         int num_tokens, const int32_t* block_lens, int32_t* context_lens,
                         int32_t* accepted, int32_t* next_tokens, int num_seqs,
                         int* device_status, struct CUstream_st* stream);

/*
 * splash_verify_attention_workspace_size — bytes of device workspace that
 * splash_verify_attention needs for these bounds on the current device
 * (depends on its SM count). Returns 0 for invalid arguments.
 */
size_t splash_verify_attention_workspace_size(int num_seqs, int num_q_tokens, int num_q_heads,
                                              int num_kv_heads, int head_dim, int max_block_len);

/*
 * splash_verify_attention — block-causal attention of every verify token over
 * its sequence's int8 paged cache (the block itself already appended).
 *
 * The target model checks a sequence's whole draft block in one forward pass
 * (Splash article on discuss.pytorch.kr, section "옵션이 아니라 기본 경로인
 * DFlash 2 추측 디코딩"); the kernel reads the 8-bit cache directly and serves
 * the G query heads of a KV head and the T verify tokens from each KV tile it
 * loads (section "형상에 맞춰 자동으로 생성하는 Metal 커널"). The mask that lets
 * verify token t see the block's tokens 0..t is this library's reading: the
 * pages do not state one.
 *
 * Verify token t of sequence b, query head hq (KV head h = hq / G) attends to
 * logical keys j = 0 .. context_lens[b] + t inclusive, dequantised as
 * code * scale:
 *   score_j = sm_scale * sum_d q[d] * k_hat_j[d]
 *   out     = sum_j softmax(score)_j * v_hat_j              -> bf16 (RNE)
 *   lse     = ln sum_j exp(score_j)   (sm_scale included)   -> fp32
 * q, out: bf16 bit patterns [num_q_tokens, Hq, D]; lse: fp32 [num_q_tokens, Hq].
 * num_q_tokens = sum(block_lens). max_block_len bounds every T_b (T_b * G must
 * be <= 128). sm_scale must be finite and > 0. The KV range of every
 * sequence is split across CTAs; partials
 * are merged by log-sum-exp in `workspace` (>= the size query's bytes, 256-byte
 * aligned). Deterministic: a fixed input, device and argument list gives
 * bitwise identical outputs, independent of the physical page numbering.
 */
int splash_verify_attention(const uint16_t* q, int num_q_tokens,
                            const int8_t* k_pages, const int8_t* v_pages,
                            const float* k_scales, const float* v_scales,
                            const int32_t* page_table, int max_pages_per_seq,
                            const int32_t* context_lens, const int32_t* block_lens, int num_seqs,
                            int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                            int num_pages, int max_block_len, float sm_scale,
                            uint16_t* out, float* lse, void* workspace, size_t workspace_bytes,
                            int* device_status, struct CUstream_st* stream);

/*
 * splash_verify_attention_tuned — splash_verify_attention with the kernel
 * choice and the split granularity fixed by the caller (tests, benchmarks).
 *   path: 0 automatic; 1 CUDA-core kernel for every sequence; 2 tensor-core
 *         kernel for every sequence; 3 the transposed tensor-core kernel
 *         (S^T = K Q'^T: keys on the MMA's M side, no row padding) for every
 *         sequence, only at head_dim 256 with T * G <= 96
 *         (SPLASH_ERR_UNSUPPORTED otherwise). Path 3 exists for comparison:
 *         it is slower than path 2 on every workload measured.
 *   ctas_per_class: 0 automatic (fills the GPU); 0 < n <= 1023 uses n
 *         persistent CTAs per kernel (1 = every sequence's KV range handled
 *         unsplit); larger n is SPLASH_ERR_INVALID_ARGUMENT. The planner
 *         splits each kernel's stream of key tiles over its CTAs by estimated
 *         cost (a tile of a unit with more query rows costs more; every unit
 *         start adds one pipeline fill), from the lengths alone.
 * Same result contract as splash_verify_attention (within rounding across
 * different choices; bitwise for a fixed choice).
 */
int splash_verify_attention_tuned(const uint16_t* q, int num_q_tokens,
                                  const int8_t* k_pages, const int8_t* v_pages,
                                  const float* k_scales, const float* v_scales,
                                  const int32_t* page_table, int max_pages_per_seq,
                                  const int32_t* context_lens, const int32_t* block_lens,
                                  int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                  int page_size, int num_pages, int max_block_len, float sm_scale,
                                  uint16_t* out, float* lse, void* workspace,
                                  size_t workspace_bytes, int* device_status,
                                  struct CUstream_st* stream, int path, int ctas_per_class);

/*
 * splash_verify_attention_swa — splash_verify_attention_tuned with a sliding
 * window: verify token t of sequence b sees only the `window` most recent keys
 * up to its own position, context_lens[b] + t - window < j <= context_lens[b]
 * + t (the draft model's windowed attention, "옵션이 아니라 기본 경로인 DFlash 2
 * 추측 디코딩" section of the Splash article on discuss.pytorch.kr). window = 0
 * is the full mask of splash_verify_attention; window < 0 is an argument error.
 * Page-table entries of pages that lie wholly below key
 * context_lens[b] - window + 1 are never read (they may be -1). Same output,
 * workspace, determinism and error contract as splash_verify_attention.
 */
int splash_verify_attention_swa(const uint16_t* q, int num_q_tokens,
                                const int8_t* k_pages, const int8_t* v_pages,
                                const float* k_scales, const float* v_scales,
                                const int32_t* page_table, int max_pages_per_seq,
                                const int32_t* context_lens, const int32_t* block_lens,
                                int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                int page_size, int num_pages, int max_block_len, float sm_scale,
                                int window, uint16_t* out, float* lse, void* workspace,
                                size_t workspace_bytes, int* device_status,
                                struct CUstream_st* stream, int path, int ctas_per_class);

/*
 * splash_verify_attention_profiled — splash_verify_attention_tuned that also
 * records two caller-created CUDA events on `stream`: `attn_begin` just before
 * the attention kernel launch(es) and `attn_end` just after, so that the
 * attention kernels can be timed apart from the split planner and the
 * log-sum-exp combine. Either event may be NULL. Same work, same results.
 */
struct CUevent_st; /* cudaEvent_t */
int splash_verify_attention_profiled(const uint16_t* q, int num_q_tokens,
                                     const int8_t* k_pages, const int8_t* v_pages,
                                     const float* k_scales, const float* v_scales,
                                     const int32_t* page_table, int max_pages_per_seq,
                                     const int32_t* context_lens, const int32_t* block_lens,
                                     int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim, int page_size, int num_pages,
                                     int max_block_len, float sm_scale, uint16_t* out, float* lse,
                                     void* workspace, size_t workspace_bytes, int* device_status,
                                     struct CUstream_st* stream, int path, int ctas_per_class,
                                     struct CUevent_st* attn_begin, struct CUevent_st* attn_end);

/*
 * splash_verify_attention_shared — splash_verify_attention for a batch whose
 * sequences share prefix pages, reading each shared prefix tile once for the
 * stacked query rows of all sequences that share it.
 *
 * The Splash article on discuss.pytorch.kr indexes the paged KV cache by
 * prefix, so requests with a common prefix point at the same pages (section
 * "배치 스케줄링과 시작 시점에 확정되는 메모리 예산"), and it measures
 * concurrent agent requests that share a long prefix (section "동시 요청에서 더
 * 벌어지는 격차"). This entry point extends the reuse of one KV tile across the
 * query rows of a sequence to the rows of every sequence sharing the tile.
 *
 *   shared_lens: int32 [num_seqs] (device, non-NULL). shared_lens[b] > 0 states
 *     that logical keys 0 .. shared_lens[b] - 1 of sequence b sit in the same
 *     pages as those of sequence b - 1 (equal page-table entries); 0 states
 *     nothing; shared_lens[0] is ignored. The caller guarantees the claim.
 *     The library only clamps it to both sequences' context_lens: a claim
 *     whose pages differ gives sequence b the keys of sequence b - 1's pages.
 *
 * A run of consecutive sequences b0 .. b1, each linked to the one before it
 * by at least 64 keys, is a prefix group. Its common prefix is the smallest
 * link, cut to every member's context and down to a multiple of 64 keys. The
 * members' query rows (sum of T_b * G), stacked in sequence order, are cut
 * into blocks of 128 rows. Each block reads the common prefix through the
 * pages of b0's page-table row. Each member reads only its own keys after
 * the prefix. The log-sum-exp combine then merges the two partial results of
 * every row. A group is stacked only when it needs fewer blocks than it has
 * members (e.g. four sequences of T * G = 96 rows: 3 blocks instead of 4
 * passes over the prefix; four of 6 rows: 1 block).
 *
 * Output, result and error contract as splash_verify_attention. The result
 * equals splash_verify_attention's within rounding, since the same scores are
 * summed in a different split. Groups apply only on the tensor-core kernel
 * (path 0 or 2, head_dim 128 or 256), and on batches of at most 1024
 * sequences. Elsewhere the call computes the same result without stacking.
 * The workspace must hold splash_verify_attention_shared_workspace_size bytes
 * (more than splash_verify_attention's: every grouped row leaves two partial
 * rows). shared_lens == NULL is SPLASH_ERR_INVALID_ARGUMENT.
 */
size_t splash_verify_attention_shared_workspace_size(int num_seqs, int num_q_tokens,
                                                     int num_q_heads, int num_kv_heads,
                                                     int head_dim, int max_block_len);
int splash_verify_attention_shared(const uint16_t* q, int num_q_tokens,
                                   const int8_t* k_pages, const int8_t* v_pages,
                                   const float* k_scales, const float* v_scales,
                                   const int32_t* page_table, int max_pages_per_seq,
                                   const int32_t* context_lens, const int32_t* block_lens,
                                   const int32_t* shared_lens, int num_seqs, int num_q_heads,
                                   int num_kv_heads, int head_dim, int page_size, int num_pages,
                                   int max_block_len, float sm_scale, uint16_t* out, float* lse,
                                   void* workspace, size_t workspace_bytes, int* device_status,
                                   struct CUstream_st* stream);
/*
 * splash_verify_attention_shared_profiled — splash_verify_attention_shared
 * with path and ctas_per_class as in splash_verify_attention_tuned, and the
 * two events of splash_verify_attention_profiled (either may be NULL).
 */
int splash_verify_attention_shared_profiled(
    const uint16_t* q, int num_q_tokens, const int8_t* k_pages, const int8_t* v_pages,
    const float* k_scales, const float* v_scales, const int32_t* page_table,
    int max_pages_per_seq, const int32_t* context_lens, const int32_t* block_lens,
    const int32_t* shared_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int page_size, int num_pages, int max_block_len, float sm_scale, uint16_t* out, float* lse,
    void* workspace, size_t workspace_bytes, int* device_status, struct CUstream_st* stream,
    int path, int ctas_per_class, struct CUevent_st* attn_begin, struct CUevent_st* attn_end);

/*
 * splash_verify_attention_fixed_scratch — splash_verify_attention without a
 * caller-provided workspace, for callers that cannot allocate device memory:
 * for example code that runs under a memory manager owning every device
 * allocation, a plugin whose host forbids allocation calls, or a serving
 * loop that cannot afford the implicit device synchronisation of cudaMalloc.
 * (The source pages describe nothing like it; it is a packaging of the same
 * operation.)
 *
 * The workspace is instead a fixed 64 MiB array (see
 * splash_verify_attention_fixed_scratch_bytes) that is part of this library's
 * device image: every GPU that loads the library holds it until the process
 * exits. Nothing is allocated or freed by the call; no allocating library
 * routine is used. The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress), so make that first call before any stream
 * capture. All calls on a device share the one array, which keeps the last
 * call's contents; the planner rewrites everything a call reads, so nothing
 * needs clearing between calls. Calls that can overlap on the same GPU (issued
 * on different streams, or from different host threads) race on the array and
 * must be serialised by the caller.
 *
 * Same arguments, results and errors as splash_verify_attention minus the
 * workspace, with one CTA per SM for each attention kernel. Returns
 * SPLASH_ERR_WORKSPACE_TOO_SMALL when the shape needs more scratch than the
 * fixed array holds (for D = 256 that is beyond about T*G = 105 rows per
 * sequence on a 152-SM GB300).
 */
size_t splash_verify_attention_fixed_scratch_bytes(void);
int splash_verify_attention_fixed_scratch(const uint16_t* q, int num_q_tokens,
                                          const int8_t* k_pages, const int8_t* v_pages,
                                          const float* k_scales, const float* v_scales,
                                          const int32_t* page_table, int max_pages_per_seq,
                                          const int32_t* context_lens, const int32_t* block_lens,
                                          int num_seqs, int num_q_heads, int num_kv_heads,
                                          int head_dim, int page_size, int num_pages,
                                          int max_block_len, float sm_scale, uint16_t* out,
                                          float* lse, int* device_status,
                                          struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPLASH_KV_H */
