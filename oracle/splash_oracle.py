"""fp64 CPU oracle for verify attention over an int8 paged KV cache.

TEST INFRASTRUCTURE ONLY. Only the test suite, the package's ``smoke()`` check
and the benchmark's CPU-baseline leg may import this module. The product path
(the CUDA library and its Python binding) never imports, calls or falls back to
it, and this module imports nothing from the product package.

What it computes, and where that is defined
-------------------------------------------
Source pages: "Splash: 범용 엔진 대신 모델마다 커널과 초안 모델을 새로 만드는 Apple
Silicon 추론 엔진" (discuss.pytorch.kr). Section "배치 스케줄링과 시작 시점에
확정되는 메모리 예산": attention state lives in a paged KV cache indexed by
prefix, and requests that share a prefix reuse its pages. Section "옵션이 아니라
기본 경로인 DFlash 2 추측 디코딩": the target model verifies a drafted block of
tokens in one forward pass; speculation runs inside the batch, each request
advancing by its own accepted count. Section "형상에 맞춰 자동으로 생성하는
Metal 커널": the decode kernel reads the 8-bit KV cache directly and reuses it
across query heads and verify tokens. The Chinese article on bnskd.com
("Splash：把推理引擎「围着模型造」…", section "技术内核：三件事撑起这个速度")
states the same three facts.

The pages give no quantisation scheme, mask, or precision. The readings used
here (the same ones the CUDA path implements):

* quantise_rows: per (token, KV head) row x of D fp32 values,
  a = max|x|, s = fl32(a / 127); s == 0 gives all-zero codes; otherwise
  c = clamp(round_half_even(fl32(x / s)), -127, 127). fl32 of a quotient is
  taken as the fp64 quotient rounded to fp32, which equals the correctly
  rounded fp32 quotient (53 >= 2*24 + 2).
* kv_append: a block of T_b new tokens goes to logical positions
  context_len .. context_len + T_b - 1 of its sequence; logical position j
  lives in physical page page_table[b][j // P], slot j % P.
* attention: verify token t of sequence b (query head hq, KV head
  hq // G) sees keys 0 .. context_len + t inclusive, i.e. the cache plus the
  block's own tokens 0..t, all read back as int8 codes times fp32 scales.
  scores = sm_scale * q . k_hat; O = softmax(scores) @ v_hat; LSE = natural
  log of sum(exp(scores)), sm_scale included.
* attention_partial / lse_combine: the split-KV form of the same quantity,
  partial (o_i, lse_i) over a key range, merged by log-sum-exp weights.
* sliding window (the draft's windowed attention, section "옵션이 아니라 기본
  경로인 DFlash 2 추측 디코딩"): with window W > 0, verify token t sees only the W
  most recent keys up to its own position, ctx + t - W < j <= ctx + t;
  W = 0 means no lower bound.
* accept_commit: each request advances by the tokens it accepted (same
  section of the discuss.pytorch.kr article). Reading: block x_0..x_{T-1}
  (x_0 = the target's previous output, x_1.. = drafts), target choices
  y_0..y_{T-1}; draft x_{i+1} is accepted while it equals y_i; with a accepted
  drafts the context grows by a + 1 and y_a is the next token.

Everything is fp64 except the quantiser, whose fp32 roundings are part of the
definition. Library primitives used as steps: numpy matmul, exp, log.
"""
from __future__ import annotations

import numpy as np

QMAX = 127


# ---------------------------------------------------------------------------
# quantiser
# ---------------------------------------------------------------------------
def _round_half_even(x: np.ndarray) -> np.ndarray:
    return np.rint(x)


def _fl32_div(a: np.ndarray, b) -> np.ndarray:
    """fp32 quotient, correctly rounded, via the exact-enough fp64 quotient."""
    return (np.asarray(a, np.float64) / np.asarray(b, np.float64)).astype(np.float32)


def quantise_rows(x: np.ndarray):
    """Symmetric absmax/127 int8 quantisation of each row of ``x``.

    x: fp32 [..., D]. Returns (codes int8 [..., D], scales fp32 [...]).
    """
    x = np.asarray(x, dtype=np.float32)
    a = np.max(np.abs(x), axis=-1)                     # exact in fp32
    s = _fl32_div(a, QMAX)                             # fl32(a / 127)
    safe = np.where(s == 0, np.float32(1), s)
    q = _fl32_div(x, safe[..., None])                  # fl32(x / s)
    c = np.clip(_round_half_even(q.astype(np.float64)), -QMAX, QMAX)
    c = np.where((s == 0)[..., None], 0, c)
    return c.astype(np.int8), s.astype(np.float32)


def dequantise(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """k_hat = code * scale, in fp64 (exact)."""
    return codes.astype(np.float64) * scales.astype(np.float64)[..., None]


# ---------------------------------------------------------------------------
# paged pool (canonical layout: codes [num_pages, Hkv, P, D], scales [num_pages, Hkv, P])
# ---------------------------------------------------------------------------
class PagedPool:
    def __init__(self, num_pages: int, num_kv_heads: int, page_size: int, head_dim: int):
        self.P = page_size
        self.k_codes = np.zeros((num_pages, num_kv_heads, page_size, head_dim), np.int8)
        self.v_codes = np.zeros_like(self.k_codes)
        self.k_scales = np.zeros((num_pages, num_kv_heads, page_size), np.float32)
        self.v_scales = np.zeros_like(self.k_scales)


def _slot(page_table_row: np.ndarray, j: int, P: int):
    return int(page_table_row[j // P]), j % P


def kv_append(pool: PagedPool, k_new: np.ndarray, v_new: np.ndarray, page_table: np.ndarray,
              context_lens: np.ndarray, block_lens: np.ndarray) -> None:
    """Quantise and write each sequence's new tokens at positions ctx..ctx+T-1.

    k_new, v_new: fp32 [sum(block_lens), Hkv, D], packed by sequence.
    """
    P = pool.P
    kc, ks = quantise_rows(k_new)
    vc, vs = quantise_rows(v_new)
    row = 0
    for b in range(len(block_lens)):
        for t in range(int(block_lens[b])):
            page, slot = _slot(page_table[b], int(context_lens[b]) + t, P)
            pool.k_codes[page, :, slot, :] = kc[row]
            pool.k_scales[page, :, slot] = ks[row]
            pool.v_codes[page, :, slot, :] = vc[row]
            pool.v_scales[page, :, slot] = vs[row]
            row += 1


def gather_keys(pool: PagedPool, page_table_row: np.ndarray, h: int, n: int):
    """Dequantised K, V of logical positions 0..n-1 of one sequence and KV head:
    fp64 [n, D] each."""
    P = pool.P
    j = np.arange(n)
    pages = page_table_row[j // P].astype(np.int64)
    slots = j % P
    k = dequantise(pool.k_codes[pages, h, slots, :], pool.k_scales[pages, h, slots])
    v = dequantise(pool.v_codes[pages, h, slots, :], pool.v_scales[pages, h, slots])
    return k, v


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------
def _visible(j: np.ndarray, ctx: int, t: int, window: int = 0) -> np.ndarray:
    """Key j is visible to verify token t iff j <= ctx + t (and, with a
    window W > 0, j > ctx + t - W)."""
    vis = j <= ctx + t
    if window > 0:
        vis = vis & (j > ctx + t - window)
    return vis


def _softmax_rows(scores: np.ndarray, visible: np.ndarray):
    """Masked softmax over the last axis; returns (p, lse)."""
    s = np.where(visible, scores, -np.inf)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.where(visible, np.exp(s - m), 0.0)
    z = np.sum(e, axis=-1, keepdims=True)
    return e / z, (m + np.log(z))[..., 0]


def attention_seq_head(q: np.ndarray, k: np.ndarray, v: np.ndarray, ctx: int, sm_scale: float,
                       window: int = 0):
    """Verify attention of one sequence and one KV head.

    q: fp64 [T, G, D] (bf16 values); k, v: fp64 [ctx + T, D] (dequantised).
    Returns O fp64 [T, G, D], LSE fp64 [T, G].
    """
    T, G, D = q.shape
    n = k.shape[0]
    scores = float(np.float32(sm_scale)) * (q.reshape(T * G, D) @ k.T)   # [T*G, n]
    j = np.arange(n)
    vis = np.stack([_visible(j, ctx, t, window) for t in range(T) for _ in range(G)])
    p, lse = _softmax_rows(scores, vis)
    return (p @ v).reshape(T, G, D), lse.reshape(T, G)


def attention(q: np.ndarray, pool: PagedPool, page_table: np.ndarray, context_lens: np.ndarray,
              block_lens: np.ndarray, num_kv_heads: int, sm_scale: float, seqs=None,
              window: int = 0):
    """Verify attention for every (sequence, KV head) (or the listed sequences).

    q: float [sum(block_lens), Hq, D] holding bf16 values. Returns O fp64
    [sum(T), Hq, D] and LSE fp64 [sum(T), Hq]; rows of unlisted sequences are NaN.
    """
    q = np.asarray(q, np.float64)
    n_tok, Hq, D = q.shape
    G = Hq // num_kv_heads
    out = np.full((n_tok, Hq, D), np.nan)
    lse = np.full((n_tok, Hq), np.nan)
    offs = np.concatenate([[0], np.cumsum(block_lens)]).astype(np.int64)
    for b in (range(len(block_lens)) if seqs is None else seqs):
        T, ctx = int(block_lens[b]), int(context_lens[b])
        if T == 0:
            continue
        r0 = offs[b]
        for h in range(num_kv_heads):
            k, v = gather_keys(pool, page_table[b], h, ctx + T)
            qs = q[r0:r0 + T, h * G:(h + 1) * G, :]
            o, l = attention_seq_head(qs, k, v, ctx, sm_scale, window)
            out[r0:r0 + T, h * G:(h + 1) * G, :] = o
            lse[r0:r0 + T, h * G:(h + 1) * G] = l
    return out, lse


def attention_partial(q: np.ndarray, k: np.ndarray, v: np.ndarray, ctx: int, sm_scale: float,
                      k0: int, k1: int, window: int = 0):
    """Split-KV partial over keys [k0, k1) of one sequence and KV head.

    Returns o_i fp64 [T, G, D] (normalised by its own sum) and lse_i [T, G]
    (-inf, with o_i = 0, for a row that sees no key in the range).
    """
    T, G, D = q.shape
    scores = float(np.float32(sm_scale)) * (q.reshape(T * G, D) @ k[k0:k1].T)
    j = np.arange(k0, k1)
    vis = np.stack([_visible(j, ctx, t, window) for t in range(T) for _ in range(G)])
    o = np.zeros((T * G, D))
    lse = np.full(T * G, -np.inf)
    any_vis = vis.any(axis=1)
    if any_vis.any():
        p, l = _softmax_rows(scores[any_vis], vis[any_vis])
        o[any_vis] = p @ v[k0:k1]
        lse[any_vis] = l
    return o.reshape(T, G, D), lse.reshape(T, G)


def lse_combine(partials):
    """Merge split partials [(o_i, lse_i), ...]: lse = log sum exp(lse_i),
    O = sum exp(lse_i - lse) o_i; splits with lse_i = -inf contribute nothing."""
    lses = np.stack([l for _, l in partials])              # [S, ...]
    m = np.max(lses, axis=0)
    w = np.exp(lses - m)
    lse = m + np.log(np.sum(w, axis=0))
    o = sum(np.exp(l - lse)[..., None] * oi for oi, l in partials)
    return o, lse


# ---------------------------------------------------------------------------
# accept / commit
# ---------------------------------------------------------------------------
def accept_commit(block_tokens, target_tokens, block_lens, context_lens):
    """Returns (accepted, new context_lens, next_tokens), one entry per sequence."""
    accepted, new_ctx, nxt = [], [], []
    off = 0
    for b, T in enumerate(block_lens):
        T = int(T)
        x = list(block_tokens[off:off + T])
        y = list(target_tokens[off:off + T])
        off += T
        if T == 0:
            accepted.append(0)
            new_ctx.append(int(context_lens[b]))
            nxt.append(-1)
            continue
        a = 0
        while a + 1 < T and x[a + 1] == y[a]:
            a += 1
        accepted.append(a)
        new_ctx.append(int(context_lens[b]) + a + 1)
        nxt.append(int(y[a]))
    return (np.array(accepted, np.int32), np.array(new_ctx, np.int32), np.array(nxt, np.int32))
