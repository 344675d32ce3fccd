"""Helpers shared by the tests: fill an oracle pool from a seeded workload,
exact-rational reference arithmetic for the quantiser pins."""
from __future__ import annotations

import math
from fractions import Fraction as F

import numpy as np

from oracle import splash_oracle as O
from speculative_verify_attention_kv_gb300 import workloads as wl


def seq_context_tokens(W: wl.Workload, b: int, start: int = 0):
    """Cached K, V of sequence b from logical position ``start``: fp32
    [ctx - start, Hkv, D] each (all KV heads stacked)."""
    ks, vs = [], []
    for h in range(W.spec.num_kv_heads):
        k, v = W.context_kv(b, h)
        ks.append(k[start:])
        vs.append(v[start:])
    return np.stack(ks, axis=1), np.stack(vs, axis=1)


def oracle_pool(W: wl.Workload, seqs=None, with_block: bool = True) -> O.PagedPool:
    """Oracle pool holding the cache (and the appended verify block) of ``seqs``."""
    s = W.spec
    pool = O.PagedPool(W.num_pages, s.num_kv_heads, s.page_size, s.head_dim)
    seqs = range(W.num_seqs) if seqs is None else seqs
    for b in seqs:
        k, v = seq_context_tokens(W, b)
        O.kv_append(pool, k, v, W.page_table[b:b + 1], np.array([0]), np.array([k.shape[0]]))
        if with_block:
            bk, bv = W.block_kv_seq(b)
            O.kv_append(pool, bk, bv, W.page_table[b:b + 1], W.context_lens[b:b + 1],
                        W.block_lens[b:b + 1])
    return pool


def q_values(W: wl.Workload) -> np.ndarray:
    return wl.f32_from_bf16_bits(W.q_bits()).astype(np.float64)


# ---- exact rational arithmetic (independent of numpy's float semantics) ----
def round_to_f32(fr: F) -> F:
    """Exact value of the fp32 nearest to ``fr`` (ties to even; normal and
    subnormal range; no overflow handling)."""
    if fr == 0:
        return F(0)
    sign = -1 if fr < 0 else 1
    fr = abs(fr)
    e = fr.numerator.bit_length() - fr.denominator.bit_length()
    while F(2) ** e > fr:
        e -= 1
    while F(2) ** (e + 1) <= fr:
        e += 1
    quantum_exp = max(e, -126) - 23
    scaled = fr / F(2) ** quantum_exp
    n = math.floor(scaled)
    rem = scaled - n
    if rem > F(1, 2) or (rem == F(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * F(2) ** quantum_exp


def round_half_even_exact(fr: F) -> int:
    n = math.floor(fr)
    rem = fr - n
    if rem > F(1, 2) or (rem == F(1, 2) and n % 2 == 1):
        n += 1
    return n


def quantise_row_exact(x):
    """The quantiser's definition evaluated with exact rationals."""
    xs = [F(float(v)) for v in np.asarray(x, np.float32)]
    a = max(abs(v) for v in xs)
    s = round_to_f32(a / 127)
    if s == 0:
        return [0] * len(xs), 0.0
    codes = [max(-127, min(127, round_half_even_exact(round_to_f32(v / s)))) for v in xs]
    return codes, float(s)


# ---- the prefix-group rule of splash_verify_attention_shared ---------------
GROUP_TILE, GROUP_MAX_ROWS = 64, 128


def expected_group_plan(ctx, T, shared_lens, G, Hkv):
    """(items, tensor-core tiles of all units) under the grouping rule the
    header states: b links to b - 1 when both have a block and
    min(shared_lens[b], ctx[b], ctx[b-1]) >= 64; a maximal linked run is a
    group whose prefix is its smallest link (cut to every context) rounded down
    to 64 keys; it is stacked when ceil(sum T*G / 128) < its size, as that many
    row blocks over the prefix, each member then reading its keys after it."""
    B = len(ctx)
    link = [0] * B
    for b in range(1, B):
        if T[b] > 0 and T[b - 1] > 0:
            s = min(shared_lens[b], ctx[b], ctx[b - 1])
            link[b] = s if s >= GROUP_TILE else 0
    pg_of = [0] * B
    blocks = []                                   # prefix keys of each row block
    b = 0
    while b < B:
        e = b + 1
        while e < B and link[e] > 0:
            e += 1
        if T[b] > 0 and e - b > 1:
            pg = min([ctx[b]] + link[b + 1:e]) // GROUP_TILE * GROUP_TILE
            rows = sum(T[i] * G for i in range(b, e))
            nblk = -(-rows // GROUP_MAX_ROWS)
            if pg >= GROUP_TILE and nblk < e - b:
                for i in range(b, e):
                    pg_of[i] = pg
                blocks += [pg] * nblk
        b = e
    tiles = 0
    for i in range(B):
        if T[i] > 0:
            tiles += -(-(ctx[i] + T[i]) // GROUP_TILE) - pg_of[i] // GROUP_TILE
    tiles += sum(pg // GROUP_TILE for pg in blocks)
    return B + len(blocks), tiles * Hkv
