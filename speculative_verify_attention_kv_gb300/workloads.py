"""Seeded synthetic inputs for the verify-attention path.

This module only draws random numbers and lays out sequences and pages. It
holds none of the method's arithmetic (no quantisation, no attention), so both
the CUDA path and the fp64 oracle can consume the same inputs without sharing
any computation.

Workloads (context scale of the Splash benchmark prompts, which are not
shipped; these seeded inputs stand in for them):

  0 ``tiny``          1 seq, 256 cached tokens, Hq/Hkv 8/2, D 128, T 4
  1 ``single_32k``    1 seq, 32768 cached tokens, Hq/Hkv 24/4, D 256, T 16
  2 ``shared_prefix`` 4 seqs sharing a 24576-token prefix (same physical
                      pages) + private 8192-token suffixes, 24/4, D 256, T 16
  3 ``batch16_32k``   16 seqs x 32768 cached tokens, 24/4, D 256, T 16,
                      1% of channels (3 per KV head) scaled x8 as outliers
  4 ``ragged64``      64 seqs, context log-uniform in [512, 131072],
                      T uniform in {1, 4, 8, 16}, 24/4, D 256

All use page size 16. K and V are fp32 N(0, 1); Q is fp32 N(0, 1) rounded to
bf16 (round to nearest even). The physical page ids are a seeded permutation
of the pool, which carries 5% slack pages that no sequence references (tests
fill them with poison).

Random streams (numpy ``default_rng`` with a list seed, so any (sequence,
head) can be regenerated on its own for sampled checks):

  [seed, 0]          structure: lengths, outlier channels, page permutation
  [seed, 1, b, h]    context K of sequence b, KV head h (private tokens)
  [seed, 2, b, h]    context V of sequence b, KV head h (private tokens)
  [seed, 5, h]       shared-prefix K of KV head h
  [seed, 6, h]       shared-prefix V of KV head h
  [seed, 3, b, h]    verify-block K then V of sequence b, KV head h
  [seed, 4, b]       Q of sequence b's verify block, all query heads
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

PAGE_SIZE = 16
SLACK_FRACTION = 0.05


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    index: int
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    num_seqs: int
    kind: str                   # "uniform" | "shared_prefix" | "ragged"
    context_len: int = 0        # uniform: cached tokens per sequence
    block_len: int = 0          # uniform / shared_prefix: verify block T
    prefix_len: int = 0         # shared_prefix: shared cached tokens
    suffix_len: int = 0         # shared_prefix: private cached tokens
    ragged_min: int = 0         # ragged: log-uniform context bounds
    ragged_max: int = 0
    ragged_blocks: tuple = ()   # ragged: T drawn uniformly from these
    outlier_scale: float = 1.0  # >1: 1% of channels per KV head scaled
    page_size: int = PAGE_SIZE

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def seed(self) -> int:
        return 1000 + self.index


SPECS = (
    WorkloadSpec(0, "tiny", 8, 2, 128, 1, "uniform", context_len=256, block_len=4),
    WorkloadSpec(1, "single_32k", 24, 4, 256, 1, "uniform", context_len=32768, block_len=16),
    WorkloadSpec(2, "shared_prefix", 24, 4, 256, 4, "shared_prefix", block_len=16,
                 prefix_len=24576, suffix_len=8192),
    WorkloadSpec(3, "batch16_32k", 24, 4, 256, 16, "uniform", context_len=32768, block_len=16,
                 outlier_scale=8.0),
    WorkloadSpec(4, "ragged64", 24, 4, 256, 64, "ragged", ragged_min=512, ragged_max=131072,
                 ragged_blocks=(1, 4, 8, 16)),
)
SPEC_BY_NAME = {s.name: s for s in SPECS}


def _normal(seed_key, shape) -> np.ndarray:
    return np.random.default_rng(seed_key).standard_normal(shape, dtype=np.float32)


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def f32_from_bf16_bits(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


class Workload:
    """One seeded instance of a workload spec (lengths, pages, tensors)."""

    def __init__(self, spec: WorkloadSpec, seed: int | None = None, *,
                 context_lens=None, block_lens=None, shared_prefix_len: int | None = None):
        self.spec = spec
        self.seed = spec.seed if seed is None else seed
        s = spec
        P = s.page_size
        rng = np.random.default_rng([self.seed, 0])
        # draw order on the structure stream: lengths -> outlier channels ->
        # physical page permutation
        self.prefix_len = 0
        if context_lens is not None:
            ctx = np.asarray(context_lens, dtype=np.int64)
            T = np.asarray(block_lens, dtype=np.int64)
            self.prefix_len = int(shared_prefix_len or 0)
        elif s.kind == "uniform":
            ctx = np.full(s.num_seqs, s.context_len, dtype=np.int64)
            T = np.full(s.num_seqs, s.block_len, dtype=np.int64)
        elif s.kind == "shared_prefix":
            ctx = np.full(s.num_seqs, s.prefix_len + s.suffix_len, dtype=np.int64)
            T = np.full(s.num_seqs, s.block_len, dtype=np.int64)
            self.prefix_len = s.prefix_len
        elif s.kind == "ragged":
            lo, hi = math.log(s.ragged_min), math.log(s.ragged_max)
            ctx = np.floor(np.exp(rng.uniform(lo, hi, size=s.num_seqs))).astype(np.int64)
            T = np.asarray(s.ragged_blocks, dtype=np.int64)[
                rng.integers(0, len(s.ragged_blocks), size=s.num_seqs)]
        else:
            raise ValueError(s.kind)
        n_out = math.ceil(0.01 * s.head_dim)
        outl = np.stack([rng.choice(s.head_dim, size=n_out, replace=False)
                         for _ in range(s.num_kv_heads)]).astype(np.int64)
        self.outlier_channels = outl if s.outlier_scale != 1.0 else None
        self.context_lens = ctx.astype(np.int32)
        self.block_lens = T.astype(np.int32)
        self.num_seqs = len(ctx)
        assert self.prefix_len % P == 0
        assert np.all(ctx >= self.prefix_len)

        # logical pages: a sequence needs ceil((ctx + T) / P) pages; the first
        # prefix_len / P are shared by every sequence when a prefix is shared.
        n_shared = self.prefix_len // P
        need = (ctx + T + P - 1) // P
        n_private = need - n_shared
        n_used = n_shared + int(n_private.sum())
        self.num_pages = n_used + max(1, int(math.ceil(SLACK_FRACTION * n_used)))
        phys = rng.permutation(self.num_pages).astype(np.int32)
        self.max_pages_per_seq = int(need.max()) if len(need) else 1
        table = np.full((self.num_seqs, self.max_pages_per_seq), -1, dtype=np.int32)
        shared_ids = phys[:n_shared]
        cur = n_shared
        for b in range(self.num_seqs):
            table[b, :n_shared] = shared_ids
            k = int(n_private[b])
            table[b, n_shared:n_shared + k] = phys[cur:cur + k]
            cur += k
        self.page_table = table
        self.used_pages = np.sort(phys[:n_used])
        self.slack_pages = np.sort(phys[n_used:])
        self.q_offsets = np.concatenate([[0], np.cumsum(T)]).astype(np.int64)
        self.num_q_tokens = int(T.sum())
        self.sm_scale = np.float32(1.0 / math.sqrt(s.head_dim))
        # key of each sequence's random streams ([seed, 1, b, h] ...): its own
        # index, or its index in the parent workload for a subset
        self.seq_ids = np.arange(self.num_seqs)

    def subset(self, seqs) -> "Workload":
        """The listed sequences as a workload of their own: the same lengths,
        outlier channels and data (every sequence keeps its random streams) on
        a compact page pool (a shared prefix stays shared)."""
        seqs = np.asarray(seqs, dtype=np.int64)
        sub = Workload(self.spec, self.seed, context_lens=self.context_lens[seqs],
                       block_lens=self.block_lens[seqs], shared_prefix_len=self.prefix_len)
        sub.outlier_channels = self.outlier_channels
        sub.seq_ids = self.seq_ids[seqs]
        return sub

    def shared_lens(self) -> np.ndarray:
        """Keys each sequence shares (same pages) with the one before it:
        int32 [num_seqs]; the shared prefix for every sequence but the first."""
        out = np.zeros(self.num_seqs, dtype=np.int32)
        if self.prefix_len and self.num_seqs > 1:
            out[1:] = self.prefix_len
        return out

    # ---- tensors --------------------------------------------------------
    def _apply_outliers(self, x: np.ndarray, h: int) -> np.ndarray:
        if self.outlier_channels is not None:
            x[..., self.outlier_channels[h]] *= np.float32(self.spec.outlier_scale)
        return x

    def prefix_kv(self, h: int):
        """Shared-prefix K, V of KV head h: fp32 [prefix_len, D] each."""
        D = self.spec.head_dim
        k = _normal([self.seed, 5, h], (self.prefix_len, D))
        v = _normal([self.seed, 6, h], (self.prefix_len, D))
        return self._apply_outliers(k, h), self._apply_outliers(v, h)

    def private_context_kv(self, b: int, h: int):
        """Context K, V of sequence b, KV head h past the shared prefix:
        fp32 [context_len - prefix_len, D] each."""
        D = self.spec.head_dim
        n = int(self.context_lens[b]) - self.prefix_len
        sid = int(self.seq_ids[b])
        k = _normal([self.seed, 1, sid, h], (n, D))
        v = _normal([self.seed, 2, sid, h], (n, D))
        return self._apply_outliers(k, h), self._apply_outliers(v, h)

    def context_kv(self, b: int, h: int):
        """All cached K, V of sequence b, KV head h: fp32 [context_len, D]."""
        k, v = self.private_context_kv(b, h)
        if self.prefix_len:
            pk, pv = self.prefix_kv(h)
            k, v = np.concatenate([pk, k]), np.concatenate([pv, v])
        return k, v

    def block_kv_seq(self, b: int):
        """Verify-block K, V of sequence b: fp32 [T_b, Hkv, D] each."""
        s = self.spec
        T = int(self.block_lens[b])
        ks, vs = [], []
        for h in range(s.num_kv_heads):
            rng = np.random.default_rng([self.seed, 3, int(self.seq_ids[b]), h])
            k = rng.standard_normal((T, s.head_dim), dtype=np.float32)
            v = rng.standard_normal((T, s.head_dim), dtype=np.float32)
            ks.append(self._apply_outliers(k, h))
            vs.append(self._apply_outliers(v, h))
        return np.stack(ks, axis=1), np.stack(vs, axis=1)

    def block_kv(self):
        """Verify-block K, V of all sequences, packed by sequence:
        fp32 [sum(T), Hkv, D] each."""
        parts = [self.block_kv_seq(b) for b in range(self.num_seqs)]
        s = self.spec
        if not parts:
            z = np.zeros((0, s.num_kv_heads, s.head_dim), np.float32)
            return z, z.copy()
        return (np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts]))

    def q_bits_seq(self, b: int) -> np.ndarray:
        s = self.spec
        T = int(self.block_lens[b])
        q = _normal([self.seed, 4, int(self.seq_ids[b])], (T, s.num_q_heads, s.head_dim))
        return bf16_bits_from_f32(q)

    def q_bits(self) -> np.ndarray:
        """Q as bf16 bit patterns, packed by sequence: uint16 [sum(T), Hq, D]."""
        s = self.spec
        parts = [self.q_bits_seq(b) for b in range(self.num_seqs)]
        if not parts:
            return np.zeros((0, s.num_q_heads, s.head_dim), np.uint16)
        return np.concatenate(parts)

    # ---- byte model (unique used KV slots + scales, Q, O) ---------------
    def unique_kv_slots(self) -> int:
        """Distinct (page, slot) positions an attention pass reads."""
        P = self.spec.page_size
        L = self.context_lens.astype(np.int64) + self.block_lens
        if self.prefix_len:
            return int(self.prefix_len + (L - self.prefix_len).sum())
        del P
        return int(L.sum())

    def logical_kv_slots(self) -> int:
        return int((self.context_lens.astype(np.int64) + self.block_lens).sum())

    def algorithmic_bytes(self, unique: bool = True) -> int:
        s = self.spec
        slots = self.unique_kv_slots() if unique else self.logical_kv_slots()
        kv = slots * s.num_kv_heads * (2 * s.head_dim + 8)
        qo = 2 * self.num_q_tokens * s.num_q_heads * s.head_dim * 2
        return kv + qo


def partition_by_kv_bytes(W: Workload, parts: int):
    """Split W's sequences into `parts` groups of nearly equal KV bytes (the
    work of a sequence is proportional to its ctx + T keys): largest first,
    each to the group with the least so far (lowest index on ties). Returns
    sorted sequence lists, one per group."""
    cost = W.context_lens.astype(np.int64) + W.block_lens
    order = sorted(range(W.num_seqs), key=lambda b: (-int(cost[b]), b))
    load = [0] * parts
    groups = [[] for _ in range(parts)]
    for b in order:
        r = min(range(parts), key=lambda i: (load[i], i))
        groups[r].append(b)
        load[r] += int(cost[b])
    return [sorted(g) for g in groups]


def make(name_or_index, seed: int | None = None) -> Workload:
    spec = SPECS[name_or_index] if isinstance(name_or_index, int) else SPEC_BY_NAME[name_or_index]
    return Workload(spec, seed)


def custom(num_q_heads, num_kv_heads, head_dim, context_lens, block_lens, seed=7,
           shared_prefix_len=0, outlier_scale=1.0) -> Workload:
    """A workload with explicit lengths (edge cases in tests)."""
    spec = WorkloadSpec(99, "custom", num_q_heads, num_kv_heads, head_dim, len(context_lens),
                        "custom", outlier_scale=outlier_scale)
    return Workload(spec, seed, context_lens=context_lens, block_lens=block_lens,
                    shared_prefix_len=shared_prefix_len)
