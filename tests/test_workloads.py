"""The seeded input recipe: shapes, lengths, page layout and byte counts that
the benchmark and the parity tests rely on (CPU only)."""
from __future__ import annotations

import math

import numpy as np
import pytest

from speculative_verify_attention_kv_gb300 import workloads as wl


def test_batch16_32k_shape_and_bytes():
    W = wl.make("batch16_32k")
    s = W.spec
    assert (W.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_dim) == (16, 24, 4, 256)
    assert np.all(W.context_lens == 32768) and np.all(W.block_lens == 16)
    # unique (page, slot)s x Hkv x (2D + 8) + Q and O in bf16
    kv = 16 * (32768 + 16) * 4 * (2 * 256 + 8)
    qo = 2 * (16 * 16) * 24 * 256 * 2
    assert W.algorithmic_bytes() == kv + qo == 1_097_342_976


def test_page_tables_are_private_except_the_shared_prefix():
    for name in ("single_32k", "batch16_32k", "ragged64", "shared_prefix"):
        W = wl.make(name)
        n_shared = W.prefix_len // 16
        need = (W.context_lens.astype(np.int64) + W.block_lens + 15) // 16
        seen = set()
        for b in range(W.num_seqs):
            row = W.page_table[b]
            assert np.all(row[:need[b]] >= 0) and np.all(row[need[b]:] == -1)
            private = row[n_shared:need[b]].tolist()
            assert not (seen & set(private)), name
            seen |= set(private)
        assert np.all(W.page_table[:, :n_shared] == W.page_table[0, :n_shared])
        used = set(W.used_pages.tolist())
        assert set(W.page_table[W.page_table >= 0].tolist()) == used
        assert not used & set(W.slack_pages.tolist())
        assert len(W.slack_pages) == max(1, math.ceil(0.05 * len(used)))


def test_shared_prefix_layout():
    W = wl.make("shared_prefix")
    assert W.prefix_len == 24576 and W.num_seqs == 4
    assert np.all(W.context_lens == 24576 + 8192)
    n_shared = 24576 // 16
    # every sequence's first 1536 pages are the same physical pages
    assert len(set(map(tuple, W.page_table[:, :n_shared].tolist()))) == 1
    assert W.algorithmic_bytes(unique=True) < W.algorithmic_bytes(unique=False)


def test_ragged_lengths():
    W = wl.make("ragged64")
    assert W.num_seqs == 64
    assert np.all(W.context_lens >= 512) and np.all(W.context_lens < 131072)
    assert set(np.unique(W.block_lens).tolist()) <= {1, 4, 8, 16}


@pytest.mark.parametrize("name", ["tiny", "single_32k"])
def test_q_is_bf16_and_seeded(name):
    W1, W2 = wl.make(name), wl.make(name)
    q1, q2 = W1.q_bits(), W2.q_bits()
    assert q1.dtype == np.uint16 and np.array_equal(q1, q2)
    x = wl.f32_from_bf16_bits(q1)
    assert np.array_equal(wl.bf16_bits_from_f32(x), q1)     # exactly representable
    assert not np.array_equal(q1, wl.make(name, seed=W1.seed + 1).q_bits())
