"""Pins of the fp64 oracle against what the definition and mathematics fix.

None of these compares the oracle with itself: the references are hand-derived
values, exact rational arithmetic, torch's float64 scaled-dot-product attention
on truncated key sets (no mask formula), closed forms and invariants. The last
group plants plausible mistakes in the oracle and checks that a pin catches
each one.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction as F

import numpy as np
import pytest
import torch

from oracle import splash_oracle as O
from speculative_verify_attention_kv_gb300 import workloads as wl

from common import oracle_pool, q_values, quantise_row_exact, round_to_f32, round_half_even_exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# quantiser
# ---------------------------------------------------------------------------
def test_quantiser_closed_form_cases():
    with open(os.path.join(GOLDEN, "quantiser_closed_form.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        x = np.array([c["x"]], np.float32)
        codes, s = O.quantise_rows(x)
        assert codes[0].tolist() == c["codes"], c["name"]
        if c["scale"] is not None:
            assert float(s[0]) == c["scale"], c["name"]


def _exact_rows(x):
    codes, scales = zip(*(quantise_row_exact(r) for r in x))
    return np.array(codes), np.array(scales, np.float64)


def test_quantiser_matches_exact_rationals_random():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((40, 64)).astype(np.float32)
    x[5:10, 3] *= 8                     # outlier channel
    x[10] = 0
    x[11, :] = 0
    x[11, 7] = -2.0 ** -140             # subnormal scale
    x[12, :] = 0
    x[12, :4] = np.float32(190 * 2.0 ** -149)   # scale rounds to 2^-149: clamp to 127
    x[12, 4] = np.float32(-64 * 2.0 ** -149)
    x[13] = np.float32(1e-30) * x[13]
    codes, scales = O.quantise_rows(x)
    ec, es = _exact_rows(x)
    assert np.array_equal(codes.astype(np.int64), ec)
    assert np.array_equal(scales.astype(np.float64), es)
    assert codes[12, 0] == 127 and scales[12] == np.float32(2.0 ** -149)


def _near_ties(n, seed=5):
    """Rows whose codes differ between x / fl32(a/127) and x * fl32(127/a)."""
    rng = np.random.default_rng(seed)
    rows = []
    while len(rows) < n:
        a = np.float32(rng.uniform(0.5, 4.0))
        k = int(rng.integers(-126, 127))
        s = round_to_f32(F(float(a)) / 127)
        x = np.float32(float((k + F(1, 2)) * s))
        div = round_half_even_exact(round_to_f32(F(float(x)) / s))
        mul = round_half_even_exact(round_to_f32(F(float(x)) * round_to_f32(F(127) / F(float(a)))))
        if div != mul:
            rows.append(np.array([a, x, 0, 0], np.float32))
    return np.stack(rows)


def test_quantiser_is_the_divide_form():
    x = _near_ties(12)
    codes, scales = O.quantise_rows(x)
    ec, es = _exact_rows(x)
    assert np.array_equal(codes.astype(np.int64), ec)
    assert np.array_equal(scales.astype(np.float64), es)


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------
def _dense_kv(pool, table_row, h, n):
    """Dequantised keys by direct indexing (torch, float64)."""
    P = pool.P
    out_k, out_v = [], []
    for j in range(n):
        p, sl = int(table_row[j // P]), j % P
        out_k.append(torch.tensor(pool.k_codes[p, h, sl], dtype=torch.float64) * float(pool.k_scales[p, h, sl]))
        out_v.append(torch.tensor(pool.v_codes[p, h, sl], dtype=torch.float64) * float(pool.v_scales[p, h, sl]))
    return torch.stack(out_k), torch.stack(out_v)


def _sdpa_truncated(W, pool, q):
    """Row (t, hq) = unmasked attention over keys 0..ctx+t (torch float64)."""
    s = W.spec
    G = s.group
    o = np.zeros(q.shape)
    lse = np.zeros(q.shape[:2])
    sm = float(W.sm_scale)
    for b in range(W.num_seqs):
        ctx, T = int(W.context_lens[b]), int(W.block_lens[b])
        for h in range(s.num_kv_heads):
            K, V = _dense_kv(pool, W.page_table[b], h, ctx + T)
            for t in range(T):
                row = int(W.q_offsets[b]) + t
                qq = torch.tensor(q[row, h * G:(h + 1) * G], dtype=torch.float64)  # [G, D]
                n = ctx + t + 1
                out = torch.nn.functional.scaled_dot_product_attention(
                    qq[None], K[None, :n], V[None, :n], scale=sm)[0]
                o[row, h * G:(h + 1) * G] = out.numpy()
                lse[row, h * G:(h + 1) * G] = torch.logsumexp(sm * qq @ K[:n].T, dim=-1).numpy()
    return o, lse


def _run_oracle(W, pool):
    q = q_values(W)
    return q, O.attention(q, pool, W.page_table, W.context_lens, W.block_lens,
                          W.spec.num_kv_heads, float(W.sm_scale))


@pytest.mark.parametrize("ctx,T,hq,hkv,D", [
    ([37], [4], 8, 2, 32), ([0, 5, 16], [3, 1, 2], 6, 3, 16), ([31, 48], [16, 5], 4, 1, 8),
])
def test_attention_matches_sdpa_on_truncated_keys(ctx, T, hq, hkv, D):
    W = wl.custom(hq, hkv, D, ctx, T, seed=3)
    pool = oracle_pool(W)
    q, (o, lse) = _run_oracle(W, pool)
    ro, rl = _sdpa_truncated(W, pool, q)
    assert np.max(np.abs(o - ro)) < 1e-12
    assert np.max(np.abs(lse - rl)) < 1e-12


def _sdpa_window(W, pool, q, window):
    """Row (t, hq) = unmasked attention over keys max(0, ctx+t-W+1) .. ctx+t."""
    s = W.spec
    G = s.group
    o = np.zeros(q.shape)
    lse = np.zeros(q.shape[:2])
    sm = float(W.sm_scale)
    for b in range(W.num_seqs):
        ctx, T = int(W.context_lens[b]), int(W.block_lens[b])
        for h in range(s.num_kv_heads):
            K, V = _dense_kv(pool, W.page_table[b], h, ctx + T)
            for t in range(T):
                row = int(W.q_offsets[b]) + t
                qq = torch.tensor(q[row, h * G:(h + 1) * G], dtype=torch.float64)
                hi = ctx + t + 1
                lo = max(0, hi - window)
                out = torch.nn.functional.scaled_dot_product_attention(
                    qq[None], K[None, lo:hi], V[None, lo:hi], scale=sm)[0]
                o[row, h * G:(h + 1) * G] = out.numpy()
                lse[row, h * G:(h + 1) * G] = torch.logsumexp(sm * qq @ K[lo:hi].T, dim=-1).numpy()
    return o, lse


@pytest.mark.parametrize("window", [1, 2, 5, 17, 40, 1000])
def test_window_matches_sdpa_on_window_keys(window):
    W = wl.custom(8, 2, 16, [37, 0, 20], [4, 3, 16], seed=5)
    pool = oracle_pool(W)
    q = q_values(W)
    o, lse = O.attention(q, pool, W.page_table, W.context_lens, W.block_lens,
                         W.spec.num_kv_heads, float(W.sm_scale), window=window)
    ro, rl = _sdpa_window(W, pool, q, window)
    assert np.max(np.abs(o - ro)) < 1e-12 and np.max(np.abs(lse - rl)) < 1e-12


def test_window_one_is_the_diagonal_key():
    W = wl.custom(4, 2, 16, [9], [3], seed=6)
    pool = oracle_pool(W)
    q = q_values(W)
    o, lse = O.attention(q, pool, W.page_table, W.context_lens, W.block_lens, 2,
                         float(W.sm_scale), window=1)
    for t in range(3):
        j = 9 + t
        p, sl = int(W.page_table[0, j // 16]), j % 16
        for hq in range(4):
            h = hq // 2
            k = pool.k_codes[p, h, sl].astype(np.float64) * float(pool.k_scales[p, h, sl])
            v = pool.v_codes[p, h, sl].astype(np.float64) * float(pool.v_scales[p, h, sl])
            assert np.max(np.abs(o[t, hq] - v)) < 1e-15
            assert abs(lse[t, hq] - float(W.sm_scale) * (q[t, hq] @ k)) < 1e-12


def test_window_covering_everything_is_full_attention():
    W = wl.custom(8, 2, 16, [37, 5], [4, 3], seed=7)
    pool = oracle_pool(W)
    q = q_values(W)
    full = O.attention(q, pool, W.page_table, W.context_lens, W.block_lens, 2, float(W.sm_scale))
    win = O.attention(q, pool, W.page_table, W.context_lens, W.block_lens, 2, float(W.sm_scale),
                      window=41)
    assert np.array_equal(full[0], win[0]) and np.array_equal(full[1], win[1])


def test_tiny_workload_matches_sdpa():
    W = wl.make("tiny")
    pool = oracle_pool(W)
    q, (o, lse) = _run_oracle(W, pool)
    ro, rl = _sdpa_truncated(W, pool, q)
    assert np.max(np.abs(o - ro)) < 1e-12 and np.max(np.abs(lse - rl)) < 1e-12


def test_single_visible_key():
    W = wl.custom(2, 1, 16, [0], [1], seed=4)
    pool = oracle_pool(W)
    q, (o, lse) = _run_oracle(W, pool)
    p = int(W.page_table[0, 0])
    k0 = pool.k_codes[p, 0, 0].astype(np.float64) * float(pool.k_scales[p, 0, 0])
    v0 = pool.v_codes[p, 0, 0].astype(np.float64) * float(pool.v_scales[p, 0, 0])
    assert np.array_equal(o[0, 0], v0) or np.max(np.abs(o[0] - v0)) < 1e-15
    sigma = float(W.sm_scale) * (q[0] @ k0)
    assert np.max(np.abs(lse[0] - sigma)) < 1e-12


def test_identical_keys_give_mean_and_log_n():
    W = wl.custom(3, 1, 16, [21], [3], seed=8)
    pool = oracle_pool(W)
    pool.k_codes[:] = pool.k_codes[int(W.page_table[0, 0]), 0, 0]
    pool.k_scales[:] = pool.k_scales[int(W.page_table[0, 0]), 0, 0]
    q, (o, lse) = _run_oracle(W, pool)
    k_hat = pool.k_codes[0, 0, 0].astype(np.float64) * float(pool.k_scales[0, 0, 0])
    for t in range(3):
        n = 21 + t + 1
        vs = []
        for j in range(n):
            p, sl = int(W.page_table[0, j // 16]), j % 16
            vs.append(pool.v_codes[p, 0, sl].astype(np.float64) * float(pool.v_scales[p, 0, sl]))
        mean = np.mean(vs, axis=0)
        assert np.max(np.abs(o[t] - mean)) < 1e-12
        sigma = float(W.sm_scale) * (q[t] @ k_hat)
        assert np.max(np.abs(lse[t] - (sigma + math.log(n)))) < 1e-12


def test_rows_sum_to_one_constant_v():
    W = wl.custom(4, 2, 32, [50, 7], [4, 2], seed=9)
    pool = oracle_pool(W)
    pool.v_codes[:] = 127
    pool.v_scales[:] = np.float32(1 / 127)
    _, (o, _) = _run_oracle(W, pool)
    const = 127 * float(np.float32(1 / 127))
    assert np.max(np.abs(o - const)) < 1e-13


def test_last_verify_token_equals_unmasked_attention():
    W = wl.custom(4, 2, 16, [40], [6], seed=10)
    pool = oracle_pool(W)
    q, (o, _) = _run_oracle(W, pool)
    for h in range(2):
        K, V = _dense_kv(pool, W.page_table[0], h, 46)
        qq = torch.tensor(q[5, 2 * h:2 * h + 2])
        ref = torch.softmax(float(W.sm_scale) * qq @ K.T, dim=-1) @ V
        assert np.max(np.abs(o[5, 2 * h:2 * h + 2] - ref.numpy())) < 1e-12


def test_future_keys_do_not_matter_and_the_diagonal_does():
    W = wl.custom(2, 1, 16, [30], [5], seed=12)
    pool = oracle_pool(W)
    q, (o, lse) = _run_oracle(W, pool)
    t = 2
    # poison every key after ctx + t
    for j in range(30 + t + 1, 35):
        p, sl = int(W.page_table[0, j // 16]), j % 16
        pool.k_codes[p, 0, sl] = 127
        pool.v_codes[p, 0, sl] = -127
        pool.v_scales[p, 0, sl] = 1e6
    _, (o2, lse2) = _run_oracle(W, pool)
    assert np.array_equal(o2[t], o[t]) and np.array_equal(lse2[t], lse[t])
    assert not np.allclose(o2[t + 1], o[t + 1])
    # the diagonal key (ctx + t) is visible to row t
    p, sl = int(W.page_table[0, (30 + t) // 16]), (30 + t) % 16
    pool.v_scales[p, 0, sl] = 1e3
    _, (o3, _) = _run_oracle(W, pool)
    assert not np.allclose(o3[t], o[t])
    assert np.array_equal(o3[t - 1], o[t - 1])


def test_t1_is_plain_decode():
    W = wl.custom(6, 2, 32, [77, 3], [1, 1], seed=13)
    pool = oracle_pool(W)
    q, (o, lse) = _run_oracle(W, pool)
    for b in range(2):
        n = int(W.context_lens[b]) + 1
        for h in range(2):
            K, V = _dense_kv(pool, W.page_table[b], h, n)
            qq = torch.tensor(q[b, 3 * h:3 * h + 3])
            ref = torch.nn.functional.scaled_dot_product_attention(
                qq[None], K[None], V[None], scale=float(W.sm_scale))[0]
            assert np.max(np.abs(o[b, 3 * h:3 * h + 3] - ref.numpy())) < 1e-12


def test_page_permutation_invariance():
    W = wl.custom(4, 2, 16, [70, 33], [4, 3], seed=14)
    pool = oracle_pool(W)
    q, (o, lse) = _run_oracle(W, pool)
    perm = np.random.default_rng(1).permutation(W.num_pages)
    pool2 = O.PagedPool(W.num_pages, 2, 16, 16)
    for name in ("k_codes", "v_codes", "k_scales", "v_scales"):
        getattr(pool2, name)[perm] = getattr(pool, name)
    table2 = np.where(W.page_table >= 0, perm[np.maximum(W.page_table, 0)], -1)
    o2, lse2 = O.attention(q, pool2, table2, W.context_lens, W.block_lens, 2, float(W.sm_scale))
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("cuts", [[0, 16, 32, 53], [0, 50, 51, 53], [0, 53], [0, 1, 53]])
def test_split_kv_equals_unsplit(cuts):
    W = wl.custom(4, 2, 16, [48], [5], seed=15)
    pool = oracle_pool(W)
    q = q_values(W)
    G = 2
    for h in range(2):
        k, v = O.gather_keys(pool, W.page_table[0], h, 53)
        qs = q[0:5, h * G:(h + 1) * G]
        o_ref, l_ref = O.attention_seq_head(qs, k, v, 48, float(W.sm_scale))
        parts = [O.attention_partial(qs, k, v, 48, float(W.sm_scale), a, b)
                 for a, b in zip(cuts[:-1], cuts[1:])]
        o, l = O.lse_combine(parts)
        assert np.max(np.abs(o - o_ref)) < 1e-12 and np.max(np.abs(l - l_ref)) < 1e-12


def test_empty_split_is_skipped():
    W = wl.custom(2, 1, 16, [8], [4], seed=16)
    pool = oracle_pool(W)
    q = q_values(W)
    k, v = O.gather_keys(pool, W.page_table[0], 0, 12)
    o_p, l_p = O.attention_partial(q[:, 0:2], k, v, 8, float(W.sm_scale), 10, 12)
    assert np.all(np.isneginf(l_p[0])) and np.all(o_p[0] == 0)   # t=0 sees keys <= 8 only
    assert np.all(np.isfinite(l_p[3]))


def test_shared_prefix_equals_separate_sequences():
    # G = 1; both sequences reference the same prefix pages
    W = wl.custom(2, 2, 16, [64, 64], [3, 2], seed=17, shared_prefix_len=48)
    assert np.array_equal(W.page_table[0, :3], W.page_table[1, :3])
    pool = oracle_pool(W)
    q, (o, lse) = _run_oracle(W, pool)
    for b in range(2):
        Wb = wl.custom(2, 2, 16, [64], [int(W.block_lens[b])], seed=99)
        pb = O.PagedPool(Wb.num_pages, 2, 16, 16)
        from common import seq_context_tokens
        k, v = seq_context_tokens(W, b)
        O.kv_append(pb, k, v, Wb.page_table, np.array([0]), np.array([64]))
        bk, bv = W.block_kv_seq(b)
        O.kv_append(pb, bk, bv, Wb.page_table, np.array([64]), Wb.block_lens)
        r0 = int(W.q_offsets[b])
        rows = q[r0:r0 + int(W.block_lens[b])]
        ob, lb = O.attention(rows, pb, Wb.page_table, Wb.context_lens, Wb.block_lens, 2,
                             float(W.sm_scale))
        assert np.array_equal(ob, o[r0:r0 + len(rows)]) and np.array_equal(lb, lse[r0:r0 + len(rows)])


def test_kv_append_positions():
    """Appended rows land at positions ctx..ctx+T-1 of the page list, nothing else moves."""
    W = wl.custom(2, 1, 8, [13, 0], [5, 2], seed=18)
    pool = O.PagedPool(W.num_pages, 1, 16, 8)
    k = np.arange(7 * 8, dtype=np.float32).reshape(7, 1, 8) + 1
    O.kv_append(pool, k, -k, W.page_table, W.context_lens, W.block_lens)
    kc, ks = O.quantise_rows(k)
    for row, (b, pos) in enumerate([(0, 13), (0, 14), (0, 15), (0, 16), (0, 17), (1, 0), (1, 1)]):
        p, sl = int(W.page_table[b, pos // 16]), pos % 16
        assert np.array_equal(pool.k_codes[p, 0, sl], kc[row, 0])
        assert np.array_equal(pool.v_codes[p, 0, sl], -kc[row, 0])
        assert pool.k_scales[p, 0, sl] == ks[row, 0]
    assert int(np.count_nonzero(pool.k_scales)) == 7


# ---------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# ---------------------------------------------------------------------------
def _pins_fail(fn) -> bool:
    try:
        fn()
    except AssertionError:
        return True
    return False


def test_planted_rounding_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(O, "_round_half_even", lambda x: np.floor(x + 0.5))
    assert _pins_fail(test_quantiser_closed_form_cases)


def test_planted_scale_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(O, "QMAX", 128)
    assert _pins_fail(test_quantiser_matches_exact_rationals_random)


def test_planted_multiply_form_is_caught(monkeypatch):
    orig = O._fl32_div

    def mul_form(a, b):
        b = np.asarray(b, np.float64)
        if b.ndim and b.shape[-1:] == (1,):          # x / s  ->  x * fl32(1/s)
            return (np.asarray(a, np.float64) * (1.0 / b).astype(np.float32)).astype(np.float32)
        return orig(a, b)
    monkeypatch.setattr(O, "_fl32_div", mul_form)
    assert _pins_fail(test_quantiser_is_the_divide_form)


def test_planted_mask_off_by_one_is_caught(monkeypatch):
    monkeypatch.setattr(O, "_visible", lambda j, ctx, t, window=0: j < ctx + t)
    assert _pins_fail(lambda: test_attention_matches_sdpa_on_truncated_keys([37], [4], 8, 2, 32))


def test_planted_mask_too_wide_is_caught(monkeypatch):
    monkeypatch.setattr(O, "_visible", lambda j, ctx, t, window=0: j <= ctx + t + 1)
    assert _pins_fail(test_future_keys_do_not_matter_and_the_diagonal_does)


def test_planted_window_off_by_one_is_caught(monkeypatch):
    # a window of W keys that starts one key early (W + 1 keys)
    monkeypatch.setattr(O, "_visible",
                        lambda j, ctx, t, window=0: (j <= ctx + t) & ((window <= 0) | (j >= ctx + t - window)))
    assert _pins_fail(lambda: test_window_matches_sdpa_on_window_keys(5))


def test_planted_dequant_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(O, "dequantise", lambda c, s: c.astype(np.float64))
    assert _pins_fail(lambda: test_attention_matches_sdpa_on_truncated_keys([37], [4], 8, 2, 32))


def test_planted_gqa_mistake_is_caught(monkeypatch):
    orig = O.attention_seq_head

    def swapped(q, k, v, ctx, sm, window=0):      # query heads paired with the wrong rows
        return orig(q[:, ::-1], k, v, ctx, sm, window)
    monkeypatch.setattr(O, "attention_seq_head", swapped)
    assert _pins_fail(lambda: test_attention_matches_sdpa_on_truncated_keys([37], [4], 8, 2, 32))


def test_planted_combine_mistake_is_caught(monkeypatch):
    def bad_combine(parts):
        lses = np.stack([l for _, l in parts])
        lse = np.max(lses, axis=0)                  # dropped the log-sum
        o = sum(np.exp(l - lse)[..., None] * oi for oi, l in parts)
        return o, lse
    monkeypatch.setattr(O, "lse_combine", bad_combine)
    assert _pins_fail(lambda: test_split_kv_equals_unsplit([0, 16, 32, 53]))


# ---------------------------------------------------------------------------
# accept / commit
# ---------------------------------------------------------------------------
def test_accept_commit_hand_cases():
    with open(os.path.join(GOLDEN, "accept_commit_cases.json")) as f:
        c = json.load(f)
    acc, ctx, nxt = O.accept_commit(c["block_tokens"], c["target_tokens"], c["block_lens"],
                                    c["context_lens"])
    assert acc.tolist() == c["accepted"]
    assert ctx.tolist() == c["new_context"]
    assert nxt.tolist() == c["next_tokens"]


def test_accept_commit_bounds_and_full_acceptance():
    rng = np.random.default_rng(3)
    T = rng.integers(0, 17, size=50)
    x = rng.integers(0, 5, size=int(T.sum()))
    y = rng.integers(0, 5, size=int(T.sum()))
    acc, ctx, nxt = O.accept_commit(x, y, T, np.zeros(50, np.int32))
    assert np.all((acc >= 0) & (acc <= np.maximum(T - 1, 0)))
    assert np.array_equal(ctx, np.where(T > 0, acc + 1, 0))
    # target agrees with every draft -> all T-1 drafts accepted
    y2 = np.concatenate([np.append(x[o + 1:o + t], 99) for o, t in
                         zip(np.concatenate([[0], np.cumsum(T)[:-1]]), T) if t > 0])
    x2 = np.concatenate([x[o:o + t] for o, t in zip(np.concatenate([[0], np.cumsum(T)[:-1]]), T) if t > 0])
    acc2, _, nxt2 = O.accept_commit(x2, y2, T, np.zeros(50, np.int32))
    assert np.array_equal(acc2, np.maximum(T - 1, 0))
    assert np.all(nxt2[T > 0] == 99)


def test_planted_accept_off_by_one_is_caught(monkeypatch):
    # compares draft x_{i+1} with the target's choice after x_{i+1} (y_{i+1}) instead of y_i
    def wrong(block_tokens, target_tokens, block_lens, context_lens):
        acc, ctx, nxt = [], [], []
        off = 0
        for b, T in enumerate(block_lens):
            T = int(T)
            x, y = list(block_tokens[off:off + T]), list(target_tokens[off:off + T])
            off += T
            if T == 0:
                acc.append(0); ctx.append(int(context_lens[b])); nxt.append(-1)
                continue
            a = 0
            while a + 1 < T and x[a + 1] == y[a + 1]:
                a += 1
            acc.append(a); ctx.append(int(context_lens[b]) + a + 1); nxt.append(int(y[a]))
        return (np.array(acc, np.int32), np.array(ctx, np.int32), np.array(nxt, np.int32))
    monkeypatch.setattr(O, "accept_commit", wrong)
    assert _pins_fail(test_accept_commit_hand_cases)


def test_lse_combine_hand_values():
    # two splits with lse 0 and ln 3: weights 1/4 and 3/4, combined lse ln 4
    o1 = np.array([[1.0, 0.0]])
    o2 = np.array([[0.0, 2.0]])
    o, lse = O.lse_combine([(o1, np.array([0.0])), (o2, np.array([np.log(3.0)]))])
    assert abs(lse[0] - np.log(4.0)) < 1e-15
    assert np.max(np.abs(o[0] - np.array([0.25, 1.5]))) < 1e-15
    # an empty split (lse = -inf) has no weight
    o, lse = O.lse_combine([(o1, np.array([0.0])), (np.full((1, 2), 7.0), np.array([-np.inf]))])
    assert lse[0] == 0.0 and np.array_equal(o[0], o1[0])
