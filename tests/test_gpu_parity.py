"""GPU parity of the CUDA path against the fp64 oracle (through the C ABI).

Bars: int8 codes and fp32 scales bit-exact; attention O (bf16) within max-abs
1e-2 and mean-abs 1e-3 of the fp64 oracle, LSE within 1e-3 absolute.
"""
from __future__ import annotations

import functools
import json

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from oracle import splash_oracle as O  # noqa: E402
from speculative_verify_attention_kv_gb300 import build as _build  # noqa: E402

import os  # noqa: E402
if not os.path.exists(_build.LIB):
    _build.build()

from speculative_verify_attention_kv_gb300 import splash_kv as sk  # noqa: E402
from speculative_verify_attention_kv_gb300 import workloads as wl  # noqa: E402

from common import oracle_pool, q_values  # noqa: E402
from gpu_common import Run, assert_parity, assert_parity_scaled, compare  # noqa: E402


def oracle_attention(W, pool, seqs=None, window=0):
    return O.attention(q_values(W), pool, W.page_table, W.context_lens, W.block_lens,
                       W.spec.num_kv_heads, float(W.sm_scale), seqs=seqs, window=window)


def written_slots(W, seqs):
    """(page, slot) of every logical position 0..ctx+T-1 of the listed sequences."""
    pages, slots = [], []
    for b in seqs:
        j = np.arange(int(W.context_lens[b] + W.block_lens[b]))
        pages.append(W.page_table[b][j // 16].astype(np.int64))
        slots.append(j % 16)
    return np.concatenate(pages), np.concatenate(slots)


def seq_rows(W, seqs):
    return np.concatenate([np.arange(W.q_offsets[b], W.q_offsets[b + 1]) for b in seqs]).astype(np.int64)


@functools.lru_cache(maxsize=None)
def _tc_probe():
    W = wl.custom(8, 2, 128, [20], [4], seed=1)
    r = Run(W)
    r.append_block()
    try:
        r.attend(path=sk.PATH_TENSOR)
    except sk.SplashError as e:
        if e.status == -2:
            return False
        raise
    return True


PATHS = [sk.PATH_AUTO, sk.PATH_SIMT, sk.PATH_TENSOR, sk.PATH_TENSOR_T]


def _path_ok(path, head_dim=256, rows=96):
    if path == sk.PATH_TENSOR:
        return sk.tensor_path_available(head_dim)
    if path == sk.PATH_TENSOR_T:
        return head_dim == 256 and rows <= 96
    return True


# ---------------------------------------------------------------------------
# kv_append: bit-exact codes and scales
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("D", [64, 128, 256])
def test_kv_append_bit_exact_edge_rows(D):
    rng = np.random.default_rng(D)
    n, hkv = 40, 2
    x = rng.standard_normal((n, hkv, D)).astype(np.float32)
    x[0] = 0
    x[1, 0, :] = 0
    x[1, 0, 5] = np.float32(-2.0 ** -140)
    x[2, 1, :] = 0
    x[2, 1, :4] = np.float32(190 * 2.0 ** -149)
    x[3, 0, :8] = np.array([127.0, 2.5, 3.5, -2.5, 0.5, 126.5, -127.0, 1.5], np.float32)
    x[3, 0, 8:] = 0
    x[4:10, :, 3] *= 8
    x[10] *= np.float32(1e-30)
    W = wl.custom(2 * hkv, hkv, D, [0, 7], [17, n - 17], seed=2)
    pool = sk.alloc_pool(W.num_pages, hkv, D)
    table = torch.from_numpy(W.page_table).cuda()
    sk.splash_kv_append(torch.from_numpy(x).cuda(), torch.from_numpy(-x).cuda(), *pool, table,
                        torch.from_numpy(W.context_lens).cuda(), torch.from_numpy(W.block_lens).cuda())
    torch.cuda.synchronize()
    opool = O.PagedPool(W.num_pages, hkv, 16, D)
    O.kv_append(opool, x, -x, W.page_table, W.context_lens, W.block_lens)
    kp, vp, ks, vs = [t.cpu().numpy() for t in pool]
    assert np.array_equal(kp, opool.k_codes) and np.array_equal(vp, opool.v_codes)
    assert np.array_equal(ks.view(np.uint32), opool.k_scales.view(np.uint32))
    assert np.array_equal(vs.view(np.uint32), opool.v_scales.view(np.uint32))


@pytest.mark.parametrize("D", [128, 256])
def test_kv_append_bf16_bit_exact(D):
    rng = np.random.default_rng(100 + D)
    n, hkv = 53, 4
    x = rng.standard_normal((n, hkv, D)).astype(np.float32) * np.float32(3.0)
    x[0, 1, :] = 0
    x[1, 2, :] = 0
    x[1, 2, 9] = np.float32(2.0 ** -133)         # a bf16 subnormal
    x[2] *= np.float32(1e20)
    xb = wl.bf16_bits_from_f32(x)
    vb = wl.bf16_bits_from_f32(-0.5 * x)
    W = wl.custom(2 * hkv, hkv, D, [5, 0, 33], [20, 1, n - 21], seed=4)
    pool = sk.alloc_pool(W.num_pages, hkv, D)
    table = torch.from_numpy(W.page_table).cuda()
    as_bf16 = lambda b: torch.from_numpy(b.view(np.int16)).cuda().view(torch.bfloat16)
    sk.splash_kv_append(as_bf16(xb), as_bf16(vb), *pool, table,
                        torch.from_numpy(W.context_lens).cuda(), torch.from_numpy(W.block_lens).cuda())
    torch.cuda.synchronize()
    opool = O.PagedPool(W.num_pages, hkv, 16, D)
    O.kv_append(opool, wl.f32_from_bf16_bits(xb), wl.f32_from_bf16_bits(vb), W.page_table,
                W.context_lens, W.block_lens)
    kp, vp, ks, vs = [t.cpu().numpy() for t in pool]
    assert np.array_equal(kp, opool.k_codes) and np.array_equal(vp, opool.v_codes)
    assert np.array_equal(ks.view(np.uint32), opool.k_scales.view(np.uint32))
    assert np.array_equal(vs.view(np.uint32), opool.v_scales.view(np.uint32))


# ---------------------------------------------------------------------------
# accept / commit: exact integers
# ---------------------------------------------------------------------------
def _accept_on_gpu(x, y, T, ctx):
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    ctx_d = i32(ctx)
    acc = torch.full((len(T),), -7, dtype=torch.int32, device="cuda")
    nxt = torch.full((len(T),), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sk.splash_accept_commit(i32(x), i32(y), i32(T), ctx_d, acc, nxt, device_status=status)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), ctx_d.cpu().numpy(), nxt.cpu().numpy(), int(status.item())


def test_accept_commit_golden_cases():
    with open(os.path.join(os.path.dirname(__file__), "golden", "accept_commit_cases.json")) as f:
        c = json.load(f)
    acc, ctx, nxt, st = _accept_on_gpu(c["block_tokens"], c["target_tokens"], c["block_lens"],
                                       c["context_lens"])
    assert st == 0
    assert acc.tolist() == c["accepted"]
    assert ctx.tolist() == c["new_context"]
    assert nxt.tolist() == c["next_tokens"]


@pytest.mark.parametrize("B", [1, 64, 1000, 5000])
def test_accept_commit_random_matches_oracle(B):
    rng = np.random.default_rng(B)
    T = rng.integers(0, 17, size=B)
    T[rng.random(B) < 0.1] = 0
    n = int(T.sum())
    x = rng.integers(0, 3, size=n)            # a small vocabulary makes long accepted runs
    y = rng.integers(0, 3, size=n)
    ctx = rng.integers(0, 40000, size=B)
    acc, new_ctx, nxt, st = _accept_on_gpu(x, y, T, ctx)
    ra, rc, rn = O.accept_commit(x, y, T, ctx)
    assert st == 0
    assert np.array_equal(acc, ra) and np.array_equal(new_ctx, rc) and np.array_equal(nxt, rn)


# ---------------------------------------------------------------------------
# attention: small cases, full oracle
# ---------------------------------------------------------------------------
SMALL = [
    dict(hq=8, hkv=2, D=128, ctx=[37, 200, 0], T=[4, 1, 3]),
    dict(hq=24, hkv=4, D=256, ctx=[130, 513, 1000], T=[16, 1, 8]),
    dict(hq=4, hkv=4, D=64, ctx=[700], T=[5]),
    dict(hq=24, hkv=4, D=256, ctx=[300, 300], T=[16, 16], prefix=256),
    dict(hq=32, hkv=4, D=128, ctx=[333], T=[16]),          # T*G = 128 rows
    dict(hq=24, hkv=4, D=256, ctx=[50, 60, 70], T=[3, 0, 2]),   # an idle sequence
    dict(hq=24, hkv=4, D=256, ctx=[4000], T=[4]),
    # more sequences than the small planner block takes (the 1024-thread planner)
    dict(hq=8, hkv=2, D=128,
         ctx=[int(x) for x in np.random.default_rng(71).integers(0, 300, 200)],
         T=[int(x) for x in np.random.default_rng(72).integers(0, 5, 200)]),
]


@pytest.mark.parametrize("case", range(len(SMALL)))
@pytest.mark.parametrize("path", PATHS)
def test_attention_small_cases(case, path):
    c = SMALL[case]
    if not _path_ok(path, c["D"], max(c["T"]) * c["hq"] // c["hkv"]):
        pytest.skip("kernel not built for this head_dim / row count")
    W = wl.custom(c["hq"], c["hkv"], c["D"], c["ctx"], c["T"], seed=20 + case,
                  shared_prefix_len=c.get("prefix", 0))
    r = Run(W)
    r.append_block()
    o_ref, l_ref = oracle_attention(W, oracle_pool(W))
    for ctas in (0, 1, 3):
        o, l = r.attend(path=path, ctas=ctas)
        torch.cuda.synchronize()
        assert_parity(o, l, o_ref, l_ref, what=f"case {case} path {path} ctas {ctas}")
    assert int(r.status.item()) == 0


# ---------------------------------------------------------------------------
# properties
# ---------------------------------------------------------------------------
def _small_run(seed=5, ctx=(900, 37, 2100), T=(16, 1, 8)):
    W = wl.custom(24, 4, 256, list(ctx), list(T), seed=seed)
    r = Run(W)
    r.append_block()
    return W, r


@pytest.mark.parametrize("path", PATHS)
def test_deterministic_and_page_permutation_bitwise(path):
    if not _path_ok(path):
        pytest.skip("tensor-core kernel not built")
    W, r = _small_run()
    o1, l1 = [t.clone() for t in r.attend(path=path)]
    o2, l2 = [t.clone() for t in r.attend(path=path)]
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    perm = torch.from_numpy(np.random.default_rng(3).permutation(W.num_pages)).cuda().long()
    newpool = sk.alloc_pool(W.num_pages, W.spec.num_kv_heads, W.spec.head_dim)
    for n, t in zip(newpool, r.pool):
        n[perm] = t
    r.pool = tuple(newpool)
    tab = r.table.long()
    r.table = torch.where(tab >= 0, perm[tab.clamp(min=0)], tab).int().contiguous()
    o3, l3 = r.attend(path=path)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


def test_split_and_unsplit_agree():
    W, r = _small_run()
    o_ref, l_ref = oracle_attention(W, oracle_pool(W))
    outs = []
    for ctas in (1, 2, 7, 0):
        o, l = [t.clone() for t in r.attend(ctas=ctas)]
        assert_parity(o, l, o_ref, l_ref, what=f"ctas={ctas}")
        outs.append((o.float(), l))
    for o, l in outs[1:]:
        assert (o - outs[0][0]).abs().max().item() <= 2 ** -7
        assert (l - outs[0][1]).abs().max().item() <= 1e-4


@pytest.mark.parametrize("path", PATHS)
def test_future_block_keys_do_not_leak(path):
    if not _path_ok(path):
        pytest.skip("tensor-core kernel not built")
    W, r = _small_run(ctx=(500,), T=(8,))
    o1, l1 = [t.clone() for t in r.attend(path=path)]
    kp, vp, ks, vs = r.pool
    for j in range(500 + 4, 508):   # poison block tokens 4..7
        page, slot = int(W.page_table[0, j // 16]), j % 16
        kp[page, :, slot] = 127
        vp[page, :, slot] = -127
        vs[page, :, slot] = 1e4
    o2, l2 = r.attend(path=path)
    assert torch.equal(o1[:4], o2[:4]) and torch.equal(l1[:4], l2[:4])
    assert not torch.equal(o1[4:], o2[4:])


def test_t1_rows_are_plain_decode():
    W = wl.custom(24, 4, 256, [777, 1500], [1, 1], seed=31)
    r = Run(W)
    r.append_block()
    o, l = r.attend()
    opool = oracle_pool(W)
    q = q_values(W)
    for b in range(2):
        n = int(W.context_lens[b]) + 1
        for h in range(4):
            k, v = O.gather_keys(opool, W.page_table[b], h, n)
            qq = torch.tensor(q[b, 6 * h:6 * h + 6])
            ref = torch.softmax(float(W.sm_scale) * qq @ torch.tensor(k).T, -1) @ torch.tensor(v)
            err = (o[b, 6 * h:6 * h + 6].float().cpu().double() - ref).abs().max().item()
            assert err <= 1e-2


def test_bad_page_sets_device_status():
    W, r = _small_run(ctx=(300,), T=(4,))
    tab = r.table.clone()
    tab[0, 5] = W.num_pages + 3
    r.table = tab
    r.status.zero_()
    r.attend()
    torch.cuda.synchronize()
    assert int(r.status.item()) == sk.DEVICE_BAD_PAGE
    r.status.zero_()
    r.table = tab
    r.append_block()       # block positions 300..303 live on page 18: valid -> no error
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0


def test_bad_length_sets_device_status():
    W, r = _small_run(ctx=(300,), T=(4,))
    r.ctx = torch.tensor([W.max_pages_per_seq * 16], dtype=torch.int32, device="cuda")
    r.status.zero_()
    r.attend()
    torch.cuda.synchronize()
    assert int(r.status.item()) == sk.DEVICE_BAD_LENGTH


def test_bad_sequence_leaves_the_others_correct():
    # the middle sequence's length exceeds its page-table capacity: it is
    # skipped, and the sequences after it keep their own Q / O rows
    W = wl.custom(24, 4, 256, [300, 500, 700], [4, 8, 16], seed=52)
    r = Run(W)
    r.append_block()
    o_ref, l_ref = oracle_attention(W, oracle_pool(W))
    ctx = r.ctx.clone()
    ctx[1] = W.max_pages_per_seq * 16
    r.ctx = ctx
    rows = seq_rows(W, [0, 2])
    for path in PATHS:
        if not _path_ok(path):
            continue
        r.status.zero_()
        o, l = r.attend(path=path)
        torch.cuda.synchronize()
        assert int(r.status.item()) == sk.DEVICE_BAD_LENGTH
        assert_parity(o, l, o_ref, l_ref, rows=rows, what=f"path {path}")


@pytest.mark.parametrize("path", [sk.PATH_TENSOR, sk.PATH_TENSOR_T])
def test_wait_timeout_is_reported_and_the_next_call_is_correct(path):
    # A wait limit of 1 ns makes the tensor-core kernel's first pipeline wait
    # run out: it must stop, let the copies and MMAs it issued complete, free
    # its tensor memory and report SPLASH_DEVICE_TIMEOUT; the following call
    # with the default limit must be unaffected.
    if not _path_ok(path):
        pytest.skip("tensor-core kernel not built")
    W, r = _small_run(seed=53)
    o_ref, l_ref = oracle_attention(W, oracle_pool(W))
    for _ in range(2):
        prev = sk.splash_set_wait_limit_ns(1)
        try:
            r.status.zero_()
            r.attend(path=path)
            torch.cuda.synchronize()
            st = int(r.status.item())
        finally:
            sk.splash_set_wait_limit_ns(prev)
        assert st == sk.DEVICE_TIMEOUT
        r.status.zero_()
        o, l = r.attend(path=path)
        torch.cuda.synchronize()
        assert int(r.status.item()) == 0
        assert_parity(o, l, o_ref, l_ref, what="after a timeout")


def test_workspace_too_small():
    W, r = _small_run(ctx=(300,), T=(4,))
    r.ws = r.ws[:1024]
    with pytest.raises(sk.SplashError) as e:
        r.attend()
    assert e.value.status == -3


def test_empty_batch_is_a_no_op():
    W = wl.custom(8, 2, 128, [10], [0], seed=3)
    r = Run(W)
    r.attend()
    torch.cuda.synchronize()


# ---------------------------------------------------------------------------
# sliding window
# ---------------------------------------------------------------------------
WINDOWS = [1, 7, 64, 65, 200, 1000, 100000]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("window", WINDOWS)
def test_sliding_window_matches_oracle(path, window):
    if not _path_ok(path):
        pytest.skip("tensor-core kernel not built")
    W = wl.custom(24, 4, 256, [900, 37, 2100, 0], [16, 1, 8, 5], seed=11)
    r = Run(W)
    r.append_block()
    o_ref, l_ref = oracle_attention(W, oracle_pool(W), window=window)
    for ctas in (0, 1, 5):
        o, l = r.attend(path=path, ctas=ctas, window=window)
        torch.cuda.synchronize()
        what = f"window {window} path {path} ctas {ctas}"
        if window >= 64:
            assert_parity(o, l, o_ref, l_ref, what=what)
        else:   # rows that see fewer than 64 keys: bound scaled with |O|
            assert_parity_scaled(o, l, o_ref, l_ref, what=what)
    assert int(r.status.item()) == 0


def test_sliding_window_never_reads_pages_below_it():
    # table entries of pages wholly below the window are -1: no error, same result
    W = wl.custom(24, 4, 256, [1000, 333], [16, 4], seed=12)
    r = Run(W)
    r.append_block()
    window = 100
    o_ref, l_ref = [t.clone() for t in r.attend(window=window)]
    table = r.table.clone()
    for b in range(W.num_seqs):
        first_key = max(0, int(W.context_lens[b]) - window + 1)
        table[b, : first_key // 16] = -1
    torch.cuda.synchronize()
    o, l = r.attend(window=window, table=table)
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    assert torch.equal(o, o_ref) and torch.equal(l, l_ref)


def test_window_zero_is_full_attention_bitwise():
    W, r = _small_run(seed=13)
    o1, l1 = [t.clone() for t in r.attend()]
    o2, l2 = [t.clone() for t in r.attend(window=0)]
    big = int(W.context_lens.max() + W.block_lens.max())
    o3, l3 = [t.clone() for t in r.attend(window=big)]
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


def test_negative_window_is_an_argument_error():
    W, r = _small_run(seed=14)
    with pytest.raises(sk.SplashError) as e:
        r.attend(window=-1)
    assert e.value.status == -1


# ---------------------------------------------------------------------------
# value magnitudes far from 1: the fp16 operand P * s_V stays accurate
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("scale", [1e3, 1e-3])
@pytest.mark.parametrize("path", [sk.PATH_AUTO, sk.PATH_TENSOR, sk.PATH_TENSOR_T])
def test_value_magnitudes_far_from_one(scale, path):
    # V scaled by `scale` (K unchanged): O scales with it, LSE does not. The
    # spec's bounds, scaled alike: max-abs 1e-2 * scale, mean-abs 1e-3 * scale.
    if not _path_ok(path):
        pytest.skip("kernel not built")
    W = wl.custom(24, 4, 256, [900, 37, 2100], [16, 1, 8], seed=61)
    s = W.spec
    r = Run(W, populate=False)
    opool = O.PagedPool(W.num_pages, s.num_kv_heads, s.page_size, s.head_dim)
    for b in range(W.num_seqs):
        ks, vs = zip(*(W.context_kv(b, h) for h in range(s.num_kv_heads)))
        k, v = np.stack(ks, 1), np.stack(vs, 1) * np.float32(scale)
        O.kv_append(opool, k, v, W.page_table[b:b + 1], np.array([0]), np.array([k.shape[0]]))
        r._append(k, v, b, 0)
    bk, bv = W.block_kv()
    bv = bv * np.float32(scale)
    O.kv_append(opool, bk, bv, W.page_table, W.context_lens, W.block_lens)
    r.v_new = torch.from_numpy(bv).cuda()
    r.append_block()
    o_ref, l_ref = oracle_attention(W, opool)
    o, l = r.attend(path=path)
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    err = np.abs(o.float().cpu().numpy().astype(np.float64) - o_ref)
    assert np.all(np.isfinite(err)) and err.max() <= 1e-2 * scale and err.mean() <= 1e-3 * scale, \
        (err.max(), err.mean())
    assert np.abs(l.cpu().numpy() - l_ref).max() <= 1e-3


def test_a_step_launches_four_kernels():
    # append, split planner, attention, log-sum-exp combine (host-side count of
    # the library's launches)
    W, r = _small_run(seed=62)
    n0 = sk.splash_launch_count()
    r.step()
    torch.cuda.synchronize()
    assert sk.splash_launch_count() - n0 == 4
