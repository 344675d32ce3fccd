"""GPU parity of the shared-prefix entry point (query rows of the sequences
that share prefix pages stacked into row blocks that read the prefix once)
against the fp64 oracle, through the C ABI.

The oracle attends every sequence on its own; the stacking is a split of the
same sums, so the bars are those of every other attention test: O within
max-abs 1e-2 / mean-abs 1e-3, LSE within 1e-3. The plan the device builds is
checked against the grouping rule the header states, recomputed here from
the lengths.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from oracle import splash_oracle as O  # noqa: E402
from speculative_verify_attention_kv_gb300 import build as _build  # noqa: E402

if not os.path.exists(_build.LIB):
    _build.build()

from speculative_verify_attention_kv_gb300 import splash_kv as sk  # noqa: E402
from speculative_verify_attention_kv_gb300 import workloads as wl  # noqa: E402

from common import expected_group_plan as expected_plan, oracle_pool, q_values  # noqa: E402
from gpu_common import Run, assert_parity  # noqa: E402

def plan_header(ws):
    """(total tensor-core tiles, items) from the plan header the prefix-group
    planner wrote (it keeps the item count in the header's first spare word)."""
    h = ws[:64].cpu().numpy().view(np.int32)
    return int(h[0]), int(h[12])


CASES = [
    # four sequences of 96 rows on a 256-key prefix: 3 row blocks instead of 4
    dict(hq=24, hkv=4, D=256, ctx=[300, 420, 300, 700], T=[16, 16, 16, 16], prefix=256),
    # single-token blocks: the four sequences' 24 rows in one block
    dict(hq=24, hkv=4, D=256, ctx=[2000, 2100, 2050, 2300], T=[1, 1, 1, 1], prefix=1984),
    # two groups cut by the links; the second one's prefix is its 200-key link
    dict(hq=24, hkv=4, D=256, ctx=[600, 700, 512, 900, 1000, 530], T=[4, 8, 1, 16, 2, 3],
         prefix=512, sl=[0, 512, 512, 0, 200, 512]),
    # 128 rows per sequence: a block per sequence, so nothing is stacked
    dict(hq=32, hkv=4, D=128, ctx=[400, 500], T=[16, 16], prefix=320),
    # head_dim 128, three sequences in one block
    dict(hq=8, hkv=2, D=128, ctx=[330, 400, 900], T=[4, 3, 5], prefix=320),
    # a prefix that is not a whole number of tiles (208 keys: 192 stacked), and
    # a sequence whose context is the prefix alone
    dict(hq=24, hkv=4, D=256, ctx=[208, 300, 260], T=[16, 16, 16], prefix=208),
    # an idle sequence inside the run breaks it
    dict(hq=24, hkv=4, D=256, ctx=[300, 300, 300], T=[4, 0, 4], prefix=256),
    # a long prefix spread over many CTAs, five sequences, ragged blocks
    dict(hq=24, hkv=4, D=256, ctx=[6000, 6100, 6500, 6050, 7000], T=[16, 8, 4, 1, 12],
         prefix=5952),
]


def _run(c, seed):
    W = wl.custom(c["hq"], c["hkv"], c["D"], c["ctx"], c["T"], seed=seed,
                  shared_prefix_len=c["prefix"])
    r = Run(W)
    r.append_block()
    sl = c.get("sl")
    sl_t = None if sl is None else torch.tensor(sl, dtype=torch.int32, device="cuda")
    sl_h = list(W.shared_lens()) if sl is None else sl
    return W, r, sl_t, sl_h


@pytest.mark.parametrize("case", range(len(CASES)))
def test_shared_prefix_matches_oracle(case):
    c = CASES[case]
    if not sk.tensor_path_available(c["D"]):
        pytest.skip("tensor-core kernel not built for this head_dim")
    W, r, sl_t, sl_h = _run(c, 40 + case)
    o_ref, l_ref = O.attention(q_values(W), oracle_pool(W), W.page_table, W.context_lens,
                               W.block_lens, W.spec.num_kv_heads, float(W.sm_scale))
    G = c["hq"] // c["hkv"]
    want = expected_plan(c["ctx"], c["T"], sl_h, G, c["hkv"])
    for ctas in (0, 1, 3, 7):
        out = torch.full_like(r.out, float("nan"))
        lse = torch.full_like(r.lse, float("nan"))
        r.attend(ctas=ctas, out=out, lse=lse, shared_lens=sl_t)
        torch.cuda.synchronize()
        assert int(r.status.item()) == 0
        assert_parity(out, lse, o_ref, l_ref, what=f"case {case} ctas {ctas}")
        tiles, items = plan_header(r.ws)
        assert (items, tiles) == want, f"case {case} ctas {ctas}: plan {(items, tiles)} != {want}"


def test_the_shared_prefix_workload_is_stacked():
    """The seeded 4 x (24K shared + 8K) workload's plan: 3 row blocks over the
    prefix, so 3 * 384 + 4 * 129 tiles per KV head instead of 4 * 513."""
    W = wl.make("shared_prefix")
    G, H = W.spec.group, W.spec.num_kv_heads
    ctx = [int(x) for x in W.context_lens]
    T = [int(x) for x in W.block_lens]
    items, tiles = expected_plan(ctx, T, list(W.shared_lens()), G, H)
    assert items == 4 + 3 and tiles == H * (3 * 384 + 4 * 129)


def test_shared_and_plain_agree():
    c = CASES[0]
    W, r, _, _ = _run(c, 7)
    o1, l1 = [t.clone() for t in r.attend(stack=False)]
    o2, l2 = [t.clone() for t in r.attend(stack=True)]
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 2 ** -7
    assert (l1 - l2).abs().max().item() <= 1e-4
    # the plain call planned one item per sequence, the shared one stacked
    _, items = plan_header(r.ws)
    assert items == len(c["ctx"]) + 3


def test_shared_deterministic_and_page_permutation_bitwise():
    c = CASES[2]
    W, r, sl_t, _ = _run(c, 9)
    o1, l1 = [t.clone() for t in r.attend(shared_lens=sl_t)]
    o2, l2 = [t.clone() for t in r.attend(shared_lens=sl_t)]
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    perm = torch.from_numpy(np.random.default_rng(4).permutation(W.num_pages)).cuda().long()
    newpool = sk.alloc_pool(W.num_pages, W.spec.num_kv_heads, W.spec.head_dim)
    for n, t in zip(newpool, r.pool):
        n[perm] = t
    r.pool = tuple(newpool)
    tab = r.table.long()
    r.table = torch.where(tab >= 0, perm[tab.clamp(min=0)], tab).int().contiguous()
    o3, l3 = r.attend(shared_lens=sl_t)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


@pytest.mark.parametrize("path", [sk.PATH_SIMT, sk.PATH_TENSOR_T])
def test_paths_without_groups_compute_the_same_result(path):
    """The CUDA-core and transposed kernels take no row blocks: the call
    plans one item per sequence and still matches the oracle."""
    c = CASES[0]
    W, r, _, _ = _run(c, 11)
    o_ref, l_ref = O.attention(q_values(W), oracle_pool(W), W.page_table, W.context_lens,
                               W.block_lens, W.spec.num_kv_heads, float(W.sm_scale))
    out, lse = r.attend(path=path)
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    assert_parity(out, lse, o_ref, l_ref, what=f"path {path}")


def test_zero_links_plan_like_the_plain_call():
    c = CASES[0]
    W, r, _, _ = _run(c, 13)
    zeros = torch.zeros(len(c["ctx"]), dtype=torch.int32, device="cuda")
    o1, l1 = [t.clone() for t in r.attend(stack=False)]
    o2, l2 = [t.clone() for t in r.attend(shared_lens=zeros)]
    # no group: the same plan (same split, same kernels), so bitwise equal
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
