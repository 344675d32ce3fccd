"""The fixed-scratch entry point, for callers that cannot allocate device
memory (an allocator that owns all device memory, a host that forbids
allocation calls, a loop that cannot take cudaMalloc's implicit device
synchronisation). It must give the same results as the workspace entry point,
call after call, while the library itself allocates nothing.

Collected last on purpose; it also runs alone in a fresh process.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from speculative_verify_attention_kv_gb300 import build as _build  # noqa: E402

if not os.path.exists(_build.LIB):
    _build.build()

from speculative_verify_attention_kv_gb300 import splash_kv as sk  # noqa: E402
from speculative_verify_attention_kv_gb300 import workloads as wl  # noqa: E402
from speculative_verify_attention_kv_gb300.device_workload import DeviceWorkload  # noqa: E402

from common import oracle_pool, q_values  # noqa: E402
from gpu_common import assert_parity  # noqa: E402
from oracle import splash_oracle as O  # noqa: E402


def _fixed(dw, out, lse):
    sk.splash_verify_attention_fixed_scratch(dw.q, *dw.pool, dw.table, dw.ctx, dw.T,
                                             float(dw.W.sm_scale), dw.max_T, out, lse,
                                             device_status=dw.status)


@pytest.mark.parametrize("case", [
    dict(hq=24, hkv=4, D=256, ctx=[900, 37, 2100], T=[16, 1, 8]),
    dict(hq=8, hkv=2, D=128, ctx=[256], T=[4]),
])
def test_fixed_scratch_matches_workspace_entry_point(case):
    W = wl.custom(case["hq"], case["hkv"], case["D"], case["ctx"], case["T"], seed=41)
    dw = DeviceWorkload(W)
    dw.append_block()
    ref_o, ref_l = [t.clone() for t in dw.attend()]
    torch.cuda.synchronize()
    o_ref, l_ref = O.attention(q_values(W), oracle_pool(W), W.page_table, W.context_lens,
                               W.block_lens, W.spec.num_kv_heads, float(W.sm_scale))
    for _ in range(2):           # two calls in a row share the scratch
        out = torch.full_like(dw.out, float("nan"))
        lse = torch.full_like(dw.lse, float("nan"))
        _fixed(dw, out, lse)
        torch.cuda.synchronize()
        # both entry points plan one tensor-core CTA per SM: same split, same bits
        assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
        assert_parity(out, lse, o_ref, l_ref, what="fixed scratch")
    assert int(dw.status.item()) == 0


def test_fixed_scratch_rejects_shapes_beyond_its_size():
    W = wl.custom(32, 4, 256, [300], [16], seed=42)     # T*G = 128 rows at D = 256
    dw = DeviceWorkload(W)
    out, lse = torch.empty_like(dw.out), torch.empty_like(dw.lse)
    with pytest.raises(sk.SplashError) as e:
        _fixed(dw, out, lse)
    assert e.value.status == -3
    assert sk.LIB.splash_verify_attention_fixed_scratch_bytes() == 64 << 20
