"""The five seeded workloads at full size, every sequence, against the fp64
oracle (through the C ABI).

Each sequence's cached K/V is drawn once and appended both to the GPU pool
(splash_kv_append) and to the oracle's pool (its own quantiser); then the
verify block is appended to both and attention runs on the GPU. Checked:
int8 codes and fp32 scales of every written slot bit for bit, and O / LSE of
every verify row within max-abs 1e-2 / mean-abs 1e-3 / LSE 1e-3. Slack pages
and the unwritten tail slots of last pages keep their poison (codes +-127,
scales NaN / inf), so any read of them would show in the outputs.
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
from speculative_verify_attention_kv_gb300.device_workload import DeviceWorkload  # noqa: E402

from common import q_values  # noqa: E402
from gpu_common import assert_parity  # noqa: E402


def _stack(pairs):
    ks, vs = zip(*pairs)
    return np.stack(ks, axis=1), np.stack(vs, axis=1)


def populate_both(W, dw, opool, chunk=16384):
    """Cached context of every sequence into both pools (a shared prefix once,
    through sequence 0's page list)."""
    H = W.spec.num_kv_heads

    def both(k, v, b, start):
        O.kv_append(opool, k, v, W.page_table[b:b + 1], np.array([start]), np.array([k.shape[0]]))
        for c0 in range(0, k.shape[0], chunk):
            dw._append(k[c0:c0 + chunk], v[c0:c0 + chunk], b, start + c0)

    if W.prefix_len:
        k, v = _stack([W.prefix_kv(h) for h in range(H)])
        both(k, v, 0, 0)
    for b in range(W.num_seqs):
        k, v = _stack([W.private_context_kv(b, h) for h in range(H)])
        if k.shape[0]:
            both(k, v, b, W.prefix_len)
    torch.cuda.synchronize()


def assert_written_slots_equal(W, dw, opool):
    kp, vp, ks, vs = dw.pool
    for b in range(W.num_seqs):
        j = np.arange(int(W.context_lens[b] + W.block_lens[b]))
        pg = W.page_table[b][j // 16].astype(np.int64)
        sl = j % 16
        pg_t, sl_t = torch.from_numpy(pg).cuda(), torch.from_numpy(sl).cuda()
        assert np.array_equal(kp[pg_t, :, sl_t].cpu().numpy(), opool.k_codes[pg, :, sl]), b
        assert np.array_equal(vp[pg_t, :, sl_t].cpu().numpy(), opool.v_codes[pg, :, sl]), b
        assert np.array_equal(ks[pg_t, :, sl_t].cpu().numpy().view(np.uint32),
                              opool.k_scales[pg, :, sl].view(np.uint32)), b
        assert np.array_equal(vs[pg_t, :, sl_t].cpu().numpy().view(np.uint32),
                              opool.v_scales[pg, :, sl].view(np.uint32)), b


@pytest.mark.parametrize("name", [s.name for s in wl.SPECS])
def test_workload_every_sequence_matches_the_oracle(name):
    W = wl.make(name)
    s = W.spec
    dw = DeviceWorkload(W, populate=False)
    opool = O.PagedPool(W.num_pages, s.num_kv_heads, s.page_size, s.head_dim)
    populate_both(W, dw, opool)
    assert int(dw.status.item()) == 0
    dw.append_block()
    bk, bv = W.block_kv()
    O.kv_append(opool, bk, bv, W.page_table, W.context_lens, W.block_lens)
    torch.cuda.synchronize()
    assert int(dw.status.item()) == 0
    assert_written_slots_equal(W, dw, opool)

    o_ref, l_ref = O.attention(q_values(W), opool, W.page_table, W.context_lens, W.block_lens,
                               s.num_kv_heads, float(W.sm_scale))
    rows_per_unit = int(W.block_lens.max()) * s.group
    # (path, stack): a shared prefix goes through the shared-prefix entry
    # point (stacked rows) by default; it is also checked without stacking
    runs = [(sk.PATH_AUTO, True)]
    if W.prefix_len:
        runs.append((sk.PATH_AUTO, False))
    if s.head_dim == 256 and rows_per_unit <= 96:
        runs.append((sk.PATH_TENSOR_T, True))
    for path, stack in runs:
        out = torch.full_like(dw.out, float("nan"))
        lse = torch.full_like(dw.lse, float("nan"))
        dw.attend(path=path, out=out, lse=lse, stack=stack)
        torch.cuda.synchronize()
        assert int(dw.status.item()) == 0
        assert_parity(out, lse, o_ref, l_ref, what=f"{name} path {path} stack {stack}")
