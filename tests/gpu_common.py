"""GPU-side helpers for the parity tests: build a poisoned pool, populate it
through the library's append, run attention through the C ABI."""
from __future__ import annotations

import numpy as np
import torch

from speculative_verify_attention_kv_gb300 import splash_kv as sk
from speculative_verify_attention_kv_gb300 import workloads as wl

from speculative_verify_attention_kv_gb300.device_workload import DeviceWorkload

class Run(DeviceWorkload):
    """A DeviceWorkload (tests keep the historical name)."""


def compare(o_gpu, lse_gpu, o_ref, lse_ref, rows=None):
    """Max/mean abs error of bf16 O and fp32 LSE against the fp64 oracle."""
    o = o_gpu.float().cpu().numpy().astype(np.float64)
    l = lse_gpu.cpu().numpy().astype(np.float64)
    if rows is not None:
        o, l, o_ref, lse_ref = o[rows], l[rows], o_ref[rows], lse_ref[rows]
    err = np.abs(o - o_ref)
    return float(err.max()), float(err.mean()), float(np.abs(l - lse_ref).max())


MAX_ABS, MEAN_ABS, LSE_ABS = 1e-2, 1e-3, 1e-3


def assert_parity(o_gpu, lse_gpu, o_ref, lse_ref, rows=None, what=""):
    mx, mean, le = compare(o_gpu, lse_gpu, o_ref, lse_ref, rows)
    assert np.isfinite(mx) and mx <= MAX_ABS, f"{what} max-abs {mx}"
    assert mean <= MEAN_ABS, f"{what} mean-abs {mean}"
    assert np.isfinite(le) and le <= LSE_ABS, f"{what} lse {le}"
    return mx, mean, le


# Bound for rows that see only a few keys (small sliding windows): O is then
# close to a single dequantised v, |O| can reach |v| ~ 6 on these inputs, and
# two roundings scale with |O|: bf16 output (half an ulp, 2^-9 relative) and
# the fp16 rounding of P * sV fed to the tensor cores (2^-11 relative).
REL_O = 2.0 ** -9 + 2.0 ** -11


def assert_parity_scaled(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """Elementwise |O - O_ref| <= MAX_ABS + REL_O * |O_ref| (and its mean for the
    mean error); LSE as usual."""
    o = o_gpu.float().cpu().numpy().astype(np.float64)
    l = lse_gpu.cpu().numpy().astype(np.float64)
    err = np.abs(o - o_ref)
    excess = err - (MAX_ABS + REL_O * np.abs(o_ref))
    assert np.all(np.isfinite(err)) and float(excess.max()) <= 0, \
        f"{what} max-abs {float(err.max())} (scaled bound exceeded by {float(excess.max())})"
    # the mean of the same bound
    mean_bound = MEAN_ABS + REL_O * float(np.abs(o_ref).mean())
    assert float(err.mean()) <= mean_bound, f"{what} mean-abs {float(err.mean())} > {mean_bound}"
    le = float(np.abs(l - lse_ref).max())
    assert np.isfinite(le) and le <= LSE_ABS, f"{what} lse {le}"
