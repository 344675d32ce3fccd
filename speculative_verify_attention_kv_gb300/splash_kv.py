"""Python binding of ``libsplashkv.so`` (ctypes; argument marshalling only).

The functions carry the C names. Tensors are torch CUDA tensors; the binding
checks dtype, device, shape and contiguity, passes raw device pointers and the
current CUDA stream, and raises :class:`SplashError` on a non-zero status. All
computation happens in the library's CUDA kernels: there is no fallback, and
importing this module fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsplashkv.so")

PAGE_SIZE = 16
DEVICE_BAD_PAGE = 1
DEVICE_BAD_LENGTH = 2
DEVICE_TIMEOUT = 3
PATH_AUTO, PATH_SIMT, PATH_TENSOR, PATH_TENSOR_T = 0, 1, 2, 3
# PATH_TENSOR: tensor-core kernel with the query rows on the MMA's M side (any
# head_dim of 128 / 256, up to 128 rows); PATH_TENSOR_T: the transposed kernel
# (keys on M, rows on N; head_dim 256, up to 96 rows per unit), which automatic
# mode picks whenever it applies


class SplashError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is missing: build it with speculative_verify_attention_kv_gb300.build.build()"
            " (there is no non-CUDA implementation)")
    lib = ctypes.CDLL(_LIB_PATH)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.splash_status_string.restype = ctypes.c_char_p
    lib.splash_status_string.argtypes = [I]
    lib.splash_abi_version.restype = I
    lib.splash_tensor_path_supported.restype = I
    lib.splash_tensor_path_supported.argtypes = [I]
    lib.splash_launch_count.restype = ctypes.c_ulonglong
    lib.splash_launch_count.argtypes = []
    lib.splash_set_wait_limit_ns.restype = ctypes.c_ulonglong
    lib.splash_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.splash_kv_append.restype = I
    lib.splash_kv_append.argtypes = [P, P, I, P, P, P, P, P, I, P, P, I, I, I, I, I, P, P]
    lib.splash_kv_append_bf16.restype = I
    lib.splash_kv_append_bf16.argtypes = [P, P, I, P, P, P, P, P, I, P, P, I, I, I, I, I, P, P]
    lib.splash_accept_commit.restype = I
    lib.splash_accept_commit.argtypes = [P, P, I, P, P, P, P, I, P, P]
    lib.splash_verify_attention_workspace_size.restype = S
    lib.splash_verify_attention_workspace_size.argtypes = [I, I, I, I, I, I]
    attn = [P, I, P, P, P, P, P, I, P, P, I, I, I, I, I, I, I, F, P, P, P, S, P, P]
    lib.splash_verify_attention.restype = I
    lib.splash_verify_attention.argtypes = attn
    lib.splash_verify_attention_tuned.restype = I
    lib.splash_verify_attention_tuned.argtypes = attn + [I, I]
    lib.splash_verify_attention_swa.restype = I
    lib.splash_verify_attention_swa.argtypes = attn[:18] + [I] + attn[18:] + [I, I]
    lib.splash_verify_attention_profiled.restype = I
    lib.splash_verify_attention_profiled.argtypes = attn + [I, I, P, P]
    lib.splash_verify_attention_shared_workspace_size.restype = S
    lib.splash_verify_attention_shared_workspace_size.argtypes = [I, I, I, I, I, I]
    # shared_lens follows block_lens
    attn_sh = attn[:10] + [P] + attn[10:]
    lib.splash_verify_attention_shared.restype = I
    lib.splash_verify_attention_shared.argtypes = attn_sh
    lib.splash_verify_attention_shared_profiled.restype = I
    lib.splash_verify_attention_shared_profiled.argtypes = attn_sh + [I, I, P, P]
    lib.splash_verify_attention_fixed_scratch_bytes.restype = S
    lib.splash_verify_attention_fixed_scratch_bytes.argtypes = []
    lib.splash_verify_attention_fixed_scratch.restype = I
    lib.splash_verify_attention_fixed_scratch.argtypes = attn[:20] + [P, P]
    return lib


LIB = _load()
EXPORTED = ("splash_status_string", "splash_abi_version", "splash_tensor_path_supported",
            "splash_set_wait_limit_ns", "splash_launch_count",
            "splash_kv_append", "splash_kv_append_bf16", "splash_accept_commit",
            "splash_verify_attention_swa",
            "splash_verify_attention_workspace_size", "splash_verify_attention",
            "splash_verify_attention_tuned", "splash_verify_attention_profiled",
            "splash_verify_attention_shared_workspace_size", "splash_verify_attention_shared",
            "splash_verify_attention_shared_profiled",
            "splash_verify_attention_fixed_scratch_bytes", "splash_verify_attention_fixed_scratch")


def tensor_path_available(head_dim: int) -> bool:
    return bool(LIB.splash_tensor_path_supported(int(head_dim)))


def splash_launch_count() -> int:
    """Kernels the library has enqueued since it was loaded."""
    return int(LIB.splash_launch_count())


def splash_set_wait_limit_ns(ns: int) -> int:
    """Limit of each internal wait of the tensor-core kernel for later launches
    (0 = the default of 1 s); returns the previous limit."""
    return int(LIB.splash_set_wait_limit_ns(int(ns)))


def status_string(status: int) -> str:
    return LIB.splash_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t: torch.Tensor, name: str, dtype, ndim: int | None = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim} dims, got {t.dim()}")


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def alloc_pool(num_pages: int, num_kv_heads: int, head_dim: int, device="cuda"):
    """Zeroed paged pool in the library's layout: (k_pages, v_pages, k_scales,
    v_scales). The codes are one allocation [num_pages, Hkv, 2, P, D]; k_pages
    and v_pages are its [:, :, 0] and [:, :, 1] views ([num_pages, Hkv, P, D]
    each, K and V codes of a (page, KV head) adjacent)."""
    codes = torch.zeros((num_pages, num_kv_heads, 2, PAGE_SIZE, head_dim), dtype=torch.int8,
                        device=device)
    scales = (num_pages, num_kv_heads, PAGE_SIZE)
    return (codes[:, :, 0], codes[:, :, 1],
            torch.zeros(scales, dtype=torch.float32, device=device),
            torch.zeros(scales, dtype=torch.float32, device=device))


def _check_pool(k_pages, v_pages):
    """k_pages / v_pages: the two halves of one [num_pages, Hkv, 2, P, D] code pool."""
    for n, t in (("k_pages", k_pages), ("v_pages", v_pages)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.int8 or not t.is_cuda or t.dim() != 4:
            raise TypeError(f"{n} must be a 4-D int8 CUDA tensor")
    num_pages, hkv, P, D = k_pages.shape
    want = (hkv * 2 * P * D, 2 * P * D, D, 1)
    if tuple(v_pages.shape) != tuple(k_pages.shape) or tuple(k_pages.stride()) != want \
            or tuple(v_pages.stride()) != want \
            or v_pages.data_ptr() != k_pages.data_ptr() + P * D:
        raise ValueError("k_pages / v_pages must be the [:, :, 0] / [:, :, 1] views of one "
                         "[num_pages, Hkv, 2, P, D] pool (see alloc_pool)")


def splash_kv_append(k_new, v_new, k_pages, v_pages, k_scales, v_scales, page_table,
                     context_lens, block_lens, device_status=None, stream=None) -> None:
    """k_new / v_new: float32 (splash_kv_append) or bfloat16 (splash_kv_append_bf16)."""
    if k_new.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("k_new must be float32 or bfloat16")
    _check(k_new, "k_new", k_new.dtype, 3)
    _check(v_new, "v_new", k_new.dtype, 3)
    _check_pool(k_pages, v_pages)
    for n, t in (("k_scales", k_scales), ("v_scales", v_scales)):
        _check(t, n, torch.float32, 3)
    _check(page_table, "page_table", torch.int32, 2)
    _check(context_lens, "context_lens", torch.int32, 1)
    _check(block_lens, "block_lens", torch.int32, 1)
    if device_status is not None:
        _check(device_status, "device_status", torch.int32)
    num_pages, hkv, P, D = k_pages.shape
    if tuple(v_pages.shape) != (num_pages, hkv, P, D) or tuple(k_new.shape[1:]) != (hkv, D) \
            or k_new.shape != v_new.shape:
        raise ValueError("shape mismatch between k_new/v_new and the pool")
    fn = LIB.splash_kv_append if k_new.dtype == torch.float32 else LIB.splash_kv_append_bf16
    st = fn(
        _ptr(k_new), _ptr(v_new), k_new.shape[0], _ptr(k_pages), _ptr(v_pages), _ptr(k_scales),
        _ptr(v_scales), _ptr(page_table), page_table.shape[1], _ptr(context_lens),
        _ptr(block_lens), context_lens.shape[0], hkv, D, P, num_pages, _ptr(device_status),
        _stream(stream))
    if st != 0:
        raise SplashError(st, "splash_kv_append")


def splash_accept_commit(block_tokens, target_tokens, block_lens, context_lens, accepted,
                         next_tokens, device_status=None, stream=None) -> None:
    """Advance context_lens (in place) by the accepted drafts plus one."""
    for n, t in (("block_tokens", block_tokens), ("target_tokens", target_tokens),
                 ("block_lens", block_lens), ("context_lens", context_lens),
                 ("accepted", accepted), ("next_tokens", next_tokens)):
        _check(t, n, torch.int32, 1)
    if device_status is not None:
        _check(device_status, "device_status", torch.int32)
    B = block_lens.shape[0]
    if context_lens.shape[0] != B or accepted.shape[0] != B or next_tokens.shape[0] != B \
            or target_tokens.shape != block_tokens.shape:
        raise ValueError("shape mismatch")
    st = LIB.splash_accept_commit(_ptr(block_tokens), _ptr(target_tokens), block_tokens.shape[0],
                                  _ptr(block_lens), _ptr(context_lens), _ptr(accepted),
                                  _ptr(next_tokens), B, _ptr(device_status), _stream(stream))
    if st != 0:
        raise SplashError(st, "splash_accept_commit")


def splash_verify_attention_workspace_size(num_seqs: int, num_q_tokens: int, num_q_heads: int,
                                           num_kv_heads: int, head_dim: int,
                                           max_block_len: int) -> int:
    return int(LIB.splash_verify_attention_workspace_size(
        num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, max_block_len))


def splash_verify_attention_shared_workspace_size(num_seqs: int, num_q_tokens: int,
                                                  num_q_heads: int, num_kv_heads: int,
                                                  head_dim: int, max_block_len: int) -> int:
    return int(LIB.splash_verify_attention_shared_workspace_size(
        num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, max_block_len))


def alloc_workspace(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, max_block_len,
                    device="cuda", ctas_per_class: int = 0, shared: bool = False) -> torch.Tensor:
    """Workspace for splash_verify_attention (``shared``: for the shared-prefix
    entry point)."""
    query = (splash_verify_attention_shared_workspace_size if shared
             else splash_verify_attention_workspace_size)
    n = query(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, max_block_len)
    if n == 0:
        raise ValueError("invalid shape for the workspace size query")
    if ctas_per_class > 0:   # a fixed CTA count may need more partial rows than the default
        rows = max_block_len * (num_q_heads // num_kv_heads)
        if shared:
            rows = max(rows, 128)
        n += 2 * rows * 2 * ctas_per_class * (head_dim + 1) * 4
    return torch.empty(n, dtype=torch.uint8, device=device)


def splash_verify_attention(q, k_pages, v_pages, k_scales, v_scales, page_table, context_lens,
                            block_lens, sm_scale: float, max_block_len: int, out, lse, workspace,
                            device_status=None, stream=None, path: int = PATH_AUTO,
                            ctas_per_class: int = 0, events=None, window: int = 0,
                            shared_lens=None) -> None:
    """``events``: optional (begin, end) torch.cuda.Event pair recorded around
    the attention kernels (the profiled entry point). ``window`` > 0: sliding
    window of that many keys (splash_verify_attention_swa). ``shared_lens``:
    int32 [num_seqs], keys each sequence shares with the one before it
    (splash_verify_attention_shared; the workspace from
    ``alloc_workspace(..., shared=True)``)."""
    _check(q, "q", torch.bfloat16, 3)
    _check(out, "out", torch.bfloat16, 3)
    _check(lse, "lse", torch.float32, 2)
    _check_pool(k_pages, v_pages)
    for n, t in (("k_scales", k_scales), ("v_scales", v_scales)):
        _check(t, n, torch.float32, 3)
    _check(page_table, "page_table", torch.int32, 2)
    _check(context_lens, "context_lens", torch.int32, 1)
    _check(block_lens, "block_lens", torch.int32, 1)
    _check(workspace, "workspace", torch.uint8, 1)
    if device_status is not None:
        _check(device_status, "device_status", torch.int32)
    num_pages, hkv, P, D = k_pages.shape
    n_tok, hq, dq = q.shape
    if dq != D or tuple(out.shape) != tuple(q.shape) or tuple(lse.shape) != (n_tok, hq):
        raise ValueError("shape mismatch between q, out, lse and the pool")
    args = (_ptr(q), n_tok, _ptr(k_pages), _ptr(v_pages), _ptr(k_scales), _ptr(v_scales),
            _ptr(page_table), page_table.shape[1], _ptr(context_lens), _ptr(block_lens),
            context_lens.shape[0], hq, hkv, D, P, num_pages, int(max_block_len), float(sm_scale),
            _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), _ptr(device_status),
            _stream(stream))
    if shared_lens is not None:
        _check(shared_lens, "shared_lens", torch.int32, 1)
        if shared_lens.shape[0] != context_lens.shape[0]:
            raise ValueError("shared_lens must have one entry per sequence")
        if window != 0:
            raise ValueError("shared_lens is taken only without a window")
        ev = [None, None] if events is None else [
            ctypes.c_void_p(e.cuda_event) if e is not None else None for e in events]
        st = LIB.splash_verify_attention_shared_profiled(*args[:10], _ptr(shared_lens), *args[10:],
                                                         int(path), int(ctas_per_class), *ev)
    elif window != 0:
        if events is not None:
            raise ValueError("events are recorded only without a window")
        st = LIB.splash_verify_attention_swa(*args[:18], int(window), *args[18:], int(path),
                                             int(ctas_per_class))
    elif events is not None:
        ev = [ctypes.c_void_p(e.cuda_event) if e is not None else None for e in events]
        st = LIB.splash_verify_attention_profiled(*args, int(path), int(ctas_per_class), *ev)
    elif path == PATH_AUTO and ctas_per_class == 0:
        st = LIB.splash_verify_attention(*args)
    else:
        st = LIB.splash_verify_attention_tuned(*args, int(path), int(ctas_per_class))
    if st != 0:
        raise SplashError(st, "splash_verify_attention")


def splash_verify_attention_fixed_scratch(q, k_pages, v_pages, k_scales, v_scales, page_table,
                                          context_lens, block_lens, sm_scale: float,
                                          max_block_len: int, out, lse, device_status=None,
                                          stream=None) -> None:
    """splash_verify_attention with the library's fixed device scratch instead
    of a workspace (for callers that cannot allocate device memory)."""
    _check(q, "q", torch.bfloat16, 3)
    _check(out, "out", torch.bfloat16, 3)
    _check(lse, "lse", torch.float32, 2)
    _check_pool(k_pages, v_pages)
    for n, t in (("k_scales", k_scales), ("v_scales", v_scales)):
        _check(t, n, torch.float32, 3)
    _check(page_table, "page_table", torch.int32, 2)
    _check(context_lens, "context_lens", torch.int32, 1)
    _check(block_lens, "block_lens", torch.int32, 1)
    if device_status is not None:
        _check(device_status, "device_status", torch.int32)
    num_pages, hkv, P, D = k_pages.shape
    n_tok, hq, dq = q.shape
    if dq != D or tuple(out.shape) != tuple(q.shape) or tuple(lse.shape) != (n_tok, hq):
        raise ValueError("shape mismatch between q, out, lse and the pool")
    st = LIB.splash_verify_attention_fixed_scratch(
        _ptr(q), n_tok, _ptr(k_pages), _ptr(v_pages), _ptr(k_scales), _ptr(v_scales),
        _ptr(page_table), page_table.shape[1], _ptr(context_lens), _ptr(block_lens),
        context_lens.shape[0], hq, hkv, D, P, num_pages, int(max_block_len), float(sm_scale),
        _ptr(out), _ptr(lse), _ptr(device_status), _stream(stream))
    if st != 0:
        raise SplashError(st, "splash_verify_attention_fixed_scratch")
