"""Host-only checks of the C ABI: the library builds, loads and exports every
symbol the header declares; argument errors come back before any launch."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "splash_kv.h")


@pytest.fixture(scope="module")
def sk():
    from speculative_verify_attention_kv_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    from speculative_verify_attention_kv_gb300 import splash_kv
    return splash_kv


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(splash_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("splash_kv_append", "splash_verify_attention",
              "splash_verify_attention_workspace_size", "splash_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(sk):
    lib = ctypes.CDLL(sk._LIB_PATH)
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(declared_functions()) <= set(sk.EXPORTED) | {"splash_abi_version"}


def test_status_strings(sk):
    assert sk.status_string(0) == "SPLASH_OK"
    assert sk.status_string(-1) == "SPLASH_ERR_INVALID_ARGUMENT"
    assert sk.status_string(-2) == "SPLASH_ERR_UNSUPPORTED"
    assert sk.status_string(-3) == "SPLASH_ERR_WORKSPACE_TOO_SMALL"
    assert sk.status_string(-4) == "SPLASH_ERR_CUDA"
    assert sk.status_string(12345) == "SPLASH_UNKNOWN_STATUS"
    assert sk.LIB.splash_abi_version() == 2


def test_wait_limit_setter_round_trips(sk):
    prev = sk.splash_set_wait_limit_ns(12345)
    try:
        assert prev == 10 ** 9
        assert sk.splash_set_wait_limit_ns(0) == 12345      # 0 restores the default
        assert sk.splash_set_wait_limit_ns(0) == 10 ** 9
    finally:
        sk.splash_set_wait_limit_ns(0)


FAKE = ctypes.c_void_p(256)  # never dereferenced: validation fails first
FAKE_V = ctypes.c_void_p(256 + 16 * 128)   # V half of the code pool at D = 128: K + P*D


def _append(sk, **kw):
    a = dict(k=FAKE, v=FAKE, n=4, kp=FAKE, vp=FAKE_V, ks=FAKE, vs=FAKE, tab=FAKE, maxp=4,
             ctx=FAKE, T=FAKE, B=1, hkv=2, D=128, P=16, pages=8, st=None, stream=None)
    a.update(kw)
    return sk.LIB.splash_kv_append(a["k"], a["v"], a["n"], a["kp"], a["vp"], a["ks"], a["vs"],
                                   a["tab"], a["maxp"], a["ctx"], a["T"], a["B"], a["hkv"],
                                   a["D"], a["P"], a["pages"], a["st"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(P=8), -2), (dict(D=96), -2), (dict(D=512), -2), (dict(hkv=0), -1), (dict(n=-1), -1),
    (dict(B=-2), -1), (dict(maxp=0), -1), (dict(k=None), -1), (dict(tab=None), -1),
    (dict(vs=None), -1), (dict(n=0), 0), (dict(B=0), 0),
    (dict(vp=FAKE), -1),              # V codes not at K + P*D of one pool
])
def test_kv_append_argument_errors(sk, kw, code):
    assert _append(sk, **kw) == code


def _attn(sk, **kw):
    a = dict(q=FAKE, n=4, kp=FAKE, vp=FAKE_V, ks=FAKE, vs=FAKE, tab=FAKE, maxp=4, ctx=FAKE,
             T=FAKE, B=1, hq=8, hkv=2, D=128, P=16, pages=8, maxT=4, sm=0.088, out=FAKE,
             lse=FAKE, ws=FAKE, wsb=1 << 30, st=None, stream=None, path=0, ctas=0)
    a.update(kw)
    args = [a[k] for k in ("q", "n", "kp", "vp", "ks", "vs", "tab", "maxp", "ctx", "T", "B", "hq",
                           "hkv", "D", "P", "pages", "maxT", "sm", "out", "lse", "ws", "wsb",
                           "st", "stream")]
    return sk.LIB.splash_verify_attention_tuned(*args, a["path"], a["ctas"])


@pytest.mark.parametrize("kw,code", [
    (dict(hq=7), -1), (dict(hkv=0), -1), (dict(D=100), -2), (dict(P=32), -2),
    (dict(maxT=40), -2),              # T*G = 160 > 128 rows
    (dict(maxT=-1), -1), (dict(n=-3), -1), (dict(maxp=0), -1), (dict(path=4), -1),
    (dict(path=3), -2),               # the transposed kernel takes head_dim 256 only
    (dict(ctas=-1), -1), (dict(q=None), -1), (dict(ws=None), -1), (dict(lse=None), -1),
    (dict(ws=ctypes.c_void_p(256 + 16)), -1),   # workspace not 256-byte aligned
    (dict(n=0), 0), (dict(B=0), 0),
    (dict(vp=FAKE), -1),              # V codes not at K + P*D of one pool
])
def test_verify_attention_argument_errors(sk, kw, code):
    assert _attn(sk, **kw) == code


def test_workspace_query_rejects_bad_shapes(sk):
    f = sk.LIB.splash_verify_attention_workspace_size
    assert f(1, 4, 7, 2, 128, 4) == 0
    assert f(1, 4, 8, 2, 100, 4) == 0
    assert f(1, 4, 8, 2, 128, 64) == 0


def _accept(sk, **kw):
    a = dict(x=FAKE, y=FAKE, n=8, T=FAKE, ctx=FAKE, acc=FAKE, nxt=FAKE, B=2, st=None, stream=None)
    a.update(kw)
    return sk.LIB.splash_accept_commit(a["x"], a["y"], a["n"], a["T"], a["ctx"], a["acc"],
                                       a["nxt"], a["B"], a["st"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(n=-1), -1), (dict(B=-1), -1), (dict(T=None), -1), (dict(ctx=None), -1),
    (dict(acc=None), -1), (dict(nxt=None), -1), (dict(x=None), -1), (dict(y=None), -1),
    (dict(B=0), 0),                   # nothing to do
])
def test_accept_commit_argument_errors(sk, kw, code):
    assert _accept(sk, **kw) == code


def test_sliding_window_argument_errors(sk):
    a = dict(q=FAKE, n=4, kp=FAKE, vp=FAKE_V, ks=FAKE, vs=FAKE, tab=FAKE, maxp=4, ctx=FAKE,
             T=FAKE, B=1, hq=8, hkv=2, D=128, P=16, pages=8, maxT=4, sm=0.088)
    args = [a[k] for k in ("q", "n", "kp", "vp", "ks", "vs", "tab", "maxp", "ctx", "T", "B", "hq",
                           "hkv", "D", "P", "pages", "maxT", "sm")]
    tail = [FAKE, FAKE, FAKE, 1 << 30, None, None, 0, 0]
    f = sk.LIB.splash_verify_attention_swa
    assert f(*args, -1, *tail) == -1                      # negative window
    assert f(*args, 5, FAKE, FAKE, FAKE, 1 << 30, None, None, 4, 0) == -1   # bad path
    args_bad_pool = list(args)
    args_bad_pool[3] = FAKE                                # V codes not at K + P*D
    assert f(*args_bad_pool, 5, *tail) == -1


def _attn_shared(sk, **kw):
    a = dict(q=FAKE, n=4, kp=FAKE, vp=FAKE_V, ks=FAKE, vs=FAKE, tab=FAKE, maxp=4, ctx=FAKE,
             T=FAKE, sl=FAKE, B=1, hq=8, hkv=2, D=128, P=16, pages=8, maxT=4, sm=0.088, out=FAKE,
             lse=FAKE, ws=FAKE, wsb=1 << 30, st=None, stream=None, path=0, ctas=0)
    a.update(kw)
    args = [a[k] for k in ("q", "n", "kp", "vp", "ks", "vs", "tab", "maxp", "ctx", "T", "sl", "B",
                           "hq", "hkv", "D", "P", "pages", "maxT", "sm", "out", "lse", "ws", "wsb",
                           "st", "stream")]
    return sk.LIB.splash_verify_attention_shared_profiled(*args, a["path"], a["ctas"], None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(sl=None), -1),              # the shared-prefix entry point needs shared_lens
    (dict(hq=7), -1), (dict(D=100), -2), (dict(P=32), -2), (dict(maxT=40), -2),
    (dict(path=4), -1), (dict(ctas=-1), -1), (dict(q=None), -1), (dict(ws=None), -1),
    (dict(ws=ctypes.c_void_p(256 + 16)), -1), (dict(vp=FAKE), -1),
    (dict(n=0), 0), (dict(B=0), 0), (dict(n=0, sl=None), 0),
])
def test_shared_prefix_argument_errors(sk, kw, code):
    assert _attn_shared(sk, **kw) == code


def test_shared_workspace_query_rejects_bad_shapes(sk):
    f = sk.LIB.splash_verify_attention_shared_workspace_size
    assert f(1, 4, 7, 2, 128, 4) == 0
    assert f(1, 4, 8, 2, 100, 4) == 0
    assert f(1, 4, 8, 2, 128, 64) == 0
