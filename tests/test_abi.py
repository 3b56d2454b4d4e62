"""The C-ABI library: it loads, exports every declared entry point, and rejects bad
arguments on the host before any launch (CPU only: no call here reaches a kernel)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def clib():
    lib_path = os.path.join(ROOT, "mla_flash_attention_gb300", "libmla_gb300.so")
    if not os.path.exists(lib_path):
        from mla_flash_attention_gb300 import build

        build.build()
    return ctypes.CDLL(lib_path)


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(mla_\w+)\s*\(", src, re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("mla_prefill", "mla_decode", "mla_decode_workspace_size", "mla_check_device_error",
              "mla_last_error", "mla_version"):
        assert n in names


def test_every_declared_symbol_is_exported(clib):
    for n in declared_functions():
        assert hasattr(clib, n), n


def _prefill(clib, **kw):
    a = dict(q_nope=16, q_rope=16, k_nope=16, k_rope=16, v=16, q_scale=None, k_scale=None,
             out=16, lse=16, B=1, H=1, S=1, dn=128, dr=64, dv=128, scale=0.1, causal=1, dt=0,
             odt=0)
    a.update(kw)
    f = clib.mla_prefill
    f.restype = ctypes.c_int
    P = ctypes.c_void_p
    return f(P(a["q_nope"]), P(a["q_rope"]), P(a["k_nope"]), P(a["k_rope"]), P(a["v"]),
             P(a["q_scale"]), P(a["k_scale"]), P(a["out"]), P(a["lse"]), a["B"], a["H"], a["S"],
             a["dn"], a["dr"], a["dv"], ctypes.c_float(a["scale"]), a["causal"], a["dt"],
             a["odt"], None)


def test_prefill_argument_checks(clib):
    # every case below is rejected before any CUDA call (pointers are never dereferenced)
    assert _prefill(clib, q_nope=None) == 1
    assert _prefill(clib, S=0) == 1
    assert _prefill(clib, B=-1) == 1
    assert _prefill(clib, dn=64) == 2
    assert _prefill(clib, dv=512) == 2
    assert _prefill(clib, dt=7) == 2
    assert _prefill(clib, odt=1) == 2
    assert _prefill(clib, dt=1) == 1           # fp8 without scales
    assert _prefill(clib, q_scale=16) == 1     # bf16 with scales
    assert _prefill(clib, q_rope=24) == 1      # misaligned
    assert _prefill(clib, scale=float("nan")) == 1
    clib.mla_last_error.restype = ctypes.c_char_p
    assert b"softmax_scale" in clib.mla_last_error()


def test_prefill_size_limits(clib):
    # the largest sizes the kernels index are enforced on the host (MLA_ERR_UNSUPPORTED)
    assert _prefill(clib, B=65536) == 2
    assert _prefill(clib, H=65536) == 2
    assert _prefill(clib, B=65535, H=65535, S=2**31 - 1) == 2   # B*S*H*128 beyond int64 indexing
    clib.mla_last_error.restype = ctypes.c_char_p
    assert b"too large" in clib.mla_last_error()


def _decode(clib, **kw):
    a = dict(ql=16, qr=16, cache=16, ks=None, pt=16, lens=16, out=16, lse=16, B=1, H=16, T=1,
             dl=512, dr=64, ps=64, mp=1, npages=1, scale=0.1, causal=1, dt=0, ws=None, wsb=0)
    a.update(kw)
    f = clib.mla_decode
    f.restype = ctypes.c_int
    P = ctypes.c_void_p
    return f(P(a["ql"]), P(a["qr"]), P(a["cache"]), P(a["ks"]), P(a["pt"]), P(a["lens"]),
             P(a["out"]), P(a["lse"]), a["B"], a["H"], a["T"], a["dl"], a["dr"], a["ps"], a["mp"],
             a["npages"], ctypes.c_float(a["scale"]), a["causal"], a["dt"], P(a["ws"]),
             ctypes.c_size_t(a["wsb"]), None)


def test_decode_argument_checks(clib):
    assert _decode(clib, ql=None) == 1
    assert _decode(clib, B=0) == 1
    assert _decode(clib, dl=256) == 2
    assert _decode(clib, ps=32) == 2
    assert _decode(clib, H=128, T=513) == 2    # more than 65536 query rows per sequence
    assert _decode(clib, dt=1) == 1            # fp8 without scales
    assert _decode(clib, ks=16) == 1           # bf16 with scales
    assert _decode(clib, out=8) == 1           # misaligned
    assert _decode(clib, npages=0) == 1


def test_decode_size_limits(clib):
    assert _decode(clib, B=65536, H=1) == 2                 # one work item per sequence: B <= 65535
    assert _decode(clib, B=65535, H=128, T=512) == 2        # B * 512 query tiles > 2^24
    assert _decode(clib, mp=2**26) == 2                     # max_pages * 64 overflows int32
    clib.mla_last_error.restype = ctypes.c_char_p
    assert b"overflows" in clib.mla_last_error()


def _backward(clib, **kw):
    names = ("qn", "qr", "kn", "kr", "v", "out", "lse", "do", "dqn", "dqr", "dkn", "dkr", "dv")
    a = {n: 16 for n in names}
    a.update(B=1, H=1, S=1, dn=128, dr=64, dvd=128, scale=0.1, causal=1, ws=None, wsb=0)
    a.update(kw)
    f = clib.mla_prefill_backward
    f.restype = ctypes.c_int
    P = ctypes.c_void_p
    return f(*[P(a[n]) for n in names], a["B"], a["H"], a["S"], a["dn"], a["dr"], a["dvd"],
             ctypes.c_float(a["scale"]), a["causal"], P(a["ws"]), ctypes.c_size_t(a["wsb"]), None)


def test_backward_argument_checks(clib):
    clib.mla_prefill_backward_workspace_size.restype = ctypes.c_size_t
    need = clib.mla_prefill_backward_workspace_size(2, 3, 300)
    assert need == 2 * ((2 * 3 * 384 * 4 + 255) // 256 * 256)
    assert clib.mla_prefill_backward_workspace_size(0, 3, 300) == 0
    assert _backward(clib, do=None) == 1
    assert _backward(clib, dkr=None) == 1
    assert _backward(clib, S=0) == 1
    assert _backward(clib, dn=64) == 2
    assert _backward(clib, dvd=512) == 2
    assert _backward(clib, dqr=40) == 1          # misaligned
    assert _backward(clib, scale=-1.0) == 1
    assert _backward(clib) == 3                  # no workspace
    assert _backward(clib, ws=16, wsb=100) == 3  # workspace too small


def test_absorb_argument_checks(clib):
    f = clib.mla_absorb
    f.restype = ctypes.c_int
    P = ctypes.c_void_p

    def call(x=16, w=16, y=16, R=4, H=2, K=64, N=128):
        return f(P(x), P(w), P(y), R, H, K, N, None)

    assert call(x=None) == 1
    assert call(R=0) == 1
    assert call(K=96) == 2           # K must be a multiple of 64
    assert call(N=64) == 2           # N must be a multiple of 128
    assert call(y=24) == 1           # misaligned
    assert call(H=70000) == 2


def test_cache_append_argument_checks(clib):
    f = clib.mla_cache_append
    f.restype = ctypes.c_int
    P = ctypes.c_void_p

    def call(c=16, cache=16, scale=None, pt=16, lens=16, B=1, T=1, dl=512, dr=64, ps=64, mp=1,
             npages=1, dt=0):
        return f(P(c), P(cache), P(scale), P(pt), P(lens), B, T, dl, dr, ps, mp, npages, dt, None)

    assert call(c=None) == 1
    assert call(B=0) == 1
    assert call(dl=256) == 2
    assert call(ps=32) == 2
    assert call(dt=1) == 1           # fp8 cache without scales
    assert call(scale=16) == 1       # bf16 cache with scales
    assert call(dt=1, scale=18) == 1  # scales not 4-byte aligned
    assert call(cache=40) == 1       # misaligned
    assert call(dt=5) == 2


def test_normal_build_has_no_bounds_checks(clib):
    # the device-side store checks exist only in the bounds-checked build (MLA_DEBUG)
    clib.mla_testing_bounds_checked.restype = ctypes.c_int
    assert clib.mla_testing_bounds_checked() == 0
