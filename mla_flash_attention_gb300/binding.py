"""Thin ctypes binding of the C ABI (include/mla.h).

Argument marshalling only: torch tensors are checked for device, dtype, shape and
contiguity, then their device pointers and the current CUDA stream are passed to
the library.  Every step of the attention runs inside the library's CUDA kernels;
there is no fallback of any kind: if the shared library is missing, importing this
module raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

# MLA_GB300_LIB selects another build of the same library, e.g. the bounds-checked
# libmla_gb300_debug.so (mla_flash_attention_gb300.build.build(debug=True))
_LIB_PATH = os.environ.get("MLA_GB300_LIB") or os.path.join(
    os.path.dirname(os.path.abspath(__file__)), "libmla_gb300.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(
        "%s is not built; run `python -c 'import __graft_entry__ as g; g.build()'`" % _LIB_PATH)
_lib = ctypes.CDLL(_LIB_PATH)

MLA_OK = 0
MLA_BF16, MLA_FP8_E4M3, MLA_FP32 = 0, 1, 2
STATUS = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED", 3: "MLA_ERR_WORKSPACE",
          4: "MLA_ERR_CUDA", 5: "MLA_ERR_TIMEOUT", 6: "MLA_ERR_DEVICE_CHECK"}

_vp, _fp, _ip = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
_i, _f, _sz = ctypes.c_int, ctypes.c_float, ctypes.c_size_t

_lib.mla_prefill.restype = _i
_lib.mla_prefill.argtypes = [_vp, _vp, _vp, _vp, _vp, _fp, _fp, _vp, _fp, _i, _i, _i, _i, _i, _i,
                             _f, _i, _i, _i, _vp]
_lib.mla_decode_workspace_size.restype = _sz
_lib.mla_decode_workspace_size.argtypes = [_i, _i, _i, _i]
_lib.mla_decode.restype = _i
_lib.mla_decode.argtypes = [_vp, _vp, _vp, _fp, _ip, _ip, _vp, _fp, _i, _i, _i, _i, _i, _i, _i, _i,
                            _f, _i, _i, _vp, _sz, _vp]
_lib.mla_decode_noalloc.restype = _i
_lib.mla_decode_noalloc.argtypes = [_vp, _vp, _vp, _fp, _ip, _ip, _vp, _fp, _i, _i, _i, _i, _i, _i,
                                    _i, _i, _f, _i, _i, _vp]
_lib.mla_decode_noalloc_max_workspace.restype = _sz
_lib.mla_decode_noalloc_max_workspace.argtypes = []
_lib.mla_absorb.restype = _i
_lib.mla_absorb.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _vp]
_lib.mla_cache_append.restype = _i
_lib.mla_cache_append.argtypes = [_vp, _vp, _fp, _ip, _ip, _i, _i, _i, _i, _i, _i, _i, _i, _vp]
_lib.mla_prefill_backward_workspace_size.restype = _sz
_lib.mla_prefill_backward_workspace_size.argtypes = [_i, _i, _i]
_lib.mla_prefill_backward.restype = _i
_lib.mla_prefill_backward.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _fp, _vp, _vp, _vp, _vp, _fp,
                                      _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp]
_lib.mla_check_device_error.restype = _i
_lib.mla_check_device_error.argtypes = [_vp]
_lib.mla_last_error.restype = ctypes.c_char_p
_lib.mla_last_error.argtypes = []
_lib.mla_version.restype = _i
_lib.mla_version.argtypes = []
_lib.mla_testing_decode_stall.restype = None
_lib.mla_testing_decode_stall.argtypes = [_i, ctypes.c_longlong]
_lib.mla_testing_bounds_checked.restype = _i
_lib.mla_testing_bounds_checked.argtypes = []
_lib.mla_testing_bounds_shrink.restype = None
_lib.mla_testing_bounds_shrink.argtypes = [ctypes.c_longlong]

EXPORTED = ("mla_prefill", "mla_decode_workspace_size", "mla_decode", "mla_decode_noalloc",
            "mla_decode_noalloc_max_workspace", "mla_cache_append", "mla_absorb",
            "mla_prefill_backward_workspace_size", "mla_prefill_backward",
            "mla_check_device_error",
            "mla_last_error", "mla_version", "mla_testing_decode_stall", "mla_testing_bounds_checked",
            "mla_testing_bounds_shrink")


class MLAError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__("%s: %s" % (STATUS.get(status, status), msg))
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def _check(st: int):
    if st != MLA_OK:
        raise MLAError(st, _lib.mla_last_error().decode(errors="replace"))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype, shape):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must have dtype %s (got %s)" % (name, dtype, t.dtype))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s (got %s)" % (name, tuple(shape), tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def version() -> int:
    return _lib.mla_version()


def testing_decode_stall(skip_unit: int = -1, wait_limit_cycles: int = 0) -> None:
    """Test hook (include/mla_testing.h): later fp8 decode calls with q_len*H <= 32 leave
    pipeline unit `skip_unit` unloaded and give each device wait `wait_limit_cycles` SM clocks.
    ``testing_decode_stall()`` restores normal calls."""
    _lib.mla_testing_decode_stall(int(skip_unit), int(wait_limit_cycles))


def testing_bounds_checked() -> bool:
    """True when the loaded library is the bounds-checked build (include/mla_testing.h)."""
    return bool(_lib.mla_testing_bounds_checked())


def testing_bounds_shrink(nbytes: int = 0) -> None:
    """Test hook (include/mla_testing.h): later launches report `out` as `nbytes` smaller to
    the store checks of the bounds-checked build; ``testing_bounds_shrink()`` restores them."""
    _lib.mla_testing_bounds_shrink(int(nbytes))


def check_device_error(stream=None) -> None:
    _check(_lib.mla_check_device_error(_stream(stream)))


def mla_prefill(q_nope, q_rope, k_nope, k_rope, v, q_scale=None, k_scale=None, *,
                softmax_scale: float, causal: bool = True, out=None, lse=None,
                out_dtype=None, stream=None):
    """Fused MLA prefill.  Returns (out [B,S,H,d_v], lse [B,H,S] fp32).

    bf16 inputs: q_nope/k_nope/v bf16.  fp8 inputs: q_nope/k_nope/v float8_e4m3fn with
    q_scale/k_scale fp32 [B,S].  Rope parts are always bf16 (k_rope [B,S,d_rope]).
    """
    B, S, H, dn = q_nope.shape
    dr = q_rope.shape[-1]
    dv = v.shape[-1]
    fp8 = q_nope.dtype == torch.float8_e4m3fn
    qkv_dt = torch.float8_e4m3fn if fp8 else torch.bfloat16
    _need(q_nope, "q_nope", qkv_dt, (B, S, H, dn))
    _need(q_rope, "q_rope", torch.bfloat16, (B, S, H, dr))
    _need(k_nope, "k_nope", qkv_dt, (B, S, H, dn))
    _need(k_rope, "k_rope", torch.bfloat16, (B, S, dr))
    _need(v, "v", qkv_dt, (B, S, H, dv))
    if fp8:
        _need(q_scale, "q_scale", torch.float32, (B, S))
        _need(k_scale, "k_scale", torch.float32, (B, S))
    elif q_scale is not None or k_scale is not None:
        raise ValueError("q_scale/k_scale are only used with fp8 inputs")
    if out_dtype is None:
        out_dtype = torch.float32 if fp8 else torch.bfloat16
    dev = q_nope.device
    if out is None:
        out = torch.empty((B, S, H, dv), dtype=out_dtype, device=dev)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    _need(out, "out", out_dtype, (B, S, H, dv))
    _need(lse, "lse", torch.float32, (B, H, S))
    st = _lib.mla_prefill(_ptr(q_nope), _ptr(q_rope), _ptr(k_nope), _ptr(k_rope), _ptr(v),
                          _ptr(q_scale), _ptr(k_scale), _ptr(out), _ptr(lse), B, H, S, dn, dr,
                          dv, float(softmax_scale), int(bool(causal)),
                          MLA_FP8_E4M3 if fp8 else MLA_BF16,
                          MLA_FP32 if out_dtype == torch.float32 else MLA_BF16, _stream(stream))
    _check(st)
    return out, lse


def prefill_backward_workspace_size(B: int, H: int, S: int) -> int:
    return int(_lib.mla_prefill_backward_workspace_size(B, H, S))


def mla_prefill_backward(q_nope, q_rope, k_nope, k_rope, v, out, lse, d_out, *,
                         softmax_scale: float, causal: bool = True, grads=None, workspace=None,
                         stream=None):
    """Gradients of bf16 MLA prefill.  Returns (dq_nope, dq_rope, dk_nope, dk_rope, dv).

    out/lse are the forward's results, d_out the upstream gradient [B,S,H,d_v] bf16.
    dk_rope [B,S,d_rope] is fp32 (summed over heads); the others are bf16 in the layouts of
    their operands.  ``grads`` may pass those five tensors preallocated.
    """
    B, S, H, dn = q_nope.shape
    dr = q_rope.shape[-1]
    dv_ = v.shape[-1]
    bf = torch.bfloat16
    _need(q_nope, "q_nope", bf, (B, S, H, dn))
    _need(q_rope, "q_rope", bf, (B, S, H, dr))
    _need(k_nope, "k_nope", bf, (B, S, H, dn))
    _need(k_rope, "k_rope", bf, (B, S, dr))
    _need(v, "v", bf, (B, S, H, dv_))
    _need(out, "out", bf, (B, S, H, dv_))
    _need(lse, "lse", torch.float32, (B, H, S))
    _need(d_out, "d_out", bf, (B, S, H, dv_))
    dev = q_nope.device
    if grads is None:
        grads = (torch.empty((B, S, H, dn), dtype=bf, device=dev),
                 torch.empty((B, S, H, dr), dtype=bf, device=dev),
                 torch.empty((B, S, H, dn), dtype=bf, device=dev),
                 torch.empty((B, S, dr), dtype=torch.float32, device=dev),
                 torch.empty((B, S, H, dv_), dtype=bf, device=dev))
    dq_n, dq_r, dk_n, dk_r, dv = grads
    _need(dq_n, "dq_nope", bf, (B, S, H, dn))
    _need(dq_r, "dq_rope", bf, (B, S, H, dr))
    _need(dk_n, "dk_nope", bf, (B, S, H, dn))
    _need(dk_r, "dk_rope", torch.float32, (B, S, dr))
    _need(dv, "dv", bf, (B, S, H, dv_))
    need = prefill_backward_workspace_size(B, H, S)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    st = _lib.mla_prefill_backward(_ptr(q_nope), _ptr(q_rope), _ptr(k_nope), _ptr(k_rope), _ptr(v),
                                   _ptr(out), _ptr(lse), _ptr(d_out), _ptr(dq_n), _ptr(dq_r),
                                   _ptr(dk_n), _ptr(dk_r), _ptr(dv), B, H, S, dn, dr, dv_,
                                   float(softmax_scale), int(bool(causal)), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st)
    return dq_n, dq_r, dk_n, dk_r, dv


def decode_workspace_size(B: int, H: int, q_len: int, d_latent: int = 512) -> int:
    return int(_lib.mla_decode_workspace_size(B, H, q_len, d_latent))


def mla_decode(q_latent, q_rope, kv_cache, page_table, cache_lens, kv_scale=None, *,
               softmax_scale: float, causal: bool = True, out=None, lse=None, workspace=None,
               stream=None):
    """Absorbed MLA decode over a paged latent cache.  Returns (out [B,T,H,dl] bf16,
    lse [B,H,T] fp32).  kv_cache bf16 or float8_e4m3fn [num_pages, page_size, dl+dr];
    kv_scale fp32 [num_pages, page_size] for fp8."""
    B, T, H, dl = q_latent.shape
    dr = q_rope.shape[-1]
    num_pages, page_size, D = kv_cache.shape
    fp8 = kv_cache.dtype == torch.float8_e4m3fn
    _need(q_latent, "q_latent", torch.bfloat16, (B, T, H, dl))
    _need(q_rope, "q_rope", torch.bfloat16, (B, T, H, dr))
    _need(kv_cache, "kv_cache", torch.float8_e4m3fn if fp8 else torch.bfloat16,
          (num_pages, page_size, dl + dr))
    if fp8:
        _need(kv_scale, "kv_scale", torch.float32, (num_pages, page_size))
    elif kv_scale is not None:
        raise ValueError("kv_scale is only used with an fp8 cache")
    max_pages = page_table.shape[1]
    _need(page_table, "page_table", torch.int32, (B, max_pages))
    _need(cache_lens, "cache_lens", torch.int32, (B,))
    dev = q_latent.device
    if out is None:
        out = torch.empty((B, T, H, dl), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, (B, T, H, dl))
    _need(lse, "lse", torch.float32, (B, H, T))
    need = decode_workspace_size(B, H, T, dl)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    st = _lib.mla_decode(_ptr(q_latent), _ptr(q_rope), _ptr(kv_cache), _ptr(kv_scale),
                         _ptr(page_table), _ptr(cache_lens), _ptr(out), _ptr(lse), B, H, T, dl,
                         dr, page_size, max_pages, num_pages, float(softmax_scale),
                         int(bool(causal)), MLA_FP8_E4M3 if fp8 else MLA_BF16, _ptr(workspace),
                         workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st)
    return out, lse


def mla_absorb(x, w, *, out=None, stream=None):
    """y[r, h, :] = x[r, h, :] @ w[h] for x [R, H, K] and w [H, K, N] (bf16); returns y [R, H, N]."""
    R, H, K = x.shape
    N = w.shape[-1]
    _need(x, "x", torch.bfloat16, (R, H, K))
    _need(w, "w", torch.bfloat16, (H, K, N))
    if out is None:
        out = torch.empty((R, H, N), dtype=torch.bfloat16, device=x.device)
    _need(out, "out", torch.bfloat16, (R, H, N))
    _check(_lib.mla_absorb(_ptr(x), _ptr(w), _ptr(out), R, H, K, N, _stream(stream)))
    return out


def mla_cache_append(c_new, kv_cache, page_table, cache_lens, kv_scale=None, *, stream=None):
    """Write the q_len new tokens' rows c_new [B, q_len, dl+dr] (bf16) into the paged cache
    (bf16, or float8_e4m3fn with per-row fp32 kv_scale [num_pages, page_size]) at positions
    cache_lens[b] - q_len + t.  Modifies kv_cache (and kv_scale) in place."""
    B, T, D = c_new.shape
    num_pages, page_size, Dc = kv_cache.shape
    fp8 = kv_cache.dtype == torch.float8_e4m3fn
    _need(c_new, "c_new", torch.bfloat16, (B, T, D))
    _need(kv_cache, "kv_cache", torch.float8_e4m3fn if fp8 else torch.bfloat16, (num_pages, page_size, D))
    if fp8:
        _need(kv_scale, "kv_scale", torch.float32, (num_pages, page_size))
    elif kv_scale is not None:
        raise ValueError("kv_scale is only used with an fp8 cache")
    max_pages = page_table.shape[1]
    _need(page_table, "page_table", torch.int32, (B, max_pages))
    _need(cache_lens, "cache_lens", torch.int32, (B,))
    st = _lib.mla_cache_append(_ptr(c_new), _ptr(kv_cache), _ptr(kv_scale), _ptr(page_table),
                               _ptr(cache_lens), B, T, D - 64, 64, page_size,
                               max_pages, num_pages, MLA_FP8_E4M3 if fp8 else MLA_BF16,
                               _stream(stream))
    _check(st)
    return kv_cache, kv_scale


def decode_noalloc_max_workspace() -> int:
    return int(_lib.mla_decode_noalloc_max_workspace())


def mla_decode_noalloc_setup() -> None:
    """The set-up call of mla_decode_noalloc on the current device (B = 0): the built-in
    scratch array is reserved and the decode kernels are loaded, so that later calls on this
    device allocate nothing.  Make it before reserving device memory and before any stream
    capture."""
    _check(_lib.mla_decode_noalloc(None, None, None, None, None, None, None, None, 0, 0, 0, 0, 0,
                                   0, 0, 0, 0.0, 1, MLA_BF16, None))


def mla_decode_noalloc(q_latent, q_rope, kv_cache, page_table, cache_lens, kv_scale=None, *,
                       softmax_scale: float, causal: bool = True, out=None, lse=None, stream=None):
    """mla_decode without a workspace: for callers that cannot allocate device memory at
    call time.  The split partials use the library's built-in scratch array (see
    include/mla.h); calls on one device must not overlap on the GPU.  ``out``/``lse`` may
    be passed in so that the call itself allocates nothing."""
    B, T, H, dl = q_latent.shape
    dr = q_rope.shape[-1]
    num_pages, page_size, _ = kv_cache.shape
    fp8 = kv_cache.dtype == torch.float8_e4m3fn
    _need(q_latent, "q_latent", torch.bfloat16, (B, T, H, dl))
    _need(q_rope, "q_rope", torch.bfloat16, (B, T, H, dr))
    _need(kv_cache, "kv_cache", torch.float8_e4m3fn if fp8 else torch.bfloat16,
          (num_pages, page_size, dl + dr))
    if fp8:
        _need(kv_scale, "kv_scale", torch.float32, (num_pages, page_size))
    elif kv_scale is not None:
        raise ValueError("kv_scale is only used with an fp8 cache")
    max_pages = page_table.shape[1]
    _need(page_table, "page_table", torch.int32, (B, max_pages))
    _need(cache_lens, "cache_lens", torch.int32, (B,))
    dev = q_latent.device
    if out is None:
        out = torch.empty((B, T, H, dl), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, (B, T, H, dl))
    _need(lse, "lse", torch.float32, (B, H, T))
    st = _lib.mla_decode_noalloc(_ptr(q_latent), _ptr(q_rope), _ptr(kv_cache), _ptr(kv_scale),
                                 _ptr(page_table), _ptr(cache_lens), _ptr(out), _ptr(lse), B, H, T,
                                 dl, dr, page_size, max_pages, num_pages, float(softmax_scale),
                                 int(bool(causal)), MLA_FP8_E4M3 if fp8 else MLA_BF16,
                                 _stream(stream))
    _check(st)
    return out, lse
