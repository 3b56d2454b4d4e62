"""Seeded input generator for MLA prefill and absorbed MLA decode.

Every tensor is drawn from numpy's PCG64 under a ``SeedSequence`` keyed by
(seed, tensor id, chunk index), so the values do not depend on the number of
threads used to draw them.  Values are returned in the storage types the CUDA
library reads:

* bf16 tensors as ``uint16`` bit patterns (round-to-nearest-even from fp32),
* fp8 tensors as ``uint8`` e4m3 codes plus one fp32 scale per token,
* page tables and cache lengths as ``int32``.

Quantisation rule for the fp8 workloads (one scale per token, shared by every
head): ``scale = amax / 448`` over the token's whole row (``1`` if the row is
all zero), ``code = e4m3_rne(clamp(x / scale, -448, 448))``.  The e4m3 cast is
torch's ``float8_e4m3fn`` conversion (round to nearest even) after the explicit
clamp.  Consumers only ever read the stored codes and scales.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

_CHUNK = 1 << 22  # elements per independently seeded chunk
E4M3_MAX = 448.0

# tensor ids (part of every SeedSequence key)
_T_QN, _T_QR, _T_KN, _T_KR, _T_V, _T_MQ, _T_MK, _T_CACHE, _T_LENS, _T_PERM, _T_DO = range(11)


def _threads() -> int:
    try:
        return max(1, min(16, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(16, os.cpu_count() or 1))


def _normal_f32(seed: int, tid: int, n: int) -> np.ndarray:
    """``n`` standard normal float32 values, chunk-seeded and drawn in parallel."""
    out = np.empty(n, dtype=np.float32)
    nchunks = max(1, math.ceil(n / _CHUNK))

    def work(i: int) -> None:
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tid, i])))
        g.standard_normal(out=out[i * _CHUNK:(i + 1) * _CHUNK], dtype=np.float32)

    if nchunks == 1:
        work(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def _rng(seed: int, tid: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tid, 1 << 30])))


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return the bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    r = ((u + bias) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = np.uint16(0x7FC0)
    return r


def _e4m3_codes(x: np.ndarray) -> np.ndarray:
    """float32 values already inside [-448, 448] -> e4m3fn codes (torch RNE cast)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def quantize_rows_e4m3(x: np.ndarray):
    """Quantise each row of a 2-D float32 array with its own fp32 scale.

    Returns (codes uint8 same shape, scale float32 [rows]).
    """
    x = np.asarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=1)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    y = np.clip(x / scale[:, None], -E4M3_MAX, E4M3_MAX).astype(np.float32)
    codes = np.empty(x.shape, dtype=np.uint8)
    step = max(1, _CHUNK // max(1, x.shape[1]))
    for r0 in range(0, x.shape[0], step):
        codes[r0:r0 + step] = _e4m3_codes(y[r0:r0 + step])
    return codes, scale


@dataclass
class PrefillInputs:
    """One MLA prefill problem.

    Shapes (innermost last): q_nope/k_nope ``[B,S,H,d_nope]``, q_rope ``[B,S,H,d_rope]``,
    k_rope ``[B,S,d_rope]`` (one rope key per token, shared by all heads),
    v ``[B,S,H,d_v]``, q_scale/k_scale ``[B,S]`` (fp8 only).
    """

    B: int
    H: int
    S: int
    d_nope: int
    d_rope: int
    d_v: int
    softmax_scale: float
    causal: bool
    fp8: bool
    q_nope: np.ndarray
    q_rope: np.ndarray
    k_nope: np.ndarray
    k_rope: np.ndarray
    v: np.ndarray
    q_scale: Optional[np.ndarray] = None
    k_scale: Optional[np.ndarray] = None
    seed: int = 0
    meta: dict = field(default_factory=dict)


@dataclass
class DecodeInputs:
    """One absorbed MLA decode problem over a paged latent cache.

    q_latent ``[B,T,H,d_latent]``, q_rope ``[B,T,H,d_rope]`` (bf16 bits);
    kv_cache ``[num_pages, page_size, d_latent + d_rope]`` (bf16 bits or e4m3 codes);
    kv_scale ``[num_pages, page_size]`` fp32 (fp8 only); page_table ``[B, max_pages]``
    int32 (-1 = unused); cache_lens ``[B]`` int32, counting the T new tokens, which sit
    at positions ``L-T .. L-1``.  Cache rows past a sequence's length hold NaN.
    """

    B: int
    H: int
    T: int
    d_latent: int
    d_rope: int
    page_size: int
    num_pages: int
    max_pages: int
    softmax_scale: float
    causal: bool
    fp8: bool
    q_latent: np.ndarray
    q_rope: np.ndarray
    kv_cache: np.ndarray
    kv_scale: Optional[np.ndarray]
    page_table: np.ndarray
    cache_lens: np.ndarray
    seed: int = 0
    meta: dict = field(default_factory=dict)


def _bf16_normal(seed, tid, shape):
    n = int(np.prod(shape))
    return bf16_bits_from_f32(_normal_f32(seed, tid, n)).reshape(shape)


def make_prefill(B, H, S, d_nope=128, d_rope=64, d_v=128, *, fp8=False, seed=0,
                 softmax_scale=None, causal=True, mag_range=(0.1, 10.0)) -> PrefillInputs:
    """Draw one prefill problem.

    bf16: every tensor ~ N(0,1) rounded to bf16.
    fp8: Q_nope, K_nope and V are N(0,1)*m with one magnitude m per token, log-uniform in
    ``mag_range`` (Q its own m; K_nope and V of one key token share m and the scale),
    quantised per token; Q_rope/K_rope stay bf16 N(0,1).
    """
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d_nope + d_rope)
    q_rope = _bf16_normal(seed, _T_QR, (B, S, H, d_rope))
    k_rope = _bf16_normal(seed, _T_KR, (B, S, d_rope))
    if not fp8:
        q_nope = _bf16_normal(seed, _T_QN, (B, S, H, d_nope))
        k_nope = _bf16_normal(seed, _T_KN, (B, S, H, d_nope))
        v = _bf16_normal(seed, _T_V, (B, S, H, d_v))
        return PrefillInputs(B, H, S, d_nope, d_rope, d_v, float(softmax_scale), bool(causal),
                             False, q_nope, q_rope, k_nope, k_rope, v, None, None, seed)
    lo, hi = math.log(mag_range[0]), math.log(mag_range[1])
    mq = np.exp(_rng(seed, _T_MQ).uniform(lo, hi, size=(B * S,))).astype(np.float32)
    mk = np.exp(_rng(seed, _T_MK).uniform(lo, hi, size=(B * S,))).astype(np.float32)
    xq = _normal_f32(seed, _T_QN, B * S * H * d_nope).reshape(B * S, H * d_nope)
    xq *= mq[:, None]
    q_nope, q_scale = quantize_rows_e4m3(xq)
    del xq
    xk = _normal_f32(seed, _T_KN, B * S * H * d_nope).reshape(B * S, H * d_nope)
    xv = _normal_f32(seed, _T_V, B * S * H * d_v).reshape(B * S, H * d_v)
    xk *= mk[:, None]
    xv *= mk[:, None]
    kv_codes, k_scale = quantize_rows_e4m3(np.concatenate([xk, xv], axis=1))
    del xk, xv
    k_nope = np.ascontiguousarray(kv_codes[:, :H * d_nope]).reshape(B, S, H, d_nope)
    v = np.ascontiguousarray(kv_codes[:, H * d_nope:]).reshape(B, S, H, d_v)
    del kv_codes
    return PrefillInputs(B, H, S, d_nope, d_rope, d_v, float(softmax_scale), bool(causal), True,
                         q_nope.reshape(B, S, H, d_nope), q_rope, k_nope, k_rope, v,
                         q_scale.reshape(B, S), k_scale.reshape(B, S), seed)


def make_grad_out(B, S, H, d_v=128, *, seed=0) -> np.ndarray:
    """Upstream gradient dO ``[B,S,H,d_v]`` of a prefill output: N(0,1) rounded to bf16 bits."""
    return _bf16_normal(seed, _T_DO, (B, S, H, d_v))


def make_decode(B, H, T, cache_lens, *, d_latent=512, d_rope=64, page_size=64, fp8=False,
                seed=0, softmax_scale=None, causal=True, extra_pages=0) -> DecodeInputs:
    """Draw one absorbed decode problem.

    ``cache_lens`` is an int, a sequence of B ints, or ``("uniform", lo, hi)`` for a seeded
    draw.  Pages of all sequences are numbered through one seeded permutation of
    ``0 .. num_pages-1``; ``extra_pages`` adds pages that no sequence owns.
    """
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(192.0)
    if isinstance(cache_lens, tuple) and cache_lens and cache_lens[0] == "uniform":
        lens = _rng(seed, _T_LENS).integers(cache_lens[1], cache_lens[2] + 1, size=B)
    elif np.isscalar(cache_lens):
        lens = np.full(B, int(cache_lens))
    else:
        lens = np.asarray(cache_lens)
    lens = lens.astype(np.int32)
    assert lens.shape == (B,) and (lens >= 0).all()
    npages = -(-lens.astype(np.int64) // page_size)
    num_pages = int(npages.sum()) + int(extra_pages)
    max_pages = max(1, int(npages.max()) if B else 1)
    perm = _rng(seed, _T_PERM).permutation(num_pages).astype(np.int32)
    page_table = np.full((B, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        page_table[b, :npages[b]] = perm[off:off + npages[b]]
        off += int(npages[b])
    D = d_latent + d_rope
    q_latent = _bf16_normal(seed, _T_QN, (B, T, H, d_latent))
    q_rope = _bf16_normal(seed, _T_QR, (B, T, H, d_rope))
    x = _normal_f32(seed, _T_CACHE, num_pages * page_size * D).reshape(num_pages * page_size, D)
    # rows past each sequence's length (and rows of unowned pages) are poisoned with NaN
    valid = np.zeros((num_pages, page_size), dtype=bool)
    for b in range(B):
        for p in range(int(npages[b])):
            n = min(page_size, int(lens[b]) - p * page_size)
            valid[page_table[b, p], :n] = True
    valid = valid.reshape(-1)
    if fp8:
        codes, scale = quantize_rows_e4m3(x)
        del x
        codes[~valid] = 0x7F
        scale[~valid] = np.nan
        kv_cache = codes.reshape(num_pages, page_size, D)
        kv_scale = scale.reshape(num_pages, page_size)
    else:
        x[~valid] = np.nan
        kv_cache = bf16_bits_from_f32(x).reshape(num_pages, page_size, D)
        kv_scale = None
        del x
    return DecodeInputs(B, H, T, d_latent, d_rope, page_size, num_pages, max_pages,
                        float(softmax_scale), bool(causal), bool(fp8), q_latent, q_rope,
                        kv_cache, kv_scale, page_table, lens, seed)


# The five workloads.  Seeds are 1000 + the workload's position in this list.
CONFIGS = {
    "prefill_tiny_b1h4s128_bf16": dict(kind="prefill", B=1, H=4, S=128, fp8=False, seed=1000),
    "prefill_b4h128s4096_bf16": dict(kind="prefill", B=4, H=128, S=4096, fp8=False, seed=1001),
    "prefill_b2h128s8192_fp8": dict(kind="prefill", B=2, H=128, S=8192, fp8=True, seed=1002),
    "decode_b64h128t1l4096_bf16": dict(kind="decode", B=64, H=128, T=1, lens=4096, fp8=False,
                                       seed=1003),
    "decode_b128h16t2_ragged_fp8": dict(kind="decode", B=128, H=16, T=2,
                                        lens=("uniform", 1, 32768), fp8=True, seed=1004),
}


def config_inputs(name: str):
    c = CONFIGS[name]
    if c["kind"] == "prefill":
        return make_prefill(c["B"], c["H"], c["S"], fp8=c["fp8"], seed=c["seed"])
    return make_decode(c["B"], c["H"], c["T"], c["lens"], fp8=c["fp8"], seed=c["seed"])
