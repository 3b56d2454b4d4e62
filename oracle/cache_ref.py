"""Reference for appending new tokens to the paged latent cache -- TEST INFRASTRUCTURE ONLY.

The step before absorbed decode: the T new tokens of every sequence (their latent and rope
rows, bf16) are written into the paged cache, at the positions decode reads them from.  An
fp8 cache stores each 576-wide row as e4m3 codes with one fp32 scale per token.

Readings (the pages are silent on the cache write; these follow the decode reading the
oracle already uses):

* ``cache_len`` counts the new tokens, so token t of sequence b goes to position
  L_b - T + t: page ``page_table[b, pos // page_size]``, row ``pos % page_size``
  (the same placement ``mla_ref.decode_gather`` reads).  Positions below 0 (L_b < T)
  are not written.
* Quantisation of one row x (the 576 values widened exactly from bf16 to fp32):
  amax = max |x|; scale = amax / 448 (scale = 1 when amax = 0); code = e4m3 of
  clamp(x / scale, -448, 448), rounded to nearest, ties to even.  The division and the
  scale are fp32 operations (the precision the code decision is taken in on the GPU).

The e4m3 encoder below is written from the format's definition (a search over the 127
non-negative finite values), not from any conversion routine of a library.
"""
from __future__ import annotations

import numpy as np

from .mla_ref import e4m3_to_f64

E4M3_MAX = 448.0

# the non-negative finite e4m3 values, in code order 0x00 .. 0x7e (increasing)
_POS_CODES = np.arange(0x7F, dtype=np.uint8)
_POS_VALUES = e4m3_to_f64(_POS_CODES)


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """fp32 values with |x| <= 448 -> e4m3 codes, round to nearest, ties to even code.

    The nearest of the representable magnitudes is found by bisection in the sorted value
    table; a value exactly half way between two neighbours takes the one whose code is
    even (its last mantissa bit is 0).  The sign bit is x's sign bit (so -0.0 -> 0x80).
    """
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x).astype(np.float64)
    if np.any(a > E4M3_MAX) or np.any(~np.isfinite(a)):
        raise ValueError("e4m3_encode expects finite |x| <= 448")
    hi = np.searchsorted(_POS_VALUES, a, side="left")      # first value >= a
    hi = np.minimum(hi, len(_POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(a == _POS_VALUES[hi], hi, code).astype(np.uint8)
    return np.where(np.signbit(x), code | np.uint8(0x80), code).astype(np.uint8)


def quantize_row(x: np.ndarray):
    """One cache row (fp32 values) -> (e4m3 codes, fp32 scale) as the reading above."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0.0)
    scale = np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(E4M3_MAX))
    y = (x / scale).astype(np.float32)
    y = np.clip(y, np.float32(-E4M3_MAX), np.float32(E4M3_MAX)).astype(np.float32)
    return e4m3_encode(y), scale


def cache_append(c_new_bits: np.ndarray, kv_cache: np.ndarray, kv_scale, page_table: np.ndarray,
                 cache_lens: np.ndarray, page_size: int, fp8: bool):
    """Write the new rows into copies of the cache (and scales); returns (kv_cache, kv_scale).

    c_new_bits: [B, T, D] bf16 bit patterns (D = d_latent + d_rope).
    kv_cache:   [num_pages, page_size, D] bf16 bits (uint16) or e4m3 codes (uint8).
    kv_scale:   [num_pages, page_size] fp32 (fp8 cache) or None.
    """
    c_new_bits = np.asarray(c_new_bits, dtype=np.uint16)
    B, T, _ = c_new_bits.shape
    cache = np.array(kv_cache, copy=True)
    scales = None if kv_scale is None else np.array(kv_scale, dtype=np.float32, copy=True)
    for b in range(B):
        L = int(cache_lens[b])
        for t in range(T):
            pos = L - T + t
            if pos < 0:
                continue
            page = int(page_table[b, pos // page_size])
            r = pos % page_size
            if fp8:
                row = (c_new_bits[b, t].astype(np.uint32) << np.uint32(16)).view(np.float32)
                codes, scale = quantize_row(row)
                cache[page, r] = codes
                scales[page, r] = scale
            else:
                cache[page, r] = c_new_bits[b, t]
    return cache, scales
