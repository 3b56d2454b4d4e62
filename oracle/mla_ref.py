"""Plain, slow fp64 reference for MLA prefill and absorbed MLA decode.

Test infrastructure only (see the package docstring).  Numpy, float64, no
tiling, no fusion, no reordering beyond the definition.

What is computed (the pages' vocabulary):

* "S = Q@K' and O += P@V" -- the two products of the attention step
  (Modular API docs, ``nn/attention/gpu/nvidia/sm100/mla_decode_utils/KVPipelineGeneric``,
  struct description and Parameters).  Written here as the closed form the online
  (flash) formulation reaches up to rounding order: P = softmax(S), O = P V.
* Q and K are each split into a "nope" part and a "rope" part stored separately
  (``.../sm100/mla_prefill_per_token_scale/MLASmemStorage``, Fields ``q_smem`` /
  ``kv_smem`` and comptime ``q_nope_bytes`` / ``q_rope_bytes``); the score is the
  sum of both dot products.
* Per-token fp32 ``q_scale`` / ``k_scale`` (same page, Fields ``q_scale_smem``,
  ``k_scale_smem``: one float per query row of a tile and per key row).

Readings where the pages are silent (the oracle pin tests exercise each one):

* softmax_scale multiplies the whole nope+rope dot product; LSE is the natural
  log-sum-exp of the scaled scores (natural log, ``[B,H,S]`` / ``[B,H,T]``).
* Prefill causal: square, query i sees keys 0..i.
* Decode ``cache_len`` counts the T new tokens, which sit at L-T .. L-1; query t
  sees keys 0 .. L-T+t (bottom-right causal).  A row that sees no key has O=0 and
  LSE=-inf.
* One rope key per token shared by every head (``k_rope [B,S,d_rope]``).
* fp8: one scale per token shared by every head; Q_nope is dequantised with
  q_scale, K_nope **and V** with k_scale (the interface has no separate V scale).
  Rope parts are bf16 and unscaled.
* Decode fp8 cache: the whole 576-wide latent+rope row of a token is e4m3 with one
  fp32 scale; V is the first ``d_latent`` columns of the same dequantised row.
"""
from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------------------
# storage decoders (from the format definitions)
# ---------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float64.

    bfloat16 is the upper half of an IEEE-754 binary32: sign, 8 exponent bits,
    7 fraction bits.  Widening therefore places the 16 bits on top of 16 zero bits.
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """OCP FP8 E4M3 ("e4m3fn") codes -> float64.

    Layout: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.  Exponent field 0
    encodes subnormals m/8 * 2^-6; exponent 1..15 encodes (1 + m/8) * 2^(e-7), except
    e=15, m=7, which is NaN (there are no infinities).  Largest finite value 448.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = (m / 8.0) * 2.0 ** -6
    val = sign * np.where(e == 0, sub, normal)
    return np.where((e == 15) & ((c & 7) == 7), np.nan, val)


# ---------------------------------------------------------------------------
# the attention definition
# ---------------------------------------------------------------------------

def attention_rows(Q: np.ndarray, K: np.ndarray, V: np.ndarray, visible: np.ndarray,
                   scale: float, return_p: bool = False):
    """softmax(scale * Q K^T) V over the visible keys of each row, in float64.

    Q [n, d], K [m, d], V [m, dv], visible bool [n, m].  Returns O [n, dv] and
    LSE [n] = log(sum_j exp(s_ij)) over visible j (natural log); a row with no
    visible key gets O = 0 and LSE = -inf.  Invisible keys are never read into the
    arithmetic (their rows may hold NaN).
    """
    Q = np.asarray(Q, dtype=np.float64)
    n, m = visible.shape
    dv = V.shape[1]
    K = np.where(visible.any(axis=0)[:, None], K, 0.0)
    V = np.where(visible.any(axis=0)[:, None], V, 0.0)
    s = scale * (Q @ K.T)
    s = np.where(visible, s, -np.inf)
    rowmax = s.max(axis=1) if m else np.full(n, -np.inf)
    empty = ~np.isfinite(rowmax)
    safe_max = np.where(empty, 0.0, rowmax)
    e = np.exp(s - safe_max[:, None])
    e = np.where(visible, e, 0.0)
    l = e.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        P = np.where(empty[:, None], 0.0, e / np.where(empty, 1.0, l)[:, None])
        lse = np.where(empty, -np.inf, safe_max + np.log(np.where(empty, 1.0, l)))
    O = P @ V if m else np.zeros((n, dv))
    if return_p:
        return O, lse, P
    return O, lse


# ---------------------------------------------------------------------------
# prefill
# ---------------------------------------------------------------------------

def _dq(x, fp8):
    """Stored values -> float64: e4m3 codes (fp8), bf16 bits, or exact float64 as given."""
    x = np.asarray(x)
    if x.dtype.kind == "f":
        return x.astype(np.float64)
    return e4m3_to_f64(x) if fp8 else bf16_to_f64(x)


def prefill_dequant_bh(inp, b: int, h: int, rows=None):
    """Dequantised operands of one (batch, head): Q [n,dn+dr], K [S,dn+dr], V [S,dv].

    fp8: Q_nope * q_scale[token], K_nope * k_scale[token], V * k_scale[token].
    """
    fp8 = inp.fp8
    rows = np.arange(inp.S) if rows is None else np.asarray(rows)
    qn = _dq(inp.q_nope[b, rows, h], fp8)
    kn = _dq(inp.k_nope[b, :, h], fp8)
    v = _dq(inp.v[b, :, h], fp8)
    if fp8:
        qn = qn * inp.q_scale[b, rows].astype(np.float64)[:, None]
        ks = inp.k_scale[b].astype(np.float64)[:, None]
        kn = kn * ks
        v = v * ks
    Q = np.concatenate([qn, _dq(inp.q_rope[b, rows, h], False)], axis=1)
    K = np.concatenate([kn, _dq(inp.k_rope[b], False)], axis=1)
    return Q, K, v


def prefill_bh(inp, b: int, h: int, rows=None, return_p: bool = False):
    """O [n, d_v] and LSE [n] for query rows ``rows`` (default: all) of one (b, h)."""
    rows = np.arange(inp.S) if rows is None else np.asarray(rows)
    Q, K, V = prefill_dequant_bh(inp, b, h, rows)
    j = np.arange(inp.S)
    visible = (j[None, :] <= rows[:, None]) if inp.causal else np.ones((len(rows), inp.S), bool)
    return attention_rows(Q, K, V, visible, inp.softmax_scale, return_p)


def mla_prefill(inp):
    """Full prefill: O [B,S,H,d_v] float64, LSE [B,H,S] float64."""
    O = np.zeros((inp.B, inp.S, inp.H, inp.d_v))
    L = np.zeros((inp.B, inp.H, inp.S))
    for b in range(inp.B):
        for h in range(inp.H):
            o, l = prefill_bh(inp, b, h)
            O[b, :, h] = o
            L[b, h] = l
    return O, L


# ---------------------------------------------------------------------------
# absorbed decode over the paged latent cache
# ---------------------------------------------------------------------------

def decode_gather(inp, b: int):
    """Dequantised cache rows 0..L_b-1 of sequence b, in token order: C [L_b, d_latent+d_rope].

    Token j lives in page ``page_table[b, j // page_size]`` at row ``j % page_size``.
    """
    L = int(inp.cache_lens[b])
    j = np.arange(L)
    pages = inp.page_table[b, j // inp.page_size].astype(np.int64)
    r = j % inp.page_size
    raw = inp.kv_cache[pages, r]
    if inp.fp8:
        return _dq(raw, True) * inp.kv_scale[pages, r].astype(np.float64)[:, None]
    return _dq(raw, False)


def decode_b(inp, b: int, key_range=None, return_p: bool = False):
    """O [T, H, d_latent] and LSE [H, T] of sequence b.

    ``key_range=(k0, k1)`` restricts the keys to positions k0..k1-1 (a split of the
    key axis, used to check split-and-combine); the causal rule is unchanged.
    """
    L = int(inp.cache_lens[b])
    C = decode_gather(inp, b)
    T, H = inp.T, inp.H
    q = np.concatenate([_dq(inp.q_latent[b], False), _dq(inp.q_rope[b], False)], axis=2)
    Q = q.reshape(T * H, -1)
    t = np.repeat(np.arange(T), H)
    j = np.arange(L)
    if inp.causal:
        visible = j[None, :] <= (L - T + t)[:, None]
    else:
        visible = np.ones((T * H, L), bool)
    if key_range is not None:
        k0, k1 = key_range
        visible = visible & (j[None, :] >= k0) & (j[None, :] < k1)
    res = attention_rows(Q, C, C[:, :inp.d_latent], visible, inp.softmax_scale, return_p)
    O = res[0].reshape(T, H, inp.d_latent)
    lse = res[1].reshape(T, H).T.copy()
    if return_p:
        return O, lse, res[2]
    return O, lse


def mla_decode(inp):
    """Full decode: O [B,T,H,d_latent] float64, LSE [B,H,T] float64."""
    O = np.zeros((inp.B, inp.T, inp.H, inp.d_latent))
    Ls = np.zeros((inp.B, inp.H, inp.T))
    for b in range(inp.B):
        O[b], Ls[b] = decode_b(inp, b)
    return O, Ls


def lse_combine(o_parts, lse_parts):
    """Merge attention results computed over disjoint key sets.

    With lse = log sum_s exp(lse_s), the merged output is sum_s exp(lse_s - lse) O_s.
    o_parts [n_split, ..., dv], lse_parts [n_split, ...].  Parts with lse_s = -inf (no
    visible key) contribute nothing; if every part is empty, O = 0 and lse = -inf.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    mx = lse_parts.max(axis=0)
    empty = ~np.isfinite(mx)
    safe = np.where(empty, 0.0, mx)
    w = np.where(np.isfinite(lse_parts), np.exp(lse_parts - safe[None]), 0.0)
    tot = w.sum(axis=0)
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, safe + np.log(np.where(empty, 1.0, tot)))
    coef = np.where(empty[None], 0.0, w / np.where(empty, 1.0, tot)[None])
    O = (coef[..., None] * o_parts).sum(axis=0)
    return O, lse
