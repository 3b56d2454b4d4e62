"""Reference for the absorption products either side of absorbed decode -- TEST INFRASTRUCTURE ONLY.

Absorbed MLA decode works on the latent: the query's nope part is first multiplied by the
key up-projection of its head (q_latent = q_nope W_UK[h]) and the latent output by the value
up-projection (o = O_latent W_UV[h]).  Both are the same per-head product

    y[r, h, :] = x[r, h, :] @ w[h]        x [R, H, K], w [H, K, N], y [R, H, N]

(R = batch x new tokens), written here as the plain definition in float64 on the decoded
inputs (bf16 bit patterns or floats).
"""
from __future__ import annotations

import numpy as np

from .mla_ref import bf16_to_f64


def _f64(a):
    a = np.asarray(a)
    return bf16_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def absorb(x, w) -> np.ndarray:
    """y[r, h, n] = sum_k x[r, h, k] w[h, k, n] in float64."""
    X, W = _f64(x), _f64(w)
    R, H, K = X.shape
    assert W.shape[:2] == (H, K), (X.shape, W.shape)
    return np.einsum("rhk,hkn->rhn", X, W)
