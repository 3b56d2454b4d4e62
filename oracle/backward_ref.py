"""Reference gradients of MLA prefill attention -- TEST INFRASTRUCTURE ONLY.

The pages define the forward step only ("S = Q@K' and O += P@V", Modular API docs,
``nn/attention/gpu/nvidia/sm100/mla_decode_utils/KVPipelineGeneric``, struct
description; nope/rope split from ``.../sm100/mla_prefill_per_token_scale/
MLASmemStorage``).  The backward pass is the exact derivative of that definition:
for an upstream gradient dO of O = softmax(s) V with s = scale * [Qn|Qr][Kn|Kr]',

    dV = P' dO                         dP = dO V'
    D_i = sum_d dO_id O_id  (= sum_j P_ij dP_ij)
    dS = P * (dP - D)                  (rows of a softmax Jacobian-vector product)
    dQ = scale * dS K                  dK = scale * dS' Q

taken per (batch, head) in float64.  The rope key is one vector per token shared by
every head, so its gradient is the sum over heads of the per-head dK rope columns.
bf16 inputs only (the fp8 forward has no backward here).
"""
from __future__ import annotations

import numpy as np

from .mla_ref import bf16_to_f64, prefill_bh, prefill_dequant_bh


def _f64(a):
    a = np.asarray(a)
    return bf16_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def prefill_backward_bh(inp, d_out_bh, b: int, h: int):
    """(dQ [S, dn+dr], dK [S, dn+dr], dV [S, dv]) of one (batch, head).

    d_out_bh: dO of this (b, h), [S, dv] (bf16 bits or floats).
    """
    Q, K, V = prefill_dequant_bh(inp, b, h)
    O, _lse, P = prefill_bh(inp, b, h, return_p=True)
    dO = _f64(d_out_bh)
    dV = P.T @ dO
    dP = dO @ V.T
    D = np.sum(dO * O, axis=1)
    dS = P * (dP - D[:, None])
    dQ = inp.softmax_scale * (dS @ K)
    dK = inp.softmax_scale * (dS.T @ Q)
    return dQ, dK, dV


def mla_prefill_backward(inp, d_out):
    """Gradients of sum(O * dO) with respect to the prefill operands, float64.

    Returns (dq_nope [B,S,H,dn], dq_rope [B,S,H,dr], dk_nope [B,S,H,dn],
    dk_rope [B,S,dr] (summed over heads), dv [B,S,H,dv]).
    """
    assert not inp.fp8, "the backward reference covers the bf16 operands"
    B, S, H, dn, dr, dv = inp.B, inp.S, inp.H, inp.d_nope, inp.d_rope, inp.d_v
    dq_n = np.zeros((B, S, H, dn))
    dq_r = np.zeros((B, S, H, dr))
    dk_n = np.zeros((B, S, H, dn))
    dk_r = np.zeros((B, S, dr))
    dv_ = np.zeros((B, S, H, dv))
    for b in range(B):
        for h in range(H):
            dQ, dK, dV = prefill_backward_bh(inp, d_out[b, :, h], b, h)
            dq_n[b, :, h] = dQ[:, :dn]
            dq_r[b, :, h] = dQ[:, dn:]
            dk_n[b, :, h] = dK[:, :dn]
            dk_r[b] += dK[:, dn:]
            dv_[b, :, h] = dV
    return dq_n, dq_r, dk_n, dk_r, dv_
