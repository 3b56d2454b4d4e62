"""Pins of the backward oracle (CPU only).

The gradient is tied to things other than its own formula: central finite differences of
the (separately pinned) forward oracle, torch autograd through scaled_dot_product_attention
in float64, and invariants that follow from softmax rows summing to one.  A dropped D term,
a missing scale, a rope gradient not summed over heads or a transposed product fails the
finite-difference and autograd pins.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import oracle.backward_ref as bref
from gen import make_grad_out, make_prefill


def small(S=5, H=2, dn=4, dr=3, dv=3, causal=True, seed=11):
    """A tiny prefill problem with float64 operands (so they can be perturbed)."""
    inp = make_prefill(1, H, S, d_nope=dn, d_rope=dr, d_v=dv, seed=seed, softmax_scale=0.37,
                       causal=causal)
    for name in ("q_nope", "q_rope", "k_nope", "k_rope", "v"):
        setattr(inp, name, oracle.bf16_to_f64(getattr(inp, name)))
    dO = oracle.bf16_to_f64(make_grad_out(1, S, H, dv, seed=seed + 1))
    return inp, dO


def loss(inp, dO):
    O, _ = oracle.mla_prefill(inp)
    return float(np.sum(O * dO))


def fd_grads(inp, dO, eps=1e-5):
    """Central differences of sum(O * dO) for every operand element."""
    out = {}
    for name in ("q_nope", "q_rope", "k_nope", "k_rope", "v"):
        x = getattr(inp, name)
        g = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            keep = x[idx]
            x[idx] = keep + eps
            up = loss(inp, dO)
            x[idx] = keep - eps
            dn = loss(inp, dO)
            x[idx] = keep
            g[idx] = (up - dn) / (2 * eps)
        out[name] = g
    return out


def analytic(inp, dO):
    dq_n, dq_r, dk_n, dk_r, dv = oracle.mla_prefill_backward(inp, dO)
    return {"q_nope": dq_n, "q_rope": dq_r, "k_nope": dk_n, "k_rope": dk_r, "v": dv}


def max_rel_gap(a, b):
    return max(np.max(np.abs(a[k] - b[k])) / (1e-3 + np.max(np.abs(b[k]))) for k in a)


@pytest.mark.parametrize("causal", [True, False])
def test_backward_equals_finite_differences(causal):
    inp, dO = small(causal=causal)
    assert max_rel_gap(analytic(inp, dO), fd_grads(inp, dO)) < 1e-7


def test_a_dropped_rope_term_is_caught(monkeypatch):
    """Planted in the oracle: the backward's K loses its rope columns."""
    inp, dO = small()
    fd = fd_grads(inp, dO)
    real = bref.prefill_dequant_bh

    def no_rope(inp_, b, h, rows=None):
        Q, K, V = real(inp_, b, h, rows)
        K = K.copy()
        K[:, inp_.d_nope:] = 0
        return Q, K, V

    monkeypatch.setattr(bref, "prefill_dequant_bh", no_rope)
    assert max_rel_gap(analytic(inp, dO), fd) > 1e-2


@pytest.mark.parametrize("causal", [True, False])
def test_backward_equals_torch_autograd(causal):
    B, H, S, dn, dr, dv = 2, 3, 37, 16, 8, 12
    inp = make_prefill(B, H, S, d_nope=dn, d_rope=dr, d_v=dv, seed=21, causal=causal)
    dO_bits = make_grad_out(B, S, H, dv, seed=22)
    f = oracle.bf16_to_f64
    qn = torch.tensor(f(inp.q_nope), requires_grad=True)
    qr = torch.tensor(f(inp.q_rope), requires_grad=True)
    kn = torch.tensor(f(inp.k_nope), requires_grad=True)
    kr = torch.tensor(f(inp.k_rope), requires_grad=True)
    v = torch.tensor(f(inp.v), requires_grad=True)
    q = torch.cat([qn, qr], dim=-1).transpose(1, 2)                       # [B,H,S,E]
    k = torch.cat([kn, kr[:, :, None, :].expand(B, S, H, dr)], dim=-1).transpose(1, 2)
    o = F.scaled_dot_product_attention(q, k, v.transpose(1, 2), is_causal=causal,
                                       scale=inp.softmax_scale)
    o.transpose(1, 2).backward(torch.tensor(f(dO_bits)))
    got = analytic(inp, dO_bits)
    for name, t in (("q_nope", qn), ("q_rope", qr), ("k_nope", kn), ("k_rope", kr), ("v", v)):
        np.testing.assert_allclose(got[name], t.grad.numpy(), rtol=1e-9, atol=1e-11, err_msg=name)


def test_backward_invariants():
    B, H, S = 1, 4, 50
    inp = make_prefill(B, H, S, d_nope=8, d_rope=4, d_v=8, seed=31)
    dO = make_grad_out(B, S, H, 8, seed=32)
    g = analytic(inp, dO)
    # rows of dS sum to zero, so the key gradients sum to zero over keys
    assert np.max(np.abs(g["k_nope"].sum(axis=1))) < 1e-10
    assert np.max(np.abs(g["k_rope"].sum(axis=1))) < 1e-10
    # rows of P sum to one, so the value gradients sum to the summed upstream gradient
    np.testing.assert_allclose(g["v"].sum(axis=1), oracle.bf16_to_f64(dO).sum(axis=1),
                               rtol=1e-10, atol=1e-10)
    # causal row 0 sees only key 0 (P = 1), so its query gets no gradient
    assert np.max(np.abs(g["q_nope"][:, 0])) < 1e-12 and np.max(np.abs(g["q_rope"][:, 0])) < 1e-12
