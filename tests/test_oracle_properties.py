"""Randomised pins of the oracle (CPU): over drawn shapes, masks, scales and cache layouts the
oracle equals torch's scaled_dot_product_attention in float64 on the same dequantised
operands, its LSE is that of torch.logsumexp over the visible scaled scores, and its
backward equals torch autograd through the same SDPA."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from gen import make_decode, make_grad_out, make_prefill
from tests.test_oracle_pins import _decode_sdpa, sdpa, t_bf16, t_e4m3

hyp = pytest.importorskip("hypothesis")
st = hyp.strategies


def _prefill_ref(inp, b):
    """(O [S,H,dv], LSE [H,S]) of batch b from torch, on the dequantised operands."""
    if inp.fp8:
        qs = torch.from_numpy(inp.q_scale[b]).double()[:, None, None]
        ks = torch.from_numpy(inp.k_scale[b]).double()[:, None, None]
        qn, kn, v = t_e4m3(inp.q_nope[b]) * qs, t_e4m3(inp.k_nope[b]) * ks, t_e4m3(inp.v[b]) * ks
    else:
        qn, kn, v = t_bf16(inp.q_nope[b]), t_bf16(inp.k_nope[b]), t_bf16(inp.v[b])
    q = torch.cat([qn, t_bf16(inp.q_rope[b])], -1)
    k = torch.cat([kn, t_bf16(inp.k_rope[b])[:, None, :].expand(-1, inp.H, -1)], -1)
    o = sdpa(q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1), inp.softmax_scale, inp.causal)
    s = inp.softmax_scale * torch.einsum("she,the->hst", q, k)
    if inp.causal:
        s = s.masked_fill(torch.ones(inp.S, inp.S, dtype=torch.bool).triu(1), -float("inf"))
    return o.transpose(0, 1).numpy(), torch.logsumexp(s, -1).numpy()


@hyp.settings(max_examples=30, deadline=None)
@hyp.given(B=st.integers(1, 2), H=st.integers(1, 3), S=st.integers(1, 40),
           dims=st.sampled_from([(16, 8, 12), (8, 4, 8), (32, 16, 16)]), causal=st.booleans(),
           fp8=st.booleans(), scale=st.sampled_from([0.05, 0.3, 1.0]), seed=st.integers(0, 10**6))
def test_prefill_matches_sdpa_on_drawn_problems(B, H, S, dims, causal, fp8, scale, seed):
    dn, dr, dv = dims
    inp = make_prefill(B, H, S, d_nope=dn, d_rope=dr, d_v=dv, fp8=fp8, seed=seed, causal=causal,
                       softmax_scale=scale)
    O, L = oracle.mla_prefill(inp)
    for b in range(B):
        o_ref, l_ref = _prefill_ref(inp, b)
        np.testing.assert_allclose(O[b], o_ref, rtol=0, atol=1e-11 * max(1.0, np.abs(o_ref).max()))
        np.testing.assert_allclose(L[b], l_ref, rtol=0, atol=1e-10)


@hyp.settings(max_examples=30, deadline=None)
@hyp.given(lens=st.lists(st.integers(0, 80), min_size=1, max_size=4), H=st.integers(1, 3),
           T=st.integers(1, 3), fp8=st.booleans(), causal=st.booleans(),
           extra=st.integers(0, 3), seed=st.integers(0, 10**6))
def test_decode_matches_sdpa_on_drawn_problems(lens, H, T, fp8, causal, extra, seed):
    inp = make_decode(len(lens), H, T, lens, d_latent=32, d_rope=8, page_size=16, fp8=fp8,
                      seed=seed, extra_pages=extra, softmax_scale=0.25, causal=causal)
    O, L = oracle.mla_decode(inp)
    for b, n in enumerate(lens):
        if causal:
            ref, mask = _decode_sdpa(inp, b)
        else:
            C = oracle.decode_gather(inp, b)  # gathered rows are pinned by the causal case
            q = torch.cat([t_bf16(inp.q_latent[b]), t_bf16(inp.q_rope[b])], -1).reshape(T * H, -1)
            Ct = torch.from_numpy(C)
            mask = torch.ones(T * H, n, dtype=torch.bool)
            ref = sdpa(q[None], Ct[None], Ct[None, :, :32], 0.25, mask=mask[None])[0].reshape(T, H, -1)
        seen = mask.any(-1).reshape(T, H).numpy()
        np.testing.assert_allclose(O[b][seen], ref.numpy()[seen], rtol=0, atol=1e-11)
        assert (O[b][~seen] == 0).all() and np.isneginf(L[b].T[~seen]).all()


@hyp.settings(max_examples=20, deadline=None)
@hyp.given(B=st.integers(1, 2), H=st.integers(1, 3), S=st.integers(1, 24),
           dims=st.sampled_from([(16, 8, 12), (8, 4, 8)]), causal=st.booleans(),
           scale=st.sampled_from([0.1, 0.37, 1.0]), seed=st.integers(0, 10**6))
def test_backward_matches_autograd_on_drawn_problems(B, H, S, dims, causal, scale, seed):
    dn, dr, dv = dims
    inp = make_prefill(B, H, S, d_nope=dn, d_rope=dr, d_v=dv, seed=seed, causal=causal,
                       softmax_scale=scale)
    dO_bits = make_grad_out(B, S, H, dv, seed=seed + 1)
    f = oracle.bf16_to_f64
    leaves = {n: torch.tensor(f(getattr(inp, n)), requires_grad=True)
              for n in ("q_nope", "q_rope", "k_nope", "k_rope", "v")}
    q = torch.cat([leaves["q_nope"], leaves["q_rope"]], -1).transpose(1, 2)
    k = torch.cat([leaves["k_nope"], leaves["k_rope"][:, :, None, :].expand(B, S, H, dr)], -1).transpose(1, 2)
    o = F.scaled_dot_product_attention(q, k, leaves["v"].transpose(1, 2), is_causal=causal, scale=scale)
    o.transpose(1, 2).backward(torch.tensor(f(dO_bits)))
    got = dict(zip(("q_nope", "q_rope", "k_nope", "k_rope", "v"), oracle.mla_prefill_backward(inp, dO_bits)))
    for name, t in leaves.items():
        g = t.grad.numpy()
        np.testing.assert_allclose(got[name], g, rtol=0, atol=1e-10 * max(1.0, np.abs(g).max()), err_msg=name)
