"""GPU parity of mla_prefill_backward (through the C ABI) against the fp64 oracle.

Tolerance, element by element, from the arithmetic of the kernels (fp32 accumulation of
bf16 products; the only coarse roundings are the bf16 operands the tensor cores take):
  - O enters D = rowsum(dO * O) as given:       |dD_i| <= u sum_d |dO_id| (|O_id| + (P|V|)_id)
    (bf16 rounding of O; from the forward kernel also its bf16 P in P V)
  - P enters dV = P' dO as bf16:                 u sum_i P_ij |dO_i|
  - dS enters dQ, dK as bf16, with the D error:  |d dS_ij| <= u |dS_ij| + P_ij |dD_i|
    so |d dQ_i| <= scale sum_j (u |dS_ij| + P_ij |dD_i|) |K_j|, and dK likewise with Q
  - bf16 outputs are rounded once more:          u |g|
with u = 2^-8 (twice the bf16 unit roundoff 2^-9, covering the fp32 exponentials, score
and accumulation errors, which are below 2^-20 relative here).  The rope-key gradient is the
sum over heads of the per-head terms, in fp32.
"""
import numpy as np
import pytest
import torch

import oracle
from gen import bf16_bits_from_f32, config_inputs, make_grad_out, make_prefill

pytestmark = pytest.mark.gpu

U = 2.0 ** -8


def _bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def run_gpu(lib, inp, dO_bits, out_bits, lse):
    from mla_flash_attention_gb300.testing import prefill_to_device

    t = prefill_to_device(inp, torch.device("cuda"))["args"][:5]
    g = lib.mla_prefill_backward(*t, _bf16_dev(out_bits), torch.from_numpy(lse).float().cuda(),
                                 _bf16_dev(dO_bits), softmax_scale=inp.softmax_scale,
                                 causal=inp.causal)
    lib.check_device_error()
    return [_f64(x) for x in g]


def bounds_bh(inp, dOb, O_use, b, h):
    """Per-element error bounds (dQ [S,192], dK [S,192], dV [S,128]) of one (b, h).

    O_use is the O the kernel was given: its error against the exact O is at most
    u (|O| + P|V|) per element (bf16 rounding of O, and of P in the forward's P V).
    """
    Q, K, V = oracle.prefill_dequant_bh(inp, b, h)
    O, _, P = oracle.prefill_bh(inp, b, h, return_p=True)
    dP = dOb @ V.T
    D = np.sum(dOb * O, axis=1)
    dS = P * (dP - D[:, None])
    errD = U * np.sum(np.abs(dOb) * (np.abs(O_use) + P @ np.abs(V)), axis=1)
    w = U * np.abs(dS) + P * errD[:, None]
    sc = inp.softmax_scale
    gq = sc * (w @ np.abs(K))
    gk = sc * (w.T @ np.abs(Q))
    gv = U * (P.T @ np.abs(dOb))
    return gq, gk, gv


def compare(inp, dO_bits, got, O_ref_bits, heads=None):
    """Check `got` (GPU gradients) against the oracle, for all (b, h) or the listed pairs;
    O_ref_bits is the forward output the kernel was given."""
    dq_n, dq_r, dk_n, dk_r, dv = got
    rel = []
    pairs = heads if heads is not None else [(b, h) for b in range(inp.B) for h in range(inp.H)]
    kr_tol = np.zeros((inp.B, inp.S, inp.d_rope))
    kr_ref = np.zeros((inp.B, inp.S, inp.d_rope))
    dn = inp.d_nope
    for b, h in pairs:
        dQ, dK, dV = oracle.prefill_backward_bh(inp, dO_bits[b, :, h], b, h)
        dOb = oracle.bf16_to_f64(dO_bits[b, :, h])
        gq, gk, gv = bounds_bh(inp, dOb, oracle.bf16_to_f64(O_ref_bits[b, :, h]), b, h)
        for name, g, ref, bnd in (("dq_nope", dq_n[b, :, h], dQ[:, :dn], gq[:, :dn]),
                                  ("dq_rope", dq_r[b, :, h], dQ[:, dn:], gq[:, dn:]),
                                  ("dk_nope", dk_n[b, :, h], dK[:, :dn], gk[:, :dn]),
                                  ("dv", dv[b, :, h], dV, gv)):
            tol = 2 * bnd + U * np.abs(ref) + 1e-6
            err = np.abs(g - ref)
            bad = np.argwhere(err > tol)
            assert bad.size == 0, "%s b=%d h=%d at %s: got %g want %g (tol %g)" % (
                name, b, h, bad[0], g[tuple(bad[0])], ref[tuple(bad[0])], tol[tuple(bad[0])])
            rel.append(np.max(err) / max(np.max(np.abs(ref)), 1e-3))  # S = 1: dQ = dK = 0
        kr_ref[b] += dK[:, dn:]
        kr_tol[b] += 2 * gk[:, dn:]
    if heads is None:
        tol = kr_tol + 1e-6 + 1e-6 * np.abs(kr_ref)
        err = np.abs(dk_r - kr_ref)
        bad = np.argwhere(err > tol)
        assert bad.size == 0, "dk_rope at %s: got %g want %g (tol %g)" % (
            bad[0], dk_r[tuple(bad[0])], kr_ref[tuple(bad[0])], tol[tuple(bad[0])])
    return max(rel)


def oracle_forward_bits(inp):
    O, L = oracle.mla_prefill(inp)
    return bf16_bits_from_f32(O.astype(np.float32)), L.astype(np.float32)


@pytest.mark.parametrize("B,H,S", [(1, 2, 300), (2, 3, 128), (1, 1, 1), (1, 2, 129), (1, 4, 513)])
@pytest.mark.parametrize("causal", [True, False])
def test_backward_matches_oracle(lib, B, H, S, causal):
    inp = make_prefill(B, H, S, seed=500 + S + H, causal=causal)
    dO = make_grad_out(B, S, H, inp.d_v, seed=600 + S)
    O_bits, L = oracle_forward_bits(inp)
    got = run_gpu(lib, inp, dO, O_bits, L)
    rel = compare(inp, dO, got, O_bits)
    assert rel < 2e-2


def test_backward_many_heads_rope_sum(lib):
    # 16 heads add into the shared rope-key gradient; 8 key tiles of 128
    inp = make_prefill(1, 16, 1024, seed=701)
    dO = make_grad_out(1, 1024, 16, inp.d_v, seed=702)
    O_bits, L = oracle_forward_bits(inp)
    got = run_gpu(lib, inp, dO, O_bits, L)
    compare(inp, dO, got, O_bits)


def test_backward_extreme_scales(lib):
    for sc in (2.0, 1e-3):
        inp = make_prefill(1, 2, 256, seed=703, softmax_scale=sc)
        dO = make_grad_out(1, 256, 2, inp.d_v, seed=704)
        O_bits, L = oracle_forward_bits(inp)
        compare(inp, dO, run_gpu(lib, inp, dO, O_bits, L), O_bits)


def test_backward_after_gpu_forward(lib):
    # the chain a training step runs: the forward kernel's O and LSE feed the backward
    from mla_flash_attention_gb300.testing import prefill_to_device

    inp = make_prefill(1, 4, 640, seed=705)
    dO = make_grad_out(1, 640, 4, inp.d_v, seed=706)
    t = prefill_to_device(inp, torch.device("cuda"))["args"]
    out, lse = lib.mla_prefill(*t, softmax_scale=inp.softmax_scale, causal=True)
    got = lib.mla_prefill_backward(*t[:5], out, lse, _bf16_dev(dO), softmax_scale=inp.softmax_scale)
    lib.check_device_error()
    O_bits = out.cpu().view(torch.int16).numpy().view(np.uint16)
    compare(inp, dO, [_f64(x) for x in got], O_bits)


@pytest.mark.slow
def test_full_size_sampled_heads(lib):
    # B4 H128 S4096 through the GPU forward and backward; four (b, h) slices compared with
    # the oracle on every element, the rope-key gradient by its zero sum over keys
    from mla_flash_attention_gb300.testing import prefill_to_device

    inp = config_inputs("prefill_b4h128s4096_bf16")
    dO = make_grad_out(inp.B, inp.S, inp.H, inp.d_v, seed=1002)
    t = prefill_to_device(inp, torch.device("cuda"))["args"]
    out, lse = lib.mla_prefill(*t, softmax_scale=inp.softmax_scale, causal=True)
    got = lib.mla_prefill_backward(*t[:5], out, lse, _bf16_dev(dO), softmax_scale=inp.softmax_scale)
    lib.check_device_error()
    O_bits = out.cpu().view(torch.int16).numpy().view(np.uint16)
    got = [_f64(x) for x in got]
    for g in got:
        assert np.isfinite(g).all()
    rng = np.random.default_rng(9)
    heads = [(0, 0), (3, 127)] + [(int(rng.integers(4)), int(rng.integers(128))) for _ in range(2)]
    compare(inp, dO, got, O_bits, heads=heads)
    dk_r = got[3]
    assert np.max(np.abs(dk_r.sum(axis=1))) <= 1e-3 * np.abs(dk_r).sum(axis=1).max() + 1e-3
