"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test ties an oracle function to a library routine, a closed form, an
invariant of attention, or brute force, so that a plausible slip in the oracle
(a dropped rope term, a wrong scale, a transposed operand, a shifted causal
diagonal, a wrong page lookup) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from gen import make_decode, make_prefill, bf16_bits_from_f32
from gen.inputs import quantize_rows_e4m3


# ---------------------------------------------------------------- helpers (library routes)

def t_bf16(bits):
    """bf16 bit patterns -> float64 through torch's own bfloat16 type."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double()


def t_e4m3(codes):
    """e4m3 codes -> float64 through torch's own float8_e4m3fn type."""
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double()


def sdpa(q, k, v, scale, causal=False, mask=None):
    """torch SDPA in float64 on [n_head, L, E] tensors."""
    return F.scaled_dot_product_attention(q[None], k[None], v[None], attn_mask=mask,
                                          is_causal=causal, scale=scale)[0]


# ---------------------------------------------------------------- storage decoders

def test_bf16_decode_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_f64(bits)
    ref = t_bf16(bits).numpy()
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all()
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_decode_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f64(codes)
    ref = t_e4m3(codes).numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert (np.isnan(ours) == nan).all()
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.nanmax(ours) == 448.0 and ours[1] == 2.0 ** -9


def test_e4m3_quantisation_round_trip_bound():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((64, 256)) * np.exp(rng.uniform(-3, 3, (64, 1)))).astype(np.float32)
    codes, scale = quantize_rows_e4m3(x)
    back = oracle.e4m3_to_f64(codes) * scale[:, None].astype(np.float64)
    y = np.abs(x.astype(np.float64))
    # e4m3 normals keep 3 fraction bits (half-ulp = 2^-4 relative); subnormals have a
    # fixed step of 2^-9 (half-step 2^-10) in units of the row scale.
    bound = np.maximum(y * 2.0 ** -4, scale[:, None] * 2.0 ** -10) * (1 + 1e-6)
    assert (np.abs(back - y * np.sign(x)) <= bound).all()
    assert np.allclose(np.abs(back).max(axis=1), np.abs(x).max(axis=1), rtol=1e-6)


# ---------------------------------------------------------------- prefill vs torch SDPA

@pytest.mark.parametrize("causal", [True, False])
def test_prefill_bf16_equals_sdpa(causal):
    inp = make_prefill(2, 3, 37, d_nope=16, d_rope=8, d_v=12, seed=5, causal=causal,
                       softmax_scale=0.3)
    O, lse = oracle.mla_prefill(inp)
    for b in range(inp.B):
        q = torch.cat([t_bf16(inp.q_nope[b]), t_bf16(inp.q_rope[b])], -1)  # [S,H,E]
        kr = t_bf16(inp.k_rope[b])[:, None, :].expand(-1, inp.H, -1)
        k = torch.cat([t_bf16(inp.k_nope[b]), kr], -1)
        v = t_bf16(inp.v[b])
        ref = sdpa(q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1), 0.3, causal)
        np.testing.assert_allclose(O[b], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)
        # LSE through torch.softmax: p_ij = exp(s_ij - lse_i) for any visible j (take j = 0)
        s = 0.3 * torch.einsum("she,the->hst", q, k)
        if causal:
            s = s.masked_fill(torch.ones(inp.S, inp.S, dtype=torch.bool).triu(1), -math.inf)
        p0 = torch.softmax(s, -1)[..., 0]
        np.testing.assert_allclose(lse[b], (s[..., 0] - torch.log(p0)).numpy(), atol=1e-9)


def test_prefill_fp8_scales_equal_sdpa_on_dequantised():
    inp = make_prefill(1, 4, 29, d_nope=32, d_rope=16, d_v=32, fp8=True, seed=9,
                       softmax_scale=0.2)
    O, lse = oracle.mla_prefill(inp)
    qs = torch.from_numpy(inp.q_scale[0]).double()[:, None, None]
    ks = torch.from_numpy(inp.k_scale[0]).double()[:, None, None]
    q = torch.cat([t_e4m3(inp.q_nope[0]) * qs, t_bf16(inp.q_rope[0])], -1)
    kr = t_bf16(inp.k_rope[0])[:, None, :].expand(-1, inp.H, -1)
    k = torch.cat([t_e4m3(inp.k_nope[0]) * ks, kr], -1)
    v = t_e4m3(inp.v[0]) * ks
    ref = sdpa(q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1), 0.2, True)
    np.testing.assert_allclose(O[0], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)
    # the per-token magnitudes span two decades, so the scales are not all alike
    assert inp.k_scale.max() / inp.k_scale.min() > 5


# ---------------------------------------------------------------- decode vs torch SDPA

def _decode_sdpa(inp, b):
    L = int(inp.cache_lens[b])
    pt = torch.from_numpy(inp.page_table[b].astype(np.int64))
    j = torch.arange(L)
    phys = pt[j // inp.page_size]
    rows = j % inp.page_size
    raw = inp.kv_cache[phys.numpy(), rows.numpy()]
    if inp.fp8:
        C = t_e4m3(raw) * torch.from_numpy(inp.kv_scale[phys.numpy(), rows.numpy()]).double()[:, None]
    else:
        C = t_bf16(raw)
    q = torch.cat([t_bf16(inp.q_latent[b]), t_bf16(inp.q_rope[b])], -1)  # [T,H,576]
    q = q.reshape(inp.T * inp.H, -1)
    t = torch.arange(inp.T).repeat_interleave(inp.H)
    mask = j[None, :] <= (L - inp.T + t)[:, None]
    out = sdpa(q[None], C[None], C[None, :, :inp.d_latent], inp.softmax_scale, mask=mask[None])[0]
    return out.reshape(inp.T, inp.H, -1), mask


@pytest.mark.parametrize("fp8", [False, True])
def test_decode_equals_sdpa(fp8):
    inp = make_decode(5, 3, 2, [1, 2, 63, 64, 130], d_latent=32, d_rope=8, page_size=16,
                      fp8=fp8, seed=11, extra_pages=3, softmax_scale=0.25)
    O, lse = oracle.mla_decode(inp)
    for b in range(inp.B):
        ref, mask = _decode_sdpa(inp, b)
        nonempty = mask.any(-1).reshape(inp.T, inp.H).numpy()
        np.testing.assert_allclose(O[b][nonempty], ref.numpy()[nonempty], rtol=0, atol=1e-12)
        assert (O[b][~nonempty] == 0).all()
        assert np.isneginf(lse[b].T[~nonempty]).all() and np.isfinite(lse[b].T[nonempty]).all()
    # b=0 has L=1 with T=2: query 0 sees nothing, query 1 sees key 0 only
    assert np.isneginf(lse[0, :, 0]).all()
    C0 = oracle.decode_gather(inp, 0)
    np.testing.assert_allclose(O[0, 1], np.broadcast_to(C0[0, :32], (3, 32)), atol=0)


# ---------------------------------------------------------------- closed forms / invariants

def test_prefill_constant_v_and_first_row():
    inp = make_prefill(1, 2, 20, d_nope=8, d_rope=8, d_v=6, seed=3)
    inp.v[:] = bf16_bits_from_f32(np.full(inp.v.shape, 1.5, np.float32))
    O, _ = oracle.mla_prefill(inp)
    assert np.allclose(O, 1.5, atol=1e-14)
    inp2 = make_prefill(1, 2, 20, d_nope=8, d_rope=8, d_v=6, seed=4)
    O2, lse2 = oracle.mla_prefill(inp2)
    # causal row 0 sees only key 0: O = V[0], LSE = s_00
    np.testing.assert_array_equal(O2[0, 0], oracle.bf16_to_f64(inp2.v[0, 0]))
    for h in range(2):
        q = np.concatenate([oracle.bf16_to_f64(inp2.q_nope[0, 0, h]),
                            oracle.bf16_to_f64(inp2.q_rope[0, 0, h])])
        k = np.concatenate([oracle.bf16_to_f64(inp2.k_nope[0, 0, h]),
                            oracle.bf16_to_f64(inp2.k_rope[0, 0])])
        assert abs(lse2[0, h, 0] - inp2.softmax_scale * float(q @ k)) < 1e-12


def test_prefill_equal_scores_is_running_mean():
    # Q = 0 makes every visible score 0: P is uniform, LSE_i = ln(i+1), O_i = mean(V_0..V_i)
    inp = make_prefill(1, 2, 25, d_nope=8, d_rope=8, d_v=5, seed=6)
    inp.q_nope[:] = 0
    inp.q_rope[:] = 0
    O, lse = oracle.mla_prefill(inp)
    V = oracle.bf16_to_f64(inp.v[0])  # [S,H,dv]
    running = np.cumsum(V, axis=0) / np.arange(1, 26)[:, None, None]
    np.testing.assert_allclose(O[0], running, atol=1e-13)
    np.testing.assert_allclose(lse[0], np.log(np.arange(1, 26))[None].repeat(2, 0), atol=1e-13)


def test_rows_of_p_sum_to_one():
    inp = make_prefill(1, 1, 33, d_nope=16, d_rope=8, d_v=8, seed=8)
    _, _, P = oracle.prefill_bh(inp, 0, 0, return_p=True)
    np.testing.assert_allclose(P.sum(1), 1.0, atol=1e-14)
    assert (np.triu(P, 1) == 0).all()


def test_brute_force_tiny():
    inp = make_prefill(1, 2, 6, d_nope=3, d_rope=2, d_v=2, seed=12, softmax_scale=0.7)
    O, lse = oracle.mla_prefill(inp)
    f = oracle.bf16_to_f64
    for h in range(2):
        for i in range(6):
            sc = []
            for j in range(i + 1):
                d = 0.0
                for c in range(3):
                    d += f(inp.q_nope[0, i, h, c]) * f(inp.k_nope[0, j, h, c])
                for c in range(2):
                    d += f(inp.q_rope[0, i, h, c]) * f(inp.k_rope[0, j, c])
                sc.append(0.7 * d)
            w = [math.exp(x) for x in sc]
            tot = sum(w)
            assert abs(lse[0, h, i] - math.log(tot)) < 1e-12
            for c in range(2):
                o = sum(w[j] * f(inp.v[0, j, h, c]) for j in range(i + 1)) / tot
                assert abs(O[0, i, h, c] - o) < 1e-12


def test_decode_single_key_returns_its_v_row():
    inp = make_decode(3, 4, 1, [1, 1, 1], d_latent=16, d_rope=8, page_size=4, seed=13)
    O, lse = oracle.mla_decode(inp)
    for b in range(3):
        C = oracle.decode_gather(inp, b)
        np.testing.assert_array_equal(O[b, 0], np.broadcast_to(C[0, :16], (4, 16)))


# ---------------------------------------------------------------- identities

def test_absorbed_decode_equals_materialised_attention():
    """q_lat = W_UK^T q_nope and V = c W_UV^T: decode over the latent equals ordinary MLA."""
    rng = np.random.default_rng(21)
    L, H, dl, dr, dn, dv = 40, 3, 24, 8, 6, 5
    dec = make_decode(1, H, 1, [L], d_latent=dl, d_rope=dr, page_size=8, seed=22,
                      softmax_scale=0.31)
    C = oracle.decode_gather(dec, 0)
    W_uk = rng.standard_normal((H, dn, dl))
    W_uv = rng.standard_normal((H, dv, dl))
    q_nope = rng.standard_normal((H, dn))
    q_rope = oracle.bf16_to_f64(dec.q_rope[0, 0])
    dec.q_latent = np.einsum("hn,hnl->hl", q_nope, W_uk)[None, None]  # exact float64 inputs
    dec.q_rope = q_rope[None, None]
    O_lat, lse_d = oracle.mla_decode(dec)
    O_abs = np.einsum("hl,hvl->hv", O_lat[0, 0], W_uv)
    # the same tokens as an ordinary (materialised) MLA prefill; its last causal row sees all keys
    pre = make_prefill(1, H, L, d_nope=dn, d_rope=dr, d_v=dv, seed=23, softmax_scale=0.31)
    pre.q_nope = np.zeros((1, L, H, dn))
    pre.q_nope[0, L - 1] = q_nope
    pre.q_rope = np.zeros((1, L, H, dr))
    pre.q_rope[0, L - 1] = q_rope
    pre.k_nope = np.einsum("jl,hnl->jhn", C[:, :dl], W_uk)[None]
    pre.k_rope = C[None, :, dl:]
    pre.v = np.einsum("jl,hvl->jhv", C[:, :dl], W_uv)[None]
    O_p, lse_p = oracle.mla_prefill(pre)
    np.testing.assert_allclose(O_abs, O_p[0, L - 1], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(lse_d[0, :, 0], lse_p[0, :, L - 1], rtol=1e-12, atol=1e-10)


@pytest.mark.parametrize("fp8", [False, True])
def test_split_and_combine_equals_unsplit(fp8):
    inp = make_decode(2, 4, 2, [77, 150], d_latent=16, d_rope=8, page_size=8, fp8=fp8, seed=31)
    for b in range(2):
        L = int(inp.cache_lens[b])
        O, lse = oracle.decode_b(inp, b)
        cuts = [0, 13, 40, L - 1, L]  # the third part holds only the last token
        parts = [oracle.decode_b(inp, b, key_range=(a, c)) for a, c in zip(cuts[:-1], cuts[1:])]
        # parts: O [T,H,dl], LSE [H,T] -> combine over [T,H]
        Oc, lc = oracle.lse_combine([p[0] for p in parts], [p[1].T for p in parts])
        np.testing.assert_allclose(Oc, O, atol=1e-12)
        np.testing.assert_allclose(lc.T, lse, atol=1e-12)
    # all parts empty -> O = 0, LSE = -inf
    Oe, le = oracle.lse_combine(np.ones((2, 3, 4)), np.full((2, 3), -np.inf))
    assert (Oe == 0).all() and np.isneginf(le).all()


def test_page_permutation_invariance():
    inp = make_decode(3, 2, 1, [20, 33, 9], d_latent=16, d_rope=8, page_size=8, seed=41,
                      extra_pages=2)
    O, lse = oracle.mla_decode(inp)
    perm = np.random.default_rng(1).permutation(inp.num_pages)
    inv = np.argsort(perm)
    inp.kv_cache = inp.kv_cache[perm]  # new page i holds old page perm[i]
    pt = inp.page_table.copy()
    pt[pt >= 0] = inv[pt[pt >= 0]]
    inp.page_table = pt
    O2, lse2 = oracle.mla_decode(inp)
    np.testing.assert_array_equal(O, O2)
    np.testing.assert_array_equal(lse, lse2)


# ---------------------------------------------------------------- planted mistakes are caught

def test_a_dropped_rope_term_is_caught(monkeypatch):
    real = oracle.mla_ref.prefill_dequant_bh

    def no_rope(inp, b, h, rows=None):
        Q, K, V = real(inp, b, h, rows)
        Q = Q.copy()
        Q[:, inp.d_nope:] = 0
        return Q, K, V

    monkeypatch.setattr(oracle.mla_ref, "prefill_dequant_bh", no_rope)
    with pytest.raises(AssertionError):
        test_prefill_bf16_equals_sdpa(True)


def test_a_shifted_decode_diagonal_is_caught(monkeypatch):
    real = oracle.mla_ref.attention_rows

    def shifted(Q, K, V, visible, scale, return_p=False):
        vis = visible.copy()
        vis[:, 1:] |= visible[:, :-1]  # one more key per row
        return real(Q, K, V, vis, scale, return_p)

    monkeypatch.setattr(oracle.mla_ref, "attention_rows", shifted)
    with pytest.raises(AssertionError):
        test_decode_equals_sdpa(False)
