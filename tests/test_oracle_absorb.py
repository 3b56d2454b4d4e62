"""Pins of the absorption oracle (CPU only): brute force, and the absorbed-decode identity.

The identity ties the product to the attention definition: decode over the latent with
q_latent = absorb(q_nope, W_UK) followed by absorb(O_latent, W_UV) must equal ordinary MLA
attention over keys W_UK c_j and values c_j W_UV (materialised per head); a transposed
weight, a wrong head or a dropped term fails it.
"""
import numpy as np

import oracle
from gen import make_decode, make_prefill


def test_absorb_matches_scalar_loops():
    rng = np.random.default_rng(5)
    R, H, K, N = 3, 2, 5, 4
    x = rng.standard_normal((R, H, K))
    w = rng.standard_normal((H, K, N))
    y = oracle.absorb(x, w)
    for r in range(R):
        for h in range(H):
            for n in range(N):
                acc = 0.0
                for k in range(K):
                    acc += x[r, h, k] * w[h, k, n]
                assert abs(y[r, h, n] - acc) <= 1e-12 * (1 + abs(acc))


def test_absorb_reads_bf16_bit_patterns():
    from gen import bf16_bits_from_f32
    rng = np.random.default_rng(6)
    x = bf16_bits_from_f32(rng.standard_normal((4, 3, 8)).astype(np.float32))
    w = bf16_bits_from_f32(rng.standard_normal((3, 8, 2)).astype(np.float32))
    np.testing.assert_array_equal(oracle.absorb(x, w),
                                  oracle.absorb(oracle.bf16_to_f64(x), oracle.bf16_to_f64(w)))


def test_absorbed_decode_through_absorb_equals_materialised_attention():
    rng = np.random.default_rng(41)
    L, H, dl, dr, dn, dv = 33, 3, 24, 8, 6, 5
    dec = make_decode(1, H, 1, [L], d_latent=dl, d_rope=dr, page_size=8, seed=42, softmax_scale=0.29)
    C = oracle.decode_gather(dec, 0)
    W_uk = rng.standard_normal((H, dn, dl))      # [H, K=dn, N=dl]
    W_uv = rng.standard_normal((H, dl, dv))      # [H, K=dl, N=dv]
    q_nope = rng.standard_normal((1, H, dn))
    q_rope = oracle.bf16_to_f64(dec.q_rope[0, 0])
    dec.q_latent = oracle.absorb(q_nope, W_uk)[None]          # [1, 1, H, dl]
    dec.q_rope = q_rope[None, None]
    O_lat, lse_d = oracle.mla_decode(dec)
    O_abs = oracle.absorb(O_lat[0], W_uv)[0]                  # [H, dv]
    pre = make_prefill(1, H, L, d_nope=dn, d_rope=dr, d_v=dv, seed=43, softmax_scale=0.29)
    pre.q_nope = np.zeros((1, L, H, dn))
    pre.q_nope[0, L - 1] = q_nope[0]
    pre.q_rope = np.zeros((1, L, H, dr))
    pre.q_rope[0, L - 1] = q_rope
    pre.k_nope = np.einsum("jl,hnl->jhn", C[:, :dl], W_uk)[None]   # k_h,j = W_UK[h] c_j
    pre.k_rope = C[None, :, dl:]
    pre.v = np.einsum("jl,hlv->jhv", C[:, :dl], W_uv)[None]        # v_h,j = c_j W_UV[h]
    O_p, lse_p = oracle.mla_prefill(pre)
    np.testing.assert_allclose(O_abs, O_p[0, L - 1], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(lse_d[0, :, 0], lse_p[0, :, L - 1], rtol=1e-12, atol=1e-10)
