"""GPU parity of mla_absorb (through the C ABI) against the fp64 oracle, every element.

Tolerance, from the arithmetic: the kernel accumulates K products in fp32 (error at most
about K * 2^-24 of sum |x w|, bounded here by 2^-14 * sum |x w| for K <= 1024) and rounds
the result to bf16 once (half a bf16 unit in the last place; one full unit allowed because
the fp32 value may sit on the other side of a rounding boundary than the exact one).
"""
import numpy as np
import pytest
import torch

import oracle
from gen import bf16_bits_from_f32

pytestmark = pytest.mark.gpu


def ulp_bf16(v):
    v = np.maximum(np.abs(v), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(v)) - 7)


def case(R, H, K, N, seed):
    rng = np.random.default_rng(seed)
    x = bf16_bits_from_f32(rng.standard_normal((R, H, K)).astype(np.float32))
    w = bf16_bits_from_f32((rng.standard_normal((H, K, N)) / np.sqrt(K)).astype(np.float32))
    return x, w


def to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("R,H,K,N", [
    (64, 128, 128, 512),   # q_nope W_UK for the bf16 decode workload (B64, T1, H128)
    (64, 128, 512, 128),   # O_latent W_UV for the same workload
    (256, 16, 128, 512),   # the ragged fp8 decode workload (B128, T2, H16)
    (1, 3, 64, 128),       # a single row, the smallest depths
    (130, 5, 192, 256),    # two row tiles with a ragged tail, 3 K chunks, 2 column tiles
    (300, 2, 1024, 128),   # long contraction
    (17, 2, 128, 384),     # N not a multiple of 256: 128-column tiles
])
def test_absorb_matches_oracle(lib, R, H, K, N):
    x, w = case(R, H, K, N, seed=R * 7 + K)
    y = lib.mla_absorb(to_dev(x), to_dev(w))
    lib.check_device_error()
    got = oracle.bf16_to_f64(y.cpu().view(torch.int16).numpy().view(np.uint16))
    ref = oracle.absorb(x, w)
    bound = oracle.absorb(np.abs(oracle.bf16_to_f64(x)), np.abs(oracle.bf16_to_f64(w)))
    tol = ulp_bf16(ref) + 2.0 ** -14 * bound
    err = np.abs(got - ref)
    assert np.all(err <= tol), "max err %.3e (tol there %.3e)" % (err.max(), tol.flat[np.argmax(err - tol)])
    # most elements are the correctly rounded bf16 of the exact value
    exact = oracle.bf16_to_f64(bf16_bits_from_f32(ref.astype(np.float32)))
    assert np.mean(got == exact) > 0.95


def test_absorb_rejects_unsupported_shapes(lib):
    x = torch.zeros((4, 2, 96), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((2, 96, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.MLAError):
        lib.mla_absorb(x, w)
