"""GPU parity of mla_prefill (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from gen import config_inputs, make_prefill
from tests.parity import TOL_O_BF16, TOL_O_FP8, check

pytestmark = pytest.mark.gpu


def run(lib, inp, out_dtype=None):
    from mla_flash_attention_gb300.testing import prefill_to_device

    t = prefill_to_device(inp, torch.device("cuda"))
    out, lse = lib.mla_prefill(*t["args"], softmax_scale=inp.softmax_scale, causal=inp.causal,
                               out_dtype=out_dtype)
    lib.check_device_error()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def test_tiny_config_full(lib):
    inp = config_inputs("prefill_tiny_b1h4s128_bf16")
    o, l = run(lib, inp)
    O, L = oracle.mla_prefill(inp)
    check(o, O, l, L, TOL_O_BF16, what="tiny")


@pytest.mark.parametrize("S", [1, 2, 37, 127, 128, 129, 300, 513])
@pytest.mark.parametrize("causal", [True, False])
def test_ragged_lengths_bf16(lib, S, causal):
    inp = make_prefill(2, 3, S, seed=100 + S, causal=causal)
    o, l = run(lib, inp)
    O, L = oracle.mla_prefill(inp)
    check(o, O, l, L, TOL_O_BF16, what="bf16 S=%d causal=%d" % (S, causal))


@pytest.mark.parametrize("S", [1, 45, 128, 259, 640])
@pytest.mark.parametrize("causal", [True, False])
def test_ragged_lengths_fp8(lib, S, causal):
    inp = make_prefill(1, 4, S, fp8=True, seed=200 + S, causal=causal)
    o, l = run(lib, inp)
    O, L = oracle.mla_prefill(inp)
    check(o, O, l, L, TOL_O_FP8, bf16_out=False, what="fp8 S=%d" % S)


def test_bf16_output_of_fp8_inputs(lib):
    inp = make_prefill(1, 2, 200, fp8=True, seed=301, mag_range=(0.5, 2.0))
    o, l = run(lib, inp, out_dtype=torch.bfloat16)
    O, L = oracle.mla_prefill(inp)
    check(o, O, l, L, TOL_O_FP8, what="fp8 in, bf16 out")


def test_fp32_output_of_bf16_inputs(lib):
    inp = make_prefill(1, 2, 150, seed=302)
    o, l = run(lib, inp, out_dtype=torch.float32)
    O, L = oracle.mla_prefill(inp)
    check(o, O, l, L, TOL_O_BF16, bf16_out=False, what="bf16 in, fp32 out")


def test_extreme_scales(lib):
    # large softmax_scale: near one-hot rows; tiny: near-uniform rows
    for sc in (2.0, 1e-4):
        inp = make_prefill(1, 2, 256, seed=303, softmax_scale=sc)
        o, l = run(lib, inp)
        O, L = oracle.mla_prefill(inp)
        check(o, O, l, L, TOL_O_BF16, what="scale %g" % sc)


def _full_rows(lib, name, tol, bf16_out):
    """Every output row of twelve (batch, head) pairs of a full-size workload -- the first and
    the last pair and ten drawn ones -- against the oracle (the kernel orders its row blocks
    longest first and skips tiles above the diagonal, so whole rows at full size are checked)."""
    inp = config_inputs(name)
    o, l = run(lib, inp)
    assert np.isfinite(o).all() and np.isfinite(l).all()
    rng = np.random.default_rng(7)
    pairs = [(0, 0), (inp.B - 1, inp.H - 1)] + [(int(rng.integers(inp.B)), int(rng.integers(inp.H)))
                                               for _ in range(10)]
    for b, h in pairs:
        O, L = oracle.prefill_bh(inp, b, h)
        check(o[b, :, h], O, l[b, h], L, tol, bf16_out=bf16_out, what="%s b=%d h=%d" % (name, b, h))


@pytest.mark.slow
def test_full_size_bf16_every_row_of_twelve_heads(lib):
    _full_rows(lib, "prefill_b4h128s4096_bf16", TOL_O_BF16, True)


@pytest.mark.slow
def test_full_size_fp8_every_row_of_twelve_heads(lib):
    _full_rows(lib, "prefill_b2h128s8192_fp8", TOL_O_FP8, False)
