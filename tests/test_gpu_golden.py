"""The CUDA path (through the C ABI) on the closed-form cases of
``tests/golden/closed_forms.json``: outputs derived by hand from the definitions, not by
the oracle."""
import numpy as np
import pytest
import torch

from tests.golden import load_cases
from tests.parity import TOL_O_BF16, TOL_O_FP8, check

pytestmark = pytest.mark.gpu

CASES = load_cases()


def _run(lib, inp):
    from mla_flash_attention_gb300.testing import decode_to_device, prefill_to_device

    dev = torch.device("cuda")
    if hasattr(inp, "S"):
        t = prefill_to_device(inp, dev)
        out, lse = lib.mla_prefill(*t["args"], softmax_scale=inp.softmax_scale, causal=inp.causal)
    else:
        d = decode_to_device(inp, dev)
        out, lse = lib.mla_decode(*d["args"], **d["kwargs"], softmax_scale=inp.softmax_scale,
                                  causal=inp.causal)
    lib.check_device_error()
    return out.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("name,inp,O,L", [(n, i, o, l) for n, i, o, l, _ in CASES], ids=[c[0] for c in CASES])
def test_closed_form(lib, name, inp, O, L):
    o, l = _run(lib, inp)
    fp8_prefill = inp.fp8 and hasattr(inp, "S")
    check(o, O, l, L, TOL_O_FP8 if inp.fp8 else TOL_O_BF16, bf16_out=not fp8_prefill, what=name)
    if name == "decode_fp8_codes":
        # one visible key with P' = 1: every output is a code value times 1/2, exact in bf16
        assert np.array_equal(o, O), np.argwhere(o != O)[:5]
