"""mla_decode_noalloc: the decode entry point that allocates nothing.

It exists for callers that cannot allocate device memory where they run decode (an engine
that owns all device memory from start-up, a plugin hook that may not allocate), so they
cannot hand mla_decode a workspace.  It must give the same results as mla_decode, call
after call, even though every call reuses (and leaves behind) the same built-in scratch
array, and after its set-up call (B = 0) it must not change the device's free memory.
This file is collected last so that a failure here cannot hide another test.
"""
import numpy as np
import pytest
import torch

import oracle
from gen import make_decode
from tests.parity import TOL_O_BF16, TOL_O_FP8, check

pytestmark = pytest.mark.gpu


def _inputs(lib_testing, inp):
    return lib_testing.decode_to_device(inp, torch.device("cuda"))


@pytest.mark.parametrize("fp8", [False, True])
def test_matches_mla_decode_on_two_calls_in_a_row(lib, fp8):
    from mla_flash_attention_gb300 import testing

    tol = TOL_O_FP8 if fp8 else TOL_O_BF16
    # two different batches back to back: the second call runs over the first call's
    # leftovers in the shared scratch array
    for seed, lens in ((51, [1, 700, 2049, 64]), (52, [3000, 65, 2])):
        inp = make_decode(len(lens), 16, 2, lens, fp8=fp8, seed=seed)
        d = _inputs(testing, inp)
        out_ref, lse_ref = lib.mla_decode(*d["args"], **d["kwargs"],
                                          softmax_scale=inp.softmax_scale)
        out = torch.empty_like(out_ref)
        lse = torch.empty_like(lse_ref)
        lib.mla_decode_noalloc(*d["args"], **d["kwargs"], softmax_scale=inp.softmax_scale,
                               out=out, lse=lse)
        lib.check_device_error()
        a, b = out.float().cpu().numpy(), out_ref.float().cpu().numpy()
        la, lb = lse.cpu().numpy(), lse_ref.cpu().numpy()
        check(a, b.astype(np.float64), la, lb.astype(np.float64), tol, what="noalloc vs decode")
        # and both agree with the oracle
        O, L = oracle.mla_decode(inp)
        check(a, O, la, L, tol, what="noalloc vs oracle")


def test_rejects_a_batch_larger_than_the_scratch(lib):
    from mla_flash_attention_gb300 import testing
    from mla_flash_attention_gb300.binding import MLAError

    cap = lib.decode_noalloc_max_workspace()
    B = 200
    assert lib.decode_workspace_size(B, 128, 1) > cap
    inp = make_decode(B, 128, 1, 1, seed=53)
    d = _inputs(testing, inp)
    with pytest.raises(MLAError, match="WORKSPACE"):
        lib.mla_decode_noalloc(*d["args"], **d["kwargs"], softmax_scale=inp.softmax_scale)


def test_allocates_nothing_after_the_setup_call(lib):
    from mla_flash_attention_gb300 import testing

    inp = make_decode(3, 16, 2, [900, 1, 4000], fp8=True, seed=54)
    d = _inputs(testing, inp)
    out = torch.empty((inp.B, inp.T, inp.H, inp.d_latent), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((inp.B, inp.H, inp.T), dtype=torch.float32, device="cuda")
    lib.mla_decode_noalloc_setup()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(2):
        lib.mla_decode_noalloc(*d["args"], **d["kwargs"], softmax_scale=inp.softmax_scale,
                               out=out, lse=lse)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0
    lib.check_device_error()
    O, L = oracle.mla_decode(inp)
    check(out.float().cpu().numpy(), O, lse.cpu().numpy(), L, TOL_O_FP8, what="noalloc after set-up")
