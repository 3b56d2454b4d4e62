"""Failure detection by timeout, without faulting the GPU: a test hook makes the decode
producer leave one pipeline unit unloaded and shortens every device wait, so the stage that
waits for it runs out.  The kernel must report MLA_ERR_TIMEOUT through the device error word,
leave nothing in flight, and the next ordinary call on the same context must be correct.

The waits are the pipeline barriers of the KVPipelineGeneric page (nn/attention/gpu/nvidia/
sm100/mla_decode_utils, Methods producer_acquire / consumer_wait), bounded here.
"""
import numpy as np
import pytest
import torch

import oracle
from gen import make_decode
from tests.parity import TOL_O_FP8, check

pytestmark = pytest.mark.gpu


def _call(lib, inp):
    from mla_flash_attention_gb300.testing import decode_to_device

    d = decode_to_device(inp, torch.device("cuda"))
    out, lse = lib.mla_decode(*d["args"], **d["kwargs"], softmax_scale=inp.softmax_scale)
    return out, lse


# (skipped unit, cache lengths): the first unit of a CTA, the first value unit of its first
# block (units 0-8 are that block's score units), and a unit deep into a CTA's work -- the
# 80,000 keys of the last case give every CTA at least 9 pages, i.e. 5 blocks and 81 units
@pytest.mark.parametrize("skip_unit,lens", [(0, [700, 3000, 65, 1500]), (9, [700, 3000, 65, 1500]),
                                            (30, [20000] * 4)])
def test_decode_wait_runs_out_and_the_next_call_is_correct(lib, skip_unit, lens):
    from mla_flash_attention_gb300.binding import MLAError

    inp = make_decode(len(lens), 16, 2, lens, fp8=True, seed=90 + skip_unit)
    lib.check_device_error()
    lib.testing_decode_stall(skip_unit, 200000)  # ~0.1 ms per wait
    try:
        _call(lib, inp)
        with pytest.raises(MLAError, match="TIMEOUT"):
            lib.check_device_error()
    finally:
        lib.testing_decode_stall()
    lib.check_device_error()  # the word was cleared and nothing else was latched
    out, lse = _call(lib, inp)
    lib.check_device_error()
    O, L = oracle.mla_decode(inp)
    check(out.float().cpu().numpy(), O, lse.cpu().numpy(), L, TOL_O_FP8, what="after a timeout")
