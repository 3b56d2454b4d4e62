"""The bounds-checked build (compiled with MLA_DEBUG): every output, LSE and workspace store
of the prefill and decode kernels is checked against its buffer on the device; a store that
would fall outside is skipped and latched as MLA_ERR_DEVICE_CHECK.

Two properties, each in a child process that loads that build (MLA_GB300_LIB):
* the kernels run clean under it -- the error word stays clear and every output equals the
  normal build's, bit for bit (the checks change no arithmetic);
* its checks are live -- with the output reported one row short (a test hook that only
  changes the size the checks compare against), the last row's stores are skipped and the
  call reports MLA_ERR_DEVICE_CHECK, while every other row is still written.  No store
  leaves the real buffer either way.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from gen import make_decode, make_prefill

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, kind, generator arguments): the bf16 and fp8 prefill, the split decode (bf16, a
# 200-row sequence in two query tiles) and the transposed fp8 decode
CASES = [
    ("prefill_bf16", "prefill", dict(B=2, H=3, S=300, fp8=False, seed=700)),
    ("prefill_fp8", "prefill", dict(B=1, H=2, S=260, fp8=True, seed=701)),
    ("decode_split", "decode", dict(B=3, H=40, T=5, lens=[5, 130, 777], fp8=False, seed=702)),
    ("decode_fp8_t", "decode", dict(B=3, H=16, T=2, lens=[900, 1, 4000], fp8=True, seed=703)),
]

CHILD = r"""
import os, sys
import numpy as np, torch
sys.path.insert(0, os.environ["MLA_REPO"])
from tests.test_gpu_bounds_build import CASES, run_case
from mla_flash_attention_gb300 import binding
assert binding.testing_bounds_checked(), "the child did not load the bounds-checked build"
mode = sys.argv[1]
res = {}
for name, kind, kw in CASES:
    if mode == "clean":
        o, l = run_case(kind, kw)
        binding.check_device_error()
    else:
        o, l = run_case(kind, kw, shrink_one_row=True)
        try:
            binding.check_device_error()
            raise SystemExit("%s: a store past the reported end was not caught" % name)
        except binding.MLAError as e:
            assert e.status == 6, e  # MLA_ERR_DEVICE_CHECK
    res[name + "_o"] = o
    res[name + "_l"] = l
np.savez(sys.argv[2], **res)
print("child ok")
"""


def run_case(kind, kw, shrink_one_row=False):
    """Run one case through the loaded library; the output starts as a 0x7f byte pattern so
    that rows the call did not write are recognisable.  Returns (out bytes, lse) on the host."""
    from mla_flash_attention_gb300 import binding
    from mla_flash_attention_gb300.testing import decode_to_device, prefill_to_device

    dev = torch.device("cuda")
    if kind == "prefill":
        inp = make_prefill(kw["B"], kw["H"], kw["S"], fp8=kw["fp8"], seed=kw["seed"])
        t = prefill_to_device(inp, dev)
        odt = torch.float32 if inp.fp8 else torch.bfloat16
        out = torch.empty((inp.B, inp.S, inp.H, inp.d_v), dtype=odt, device=dev)
        lse = torch.empty((inp.B, inp.H, inp.S), dtype=torch.float32, device=dev)
        out.view(torch.uint8).fill_(0x7F)
        row = inp.d_v * out.element_size()
        binding.testing_bounds_shrink(row if shrink_one_row else 0)
        try:
            binding.mla_prefill(*t["args"], softmax_scale=inp.softmax_scale, causal=True, out=out, lse=lse)
        finally:
            binding.testing_bounds_shrink(0)
    else:
        inp = make_decode(len(kw["lens"]), kw["H"], kw["T"], kw["lens"], fp8=kw["fp8"], seed=kw["seed"])
        d = decode_to_device(inp, dev)
        out = torch.empty((inp.B, inp.T, inp.H, inp.d_latent), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((inp.B, inp.H, inp.T), dtype=torch.float32, device=dev)
        out.view(torch.uint8).fill_(0x7F)
        row = inp.d_latent * 2
        binding.testing_bounds_shrink(row if shrink_one_row else 0)
        try:
            binding.mla_decode(*d["args"], **d["kwargs"], softmax_scale=inp.softmax_scale, out=out, lse=lse)
        finally:
            binding.testing_bounds_shrink(0)
    torch.cuda.synchronize()
    return out.view(torch.uint8).cpu().numpy().reshape(-1, row), lse.cpu().numpy()


@pytest.fixture(scope="module")
def debug_lib():
    from mla_flash_attention_gb300 import build

    return build.build(debug=True)


def _child(debug_lib, mode, tmp_path):
    path = str(tmp_path / ("%s.npz" % mode))
    env = dict(os.environ, MLA_GB300_LIB=debug_lib, MLA_REPO=ROOT)
    r = subprocess.run([sys.executable, "-c", CHILD, mode, path], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    return np.load(path)


def test_normal_build_has_no_checks(lib):
    assert not lib.testing_bounds_checked()


def test_kernels_run_clean_and_identical_under_the_checks(lib, debug_lib, tmp_path):
    got = _child(debug_lib, "clean", tmp_path)
    for name, kind, kw in CASES:
        o, l = run_case(kind, kw)
        lib.check_device_error()
        assert np.array_equal(got[name + "_o"], o), name
        assert np.array_equal(got[name + "_l"], l, equal_nan=True), name


def test_checks_catch_a_store_past_the_reported_end(lib, debug_lib, tmp_path):
    got = _child(debug_lib, "shrunk", tmp_path)
    for name, kind, kw in CASES:
        o, _ = run_case(kind, kw)
        lib.check_device_error()
        g = got[name + "_o"]
        assert (g[-1] == 0x7F).all(), "%s: the last row was written past the reported end" % name
        assert np.array_equal(g[:-1], o[:-1]), "%s: rows before the end differ" % name
