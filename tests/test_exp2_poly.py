"""The polynomial 2^x used for part of the prefill exponentials (CPU check of its error bound).

The kernel evaluates the cubic in fp32 after the round-to-nearest reduction; this test reads
the coefficients from the CUDA header and replays the same fp32 steps in numpy against
numpy's exp2 over the whole range the softmax feeds it.
"""
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _coeffs():
    src = open(os.path.join(ROOT, "mla_flash_attention_gb300", "csrc", "sm103_ptx.cuh")).read()
    return [np.float32(float(re.search(r"kEx2C%d = ([0-9.eE+-]+)f;" % k, src).group(1)))
            for k in range(4)]


def _ex2_poly(x):
    c0, c1, c2, c3 = _coeffs()
    x = np.maximum(x.astype(np.float32), np.float32(-125.0))
    t = (x + np.float32(12582912.0)).astype(np.float32)
    n = (t - np.float32(12582912.0)).astype(np.float32)
    f = (x - n).astype(np.float32)
    p = (f * c3 + c2).astype(np.float32)
    p = (p * f + c1).astype(np.float32)
    p = (p * f + c0).astype(np.float32)
    return (p.view(np.int32) + (t.view(np.int32) << 23)).view(np.float32)


def test_relative_error_bound_over_the_softmax_range():
    x = np.concatenate([np.linspace(-125, 8, 3_000_001), np.arange(-125, 9)]).astype(np.float32)
    got = _ex2_poly(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(got - ref) / ref
    assert rel.max() <= 1.5e-4, rel.max()
    # far below the 2^-9 relative rounding of the bf16 probabilities it feeds
    assert rel.max() < 2.0 ** -9 / 10


def test_masked_scores_vanish():
    got = _ex2_poly(np.array([-np.inf, -1e30, -200.0], dtype=np.float32))
    assert np.all(got > 0) and np.all(got < 3e-38)
