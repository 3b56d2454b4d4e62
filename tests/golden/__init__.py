"""Closed-form MLA cases (``closed_forms.json``, written by ``make_golden.py``) turned into the
input objects the oracle and the CUDA path's tests take, plus their expected outputs.

Loading is storage conversion only: every stored input value must be exactly representable
in its storage type (bf16, fp32; e4m3 and int32 are stored as codes), which is checked.
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np

from gen import DecodeInputs, PrefillInputs, bf16_bits_from_f32

HERE = os.path.dirname(os.path.abspath(__file__))
PATH = os.path.join(HERE, "closed_forms.json")


def _num(v) -> float:
    if isinstance(v, (int, float)):
        return float(v)
    if v in ("nan", "inf", "-inf"):
        return float(v)
    return float(Fraction(v))


def _bf16_value(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _dense(t):
    """The stored array of a sparse tensor description, in its storage type."""
    shape = tuple(t["shape"])
    dt = t["dtype"]
    if dt in ("e4m3", "i32"):
        a = np.full(shape, int(t["fill"]), dtype=np.int64)
        for z in t["zero"]:
            a[tuple(z)] = 0
        for idx, v in t["entries"]:
            a[tuple(idx)] = int(v)
        return a.astype(np.uint8 if dt == "e4m3" else np.int32)
    a = np.full(shape, _num(t["fill"]), dtype=np.float64)
    for z in t["zero"]:
        a[tuple(z)] = 0.0
    for idx, v in t["entries"]:
        a[tuple(idx)] = _num(v)
    if dt == "f64":
        return a
    f32 = a.astype(np.float32)
    if dt == "f32":
        stored = f32.astype(np.float64)
        ok = (stored == a) | (np.isnan(stored) & np.isnan(a))
        assert ok.all(), "value not exact in fp32"
        return f32
    assert dt == "bf16", dt
    bits = bf16_bits_from_f32(f32)
    back = _bf16_value(bits).astype(np.float64)
    ok = (back == a) | (np.isnan(back) & np.isnan(a))
    assert ok.all(), "value not exact in bf16"
    return bits


def load_cases():
    """[(name, inputs, O expected float64, LSE expected float64, case dict)]."""
    with open(PATH) as f:
        raw = json.load(f)["cases"]
    out = []
    for c in raw:
        t = {k: (_dense(v) if v is not None else None) for k, v in c["inputs"].items()}
        if c["kind"] == "prefill":
            inp = PrefillInputs(B=c["B"], H=c["H"], S=c["S"], d_nope=128, d_rope=64, d_v=128,
                                softmax_scale=c["softmax_scale"], causal=c["causal"], fp8=c["fp8"],
                                q_nope=t["q_nope"], q_rope=t["q_rope"], k_nope=t["k_nope"],
                                k_rope=t["k_rope"], v=t["v"], q_scale=t.get("q_scale"),
                                k_scale=t.get("k_scale"), meta={"golden": c["name"]})
        else:
            inp = DecodeInputs(B=c["B"], H=c["H"], T=c["T"], d_latent=512, d_rope=64, page_size=64,
                               num_pages=c["num_pages"], max_pages=c["max_pages"],
                               softmax_scale=c["softmax_scale"], causal=c["causal"], fp8=c["fp8"],
                               q_latent=t["q_latent"], q_rope=t["q_rope"], kv_cache=t["kv_cache"],
                               kv_scale=t["kv_scale"], page_table=t["page_table"],
                               cache_lens=t["cache_lens"], meta={"golden": c["name"]})
        O = _dense(c["expected"]["O"])
        L = np.array([[[_num(x) for x in row] for row in mat] for mat in c["expected"]["LSE"]["values"]])
        assert L.shape == tuple(c["expected"]["LSE"]["shape"])
        out.append((c["name"], inp, O, L, c))
    return out
