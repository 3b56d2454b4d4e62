"""Seeded synthetic inputs for fused MLA attention (prefill and absorbed decode).

This package is shared by the fp64 oracle and by the CUDA path's tests and
benchmark.  It only draws random numbers and stores them in the storage types
the kernels read (bf16 bit patterns, fp8 e4m3 bytes with fp32 per-token scales,
int32 page tables); it contains none of the attention arithmetic.
"""
from .inputs import (  # noqa: F401
    PrefillInputs,
    DecodeInputs,
    make_prefill,
    make_grad_out,
    make_decode,
    CONFIGS,
    config_inputs,
    bf16_bits_from_f32,
)
