"""fp64 CPU oracle for fused MLA attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  The CUDA library never calls it and
shares no code with it; the two meet only in the seeded input generator
(``gen/``), which holds none of the attention arithmetic.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(library special cases, closed forms, invariants and brute force).  Nothing in
this package is "parity unpinned".
"""
from .mla_ref import (  # noqa: F401
    bf16_to_f64,
    e4m3_to_f64,
    attention_rows,
    prefill_dequant_bh,
    prefill_bh,
    mla_prefill,
    decode_gather,
    decode_b,
    mla_decode,
    lse_combine,
)
from .cache_ref import (  # noqa: F401
    e4m3_encode,
    quantize_row,
    cache_append,
)
from .absorb_ref import absorb  # noqa: F401
from .backward_ref import prefill_backward_bh, mla_prefill_backward  # noqa: F401
