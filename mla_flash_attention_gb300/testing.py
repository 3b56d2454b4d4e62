"""Upload generator outputs (numpy storage arrays) to device tensors of the types the
library reads.  Pure data movement: bf16 bit patterns are viewed as bfloat16, e4m3
codes as float8_e4m3fn."""
from __future__ import annotations

import numpy as np
import torch


def _bf16(a, dev, pin=False):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pin else t.to(dev)


def _e4m3(a, dev, pin=False):
    t = torch.from_numpy(np.ascontiguousarray(a)).view(torch.float8_e4m3fn)
    return t.pin_memory() if pin else t.to(dev)


def _plain(a, dev, pin=False):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.pin_memory() if pin else t.to(dev)


def prefill_to_device(inp, dev, pin=False):
    """Tensors for binding.mla_prefill (on ``dev``, or pinned host memory if ``pin``)."""
    nope = _e4m3 if inp.fp8 else _bf16
    args = [nope(inp.q_nope, dev, pin), _bf16(inp.q_rope, dev, pin), nope(inp.k_nope, dev, pin),
            _bf16(inp.k_rope, dev, pin), nope(inp.v, dev, pin)]
    if inp.fp8:
        args += [_plain(inp.q_scale, dev, pin), _plain(inp.k_scale, dev, pin)]
    else:
        args += [None, None]
    return {"args": args}


def decode_to_device(inp, dev, pin=False):
    """Tensors for binding.mla_decode (on ``dev``, or pinned host memory if ``pin``)."""
    cache = _e4m3(inp.kv_cache, dev, pin) if inp.fp8 else _bf16(inp.kv_cache, dev, pin)
    args = [_bf16(inp.q_latent, dev, pin), _bf16(inp.q_rope, dev, pin), cache,
            _plain(inp.page_table, dev, pin), _plain(inp.cache_lens, dev, pin)]
    kwargs = {"kv_scale": _plain(inp.kv_scale, dev, pin) if inp.fp8 else None}
    return {"args": args, "kwargs": kwargs}
