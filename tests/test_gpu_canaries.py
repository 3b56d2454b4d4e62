"""Out-of-bounds writes, caught with guard regions: every buffer a kernel writes (outputs, LSE,
workspaces, gradients, the cache) is placed inside a larger allocation whose margins hold a
known byte pattern; after the call, synchronised and with the device error word clear, the
margins must be unchanged.  This stands in for a memory checker, which these tests cannot
run; the outputs themselves are checked against the oracle elsewhere."""
import numpy as np
import pytest
import torch

from gen import make_decode, make_prefill, make_grad_out

pytestmark = pytest.mark.gpu

MARGIN = 4096  # bytes of guard on each side (a multiple of 16: the views stay 16-byte aligned)
PATTERN = 0xA5


class Guarded:
    """A tensor of `shape` and `dtype` inside a byte buffer with MARGIN guard bytes each side."""

    def __init__(self, shape, dtype, fill=None):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((n + 2 * MARGIN,), PATTERN, dtype=torch.uint8, device="cuda")
        self.t = self.buf[MARGIN:MARGIN + n].view(dtype).view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def intact(self):
        torch.cuda.synchronize()
        head = self.buf[:MARGIN].cpu().numpy()
        tail = self.buf[-MARGIN:].cpu().numpy()
        return bool((head == PATTERN).all() and (tail == PATTERN).all())


def _bytes(n):
    return Guarded((n,), torch.uint8)


@pytest.mark.parametrize("fp8", [False, True])
def test_prefill_writes_only_out_and_lse(lib, fp8):
    from mla_flash_attention_gb300.testing import prefill_to_device

    inp = make_prefill(2, 3, 300, fp8=fp8, seed=400 + fp8)
    t = prefill_to_device(inp, torch.device("cuda"))
    odt = torch.float32 if fp8 else torch.bfloat16
    out = Guarded((inp.B, inp.S, inp.H, inp.d_v), odt)
    lse = Guarded((inp.B, inp.H, inp.S), torch.float32)
    lib.mla_prefill(*t["args"], softmax_scale=inp.softmax_scale, causal=True, out=out.t, lse=lse.t)
    lib.check_device_error()
    assert out.intact() and lse.intact()


@pytest.mark.parametrize("fp8,H,T,lens", [
    (True, 16, 2, [1, 700, 3000, 65, 0]),     # transposed kernel (q_len*H <= 32), an empty sequence
    (False, 128, 1, [1, 700, 3000, 65]),      # split-pair kernel
    (False, 40, 5, [5, 130, 777]),            # 200 query rows: a full tile and a 72-row tail
])
def test_decode_writes_only_out_lse_and_workspace(lib, fp8, H, T, lens):
    from mla_flash_attention_gb300.testing import decode_to_device

    inp = make_decode(len(lens), H, T, lens, fp8=fp8, seed=410 + H + T, extra_pages=1)
    d = decode_to_device(inp, torch.device("cuda"))
    out = Guarded((inp.B, inp.T, inp.H, inp.d_latent), torch.bfloat16)
    lse = Guarded((inp.B, inp.H, inp.T), torch.float32)
    ws = _bytes(lib.decode_workspace_size(inp.B, inp.H, inp.T))
    cache = d["args"][2]
    cache_copy = cache.clone()
    lib.mla_decode(*d["args"], **d["kwargs"], softmax_scale=inp.softmax_scale, out=out.t, lse=lse.t,
                   workspace=ws.t)
    lib.check_device_error()
    assert out.intact() and lse.intact() and ws.intact()
    assert torch.equal(cache.view(torch.uint8), cache_copy.view(torch.uint8))  # inputs are read only


def test_decode_noalloc_writes_only_out_and_lse(lib):
    from mla_flash_attention_gb300.testing import decode_to_device

    inp = make_decode(3, 16, 2, [900, 1, 4000], fp8=True, seed=420)
    d = decode_to_device(inp, torch.device("cuda"))
    out = Guarded((inp.B, inp.T, inp.H, inp.d_latent), torch.bfloat16)
    lse = Guarded((inp.B, inp.H, inp.T), torch.float32)
    lib.mla_decode_noalloc(*d["args"], **d["kwargs"], softmax_scale=inp.softmax_scale, out=out.t, lse=lse.t)
    lib.check_device_error()
    assert out.intact() and lse.intact()


@pytest.mark.parametrize("fp8", [False, True])
def test_cache_append_writes_only_the_cache(lib, fp8):
    from mla_flash_attention_gb300.testing import decode_to_device

    inp = make_decode(3, 16, 2, [65, 300, 2], fp8=fp8, seed=430 + fp8)
    d = decode_to_device(inp, torch.device("cuda"))
    cache = Guarded(tuple(d["args"][2].shape), d["args"][2].dtype, fill=d["args"][2])
    scale = None
    if fp8:
        scale = Guarded(tuple(d["kwargs"]["kv_scale"].shape), torch.float32, fill=d["kwargs"]["kv_scale"])
    c_new = torch.randn((inp.B, inp.T, 576), device="cuda").to(torch.bfloat16)
    lib.mla_cache_append(c_new, cache.t, d["args"][3], d["args"][4], kv_scale=None if scale is None else scale.t)
    lib.check_device_error()
    assert cache.intact() and (scale is None or scale.intact())


def test_absorb_writes_only_y(lib):
    x = torch.randn((70, 3, 128), device="cuda").to(torch.bfloat16)
    w = (torch.randn((3, 128, 512), device="cuda") / 11).to(torch.bfloat16)
    y = Guarded((70, 3, 512), torch.bfloat16)
    lib.mla_absorb(x, w, out=y.t)
    lib.check_device_error()
    assert y.intact()


def test_prefill_backward_writes_only_gradients_and_workspace(lib):
    from mla_flash_attention_gb300.testing import prefill_to_device

    inp = make_prefill(1, 2, 200, seed=440)
    bt = prefill_to_device(inp, torch.device("cuda"))["args"][:5]
    o, l = lib.mla_prefill(*bt, None, None, softmax_scale=inp.softmax_scale, causal=True)
    d_out = torch.from_numpy(make_grad_out(1, 200, 2, 128, seed=441).view(np.int16)).view(torch.bfloat16).cuda()
    B, S, H = 1, 200, 2
    g = [Guarded((B, S, H, 128), torch.bfloat16), Guarded((B, S, H, 64), torch.bfloat16),
         Guarded((B, S, H, 128), torch.bfloat16), Guarded((B, S, 64), torch.float32),
         Guarded((B, S, H, 128), torch.bfloat16)]
    ws = _bytes(lib.prefill_backward_workspace_size(B, H, S))
    lib.mla_prefill_backward(*bt, o, l, d_out, softmax_scale=inp.softmax_scale, causal=True,
                             grads=tuple(x.t for x in g), workspace=ws.t)
    lib.check_device_error()
    assert all(x.intact() for x in g) and ws.intact()
