"""GPU parity of mla_cache_append (through the C ABI) against the oracle: bit-exact.

Appending is integer/byte work once the fp32 decisions are taken (same IEEE fp32 division
and scale on both sides), so the whole cache (codes or bf16 bits) and every scale must be
identical to the oracle's, including the rows that must not be touched (which hold NaN
past each sequence's end).
"""
import numpy as np
import pytest
import torch

import oracle
from gen import bf16_bits_from_f32, config_inputs, make_decode
from tests.parity import TOL_O_BF16, TOL_O_FP8, check

pytestmark = pytest.mark.gpu


def new_rows(B, T, seed, mag=1.0, zero_rows=()):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, T, 576)).astype(np.float32) * np.float32(mag)
    for b, t in zero_rows:
        x[b, t] = 0
    return bf16_bits_from_f32(x)


def run(lib, inp, c_new_bits):
    """(cache bits/codes, scales) after the GPU append, as numpy."""
    dev = torch.device("cuda")
    c_new = torch.from_numpy(np.ascontiguousarray(c_new_bits).view(np.int16)).view(torch.bfloat16).to(dev)
    if inp.fp8:
        cache = torch.from_numpy(np.ascontiguousarray(inp.kv_cache)).view(torch.float8_e4m3fn).to(dev)
        scale = torch.from_numpy(np.ascontiguousarray(inp.kv_scale)).to(dev)
    else:
        cache = torch.from_numpy(np.ascontiguousarray(inp.kv_cache).view(np.int16)).view(torch.bfloat16).to(dev)
        scale = None
    pt = torch.from_numpy(inp.page_table).to(dev)
    lens = torch.from_numpy(inp.cache_lens).to(dev)
    lib.mla_cache_append(c_new, cache, pt, lens, kv_scale=scale)
    lib.check_device_error()
    if inp.fp8:
        return cache.view(torch.uint8).cpu().numpy(), scale.cpu().numpy()
    return cache.view(torch.int16).cpu().numpy().view(np.uint16), None


def expect(inp, c_new_bits):
    return oracle.cache_append(c_new_bits, inp.kv_cache, inp.kv_scale, inp.page_table,
                               inp.cache_lens, inp.page_size, inp.fp8)


def same(got, want):
    assert got[0].shape == want[0].shape
    bad = np.argwhere(got[0] != want[0])
    assert bad.size == 0, "cache differs at %s (got %s, want %s)" % (
        bad[0], got[0][tuple(bad[0])], want[0][tuple(bad[0])])
    if want[1] is not None:
        assert np.array_equal(got[1].view(np.uint32), want[1].view(np.uint32))


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("T", [1, 2, 5])
def test_page_edges_and_short_sequences(lib, fp8, T):
    lens = [1, 2, 63, 64, 65, 127, 128, 129, 3000]  # includes L < T (nothing before position 0)
    inp = make_decode(len(lens), 4, T, lens, fp8=fp8, seed=31 + T, extra_pages=2)
    c = new_rows(inp.B, T, seed=7 + T)
    same(run(lib, inp, c), expect(inp, c))


@pytest.mark.parametrize("mag", [1e-3, 1.0, 40.0, 1e4])
def test_fp8_magnitudes_and_zero_rows(lib, mag):
    inp = make_decode(6, 4, 3, [3, 64, 65, 500, 2, 9], fp8=True, seed=41)
    c = new_rows(6, 3, seed=int(mag * 1000) % 97, mag=mag, zero_rows=[(0, 1), (3, 2)])
    got, want = run(lib, inp, c), expect(inp, c)
    same(got, want)
    # the all-zero rows got scale 1 and zero codes
    for b, t in [(0, 1), (3, 2)]:
        pos = int(inp.cache_lens[b]) - 3 + t
        page, r = inp.page_table[b, pos // 64], pos % 64
        assert got[1][page, r] == 1.0 and not got[0][page, r].any()


def test_bad_page_is_reported_and_skipped(lib):
    inp = make_decode(3, 4, 1, [10, 70, 5], fp8=True, seed=43)
    inp.page_table[1, 1] = inp.num_pages + 5  # sequence 1 appends into its second page
    c = new_rows(3, 1, seed=3)
    dev = torch.device("cuda")
    c_new = torch.from_numpy(c.view(np.int16)).view(torch.bfloat16).to(dev)
    cache = torch.from_numpy(inp.kv_cache.copy()).view(torch.float8_e4m3fn).to(dev)
    scale = torch.from_numpy(inp.kv_scale.copy()).to(dev)
    lib.mla_cache_append(c_new, cache, torch.from_numpy(inp.page_table).to(dev),
                         torch.from_numpy(inp.cache_lens).to(dev), kv_scale=scale)
    with pytest.raises(lib.MLAError):
        lib.check_device_error()
    # the other two sequences were still written; nothing was written for sequence 1
    inp_ok = make_decode(3, 4, 1, [10, 70, 5], fp8=True, seed=43)
    want_cache, want_scale = oracle.cache_append(c[[0, 2]], inp_ok.kv_cache, inp_ok.kv_scale,
                                                 inp_ok.page_table[[0, 2]], inp_ok.cache_lens[[0, 2]],
                                                 64, True)
    assert np.array_equal(cache.view(torch.uint8).cpu().numpy(), want_cache)
    assert np.array_equal(scale.cpu().numpy().view(np.uint32), want_scale.view(np.uint32))


@pytest.mark.slow
def test_full_size_fp8_cache(lib):
    # the ragged fp8 decode workload: 128 sequences, 2 new tokens each, 1.2 GB cache
    inp = config_inputs("decode_b128h16t2_ragged_fp8")
    c = new_rows(inp.B, inp.T, seed=1004)
    same(run(lib, inp, c), expect(inp, c))


@pytest.mark.parametrize("fp8", [False, True])
def test_append_then_decode(lib, fp8):
    from mla_flash_attention_gb300.testing import decode_to_device

    inp = make_decode(4, 16, 2, [2, 65, 700, 1500], fp8=fp8, seed=53)
    c = new_rows(4, 2, seed=9)
    cache, scale = run(lib, inp, c)
    inp.kv_cache, inp.kv_scale = cache, scale
    d = decode_to_device(inp, torch.device("cuda"))
    out, lse = lib.mla_decode(*d["args"], **d["kwargs"], softmax_scale=inp.softmax_scale, causal=True)
    lib.check_device_error()
    want = expect(make_decode(4, 16, 2, [2, 65, 700, 1500], fp8=fp8, seed=53), c)
    inp.kv_cache, inp.kv_scale = want
    O, L = oracle.mla_decode(inp)
    check(out.float().cpu().numpy(), O, lse.cpu().numpy(), L, TOL_O_FP8 if fp8 else TOL_O_BF16,
          what="append+decode fp8=%d" % fp8)
