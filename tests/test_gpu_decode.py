"""GPU parity of mla_decode (split-KV with the merge of the splits fused in, through the C ABI)
against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from gen import config_inputs, make_decode
from tests.parity import TOL_O_BF16, TOL_O_FP8, check

pytestmark = pytest.mark.gpu


def run(lib, inp, causal=None):
    from mla_flash_attention_gb300.testing import decode_to_device

    d = decode_to_device(inp, torch.device("cuda"))
    out, lse = lib.mla_decode(*d["args"], **d["kwargs"], softmax_scale=inp.softmax_scale,
                              causal=inp.causal if causal is None else causal)
    lib.check_device_error()
    return out.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("lens", [[1], [63], [64], [65], [1, 63, 64, 65, 129, 4000]])
def test_page_boundaries(lib, fp8, lens):
    inp = make_decode(len(lens), 16, 1, lens, fp8=fp8, seed=sum(lens))
    o, l = run(lib, inp)
    O, L = oracle.mla_decode(inp)
    check(o, O, l, L, TOL_O_FP8 if fp8 else TOL_O_BF16, what="lens=%s fp8=%d" % (lens, fp8))


@pytest.mark.parametrize("fp8", [False, True])
def test_two_new_tokens_with_empty_row(lib, fp8):
    # L=1 with q_len=2: new token 0 sees no key (O=0, LSE=-inf)
    inp = make_decode(4, 16, 2, [1, 2, 3, 1000], fp8=fp8, seed=17)
    o, l = run(lib, inp)
    O, L = oracle.mla_decode(inp)
    assert np.isneginf(L[0, :, 0]).all()
    check(o, O, l, L, TOL_O_FP8 if fp8 else TOL_O_BF16, what="q_len=2")


@pytest.mark.parametrize("H,T", [(128, 1), (64, 2), (3, 3), (1, 1), (32, 4)])
def test_head_and_token_counts(lib, H, T):
    inp = make_decode(3, H, T, [T, 700, 2049], seed=H * 10 + T)
    o, l = run(lib, inp)
    O, L = oracle.mla_decode(inp)
    check(o, O, l, L, TOL_O_BF16, what="H=%d T=%d" % (H, T))


def test_non_causal(lib):
    inp = make_decode(2, 8, 3, [5, 300], seed=23, causal=False)
    o, l = run(lib, inp)
    O, L = oracle.mla_decode(inp)
    check(o, O, l, L, TOL_O_BF16, what="non-causal")


def test_zero_length_sequence(lib):
    inp = make_decode(3, 8, 1, [0, 70, 0], seed=29, extra_pages=1)
    o, l = run(lib, inp)
    O, L = oracle.mla_decode(inp)
    assert (O[0] == 0).all() and np.isneginf(L[0]).all()
    check(o, O, l, L, TOL_O_BF16, what="L=0")


def test_many_short_sequences(lib):
    # more sequences than work CTAs: one CTA walks through several sequences
    lens = list(np.random.default_rng(3).integers(1, 130, size=400))
    inp = make_decode(400, 4, 1, lens, seed=31)
    o, l = run(lib, inp)
    O, L = oracle.mla_decode(inp)
    check(o, O, l, L, TOL_O_BF16, what="400 short")


def test_one_long_sequence(lib):
    # one sequence split across every work CTA
    inp = make_decode(1, 128, 1, [32768], seed=37)
    o, l = run(lib, inp)
    O, L = oracle.mla_decode(inp)
    check(o, O, l, L, TOL_O_BF16, what="one long")


def test_bad_page_is_reported(lib):
    inp = make_decode(2, 4, 1, [100, 100], seed=41)
    inp.page_table[1, 1] = inp.num_pages + 5  # out of range: skipped and reported
    from mla_flash_attention_gb300.binding import MLAError
    from mla_flash_attention_gb300.testing import decode_to_device

    d = decode_to_device(inp, torch.device("cuda"))
    lib.mla_decode(*d["args"], **d["kwargs"], softmax_scale=inp.softmax_scale)
    with pytest.raises(MLAError, match="DEVICE_CHECK"):
        lib.check_device_error()
    lib.check_device_error()  # the word was cleared


@pytest.mark.slow
@pytest.mark.parametrize("name,tol", [("decode_b64h128t1l4096_bf16", TOL_O_BF16),
                                      ("decode_b128h16t2_ragged_fp8", TOL_O_FP8)])
def test_full_size_configs(lib, name, tol):
    inp = config_inputs(name)
    o, l = run(lib, inp)
    O, L = oracle.mla_decode(inp)
    check(o, O, l, L, tol, what=name)


def test_fp8_widening_is_exact_for_every_code(lib):
    # One visible key whose latent columns hold every finite e4m3 code (subnormals and both
    # zeros included) with scale 1: P' = 1 and O is that row, so the bf16 output must equal
    # the decoded codes exactly (each e4m3 value is a bf16 value).
    inp = make_decode(1, 1, 1, [1], fp8=True, seed=61)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    row = np.resize(finite, 576).astype(np.uint8)
    row[512:] = 0  # rope columns: no contribution needed
    page = int(inp.page_table[0, 0])
    inp.kv_cache[page, 0] = row
    inp.kv_scale[page, 0] = 1.0
    o, l = run(lib, inp)
    want = oracle.e4m3_to_f64(row[:512])
    assert np.array_equal(o[0, 0, 0], want), np.argwhere(o[0, 0, 0] != want)[:5]


# ---------------------------------------------------------------- query rows beyond one tile
# q_len * H > 128: the rows of a sequence are processed in tiles of 128 (each planned as its
# own work item); q_len new tokens over a paged prefix is chunked prefill in absorbed form.

@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("B,H,T,lens", [
    (2, 128, 4, [300, 1000]),          # 512 rows: 4 full tiles
    (3, 40, 5, [5, 130, 777]),         # 200 rows: a full tile and a 72-row tail
    (2, 16, 64, [64, 2000]),           # 1024 rows: a 64-token chunk over a prefix
    (1, 3, 50, [49]),                  # 150 rows, L < q_len (the first token sees nothing)
])
def test_query_rows_beyond_one_tile(lib, fp8, B, H, T, lens):
    inp = make_decode(B, H, T, lens, fp8=fp8, seed=B * 100 + H + T)
    o, l = run(lib, inp)
    O, L = oracle.mla_decode(inp)
    check(o, O, l, L, TOL_O_FP8 if fp8 else TOL_O_BF16, what="B=%d H=%d T=%d fp8=%d" % (B, H, T, fp8))


def test_chunked_prefill_chunk_of_32_tokens_at_128_heads(lib):
    inp = make_decode(2, 128, 32, [1024, 3000], seed=77)
    o, l = run(lib, inp)
    O, L = oracle.mla_decode(inp)
    check(o, O, l, L, TOL_O_BF16, what="chunk T=32 H=128")
