"""Pins of the cache-append oracle (CPU only).

The e4m3 encoder is tied to torch's own float8_e4m3fn conversion (an independent library
route) on every representable value, every half-way point between neighbours and random
values; the row quantisation to the e4m3 error bounds and its special cases; the append to
the decode oracle's own page lookup (so a wrong page, row or position fails), to rows that
must stay untouched, and to a brute-force scalar re-statement of the quantisation.
"""
from types import SimpleNamespace

import numpy as np
import torch

import oracle
from gen import bf16_bits_from_f32


def torch_e4m3(x):
    """float32 -> e4m3 codes through torch's float8_e4m3fn cast (round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_encode_matches_torch_on_all_values_and_midpoints():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_to_f64(codes)
    finite = np.isfinite(vals)
    # every finite value round-trips to its own code (+0 / -0 keep their sign bit)
    v32 = vals[finite].astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(v32), codes[finite])
    assert np.array_equal(torch_e4m3(v32), codes[finite])
    # half-way points between neighbouring magnitudes: ties go to the even code
    pos = np.sort(vals[(codes < 0x7F) & finite & (vals >= 0)])
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.all(mids.astype(np.float64) == (pos[:-1] + pos[1:]) / 2)  # exact in fp32
    for m in (mids, -mids):
        got = oracle.e4m3_encode(m)
        assert np.array_equal(got, torch_e4m3(m))
        assert np.all((got & 1) == 0)


def test_encode_matches_torch_on_random_values():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.uniform(-448, 448, 200_000),
                        rng.standard_normal(100_000) * np.exp2(rng.uniform(-12, 3, 100_000))])
    x = x.astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(x), torch_e4m3(x))


def test_quantize_row_error_bounds_and_special_cases():
    rng = np.random.default_rng(3)
    for mag in (1e-3, 1.0, 37.0, 1e4):
        x = (rng.standard_normal(576) * mag).astype(np.float32)
        codes, scale = oracle.quantize_row(x)
        assert scale == np.float32(np.max(np.abs(x)) / np.float32(448.0))
        back = oracle.e4m3_to_f64(codes) * np.float64(scale)
        err = np.abs(back - x.astype(np.float64))
        y = np.abs(x.astype(np.float64)) / np.float64(scale)
        normal = y >= 2.0 ** -6
        # half a unit in the last place: 2^-4 relative for normals, 2^-10 (times scale) below
        assert np.all(err[normal] <= 2.0 ** -4 * np.abs(x[normal]) * (1 + 1e-6))
        assert np.all(err[~normal] <= 2.0 ** -10 * scale * (1 + 1e-6))
        # the largest magnitude maps to 448 (code 0x7e, with the sign)
        k = int(np.argmax(np.abs(x)))
        assert codes[k] & 0x7F == 0x7E
    codes, scale = oracle.quantize_row(np.zeros(576, np.float32))
    assert scale == 1.0 and not codes.any()


def test_quantize_row_matches_scalar_restatement():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(64) * 3).astype(np.float32)
    codes, scale = oracle.quantize_row(x)
    table = {int(c): float(v) for c, v in zip(range(0x7F), oracle.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8)))}
    for xi, ci in zip(x, codes):
        y = float(np.float32(xi / scale))
        best = min(table, key=lambda c: (abs(table[c] - abs(y)), c & 1))
        assert int(ci) == (best | (0x80 if y < 0 else 0))


def _cache_case(fp8, seed=5):
    rng = np.random.default_rng(seed)
    B, T, D, P = 5, 2, 576, 64
    lens = np.array([1, 2, 64, 65, 130], np.int32)          # L < T, page edges, second page
    max_pages = 3
    num_pages = 16
    perm = rng.permutation(num_pages)
    pt = np.full((B, max_pages), -1, np.int32)
    k = 0
    for b in range(B):
        for p in range((lens[b] + P - 1) // P):
            pt[b, p] = perm[k]
            k += 1
    new = bf16_bits_from_f32(rng.standard_normal((B, T, D)).astype(np.float32) * 2)
    if fp8:
        cache = rng.integers(0, 0x7E, (num_pages, P, D)).astype(np.uint8)
        scales = rng.uniform(0.5, 2, (num_pages, P)).astype(np.float32)
    else:
        cache = bf16_bits_from_f32(rng.standard_normal((num_pages, P, D)).astype(np.float32))
        scales = None
    return SimpleNamespace(B=B, T=T, lens=lens, pt=pt, new=new, cache=cache, scales=scales, P=P)


def _gather(c, cache, scales, fp8):
    return SimpleNamespace(cache_lens=c.lens, page_table=c.pt, page_size=c.P, kv_cache=cache,
                           kv_scale=scales, fp8=fp8)


def test_append_lands_where_decode_reads_and_touches_nothing_else():
    for fp8 in (False, True):
        c = _cache_case(fp8)
        cache, scales = oracle.cache_append(c.new, c.cache, c.scales, c.pt, c.lens, c.P, fp8)
        written = np.zeros(cache.shape[:2], bool)
        for b in range(c.B):
            rows = oracle.decode_gather(_gather(c, cache, scales, fp8), b)   # [L_b, D]
            for t in range(c.T):
                pos = int(c.lens[b]) - c.T + t
                if pos < 0:
                    continue
                want = oracle.bf16_to_f64(c.new[b, t])
                got = rows[pos]
                if fp8:
                    codes, sc = oracle.quantize_row(want.astype(np.float32))
                    assert np.array_equal(got, oracle.e4m3_to_f64(codes) * np.float64(sc))
                    assert np.all(np.abs(got - want) <= 2.0 ** -4 * np.abs(want) + 2.0 ** -10 * sc)
                else:
                    assert np.array_equal(got, want)
                written[c.pt[b, pos // c.P], pos % c.P] = True
        assert written.sum() == sum(max(0, min(c.T, int(L))) for L in c.lens)
        assert np.array_equal(cache[~written], c.cache[~written])
        if fp8:
            assert np.array_equal(scales[~written], c.scales[~written])
