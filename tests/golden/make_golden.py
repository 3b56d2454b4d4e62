"""Writes ``closed_forms.json``: small MLA problems whose exact outputs follow by hand from
the definitions, with their inputs.

The pages print no worked example (no input/output values), so these cases are built so
that the answer is a closed form: all visible scores equal (softmax weights 1/n, O the
mean of the visible value rows, LSE = s + ln n), a single visible key (O = that key's
value row, LSE = its score), or one key whose score exceeds all others by 200 (O = that
row and LSE = 200 to within e^-200 < 1e-86 relative, far below float64 resolution).
Expected values are computed here with exact rationals (``fractions``) and ``math.log``
of small integers; nothing here calls the oracle or the CUDA library.

What the cases rest on (the pages' definitions, restated):

* attention step "S = Q@K' and O += P@V" with P the softmax of S (Modular API docs,
  ``nn/attention/gpu/nvidia/sm100/mla_decode_utils/KVPipelineGeneric``, struct
  description), the score being the sum of the nope and the rope dot products
  (``.../sm100/mla_prefill_per_token_scale/MLASmemStorage``, Fields ``q_smem`` /
  ``kv_smem``);
* per-token fp32 ``q_scale`` / ``k_scale`` on the fp8 nope parts (same page, Fields
  ``q_scale_smem`` / ``k_scale_smem``);
* e4m3 codes: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is subnormal
  (m/8 * 2^-6), S.1111.111 is NaN (OCP 8-bit floating point, E4M3).

Readings the cases exercise (the same ones the oracle documents): LSE is the natural
log-sum-exp of the scaled scores, [B, H, S] / [B, H, T]; prefill causal is square (query
i sees keys 0..i); decode cache_len counts the T new tokens, query t sees keys
0..L-T+t; a row that sees no key has O = 0 and LSE = -inf; fp8 scales dequantise
K_nope and V alike; the fp8 decode cache row (latent and rope) shares one scale.

Run ``python tests/golden/make_golden.py`` to rewrite the file; ``tests/test_golden.py``
checks that the committed file is what this script writes.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction as F

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(HERE, "closed_forms.json")

DN, DR, DV, DL, PAGE = 128, 64, 128, 512, 64

# e4m3 codes used below and their values, from the format: (-1)^s 2^(e-7) (1 + m/8),
# or (-1)^s 2^-6 m/8 when e = 0
E4M3 = {
    0x01: F(1, 512),          # e=0 m=1: 2^-9, the smallest subnormal
    0x07: F(7, 512),          # e=0 m=7: the largest subnormal
    0x08: F(1, 64),           # e=1 m=0: 2^-6, the smallest normal
    0x0F: F(15, 512),         # e=1 m=7: 1.875 * 2^-6
    0x38: F(1),               # e=7 m=0
    0x3F: F(15, 8),           # e=7 m=7
    0x40: F(2),               # e=8 m=0
    0x48: F(4),               # e=9 m=0
    0x70: F(128),             # e=14 m=0
    0x7E: F(448),             # e=15 m=6: the largest finite value
    0x80: F(0),               # negative zero
    0xB8: F(-1),
    0xC8: F(-4),
    0xFE: F(-448),
}


def _s(x: F) -> str:
    return str(x.numerator) if x.denominator == 1 else "%d/%d" % (x.numerator, x.denominator)


def tensor(dtype, shape, entries, fill="0", zero=()):
    """A sparse tensor: ``fill`` everywhere, then 0 on the sub-arrays whose leading indices
    are listed in ``zero``, then ``entries`` ({index tuple: value})."""
    return {"dtype": dtype, "shape": list(shape), "fill": fill, "zero": [list(z) for z in zero],
            "entries": [[list(k), v if isinstance(v, int) and dtype in ("e4m3", "i32") else _s(F(v))]
                        for k, v in sorted(entries.items())]}


def mean(rows):
    """Exact mean of equal-length lists of Fractions."""
    n = len(rows)
    return [sum(col, F(0)) / n for col in zip(*rows)]


# ---------------------------------------------------------------------------- prefill

def _prefill_values(S, H):
    """Sparse V rows (columns 0, 1, 64, 127) and K entries that the zero query ignores."""
    cols = (0, 1, 64, 127)

    def v_row(j, h):
        return {0: F(j + 1 + 10 * h), 1: F((-1) ** j * (h + 1)), 64: F(j * j, 4), 127: F(3 - 2 * j)}

    v = {(0, j, h, c): val for j in range(S) for h in range(H) for c, val in v_row(j, h).items()}
    k_nope = {(0, j, h, c): F((j + c + h) % 5 - 2) for j in range(S) for h in range(H) for c in range(4)}
    k_rope = {(0, j, c): F((2 * j + c) % 7 - 3, 2) for j in range(S) for c in range(3)}
    return cols, v_row, v, k_nope, k_rope


def _o_entries(rows_by_index, cols):
    out = {}
    for idx, row in rows_by_index.items():
        for c, val in zip(cols, row):
            if val != 0:
                out[idx + (c,)] = val
    return out


def case_prefill_zero_query(causal):
    S, H = 6, 2
    cols, v_row, v, k_nope, k_rope = _prefill_values(S, H)
    o, lse = {}, []
    for h in range(H):
        lrow = []
        for i in range(S):
            n = i + 1 if causal else S
            o[(0, i, h)] = mean([[v_row(j, h)[c] for c in cols] for j in range(n)])
            lrow.append(math.log(n))
        lse.append(lrow)
    return {
        "name": "prefill_zero_query_" + ("causal" if causal else "full"),
        "kind": "prefill",
        "derivation": "Q = 0, so every score is 0 and each query row gives equal weight to its "
                      "n visible keys: O_i = mean of the visible V rows, LSE_i = ln n "
                      "(n = i + 1 causal, n = S otherwise); K holds values the zero query ignores.",
        "B": 1, "H": H, "S": S, "fp8": False, "causal": causal, "softmax_scale": 1 / math.sqrt(192),
        "inputs": {
            "q_nope": tensor("bf16", (1, S, H, DN), {}),
            "q_rope": tensor("bf16", (1, S, H, DR), {}),
            "k_nope": tensor("bf16", (1, S, H, DN), k_nope),
            "k_rope": tensor("bf16", (1, S, DR), k_rope),
            "v": tensor("bf16", (1, S, H, DV), v),
        },
        "expected": {"O": tensor("f64", (1, S, H, DV), _o_entries(o, cols)),
                     "LSE": {"shape": [1, H, S], "values": [lse]}},
    }


def case_prefill_dominant_key():
    S, H, key = 6, 1, 3
    cols, v_row, v, _, _ = _prefill_values(S, H)
    # score of key 3 = sigma (16 * 150 + 8 * 100) = 200 with sigma = 1/16; every other score 0
    q_nope = {(0, i, 0, 0): F(16) for i in range(S)}
    q_rope = {(0, i, 0, 0): F(8) for i in range(S)}
    k_nope = {(0, key, 0, 0): F(150)}
    k_rope = {(0, key, 0): F(100)}
    o, lse = {}, []
    for i in range(S):
        if i < key:
            o[(0, i, 0)] = mean([[v_row(j, 0)[c] for c in cols] for j in range(i + 1)])
            lse.append(math.log(i + 1))
        else:
            o[(0, i, 0)] = [v_row(key, 0)[c] for c in cols]
            lse.append(200.0)
    return {
        "name": "prefill_dominant_key",
        "kind": "prefill",
        "derivation": "sigma = 1/16; key 3 scores sigma (16*150 + 8*100) = 200 (nope 150, rope 50), "
                      "every other key 0.  Rows i < 3 do not see key 3: O = mean of V[0..i], "
                      "LSE = ln(i+1).  Rows i >= 3: O = V[3] and LSE = 200 + ln(1 + i e^-200) = 200 "
                      "(the other keys weigh e^-200 < 1e-86).  Dropping the rope term gives LSE 150.",
        "B": 1, "H": H, "S": S, "fp8": False, "causal": True, "softmax_scale": 0.0625,
        "inputs": {
            "q_nope": tensor("bf16", (1, S, H, DN), q_nope),
            "q_rope": tensor("bf16", (1, S, H, DR), q_rope),
            "k_nope": tensor("bf16", (1, S, H, DN), k_nope),
            "k_rope": tensor("bf16", (1, S, DR), k_rope),
            "v": tensor("bf16", (1, S, H, DV), v),
        },
        "expected": {"O": tensor("f64", (1, S, H, DV), _o_entries(o, cols)),
                     "LSE": {"shape": [1, H, S], "values": [[lse]]}},
    }


def case_prefill_fp8_scales():
    S, H, key = 5, 1, 2
    k_scale = [F(1), F(2), F(75, 64), F(4), F(5)]
    q_scale = [F(4)] * S
    # q_nope code 0x48 = 4, times q_scale 4 = 16; key 2's k_nope code 0x70 = 128 times
    # k_scale 75/64 = 150; rope bf16 8 and 100: score sigma (16*150 + 8*100) = 200
    q_nope = {(0, i, 0, 0): 0x48 for i in range(S)}
    q_rope = {(0, i, 0, 0): F(8) for i in range(S)}
    k_nope = {(0, key, 0, 0): 0x70}
    k_rope = {(0, key, 0): F(100)}
    vcodes = {0: 0x38, 1: 0x7E, 2: 0x01, 3: 0xB8, 100: 0x3F}
    cols = tuple(sorted(vcodes))
    v = {(0, j, 0, c): code for j in range(S) for c, code in vcodes.items()}

    def v_deq(j):
        return [E4M3[vcodes[c]] * k_scale[j] for c in cols]

    o, lse = {}, []
    for i in range(S):
        if i < key:
            o[(0, i, 0)] = mean([v_deq(j) for j in range(i + 1)])
            lse.append(math.log(i + 1))
        else:
            o[(0, i, 0)] = v_deq(key)
            lse.append(200.0)
    return {
        "name": "prefill_fp8_scales",
        "kind": "prefill",
        "derivation": "e4m3 nope parts with per-token scales, sigma = 1/16.  Q_nope = code 0x48 (4) "
                      "x q_scale 4 = 16; key 2: K_nope code 0x70 (128) x k_scale 75/64 = 150, rope "
                      "8 x 100: score 200; other keys score 0.  V = codes x k_scale of their token "
                      "(0x38 = 1, 0x7E = 448, 0x01 = 2^-9, 0xB8 = -1, 0x3F = 1.875).  Rows 0, 1: "
                      "mean of the visible dequantised V rows, LSE ln(i+1); rows >= 2: V row 2, LSE 200.",
        "B": 1, "H": H, "S": S, "fp8": True, "causal": True, "softmax_scale": 0.0625,
        "inputs": {
            "q_nope": tensor("e4m3", (1, S, H, DN), q_nope),
            "q_rope": tensor("bf16", (1, S, H, DR), q_rope),
            "k_nope": tensor("e4m3", (1, S, H, DN), k_nope),
            "k_rope": tensor("bf16", (1, S, DR), k_rope),
            "v": tensor("e4m3", (1, S, H, DV), v),
            "q_scale": tensor("f32", (1, S), {(0, i): q_scale[i] for i in range(S)}),
            "k_scale": tensor("f32", (1, S), {(0, j): k_scale[j] for j in range(S)}),
        },
        "expected": {"O": tensor("f64", (1, S, H, DV), _o_entries(o, cols)),
                     "LSE": {"shape": [1, H, S], "values": [[lse]]}},
    }


# ---------------------------------------------------------------------------- decode

def _decode_case(name, derivation, *, B, T, H, fp8, causal, sigma, num_pages, page_table,
                 cache_lens, cache, kv_scale, q_latent, q_rope, o, lse, cache_fill, cache_rows):
    return {
        "name": name, "kind": "decode", "derivation": derivation,
        "B": B, "T": T, "H": H, "fp8": fp8, "causal": causal, "softmax_scale": sigma,
        "num_pages": num_pages, "max_pages": len(page_table[0]),
        "inputs": {
            "q_latent": tensor("bf16", (B, T, H, DL), q_latent),
            "q_rope": tensor("bf16", (B, T, H, DR), q_rope),
            "kv_cache": tensor("e4m3" if fp8 else "bf16", (num_pages, PAGE, DL + DR), cache,
                               fill=cache_fill, zero=cache_rows),
            "kv_scale": tensor("f32", (num_pages, PAGE), kv_scale, fill="nan") if fp8 else None,
            "page_table": tensor("i32", (B, len(page_table[0])),
                                 {(b, p): v for b, row in enumerate(page_table) for p, v in enumerate(row)},
                                 fill="-1"),
            "cache_lens": tensor("i32", (B,), {(b,): v for b, v in enumerate(cache_lens)}),
        },
        "expected": {"O": tensor("f64", (B, T, H, DL), o), "LSE": {"shape": [B, H, T], "values": lse}},
    }


def case_decode_single_key_and_empty():
    # sequence 0: one cached token in page 2, row 0; sequence 1: no token
    c0 = {0: F(1, 2), 7: F(3), 300: F(-2), 511: F(5, 4), DL + 1: F(1)}
    cache = {(2, 0, c): v for c, v in c0.items()}
    q_latent = {(0, 0, 0, 7): F(2), (0, 0, 1, 0): F(-1), (1, 0, 0, 0): F(1)}
    q_rope = {(0, 0, 0, 1): F(4)}
    o = {(0, 0, h, c): v for h in range(2) for c, v in c0.items() if c < DL}
    lse = [[[0.625], [-0.03125]], [["-inf"], ["-inf"]]]
    return _decode_case(
        "decode_single_key_and_empty",
        "sigma = 1/16.  Sequence 0 holds one token (page 2, row 0), so each head's O is that "
        "token's latent row and LSE its score: head 0 sigma (2*3 + 4*1) = 0.625 (latent column 7 "
        "and rope column 1), head 1 sigma (-1 * 0.5) = -0.03125.  Sequence 1 holds none: O = 0, "
        "LSE = -inf.  Every other cache row is NaN, so reading one shows.",
        B=2, T=1, H=2, fp8=False, causal=True, sigma=0.0625, num_pages=3,
        page_table=[[2, -1], [-1, -1]], cache_lens=[1, 0], cache=cache, kv_scale=None,
        q_latent=q_latent, q_rope=q_rope, o=o, lse=lse, cache_fill="nan", cache_rows=[(2, 0)])


def case_decode_two_new_tokens(causal):
    L, T = 3, 2

    def c_row(j):
        return {0: F(j + 1), 100: F((-2) ** j), 511: F(j, 4), DL: F(7 - j), DL + 63: F(-j)}

    cache = {(0, j, c): v for j in range(L) for c, v in c_row(j).items()}
    lat = [c for c in sorted(c_row(0)) if c < DL]
    o, lse = {}, [[[]]]
    for t in range(T):
        n = (L - T + t + 1) if causal else L
        m = mean([[c_row(j)[c] for c in lat] for j in range(n)])
        o.update({(0, t, 0, c): v for c, v in zip(lat, m) if v != 0})
        lse[0][0].append(math.log(n))
    return _decode_case(
        "decode_two_new_tokens_" + ("causal" if causal else "full"),
        "q = 0, so all visible keys weigh alike.  L = 3 counts the 2 new tokens (positions 1, 2); "
        + ("causal: token 0 sees keys 0..1 (O = mean, LSE ln 2), token 1 keys 0..2 (LSE ln 3)."
           if causal else "non-causal: both tokens see keys 0..2 (O = mean, LSE ln 3)."),
        B=1, T=T, H=1, fp8=False, causal=causal, sigma=0.0625, num_pages=1, page_table=[[0]],
        cache_lens=[L], cache=cache, kv_scale=None, q_latent={}, q_rope={}, o=o, lse=lse,
        cache_fill="nan", cache_rows=[(0, j) for j in range(L)])


def case_decode_fp8_codes():
    codes = {0: 0x01, 1: 0x07, 2: 0x08, 3: 0x38, 4: 0x7E, 5: 0xFE, 6: 0x80, 7: 0x3F, 8: 0x40,
             9: 0x0F, 511: 0xC8, DL: 0x48}
    scale = F(1, 2)
    cache = {(1, 0, c): code for c, code in codes.items()}
    o = {(0, 0, 0, c): E4M3[code] * scale for c, code in codes.items() if c < DL and E4M3[code] != 0}
    # score: latent column 3 (code 1.0 x 0.5) times q 2, plus rope column 0 (code 4 x 0.5)
    # times q 1: sigma (1 + 2) = 3/16
    return _decode_case(
        "decode_fp8_codes",
        "fp8 cache, one token (page 1, row 0) with scale 1/2: O = code value x 1/2 for every "
        "latent column (subnormals 0x01, 0x07, smallest normal 0x08, 0x0F, 1.0, +-448, -0, 1.875, "
        "2, -4), LSE = sigma (2 * 0.5 + 1 * 2) = 3/16 with sigma = 1/16.  Rows past the token "
        "hold the NaN code 0x7F and NaN scales.",
        B=1, T=1, H=1, fp8=True, causal=True, sigma=0.0625, num_pages=2, page_table=[[1]],
        cache_lens=[1], cache=cache, kv_scale={(1, 0): scale},
        q_latent={(0, 0, 0, 3): F(2)}, q_rope={(0, 0, 0, 0): F(1)}, o=o, lse=[[[0.1875]]],
        cache_fill="127", cache_rows=[(1, 0)])


def cases():
    return [
        case_prefill_zero_query(True),
        case_prefill_zero_query(False),
        case_prefill_dominant_key(),
        case_prefill_fp8_scales(),
        case_decode_single_key_and_empty(),
        case_decode_two_new_tokens(True),
        case_decode_two_new_tokens(False),
        case_decode_fp8_codes(),
    ]


def render() -> str:
    """One case per line (compact JSON), inside ``{"cases": [...]}``."""
    body = ",\n".join(json.dumps(c, sort_keys=True, separators=(",", ":")) for c in cases())
    return '{"cases": [\n' + body + "\n]}\n"


if __name__ == "__main__":
    with open(OUT, "w") as f:
        f.write(render())
    print("wrote", OUT)
