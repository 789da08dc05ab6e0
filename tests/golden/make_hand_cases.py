"""Writes the hand-derived fixtures of tests/golden/.  Run from the repo root:
`python tests/golden/make_hand_cases.py`.

These cases are worked out by hand from the definitions in the pages (no
oracle code is called), and chosen so that every intermediate value is exact
in fp32 and fp64, so the expected codes, scales and bf16 words are unique:

hand_case_pow2.json  (dual RMSNorm + per-1x128 quant, vLLM PR #53540 "Purpose")
  Kq = Kkv = 128, eps = 0.
  q[k] = +4 or -4 (minus when k % 3 == 2): mean(q^2) = 16, r_q = 1/4 exactly.
  gamma_q[k] = 2**(k % 8 - 4): x_hat_q[k] = sign * 2**(k % 8 - 4), amax = 8.
  scale = fp32(8 / 448) = fp32(1/56); x_hat / scale = sign * 56 * 2**(k%8-4)
  (to within the fp32 rounding of 1/56, far from any E4M3 rounding boundary):
  |value| 3.5, 7, 14, 28, 56, 112, 224, 448 -> E4M3FN codes
  0x46, 0x4E, 0x56, 0x5E, 0x66, 0x6E, 0x76, 0x7E (value = 2**(E-7)*(1+m/8),
  code = E<<3 | m), with 0x80 set for negative entries.
  kv[k] = +2 or -2 (minus when k is odd): mean = 4, r_kv = 1/2;
  gamma_kv[k] = 1 + k/128 (7 fraction bits, exact in bf16), so
  kv_out[k] = sign * (1 + k/128) exactly; its bf16 word is sign<<15 |
  127<<7 | k.

hand_case_ties.json  (round to nearest, ties to even, on the fused path)
  Kq = 128, Kkv = 8, eps = 0, q[k] = 1 (r_q = 1), gamma_q chosen so that
  x_hat_q = gamma_q, with amax = 7 -> scale = 7/448 = 1/64 exactly and
  x_hat/scale = 64 * gamma_q exactly:
    64*g = 17  lies halfway between 16 (0x58) and 18 (0x59): even -> 0x58
    64*g = 19  between 18 (0x59) and 20 (0x5A): even -> 0x5A
    64*g = 3*2**-10 between 2**-9 (0x01) and 2*2**-9 (0x02): even -> 0x02
    64*g = 25  between 24 (0x5C) and 26 (0x5D): even -> 0x5C
    64*g = 448 (g = 7, the amax) -> 0x7E
    64*g = 2**-10 between 0 and 2**-9: even -> 0x00 (0x80 when negative)
  and negatives of the same (sign bit 0x80).  The remaining entries are 0.
  kv = 1 with gamma_kv = 1: kv_out = 1.0 (0x3F80) everywhere.
"""

from __future__ import annotations

import json
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def bf16_word(sign: int, exp: int, frac7: int) -> int:
    return (sign << 15) | (exp << 7) | frac7


def pow2_case():
    Kq = Kkv = 128
    q = [(-4.0 if k % 3 == 2 else 4.0) for k in range(Kq)]
    gq = [2.0 ** (k % 8 - 4) for k in range(Kq)]
    mag_code = [0x46, 0x4E, 0x56, 0x5E, 0x66, 0x6E, 0x76, 0x7E]   # 3.5 .. 448
    codes = [mag_code[k % 8] | (0x80 if k % 3 == 2 else 0) for k in range(Kq)]
    kv = [(-2.0 if k % 2 else 2.0) for k in range(Kkv)]
    gkv = [1.0 + k / 128.0 for k in range(Kkv)]
    kv_out = [bf16_word(k % 2, 127, k) for k in range(Kkv)]
    return {
        "citation": "vLLM PR #53540, Purpose: dual RMSNorm with fp32 accumulation, per-1x128 "
                    "FP8 group quant from the fp32 values; hand derivation in make_hand_cases.py",
        "M": 1, "Kq": Kq, "Kkv": Kkv, "eps": 0.0,
        "q": [q], "kv": [kv], "gamma_q": gq, "gamma_kv": gkv,
        "expected_codes": [codes],
        "expected_scale": {"numerator": 1, "denominator": 56, "rounding": "fp32 round-to-nearest-even"},
        "expected_kv_bf16_words": [kv_out],
    }


def ties_case():
    Kq, Kkv = 128, 8
    entries = {  # position -> (gamma value, expected code)
        0: (7.0, 0x7E),             # amax: 448
        1: (17 / 64, 0x58),         # tie 16|18 -> 16
        2: (19 / 64, 0x5A),         # tie 18|20 -> 20
        3: (3 * 2.0 ** -16, 0x02),  # tie 1*2^-9 | 2*2^-9 -> 2*2^-9 (subnormal)
        4: (25 / 64, 0x5C),         # tie 24|26 -> 24
        5: (-17 / 64, 0xD8),
        6: (-19 / 64, 0xDA),
        7: (-3 * 2.0 ** -16, 0x82),
        8: (-7.0, 0xFE),            # |amax| again, negative: -448
        9: (2.0 ** -16, 0x00),      # 64*g = 2^-10: tie 0 | 2^-9 -> 0
        10: (-(2.0 ** -16), 0x80),  # negative value rounding to zero keeps its sign
    }
    gq = [0.0] * Kq
    codes = [0x00] * Kq
    for k, (g, c) in entries.items():
        gq[k], codes[k] = g, c
    return {
        "citation": "vLLM PR #53540, Purpose (per-1x128 FP8 quant from fp32); OCP E4M3FN "
                    "round-to-nearest-even; hand derivation in make_hand_cases.py",
        "M": 1, "Kq": Kq, "Kkv": Kkv, "eps": 0.0,
        "q": [[1.0] * Kq], "kv": [[1.0] * Kkv], "gamma_q": gq, "gamma_kv": [1.0] * Kkv,
        "expected_codes": [codes],
        "expected_scale": {"numerator": 1, "denominator": 64, "rounding": "exact"},
        "expected_kv_bf16_words": [[0x3F80] * Kkv],
    }


if __name__ == "__main__":
    for name, case in (("hand_case_pow2.json", pow2_case()), ("hand_case_ties.json", ties_case())):
        with open(os.path.join(HERE, name), "w") as f:
            json.dump(case, f, indent=1)
        print("wrote", name)
