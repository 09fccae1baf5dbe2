"""Exact rational models of the few IEEE binary32 operations and the two
encoders the NVFP4 quantiser is built from. They pin the oracle's quantiser
from outside: nothing here calls the oracle or the CUDA library.

Every value is a fractions.Fraction. rn32(q) is the binary32 number nearest
to q (ties to the even significand), with subnormals (quantum 2^-149); the
inputs here never overflow. The E4M3 and E2M1 encoders pick the nearest
representable value of the OCP formats (E4M3 "FN": bias 7, subnormals m 2^-9,
largest finite 448; E2M1: 0, 0.5, 1, 1.5, 2, 3, 4, 6), ties to the even code,
values beyond the largest saturating to it (satfinite).

The quantiser of a 16-element block with per-tensor global g, as the library
reads the NVFP4 recipe (blockamax / 6 / global, then x over the decoded scale
times the global; "Let's optimize Nemotron 3.5 Lightning - a worklog",
Step 1, block size 16):
    s = E4M3( rn32( rn32(amax_b / 6) / g ) ),  d = rn32( E4M3value(s) * g ),
    code_i = E2M1( rn32(x_i / d) ),             g = rn32(amax / 2688).
The variants below are the plausible misreadings a pin has to tell apart.
"""
from fractions import Fraction

import numpy as np


def f32(x) -> Fraction:
    """Exact value of a binary32 number (a Python/numpy float that is one)."""
    v = np.float32(x)
    assert float(v) == float(x), "not a binary32 value"
    return Fraction(float(v))


def bits_to_fraction(b: int) -> Fraction:
    return Fraction(float(np.array([b], np.uint32).view(np.float32)[0]))


def fraction_to_bits(q: Fraction) -> int:
    f = np.float32(float(q))
    assert Fraction(float(f)) == q, "not a binary32 value"
    return int(np.array([f], np.float32).view(np.uint32)[0])


def _floor_log2(a: Fraction) -> int:
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


def _round_half_even(q: Fraction) -> int:
    n, r = divmod(q.numerator, q.denominator)
    twice = 2 * r
    if twice > q.denominator or (twice == q.denominator and n % 2 == 1):
        n += 1
    return n


def rn32(q: Fraction) -> Fraction:
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = max(_floor_log2(a), -126)
    quantum = Fraction(2) ** (e - 23)
    return sign * _round_half_even(a / quantum) * quantum


def e4m3_value(s: int) -> Fraction:
    e, m = (s >> 3) & 15, s & 7
    if e == 0:
        return Fraction(m, 512)
    return (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


E4M3_POS = [(e4m3_value(s), s) for s in range(0x7F)]  # 0x00 .. 0x7E (0x7F is NaN)


def _nearest_even(v: Fraction, table):
    best = None
    for val, code in table:
        d = abs(v - val)
        if best is None or d < best[0] or (d == best[0] and code % 2 == 0 and best[1] % 2 == 1):
            best = (d, code)
    return best[1]


def e4m3_encode(v: Fraction) -> int:
    """Non-negative v -> E4M3 byte, nearest, ties to even, saturating at 448."""
    assert v >= 0
    if v >= 448:
        return 0x7E
    return _nearest_even(v, E4M3_POS)


E2M1_POS = [(Fraction(v), c) for c, v in enumerate([0, 0.5, 1, 1.5, 2, 3, 4, 6])]


def e2m1_encode(v: Fraction) -> int:
    """v -> E2M1 code (bit 3 the sign, kept for a zero result), nearest, ties
    to even, saturating at 6."""
    sign = 8 if v < 0 else 0
    a = abs(v)
    mag = 7 if a >= 6 else _nearest_even(a, E2M1_POS)
    return sign | mag


def global_scale(amax: Fraction, variant: str = "A") -> Fraction:
    if variant == "A":    # one division by the exact constant 6 * 448
        return rn32(amax / 2688)
    if variant == "B":    # two divisions, by 6 then by 448
        return rn32(rn32(amax / 6) / 448)
    if variant == "C":    # multiplication by the rounded reciprocal
        return rn32(amax * rn32(Fraction(1, 2688)))
    raise ValueError(variant)


def quantize_block(x, g: Fraction, variant: str = "A"):
    """x: 16 Fractions (binary32 values). Returns (scale byte, 16 codes).
    variant A: the reading above; B: scale from amax_b / rn32(6 g);
    C: codes from x * rn32(1 / d); D: scale from the exact amax_b / (6 g)
    rounded once."""
    amax_b = max(abs(v) for v in x)
    s = 0
    if g > 0:
        if variant == "B":
            q = rn32(amax_b / rn32(6 * g))
        elif variant == "D":
            q = rn32(amax_b / (6 * g))
        else:
            q = rn32(rn32(amax_b / 6) / g)
        s = e4m3_encode(q)
    d = rn32(e4m3_value(s) * g)
    codes = []
    for v in x:
        if d == 0:
            codes.append(0)
        elif variant == "C":
            codes.append(e2m1_encode(rn32(v * rn32(1 / d))))
        else:
            codes.append(e2m1_encode(rn32(v / d)))
    return s, codes


def pack_codes(codes):
    """16 codes -> 8 bytes, element 2j in the low nibble of byte j."""
    return bytes(codes[2 * j] | (codes[2 * j + 1] << 4) for j in range(len(codes) // 2))
