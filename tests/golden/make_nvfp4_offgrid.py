"""Writes nvfp4_offgrid.txt: quantiser cases whose inputs sit next to a
rounding boundary, so that the reading of the NVFP4 recipe (one division of
the tensor amax by 2688; the block scale as (blockamax / 6) / global, two
binary32 divisions; codes from x / d by division) gives a different result
from a plausible misreading of it. Expected values come from the exact
rational model in tests/exact_fp.py, never from the oracle or the GPU.

    python tests/golden/make_nvfp4_offgrid.py   (deterministic; seed 20261202)
"""
import os
import random
import sys
from fractions import Fraction

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
import exact_fp as X  # noqa: E402

OUT = os.path.join(HERE, "nvfp4_offgrid.txt")


def f32_near(q: Fraction, k: int) -> Fraction:
    """The binary32 number k ulps away from rn32(q) (k may be negative)."""
    b = X.fraction_to_bits(X.rn32(q)) + k
    return X.bits_to_fraction(b)


def rand_f32(rng, lo_exp, hi_exp) -> Fraction:
    e = rng.randint(lo_exp, hi_exp)
    m = rng.randint(1 << 23, (1 << 24) - 1)
    return Fraction(m, 1 << 23) * Fraction(2) ** e


def hexf(q: Fraction) -> str:
    return "%08x" % X.fraction_to_bits(q)


def filler(rng, amax: Fraction, n: int):
    out = []
    for _ in range(n):
        v = X.rn32(amax * Fraction(rng.randint(1, 999), 1000))
        out.append(-v if rng.random() < 0.5 else v)
    return out


def main():
    rng = random.Random(20261202)
    lines = ["# NVFP4 quantiser cases next to rounding boundaries (expected: exact model, variant A).",
             "# global <amax> <g>                       : PER_TENSOR of a 16-element row holding amax",
             "# block <variant> <g> <x0..x15> <scale> <codes>: GIVEN global g; <variant> names the misreading",
             "#   (B: scale from blockamax / (6 g) with 6 g rounded; C: codes from x * rn(1/d);",
             "#    D: scale from blockamax / (6 g) rounded once) that gives a different scale or codes.",
             "# All numbers are binary32 bit patterns in hex; codes are 8 bytes, element 2j low nibble of byte j."]
    # 1. tensor globals where one division by 2688 differs from /6 then /448 or from * rn(1/2688)
    want = {"B": 3, "C": 3}
    while any(want.values()):
        a = rand_f32(rng, -12, 10)
        gA = X.global_scale(a, "A")
        for v in ("B", "C"):
            if want[v] and X.global_scale(a, v) != gA:
                lines.append("global %s %s %s" % (v, hexf(a), hexf(gA)))
                want[v] -= 1
                break
    # 2. block scales next to an E4M3 midpoint
    want = {"B": 4, "D": 2}
    while any(want.values()):
        g = rand_f32(rng, -14, -6)
        s = rng.randint(0x10, 0x70)
        mid = (X.e4m3_value(s) + X.e4m3_value(s + 1)) / 2
        found = None
        for k in range(-40, 41):
            a = f32_near(mid * 6 * g, k)
            x = [a] + filler(rng, a, 15)
            rng.shuffle(x)
            sa, ca = X.quantize_block(x, g, "A")
            for v in ("B", "D"):
                if want[v] and X.quantize_block(x, g, v)[0] != sa:
                    found = (v, x, sa, ca)
                    break
            if found:
                break
        if found:
            v, x, sa, ca = found
            lines.append("block %s %s %s %02x %s" % (v, hexf(g), " ".join(hexf(q) for q in x), sa,
                                                     X.pack_codes(ca).hex()))
            want[v] -= 1
    # 3. codes next to an E2M1 midpoint (division vs reciprocal)
    want = 8
    mids = [Fraction(1, 4), Fraction(3, 4), Fraction(5, 4), Fraction(7, 4), Fraction(5, 2), Fraction(7, 2),
            Fraction(5)]
    while want:
        g = rand_f32(rng, -14, -6)
        amax = rand_f32(rng, -4, 2)
        x = [amax] + filler(rng, amax, 15)
        s, _ = X.quantize_block(x, g, "A")
        d = X.rn32(X.e4m3_value(s) * g)
        if d == 0:
            continue
        m = mids[rng.randrange(len(mids))]
        for k in range(-8, 9):
            y = f32_near(m * d, k)
            if y >= amax:
                continue
            x2 = list(x)
            x2[1 + rng.randrange(15)] = -y if rng.random() < 0.5 else y
            sa, ca = X.quantize_block(x2, g, "A")
            sc, cc = X.quantize_block(x2, g, "C")
            if sa == s and cc != ca:
                lines.append("block C %s %s %02x %s" % (hexf(g), " ".join(hexf(q) for q in x2), sa,
                                                        X.pack_codes(ca).hex()))
                want -= 1
                break
    with open(OUT, "w") as f:
        f.write("\n".join(lines) + "\n")
    print(OUT, len(lines), "lines")


if __name__ == "__main__":
    main()
