"""Pins of the oracle's NVFP4 quantiser off the grid, from exact arithmetic.

The round-trip pins use values already on the grid, where every reading of the
recipe gives the same codes. Here the inputs sit next to rounding boundaries
(tests/golden/nvfp4_offgrid.txt, written by make_nvfp4_offgrid.py from the
rational model in tests/exact_fp.py) so that the reading - tensor global
amax / 2688 in one division, block scale (blockamax / 6) / global in two,
codes x / d by division ("Let's optimize Nemotron 3.5 Lightning - a
worklog", Step 1) - differs from each plausible misreading, and the oracle
must give the reading's result bit for bit. The rational model itself is
pinned against numpy's binary32 arithmetic and torch's E4M3 conversion."""
import os
import random
from fractions import Fraction

import numpy as np
import torch

import exact_fp as X
from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "nvfp4_offgrid.txt")


def _f(h):
    return X.bits_to_fraction(int(h, 16))


def _cases():
    out = []
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            t = line.split()
            if t[0] == "global":
                out.append(("global", t[1], _f(t[2]), _f(t[3])))
            else:
                g = _f(t[2])
                x = [_f(h) for h in t[3:19]]
                out.append(("block", t[1], g, x, int(t[19], 16), bytes.fromhex(t[20])))
    return out


def test_rn32_matches_numpy_binary32():
    rng = np.random.default_rng(7)
    a = (rng.standard_normal(3000) * np.exp(rng.uniform(-30, 30, 3000))).astype(np.float32)
    b = (rng.standard_normal(3000) * np.exp(rng.uniform(-30, 30, 3000))).astype(np.float32)
    q = a / b  # IEEE binary32 division, round to nearest even
    p = a * b
    for i in range(3000):
        fa, fb = Fraction(float(a[i])), Fraction(float(b[i]))
        assert X.rn32(fa / fb) == Fraction(float(q[i]))
        assert X.rn32(fa * fb) == Fraction(float(p[i]))


def test_e4m3_encoder_matches_torch():
    rng = np.random.default_rng(8)
    v = np.concatenate([np.exp(rng.uniform(np.log(2.0 ** -12), np.log(440.0), 4000)),
                        [X.e4m3_value(s) for s in range(0x7F)],
                        [(X.e4m3_value(s) + X.e4m3_value(s + 1)) / 2 for s in range(0x7E)]]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for i in range(v.size):
        assert X.e4m3_encode(Fraction(float(v[i]))) == int(ref[i]), float(v[i])
    assert X.e4m3_encode(Fraction(500)) == 0x7E


def test_e2m1_encoder_midpoints_and_sign():
    # ties to the even code: 0.25 -> 0, 0.75 -> 1.0, 1.25 -> 1.0, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4
    mids = {Fraction(1, 4): 0, Fraction(3, 4): 2, Fraction(5, 4): 2, Fraction(7, 4): 4, Fraction(5, 2): 4,
            Fraction(7, 2): 6, Fraction(5): 6}
    for m, c in mids.items():
        assert X.e2m1_encode(m) == c and X.e2m1_encode(-m) == 8 | c
    assert X.e2m1_encode(Fraction(-1, 10)) == 8  # a negative value that rounds to 0 keeps its sign
    assert X.e2m1_encode(Fraction(100)) == 7


def test_golden_cases_discriminate_and_agree_with_model():
    cases = _cases()
    kinds = {(c[0], c[1]) for c in cases}
    assert {("global", "B"), ("global", "C"), ("block", "B"), ("block", "C"), ("block", "D")} <= kinds
    for c in cases:
        if c[0] == "global":
            _, v, amax, g = c
            assert X.global_scale(amax, "A") == g
            assert X.global_scale(amax, v) != g
        else:
            _, v, g, x, s, codes = c
            sa, ca = X.quantize_block(x, g, "A")
            assert sa == s and X.pack_codes(ca) == codes
            sv, cv = X.quantize_block(x, g, v)
            assert (sv, X.pack_codes(cv)) != (s, codes)


def test_oracle_matches_offgrid_golden():
    for c in _cases():
        if c[0] == "global":
            _, _, amax, g = c
            row = np.zeros((1, 16), np.float32)
            row[0, 5] = np.float32(float(amax))
            _, _, gq = orc.quantize(row, orc.PER_TENSOR)
            assert Fraction(float(gq[0])) == g
        else:
            _, _, g, x, s, codes = c
            xa = np.array([[float(v) for v in x]], np.float32)
            cq, sq, _ = orc.quantize(xa, orc.GIVEN, g=float(g))
            assert int(sq[0, 0]) == s
            assert bytes(cq[0]) == codes


def test_oracle_matches_exact_model_on_random_blocks():
    rng = random.Random(5)
    nrng = np.random.default_rng(5)
    for _ in range(150):
        g = Fraction(float(np.float32(np.exp(nrng.uniform(np.log(1e-6), np.log(1e-1))))))
        x = (nrng.standard_normal(16) * np.exp(nrng.uniform(-8, 4))).astype(np.float32)
        if rng.random() < 0.2:
            x[rng.randrange(16)] = 0.0
        cq, sq, _ = orc.quantize(x[None, :], orc.GIVEN, g=float(g))
        s, codes = X.quantize_block([Fraction(float(v)) for v in x], g, "A")
        assert int(sq[0, 0]) == s
        assert bytes(cq[0]) == X.pack_codes(codes)
