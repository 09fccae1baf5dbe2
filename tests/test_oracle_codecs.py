"""Pins for the oracle's E2M1 / E4M3 / bf16 codecs against definitions that do
not come from the oracle: the OCP value lists, torch's float8_e4m3fn
conversion, and the nearest-value property checked by brute force."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc

E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # OCP MX spec FP4 E2M1


def test_e2m1_table():
    for c in range(16):
        v = orc.e2m1_value(c)
        mag = E2M1_MAGNITUDES[c & 7]
        assert v == (-mag if c & 8 else mag) or (mag == 0 and v == 0)


def test_e4m3_table_matches_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    for b in range(256):
        v = orc.e4m3_value(b)
        if np.isnan(ref[b]):
            assert np.isnan(v) and (b & 0x7F) == 0x7F
        else:
            assert v == ref[b], b
    assert orc.e4m3_value(0x7E) == 448.0
    assert orc.e4m3_value(0x01) == 2.0 ** -9
    assert orc.e4m3_value(0x38) == 1.0


def test_e4m3_encoder_matches_torch_rne():
    rng = np.random.default_rng(0)
    finite = np.array([orc.e4m3_value(b) for b in range(0x7F)])
    mids = (finite[1:] + finite[:-1]) / 2          # every tie point
    vals = np.concatenate([finite, mids, rng.uniform(0, 464, 20000),
                           np.exp(rng.uniform(np.log(1e-4), np.log(448), 20000))])
    vals = vals[vals < 464].astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(v)) for v in vals])
    assert np.array_equal(got, ref)


def test_e4m3_encoder_saturates():
    for v in [448.0, 460.0, 464.0, 500.0, 1e6, float("inf")]:
        assert orc.e4m3_encode(v) == 0x7E


def test_e2m1_encoder_nearest_and_ties():
    grid = np.array(E2M1_MAGNITUDES)
    mids = (grid[1:] + grid[:-1]) / 2
    rng = np.random.default_rng(1)
    xs = np.concatenate([grid, mids, -grid, -mids, rng.uniform(-8, 8, 5000),
                         np.nextafter(mids, 0), np.nextafter(mids, 10)]).astype(np.float32)
    for x in xs:
        c = orc.e2m1_encode(float(x))
        v = orc.e2m1_value(c)
        a = abs(float(x))
        d = np.abs(grid - min(a, 6.0))
        # nearest value (saturating at 6)
        assert abs(abs(v) - min(a, 6.0)) == d.min()
        # exact ties pick the even code
        if np.sum(d == d.min()) > 1:
            assert (c & 1) == 0
        # sign kept, also when the magnitude rounds to zero
        assert bool(c & 8) == bool(np.signbit(x))
    assert orc.e2m1_encode(0.25) == 0 and orc.e2m1_encode(0.75) == 2
    assert orc.e2m1_encode(1.25) == 2 and orc.e2m1_encode(1.75) == 4
    assert orc.e2m1_encode(2.5) == 4 and orc.e2m1_encode(3.5) == 6
    assert orc.e2m1_encode(5.0) == 6 and orc.e2m1_encode(1e9) == 7
    assert orc.e2m1_encode(-0.2) == 8


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(2)
    xs = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 6, 20000),
                         [0.0, -0.0, 1.0, -3.5]])
    # torch rounds float32 -> bf16 RNE; feed values exact in float32 to avoid double rounding
    xs = xs.astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(xs.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    ref = ref.astype(np.uint16)
    got = np.array([orc.bf16_round(float(x)) for x in xs], np.uint16)
    assert np.array_equal(got, ref)
    # a tie in binary64 that is not representable in binary32 is rounded once
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40   # just above the midpoint between 1 and 1+2^-7
    assert orc.bf16_value(orc.bf16_round(x)) == 1.0 + 2.0 ** -7
    x = 1.0 + 2.0 ** -8                # exact midpoint: even mantissa (1.0)
    assert orc.bf16_value(orc.bf16_round(x)) == 1.0
