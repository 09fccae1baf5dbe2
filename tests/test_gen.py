"""The synthetic-input generator: pinned to the published Philox4x32-10 known
answers, and checked for the distributions the workloads ask for."""
import math
import os

import numpy as np

from gen import gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def test_philox_known_answers():
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        v = [int(x, 16) for x in r]
        out = gen.philox(v[0:4], v[4:6])
        assert [int(x) for x in out] == v[6:10]


def test_log_is_accurate():
    for x in [1.0, 0.5, 0.25, 0.1, 1e-3, 0.9999, 1e-20, 0.7071, 0.3, 2.0 ** -40]:
        assert abs(gen.host().gen_log_test(x) - math.log(x)) <= 2e-6 * max(1.0, abs(math.log(x)))


def test_normal_moments():
    x = gen.normal_f32(1 << 21, 0, gen.tensor_id(gen.KIND_HIDDEN, 7, 3)).astype(np.float64)
    assert abs(x.mean()) < 5e-3
    assert abs(x.std() - 1.0) < 5e-3
    # fourth moment of a normal is 3; tails reach past 4.5 sigma at this size
    assert abs((x ** 4).mean() - 3.0) < 0.05
    assert np.abs(x).max() > 4.5
    # fraction inside one sigma
    assert abs((np.abs(x) < 1).mean() - 0.682689) < 2e-3


def test_uniform_range_and_mean():
    u = gen.uniform_f32(1 << 18, 0, 99, -0.1, 0.1).astype(np.float64)
    assert u.min() >= -0.1 - 1e-7 and u.max() < 0.1 + 1e-7
    assert abs(u.mean()) < 1e-3


def test_slices_regenerate_exactly():
    tid = gen.tensor_id(gen.KIND_UP, 3, 17)
    full = gen.normal_bf16(4097, 5, tid, 0.02)
    part = gen.normal_bf16_range(1001, 3000, 5, tid, 0.02)
    assert np.array_equal(full[1001:4001], part)


def test_hidden_correlation():
    T, H = 5, 1 << 15
    h = gen.bf16_bits_to_f32(gen.hidden_bf16(T, H, 0, layer=0, rho=0.5)).astype(np.float64)
    c = np.corrcoef(h)
    off = c[~np.eye(T, dtype=bool)]
    assert np.all(np.abs(off - 0.5) < 0.03)
    h0 = gen.bf16_bits_to_f32(gen.hidden_bf16(T, H, 0, layer=0, rho=0.0)).astype(np.float64)
    off0 = np.corrcoef(h0)[~np.eye(T, dtype=bool)]
    assert np.all(np.abs(off0) < 0.03)
