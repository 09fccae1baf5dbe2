"""Pins for the oracle's NVFP4 quantiser: exact round trips for values already
on the grid, power-of-two scale invariance, mode equivalences, degenerate
inputs, and dequantisation against an independent torch-based decoder."""
import numpy as np
import torch

from oracle import oracle as orc

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _decode_independent(codes, scales, g, cols):
    """Dequantise with numpy + torch's float8_e4m3fn decoder (not the oracle)."""
    lo = codes & 15
    hi = codes >> 4
    c = np.empty((codes.shape[0], cols), np.int64)
    c[:, 0::2] = lo
    c[:, 1::2] = hi
    mag = E2M1[c & 7] * np.where(c & 8, -1.0, 1.0)
    s = torch.from_numpy(scales.copy()).view(torch.float8_e4m3fn).double().numpy()
    s = np.repeat(s, 16, axis=1)
    return mag * s * np.asarray(g, np.float64).reshape(-1, 1)


def _on_grid(rng, rows, cols, g):
    """Values exactly representable as e2m1 * e4m3 * g with a +-6 in every block
    and 6 * 448 * g somewhere, so the quantiser must reproduce them exactly."""
    nb = cols // 16
    codes = rng.integers(0, 16, (rows, cols))
    scl = rng.integers(0x08, 0x7E, (rows, nb))          # normal E4M3 scales
    pos = rng.integers(0, 16, (rows, nb))
    for r in range(rows):
        for b in range(nb):
            codes[r, b * 16 + pos[r, b]] = 7 | (8 * rng.integers(0, 2))
    scl[0, 0] = 0x7E
    sv = torch.from_numpy(scl.astype(np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    x = E2M1[codes & 7] * np.where(codes & 8, -1.0, 1.0) * np.repeat(sv, 16, axis=1) * g
    return x.astype(np.float32), codes, scl


def test_round_trip_exact_on_grid():
    rng = np.random.default_rng(0)
    g = 2.0 ** -10
    x, codes, scl = _on_grid(rng, 7, 96, g)
    c, s, gq = orc.quantize(x, orc.PER_TENSOR)
    assert gq[0] == np.float32(g)
    assert np.array_equal(s, scl.astype(np.uint8))
    xr = orc.dequantize(c, s, gq)
    assert np.array_equal(xr.astype(np.float32), x)
    assert np.array_equal(_decode_independent(c, s, gq, 96).astype(np.float32), x)


def test_scale_invariance_power_of_two():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((5, 64)) * 0.02).astype(np.float32)
    c0, s0, g0 = orc.quantize(x)
    for j in [-20, -3, 1, 7, 30]:
        c1, s1, g1 = orc.quantize((x * np.float32(2.0 ** j)).astype(np.float32))
        assert np.array_equal(c0, c1) and np.array_equal(s0, s1)
        assert g1[0] == np.float32(g0[0] * 2.0 ** j)


def test_modes_agree():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((6, 48)) * 3).astype(np.float32)
    ct, st, gt = orc.quantize(x, orc.PER_TENSOR)
    cg, sg, _ = orc.quantize(x, orc.GIVEN, g=float(gt[0]))
    assert np.array_equal(ct, cg) and np.array_equal(st, sg)
    for r in range(6):
        c1, s1, g1 = orc.quantize(x[r:r + 1], orc.PER_TENSOR)
        cr, sr, gr = orc.quantize(x, orc.PER_ROW)
        assert np.array_equal(cr[r], c1[0]) and np.array_equal(sr[r], s1[0]) and gr[r] == g1[0]
    assert gt[0] == np.float32(np.abs(x).max() / np.float32(2688.0))


def test_dequantize_matches_independent_decoder():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((9, 160)) * 0.02).astype(np.float32)
    c, s, g = orc.quantize(x)
    assert np.array_equal(orc.dequantize(c, s, g), _decode_independent(c, s, g, 160))
    c, s, g = orc.quantize(x, orc.PER_ROW)
    assert np.array_equal(orc.dequantize(c, s, g), _decode_independent(c, s, g, 160))


def test_nibble_order_low_first():
    x = np.zeros((1, 16), np.float32)
    x[0, 0] = 6.0    # element 0 -> low nibble of byte 0
    x[0, 1] = -1.0   # element 1 -> high nibble of byte 0
    c, s, g = orc.quantize(x)
    assert c[0, 0] == (0x7 | (0xA << 4))


def test_quantisation_error_is_bounded():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((32, 256)) * 0.02).astype(np.float32)
    c, s, g = orc.quantize(x)
    xr = orc.dequantize(c, s, g)
    sv = np.repeat(torch.from_numpy(s).view(torch.float8_e4m3fn).double().numpy(), 16, axis=1)
    d = sv * float(g[0])
    # |x/d| <= 6 up to scale rounding; the E2M1 grid step there is at most 2,
    # so the error is at most one step (2 d) and on average far less
    assert np.all(np.abs(xr - x) <= 2.0 * d + 1e-12)
    rel = np.sqrt(np.mean((xr - x) ** 2) / np.mean(x.astype(np.float64) ** 2))
    assert 0.02 < rel < 0.2


def test_degenerate_inputs():
    c, s, g = orc.quantize(np.zeros((2, 32), np.float32))
    assert g[0] == 0 and not c.any() and not s.any()
    x = np.zeros((1, 32), np.float32)
    x[0, 20] = 1.0
    c, s, g = orc.quantize(x)
    assert not c[0, :8].any() and s[0, 0] == 0   # zero block: scale 0, codes 0
    assert s[0, 1] == 0x7E                       # the amax block takes scale 448
