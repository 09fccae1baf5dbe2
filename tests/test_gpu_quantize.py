"""nvfp4_quantize on the GPU against the oracle: codes, scales and globals
bit-exact, for weights (per tensor), activations (per row) and given globals,
including every E2M1 tie point, sign-kept zeros, zero blocks and the pages'
full-size expert and lm_head matrices."""
import numpy as np
import pytest
import torch

from gen import configs, gen
from oracle import oracle as orc
from tests.gpu_fixtures import nm  # noqa: F401
from tests.helpers import to_dev_bf16

pytestmark = pytest.mark.gpu

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def gpu_quant(nm, x, mode, g=None):
    if x.dtype == np.uint16:
        xd = to_dev_bf16(x)
    else:
        xd = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    gs = None if g is None else torch.tensor([g], dtype=torch.float32, device="cuda")
    m = nm.nvfp4_quantize(xd, mode, global_scale=gs)
    torch.cuda.synchronize()
    return m.codes.cpu().numpy(), m.scales.cpu().numpy(), m.global_scale.cpu().numpy()


def same(nm, x, mode, g=None):
    c1, s1, g1 = gpu_quant(nm, x, mode, g)
    c0, s0, g0 = orc.quantize(x, mode, g)
    assert np.array_equal(g1.view(np.uint32), g0.view(np.uint32)), "global differs"
    assert np.array_equal(s1, s0), f"scales differ in {np.sum(s1 != s0)} places"
    assert np.array_equal(c1, c0), f"codes differ in {np.sum(c1 != c0)} bytes"


@pytest.mark.parametrize("rows,cols", [(1, 16), (5, 48), (16, 64), (37, 2688), (64, 1856), (3, 3712)])
def test_weights_bf16_per_tensor(nm, rows, cols):
    x = gen.normal_bf16(rows * cols, 1, 1000 + rows, 0.02).reshape(rows, cols)
    same(nm, x, orc.PER_TENSOR)


def test_float32_input_and_given_global(nm):
    x = (gen.normal_f32(7 * 96, 2, 5) * 3.0).astype(np.float32).reshape(7, 96)
    same(nm, x, orc.PER_TENSOR)
    same(nm, x, orc.GIVEN, g=0.0011)


def test_activation_rows_per_row(nm):
    h = gen.hidden_bf16(9, 2688, 0, layer=3)
    same(nm, h, orc.PER_ROW)
    # relu^2-shaped rows (heavy right tail, many zeros)
    u = gen.normal_f32(4 * 1856, 3, 9).reshape(4, 1856)
    a = np.maximum(u, 0) ** 2
    same(nm, a.astype(np.float32), orc.PER_ROW)


def test_tie_points_signed_zero_and_zero_blocks(nm):
    rng = np.random.default_rng(0)
    g = 2.0 ** -10
    rows, cols = 8, 256
    nb = cols // 16
    scl = rng.integers(0x08, 0x7E, (rows, nb)).astype(np.uint8)
    scl[0, 0] = 0x7E
    sv = torch.from_numpy(scl).view(torch.float8_e4m3fn).double().numpy()
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.1, 0.2, 7.0])
    vals = rng.choice(np.concatenate([mids, E2M1]), (rows, cols)) * rng.choice([-1.0, 1.0], (rows, cols))
    vals[:, ::16] = 6.0 * rng.choice([-1.0, 1.0], (rows, nb))  # every block recomputes its scale
    x = vals * np.repeat(sv, 16, axis=1) * g
    x[3, 32:48] = 0.0                                           # a zero block
    x[4, 48:64] = -0.0
    x = x.astype(np.float32)
    same(nm, x, orc.PER_TENSOR)
    same(nm, x, orc.PER_ROW)
    # the ties really are exercised: codes of exact midpoints are even
    c, s, _ = orc.quantize(x, orc.PER_TENSOR)
    assert s[0, 0] == 0x7E


def test_full_size_expert_and_shared_matrices(nm):
    c = configs.shape(1)
    H, I, S = c["H"], c["I"], c["S"]
    for kind, idx, n, k in [(gen.KIND_UP, 0, I, H), (gen.KIND_DOWN, 77, H, I), (gen.KIND_SH_UP, 0, S, H)]:
        tid = gen.tensor_id(kind, 5, idx)
        host = gen.normal_bf16(n * k, 0, tid, gen.WEIGHT_SIGMA).reshape(n, k)
        dev = torch.empty((n, k), dtype=torch.bfloat16, device="cuda")
        gen.dev_normal_bf16(dev, 0, tid, gen.WEIGHT_SIGMA)
        torch.cuda.synchronize()
        assert np.array_equal(dev.view(torch.int16).cpu().numpy().astype(np.uint16), host), \
            "device generator differs from host generator"
        m = nm.nvfp4_quantize(dev, nm.PER_TENSOR)
        c0, s0, g0 = orc.quantize(host, orc.PER_TENSOR)
        torch.cuda.synchronize()
        assert np.array_equal(m.global_scale.cpu().numpy().view(np.uint32), g0.view(np.uint32))
        assert np.array_equal(m.scales.cpu().numpy(), s0)
        assert np.array_equal(m.codes.cpu().numpy(), c0)


def test_full_size_lm_head_matrix(nm):
    V, H = configs.V, configs.H
    tid = gen.tensor_id(gen.KIND_LM_HEAD, 0, 0)
    dev = torch.empty((V, H), dtype=torch.bfloat16, device="cuda")
    gen.dev_normal_bf16(dev, 0, tid, gen.WEIGHT_SIGMA)
    m = nm.nvfp4_quantize(dev, nm.PER_TENSOR)
    host = gen.lm_head_master(0, V, H)
    amax = np.abs(gen.bf16_bits_to_f32(host)).max()
    g0 = np.float32(amax) / np.float32(2688.0)
    torch.cuda.synchronize()
    assert m.global_scale.cpu().numpy()[0] == g0
    rows = np.unique(np.concatenate([np.arange(64), V - 64 + np.arange(64),
                                     np.random.default_rng(0).integers(0, V, 2048)]))
    c0, s0, _ = orc.quantize(host[rows], orc.GIVEN, g=float(g0))
    assert np.array_equal(m.codes[torch.from_numpy(rows).cuda()].cpu().numpy(), c0)
    assert np.array_equal(m.scales[torch.from_numpy(rows).cuda()].cpu().numpy(), s0)


def test_offgrid_boundary_cases_exact(nm):
    """The quantiser cases next to rounding boundaries (tests/golden/nvfp4_offgrid.txt,
    expected values from exact arithmetic): the kernels' corrected-reciprocal
    division and scale arithmetic must give the reading's codes bit for bit."""
    from fractions import Fraction
    from tests.test_oracle_quant_exact import _cases
    for c in _cases():
        if c[0] == "global":
            _, _, amax, g = c
            row = np.zeros((1, 16), np.float32)
            row[0, 5] = np.float32(float(amax))
            _, _, gq = gpu_quant(nm, row, orc.PER_TENSOR)
            assert Fraction(float(gq[0])) == g
        else:
            _, _, g, x, s, codes = c
            xa = np.array([[float(v) for v in x]], np.float32)
            cq, sq, _ = gpu_quant(nm, xa, orc.GIVEN, float(g))
            assert int(sq[0, 0]) == s
            assert bytes(cq[0]) == codes


def test_division_next_to_every_midpoint_for_many_divisors(nm):
    """x / d with d = E4M3 scale x global (binary32 products) for 300 random
    globals and every positive finite E4M3 scale, x within two ulps of each
    E2M1 rounding midpoint m d: the kernels' division (a corrected
    reciprocal) must give the codes of a correctly rounded binary32 quotient,
    which the oracle takes by plain division. Many quotients land exactly on
    a midpoint (even-code ties), the rest one or two ulps to either side."""
    rng = np.random.default_rng(17)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    e4m3 = np.array([orc.e4m3_value(b) for b in range(1, 127)], np.float32)
    exact_ties = 0
    for _ in range(300):
        g = np.float32(np.ldexp(rng.uniform(1.0, 2.0), int(rng.integers(-16, 0))))
        blocks = []
        for s in e4m3:
            d = np.float32(s * g)
            x0 = (mids * d).astype(np.float32)
            near = [x0]
            up, dn = x0.copy(), x0.copy()
            for _k in range(2):
                up = np.nextafter(up, np.float32(np.inf))
                dn = np.nextafter(dn, np.float32(0))
                near += [up, dn]
            x = np.concatenate(near) * rng.choice(np.float32([-1, 1]), 35)
            amax = np.float32(6 * d)
            x = np.concatenate([x, np.zeros(10, np.float32)]).reshape(3, 15)
            blocks.append(np.concatenate([np.full((3, 1), amax, np.float32), x], axis=1))
            q = np.abs(np.concatenate(near)) / d
            exact_ties += int(np.isin(q, mids).sum())
        row = np.concatenate(blocks).reshape(1, -1).astype(np.float32)
        same(nm, row, orc.GIVEN, g=float(g))
    assert exact_ties > 300 * 126 * 2
