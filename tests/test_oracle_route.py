"""Pins for the oracle's sigmoid router: special cases whose answer is fixed
by the definition, and the logits against a numpy float64 matmul."""
import numpy as np
from scipy.special import expit

from gen import gen
from oracle import oracle as orc


def _setup(T=3, H=64, E=16, seed=0):
    h = gen.hidden_bf16(T, H, seed, layer=9)
    Wg = gen.router_w(seed, 9, E, H)
    bias = gen.router_bias(seed, 9, E, -0.1, 0.1)
    return h, Wg, bias


def test_logits_and_scores_match_numpy():
    h, Wg, bias = _setup()
    r = orc.route(h, Wg, bias, 4)
    hf = gen.bf16_bits_to_f32(h).astype(np.float64)
    z = hf @ Wg.astype(np.float64).T
    assert np.allclose(r["z"], z, rtol=1e-12, atol=1e-12)
    assert np.allclose(r["c"], expit(z) + bias.astype(np.float64), rtol=1e-12, atol=1e-12)


def test_selection_is_top_k_of_biased_scores():
    h, Wg, bias = _setup(T=5, E=32)
    r = orc.route(h, Wg, bias, 6)
    for t in range(5):
        order = np.lexsort((np.arange(32), -r["c"][t]))   # c desc, index asc
        assert list(r["idx"][t]) == list(order[:6])
        sig = expit(r["z"][t][r["idx"][t]])
        assert np.allclose(r["w"][t], sig / sig.sum(), rtol=1e-12)
        assert abs(r["w"][t].sum() - 1.0) < 1e-12


def test_zero_hidden_selects_by_bias_with_equal_weights():
    _, Wg, bias = _setup(E=16)
    h = np.zeros((1, 64), np.uint16)
    r = orc.route(h, Wg, bias, 6)
    assert list(r["idx"][0]) == list(np.argsort(-bias.astype(np.float64), kind="stable")[:6])
    assert np.allclose(r["w"][0], 1.0 / 6.0, rtol=0, atol=1e-15)


def test_k_equals_E_is_a_permutation_and_k1_is_argmax():
    h, Wg, bias = _setup(T=2, E=16)
    r = orc.route(h, Wg, bias, 16)
    for t in range(2):
        assert sorted(r["idx"][t]) == list(range(16))
        assert np.all(np.diff(r["c"][t][r["idx"][t]]) <= 0)
    r1 = orc.route(h, Wg, bias, 1)
    assert list(r1["idx"][:, 0]) == list(np.argmax(r["c"], axis=1))
    assert np.all(r1["w"] == 1.0)


def test_ties_go_to_lower_index():
    Wg = np.zeros((8, 32), np.float32)
    bias = np.array([0.1, 0.3, 0.3, 0.0, 0.3, 0.2, 0.2, 0.0], np.float32)
    h = np.zeros((1, 32), np.uint16)
    r = orc.route(h, Wg, bias, 4)
    assert list(r["idx"][0]) == [1, 2, 4, 5]


def test_rms_norm_matches_numpy_and_torch_rounding():
    import torch
    h = gen.hidden_bf16(3, 2688, 0, layer=4)
    hf = gen.bf16_bits_to_f32(h).astype(np.float64) * np.array([[1.0], [37.0], [1e-3]])
    hb = torch.from_numpy(hf).to(torch.float32).to(torch.bfloat16)
    h = hb.view(torch.int16).numpy().astype(np.uint16)
    x = gen.bf16_bits_to_f32(h).astype(np.float64)
    ref = x / np.sqrt((x ** 2).mean(axis=1, keepdims=True) + 1e-5)
    got = gen.bf16_bits_to_f32(orc.rms_norm(h, 1e-5)).astype(np.float64)
    # one bf16 rounding of the exact value: within half an ulp (2^-8 relative)
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30)
    # and it is the nearest bf16: torch's RNE of the float32 value agrees where
    # the float32 rounding cannot straddle a bf16 midpoint
    near = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).float().numpy()
    assert np.mean(near == got) > 0.999
    assert np.allclose(np.sqrt((got[:2] ** 2).mean(axis=1)), 1.0, atol=5e-3)  # row 3: eps dominates


def test_rms_norm_slack_counts_only_elements_at_a_rounding_midpoint():
    """rms_norm_slack: an all-ones row normalised to exactly the midpoint
    between the bf16 neighbours 0.99609375 and 1.0 (eps = 1/m^2 - 1 with
    m = 0.998046875) may round either way in every element: the slack of a
    router row is then sum_i |Wg_i| * 2^-8. Away from a midpoint, for a zero
    row, and without a norm, the slack is zero."""
    ones = np.full((1, 4), 0x3F80, np.uint16)  # bf16 1.0
    Wg = np.array([[1.0, -2.0, 0.5, 0.25], [0.0, 0.0, 0.0, 0.0]])
    m = 0.998046875
    s = orc.rms_norm_slack(ones, 1.0 / m ** 2 - 1.0, Wg)
    np.testing.assert_allclose(s, [[3.75 * 2.0 ** -8, 0.0]], rtol=1e-12)
    assert not orc.rms_norm_slack(ones, 1e-5, Wg).any()            # x = 0.999995: far from a midpoint
    assert not orc.rms_norm_slack(np.zeros((1, 4), np.uint16), 1e-5, Wg).any()
    assert not orc.rms_norm_slack(ones, 0.0, Wg).any()             # no norm
    # real rows: a handful of near-midpoint elements at most
    h, Wg2, _ = _setup(T=4, H=2688, E=8)
    s2 = orc.rms_norm_slack(h, 1e-5, Wg2)
    assert s2.shape == (4, 8) and (s2 >= 0).all() and s2.max() < 1e-2
