"""Pins for the oracle's expert MLP, MoE layer and lm_head: numpy float64
dense matmuls over weights dequantised by an independent decoder, at tiny
shapes and at one full-size layer (hidden 2688, 128 experts, top-6)."""
import numpy as np
import pytest
import torch

from gen import configs, gen
from oracle import oracle as orc
from oracle.workload import OracleLayer

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def deq(m: orc.Mat):
    c = np.empty((m.n, m.k), np.int64)
    c[:, 0::2] = m.codes & 15
    c[:, 1::2] = m.codes >> 4
    mag = E2M1[c & 7] * np.where(c & 8, -1.0, 1.0)
    s = torch.from_numpy(m.scales.copy()).view(torch.float8_e4m3fn).double().numpy()
    return mag * np.repeat(s, 16, axis=1) * m.g


def bf16(x):
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16).double().numpy()


def act(x, w4a4):
    if not w4a4:
        return x
    c, s, g = orc.quantize(x.astype(np.float32)[None, :], orc.PER_ROW)
    return deq(orc.Mat(c, s, g[0]))[0]


def ref_layer(L: OracleLayer, h, r, w4a4, residual):
    out = []
    for t in range(h.shape[0]):
        x = gen.bf16_bits_to_f32(h[t]).astype(np.float64)
        xa = act(x, w4a4)

        def mlp(up, down):
            u = deq(up) @ xa
            a = bf16(np.maximum(u, 0.0) ** 2)
            return deq(down) @ act(a, w4a4)

        acc = mlp(L.sh_up, L.sh_down)
        for j, e in enumerate(r["idx"][t]):
            acc = acc + r["w"][t][j] * mlp(L.up[int(e)], L.down[int(e)])
        if residual:
            acc = acc + x
        out.append(acc)
    return np.array(out)


@pytest.mark.parametrize("w4a4,residual", [(False, False), (True, False), (True, True)])
@pytest.mark.parametrize("H,I,S,E,k", [(32, 16, 48, 8, 2), (80, 48, 112, 8, 3)])
def test_tiny_layer_matches_dense_numpy(w4a4, residual, H, I, S, E, k):
    L = OracleLayer(3, 1, H, I, S, E, (-0.1, 0.1))
    h = gen.hidden_bf16(4, H, 3, layer=1)
    out, outf, r = L.forward(h, k, w4a4, residual)
    ref = ref_layer(L, h, r, w4a4, residual)
    assert np.allclose(outf, ref, rtol=1e-12, atol=1e-13)
    assert np.array_equal(out, bf16(ref).astype(np.float32).view(np.uint32).__rshift__(16)
                          .astype(np.uint16))


def test_lm_head_matches_dense_numpy():
    W = orc.Mat.from_master(gen.normal_bf16(40 * 64, 1, 77, 0.02).reshape(40, 64))
    h = gen.hidden_bf16(3, 64, 1, layer=5)
    got = orc.lm_head(W, h)
    ref = gen.bf16_bits_to_f32(h).astype(np.float64) @ deq(W).T
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)
    rows = np.array([0, 7, 39])
    assert np.allclose(orc.lm_head_rows(W, h, rows), ref[:, rows], rtol=1e-12, atol=1e-13)


def test_full_size_layer_matches_dense_numpy():
    c = configs.shape(0)
    L = OracleLayer(0, 0, c["H"], c["I"], c["S"], c["E"], c["bias"])
    h = gen.hidden_bf16(1, c["H"], 0, layer=configs.HIDDEN_LAYER)
    for w4a4 in (False, True):
        out, outf, r = L.forward(h, c["K"], w4a4, False)
        ref = ref_layer(L, h, r, w4a4, False)
        assert np.allclose(outf, ref, rtol=1e-10, atol=1e-10)
