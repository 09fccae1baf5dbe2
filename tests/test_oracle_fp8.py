"""Pins for the oracle's FP8 (E4M3) per-tensor W8A8 path (the shared expert
of the W4A4 card's precision table): the quantiser against torch's
float8_e4m3fn conversion of binary32 quotients, and the shared expert
against a numpy float64 dense computation over independently decoded
weights."""
import numpy as np
import pytest
import torch

from gen import gen
from oracle import oracle as orc


def e4m3_torch(x32):
    """E4M3 codes of binary32 values (|x| < 464: torch rounds to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def e4m3_values(q):
    return torch.from_numpy(np.ascontiguousarray(q, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def bf16(x):
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("rows,cols", [(1, 16), (7, 96), (64, 2688)])
def test_quantize_per_tensor_matches_torch(rows, cols):
    x = gen.bf16_bits_to_f32(gen.normal_bf16(rows * cols, 4, 100 + rows, 0.02)).reshape(rows, cols)
    q, g = orc.fp8_quantize(x, orc.PER_TENSOR)
    g0 = np.float32(np.abs(x).max()) / np.float32(448.0)
    assert g[0] == g0
    assert np.array_equal(q, e4m3_torch(x / g0))
    # the element at the amax is 448 (code 0x7E) up to its sign
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert q[r, c] & 0x7F == 0x7E


def test_quantize_per_row_and_given_scale_match_torch():
    x = gen.bf16_bits_to_f32(gen.hidden_bf16(5, 2688, 0, layer=3))
    q, g = orc.fp8_quantize(x, orc.PER_ROW)
    for r in range(5):
        gr = np.float32(np.abs(x[r]).max()) / np.float32(448.0)
        assert g[r] == gr
        assert np.array_equal(q[r], e4m3_torch(x[r] / gr))
    q2, _ = orc.fp8_quantize(x, orc.GIVEN, g=0.0123)
    assert np.array_equal(q2, e4m3_torch(np.clip(x / np.float32(0.0123), -448, 448)))


def test_quantize_subnormals_ties_and_zero_rows():
    g = np.float32(1.0)
    # E4M3 subnormals are multiples of 2^-9; midpoints go to the even code
    x = np.array([[2.0 ** -10, 3 * 2.0 ** -10, 5 * 2.0 ** -10, -(2.0 ** -10), 0.0, -0.0, 448.0, 460.0]], np.float32)
    q, _ = orc.fp8_quantize(x, orc.GIVEN, g=float(g))
    assert list(q[0]) == [0x00, 0x02, 0x02, 0x80, 0x00, 0x80, 0x7E, 0x7E]
    z = np.zeros((2, 32), np.float32)
    z[1, 3] = -0.0
    q, gz = orc.fp8_quantize(z, orc.PER_ROW)
    assert np.all(gz == 0) and q[0].max() == 0 and q[1, 3] == 0x80


def dense_shared(x_bits, wu, gu, wd, gd):
    """numpy float64 reference: per-row E4M3 activations via torch."""
    out, acts = [], []
    Wu, Wd = e4m3_values(wu), e4m3_values(wd)
    for t in range(x_bits.shape[0]):
        x = gen.bf16_bits_to_f32(x_bits[t])
        gx = np.float32(np.abs(x).max()) / np.float32(448.0)
        xq = e4m3_values(e4m3_torch(x / gx))
        u = (Wu @ xq) * np.float64(gu) * np.float64(gx)
        a = bf16(np.maximum(u, 0.0) ** 2)
        a32 = a.astype(np.float32)
        ga = np.float32(np.abs(a32).max()) / np.float32(448.0)
        aq = e4m3_values(e4m3_torch(a32 / ga))
        out.append((Wd @ aq) * np.float64(gd) * np.float64(ga))
        acts.append(a)
    return np.array(out), np.array(acts)


@pytest.mark.parametrize("T,H,S", [(3, 128, 96), (1, 2688, 3712)])
def test_shared_expert_matches_dense_numpy(T, H, S):
    wu_m = gen.bf16_bits_to_f32(gen.normal_bf16(S * H, 6, 11, 0.02)).reshape(S, H)
    wd_m = gen.bf16_bits_to_f32(gen.normal_bf16(H * S, 6, 12, 0.02)).reshape(H, S)
    wu, gu = orc.fp8_quantize(wu_m, orc.PER_TENSOR)
    wd, gd = orc.fp8_quantize(wd_m, orc.PER_TENSOR)
    x = gen.hidden_bf16(T, H, 6, layer=2)
    y, act = orc.shared_fp8(x, wu, gu[0], wd, gd[0])
    ref, ref_act = dense_shared(x, wu, gu[0], wd, gd[0])
    assert np.array_equal(gen.bf16_bits_to_f32(act).astype(np.float64), ref_act)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-14)
    # the W8A8 expert approximates the bf16 expert it was quantised from
    xf = gen.bf16_bits_to_f32(x).astype(np.float64)
    full = (wd_m.astype(np.float64) @ (np.maximum(wu_m.astype(np.float64) @ xf.T, 0.0) ** 2)).T
    rel = np.linalg.norm(y - full) / np.linalg.norm(full)
    assert rel < 0.1
