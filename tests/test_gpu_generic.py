"""moe_expert_forward on layer widths that are multiples of 16 but not of 64
(the generic kernels) against the oracle, elementwise within
|err| <= 1e-2 + 2e-2 |ref|: each width off the 64 grid in turn, W4A16 and
W4A4, with and without the residual and the RMS norm, at token counts on
both sides of the decode / grouped threshold the fast paths use."""
import numpy as np
import pytest

from gen import gen
from oracle.workload import OracleLayer
from tests.gpu_fixtures import device_layer, nm  # noqa: F401
from tests.test_gpu_moe import run_layer

pytestmark = pytest.mark.gpu

SHAPES = [  # (E, H, I, S): hidden, intermediate and shared widths off the 64 grid in turn
    (8, 80, 128, 192),
    (8, 128, 48, 192),
    (8, 128, 128, 112),
    (6, 208, 144, 272),
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("T", [1, 3, 6])
@pytest.mark.parametrize("w4a4", [False, True])
def test_generic_widths(nm, shape, T, w4a4):
    E, H, I, S = shape
    L = device_layer(nm, 11, 1, E, H, I, S, (-0.1, 0.1))
    OL = OracleLayer(11, 1, H, I, S, E, (-0.1, 0.1))
    h = gen.hidden_bf16(T, H, 11, layer=1, rho=0.5)
    run_layer(nm, L, OL, h, 3, w4a4, residual=T != 3)


def test_generic_rms_norm_residual(nm):
    """The pre-normed block: x = RMSNorm(3 h), residual 3 h."""
    E, H, I, S = 8, 80, 48, 112
    L = device_layer(nm, 12, 0, E, H, I, S, (-0.1, 0.1))
    OL = OracleLayer(12, 0, H, I, S, E, (-0.1, 0.1))
    h = gen.hidden_bf16(4, H, 12, layer=0, rho=0.5)
    h3 = (gen.bf16_bits_to_f32(h) * 3.0).astype(np.float32).view(np.uint32) >> 16
    for w4a4 in (False, True):
        run_layer(nm, L, OL, h3.astype(np.uint16), 2, w4a4, True, rms_eps=1e-5)


@pytest.mark.parametrize("V,H", [(48, 80), (160, 208)])
@pytest.mark.parametrize("T", [1, 5, 11])
@pytest.mark.parametrize("eps", [0.0, 1e-5])
def test_generic_lm_head(nm, V, H, T, eps):
    """lm_head_gemv and lm_head_forward at a hidden width off the 64 grid (the
    generic kernel, any token count) against the oracle."""
    import torch
    from gen import configs
    from oracle import oracle as orc
    from tests.helpers import assert_close, to_dev_bf16
    tid = gen.tensor_id(gen.KIND_LM_HEAD, 3, V)
    master = gen.normal_bf16(V * H, 5, tid, gen.WEIGHT_SIGMA).reshape(V, H)
    W = orc.Mat.from_master(master)
    m = nm.nvfp4_quantize(to_dev_bf16(master), nm.PER_TENSOR)
    h = gen.hidden_bf16(T, H, 5, layer=configs.LM_INPUT_LAYER)
    x = orc.rms_norm(h, eps) if eps > 0 else h
    ref = orc.lm_head(W, x)
    got = nm.lm_head_forward(m, to_dev_bf16(h), rms_eps=eps)
    torch.cuda.synchronize()
    assert nm.nvfp4_last_device_error() == 0
    assert_close(got.cpu().numpy(), ref, "logits")
    if T <= 8:
        got2 = nm.lm_head_gemv(m, to_dev_bf16(h), rms_eps=eps)
        torch.cuda.synchronize()
        assert np.array_equal(got2.cpu().numpy(), got.cpu().numpy())
