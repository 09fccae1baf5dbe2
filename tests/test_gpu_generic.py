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
