"""lm_head_gemv on the GPU against the oracle: small shapes (several tiles,
token counts across the 8-column groups) and the pages' full 131072 x 2688
matrix on sampled rows."""
import numpy as np
import pytest
import torch

from gen import configs, gen
from oracle import oracle as orc
from tests.gpu_fixtures import nm  # noqa: F401
from tests.helpers import assert_close, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [1, 3, 8, 11])
@pytest.mark.parametrize("V,H", [(512, 256), (48, 1856), (1024, 2688)])
def test_small_lm_head(nm, T, V, H):
    tid = gen.tensor_id(gen.KIND_LM_HEAD, 1, V)
    master = gen.normal_bf16(V * H, 4, tid, gen.WEIGHT_SIGMA).reshape(V, H)
    W = orc.Mat.from_master(master)
    m = nm.nvfp4_quantize(to_dev_bf16(master), nm.PER_TENSOR)
    h = gen.hidden_bf16(T, H, 4, layer=configs.LM_INPUT_LAYER)
    got = nm.lm_head_gemv(m, to_dev_bf16(h))
    torch.cuda.synchronize()
    assert_close(got.cpu().numpy(), orc.lm_head(W, h), "logits")


@pytest.mark.parametrize("T", [1, 4])
def test_full_lm_head_sampled_rows(nm, T):
    V, H = configs.V, configs.H
    dev = torch.empty((V, H), dtype=torch.bfloat16, device="cuda")
    gen.dev_normal_bf16(dev, 0, gen.tensor_id(gen.KIND_LM_HEAD, 0, 0), gen.WEIGHT_SIGMA)
    m = nm.nvfp4_quantize(dev, nm.PER_TENSOR)
    del dev
    h = gen.hidden_bf16(T, H, 0, layer=configs.LM_INPUT_LAYER)
    got = nm.lm_head_gemv(m, to_dev_bf16(h))
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    assert np.isfinite(got).all()
    rows = np.unique(np.concatenate([np.arange(32), V - 32 + np.arange(32),
                                     np.random.default_rng(1).integers(0, V, 1024)]))
    host = gen.lm_head_master(0, V, H)
    g = np.float32(np.abs(gen.bf16_bits_to_f32(host)).max()) / np.float32(2688.0)
    c, s, _ = orc.quantize(host[rows], orc.GIVEN, g=float(g))
    ref = orc.lm_head(orc.Mat(c, s, g), h)
    assert_close(got[:, rows], ref, "sampled logits")


@pytest.mark.parametrize("T", [9, 64, 100, 300])
@pytest.mark.parametrize("eps", [0.0, 1e-5])
@pytest.mark.parametrize("V", [1024, 1152, 128])
def test_small_lm_head_forward_gemm(nm, T, eps, V):
    """lm_head_forward above 8 tokens (the tensor-core GEMM: N = tokens rounded
    up to 16, up to 256 per launch; 300 tokens take two launches; 1152 and
    128 rows give fewer 128-row tiles than CTAs) against the oracle, with and
    without the final RMS norm."""
    H = 2688
    tid = gen.tensor_id(gen.KIND_LM_HEAD, 2, V)
    master = gen.normal_bf16(V * H, 4, tid, gen.WEIGHT_SIGMA).reshape(V, H)
    W = orc.Mat.from_master(master)
    m = nm.nvfp4_quantize(to_dev_bf16(master), nm.PER_TENSOR)
    h = gen.hidden_bf16(T, H, 4, layer=configs.LM_INPUT_LAYER + 1)
    got = nm.lm_head_forward(m, to_dev_bf16(h), rms_eps=eps)
    torch.cuda.synchronize()
    assert nm.nvfp4_last_device_error() == 0
    x = orc.rms_norm(h, eps) if eps > 0 else h
    assert_close(got.cpu().numpy(), orc.lm_head(W, x), "logits")


def test_full_lm_head_forward_256_tokens(nm):
    """The 131072 x 2688 head for 256 concurrent tokens; sampled rows and tokens."""
    V, H, T = configs.V, configs.H, 256
    dev = torch.empty((V, H), dtype=torch.bfloat16, device="cuda")
    gen.dev_normal_bf16(dev, 0, gen.tensor_id(gen.KIND_LM_HEAD, 0, 0), gen.WEIGHT_SIGMA)
    m = nm.nvfp4_quantize(dev, nm.PER_TENSOR)
    del dev
    h = gen.hidden_bf16(T, H, 0, layer=configs.LM_INPUT_LAYER)
    got = nm.lm_head_forward(m, to_dev_bf16(h), rms_eps=1e-5)
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    assert np.isfinite(got).all()
    rows = np.unique(np.concatenate([np.arange(16), V - 16 + np.arange(16),
                                     np.random.default_rng(2).integers(0, V, 256)]))
    toks = np.array([0, 1, 63, 64, 128, 200, 255])
    host = gen.lm_head_master(0, V, H)
    g = np.float32(np.abs(gen.bf16_bits_to_f32(host)).max()) / np.float32(2688.0)
    c, s, _ = orc.quantize(host[rows], orc.GIVEN, g=float(g))
    ref = orc.lm_head(orc.Mat(c, s, g), orc.rms_norm(h[toks], 1e-5))
    assert_close(got[np.ix_(toks, rows)], ref, "sampled logits")
