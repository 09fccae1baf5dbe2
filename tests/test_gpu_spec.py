"""The MTP drafter's MoE on the GPU (worklog Step 6: the drafter's 128
experts quantised to NVFP4, run by the same kernels with its own weights),
against the oracle, and one speculative step: k draft passes at one token,
then the main stack's verify pass over k + 1 tokens."""
import numpy as np
import pytest
import torch

from gen import configs, fill, gen
from oracle.workload import OracleLayer
from tests.gpu_fixtures import nm  # noqa: F401
from tests.helpers import assert_close, bf16_bits, bf16_to_f64, check_routing, to_dev_bf16

pytestmark = pytest.mark.gpu


def drafter_layer(nm, E, H, I, S, seed=0):
    from nvfp4_quantized_moe_sigmoid_gb300.model import register_layer
    L = nm.MoELayer(E, H, I, S)
    register_layer(L, configs.DRAFTER_LAYER, *fill.fillers(seed, (-0.1, 0.1)))
    torch.cuda.synchronize()
    return L


def test_drafter_moe_full_shape(nm):
    """The drafter layer at the pages' shapes, one token, W4A4 with the
    pre-norm, as one stack call: routing and output against the oracle."""
    c = configs.shape(1)
    L = drafter_layer(nm, c["E"], c["H"], c["I"], c["S"])
    OL = OracleLayer(0, configs.DRAFTER_LAYER, c["H"], c["I"], c["S"], c["E"], (-0.1, 0.1))
    h = gen.hidden_bf16(1, c["H"], 0, layer=configs.DRAFTER_LAYER)
    hout, idx, w = nm.moe_stack_forward([L], to_dev_bf16(h), c["K"], nm.W4A4, rms_eps=c["rms_eps"])
    torch.cuda.synchronize()
    assert nm.nvfp4_last_device_error() == 0
    ref, _, r = OL.forward(h, c["K"], True, True, rms_eps=c["rms_eps"])
    if check_routing(idx[0].cpu().numpy(), w[0].cpu().numpy(), r, c["K"]) == 0:
        assert_close(bf16_to_f64(bf16_bits(hout[0])), bf16_to_f64(ref), "drafter layer")


def test_spec_step_small(nm):
    """A small model (16 experts, hidden 256, two main layers): the draft
    chain of the step matches the oracle pass by pass (teacher-forced), and
    its verify pass is exactly the main stack's own step on the same input."""
    from nvfp4_quantized_moe_sigmoid_gb300.model import MoEDecodeStack, SpecDecodeStep
    E, H, I, S, k, V, K = 16, 256, 128, 192, 4, 512, configs.SPEC_K
    main = MoEDecodeStack(2, E, H, I, S, k, K + 1, w4a4=True, V=V)
    main.register(*fill.fillers(9, (-0.1, 0.1)))
    d = drafter_layer(nm, E, H, I, S, seed=9)
    step = SpecDecodeStep(main, d, K)
    fill.hidden(main.h[0], 9, layer=0, rho=0.5)
    h0 = gen.hidden_bf16(1, H, 9, layer=configs.DRAFTER_LAYER)
    step.hd[0].copy_(to_dev_bf16(h0))
    step.capture()
    step.graph.replay()
    torch.cuda.synchronize()
    assert nm.nvfp4_last_device_error() == 0
    OL = OracleLayer(9, configs.DRAFTER_LAYER, H, I, S, E, (-0.1, 0.1))
    hs = [bf16_bits(step.hd[j]) for j in range(K + 1)]
    for j in range(K):
        ref, _, r = OL.forward(hs[j], k, True, True, rms_eps=main.rms_eps)
        if check_routing(step.d_idx[j, 0].cpu().numpy(), step.d_w[j, 0].cpu().numpy(), r, k) == 0:
            assert_close(bf16_to_f64(hs[j + 1]), bf16_to_f64(ref), f"draft pass {j}")
    got = main.h[main.L].clone()
    main.step()
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), main.h[main.L].view(torch.int16))
    assert np.isfinite(step.d_logits.cpu().numpy()).all()
