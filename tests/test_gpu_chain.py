"""The full-depth decode step at the pages' sizes (23 W4A4 MoE layers +
131072 x 2688 lm_head), in the launch configuration the benchmark times.

The per-layer calls are teacher-forced from the oracle to the GPU: the oracle
runs its own chain h_0 -> h_23; for every layer the GPU is given its h_l and must
reproduce the oracle's routing (bit-exact up to near-ties) and h_{l+1}
(within tolerance); the lm_head is checked on the oracle's h_23 at sampled
rows. The benchmark's own path (all layers in one moe_stack_forward call) is
checked the other way round: the oracle is teacher-forced on the GPU's h_l.
The free-running GPU chain (CUDA graph, as timed) must be deterministic and
stay finite."""
import numpy as np
import pytest
import torch

from gen import configs, fill, gen
from oracle import oracle as orc
from oracle.workload import OracleLayer
from tests.gpu_fixtures import nm  # noqa: F401
from tests.helpers import assert_close, bf16_bits, bf16_to_f64, check_routing, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def stack(nm):
    from nvfp4_quantized_moe_sigmoid_gb300.model import MoEDecodeStack
    c = configs.shape(1)
    st = MoEDecodeStack(c["layers"], c["E"], c["H"], c["I"], c["S"], c["K"], 4, w4a4=True, V=c["V"],
                        rms_eps=c["rms_eps"])
    st.register(*fill.fillers(c["seed"], c["bias"]))
    torch.cuda.synchronize()
    return c, st


@pytest.mark.parametrize("cfg", [1, 2])
def test_chain_teacher_forced(nm, stack, cfg):
    c0, st = stack
    c = configs.shape(cfg)
    T = c["T"]
    h = gen.hidden_bf16(T, c["H"], c["seed"], layer=configs.HIDDEN_LAYER, rho=c["rho"])
    assert np.isfinite(bf16_to_f64(h)).all(), "generated hidden state is not finite"
    ws = nm.make_workspace(st.layers[0], T, c["K"], nm.W4A4)
    lws = nm.make_layer_workspace(st.layers[0], T, c["K"], nm.W4A4)
    exempt = 0
    for l in range(c["layers"]):
        OL = OracleLayer(c["seed"], l, c["H"], c["I"], c["S"], c["E"], c["bias"])
        assert np.isfinite(OL.Wg).all() and np.isfinite(OL.bias).all(), f"layer {l} router not finite"
        ref, _, r = OL.forward(h, c["K"], True, True, rms_eps=c["rms_eps"])
        assert np.isfinite(bf16_to_f64(ref)).all(), f"oracle layer {l} output not finite" 
        hd = to_dev_bf16(h)
        idx, w = nm.moe_route_topk(hd, st.layers[l].router_w, st.layers[l].router_b, c["K"],
                                   rms_eps=c["rms_eps"])
        torch.cuda.synchronize()
        e = check_routing(idx.cpu().numpy(), w.cpu().numpy(), r, c["K"])
        exempt += e
        if e == 0:
            out = nm.moe_expert_forward(st.layers[l], hd, idx, w, nm.W4A4, residual=hd, workspace=ws,
                                        rms_eps=c["rms_eps"])
            torch.cuda.synchronize()
            assert_close(bf16_to_f64(bf16_bits(out)), bf16_to_f64(ref), f"layer {l}")
            # the fused layer call, as the benchmark's step runs it
            outf, idxf, _ = nm.moe_layer_forward(st.layers[l], hd, c["K"], nm.W4A4, residual=hd,
                                                 workspace=lws, rms_eps=c["rms_eps"])
            torch.cuda.synchronize()
            assert torch.equal(idxf, idx)
            assert_close(bf16_to_f64(bf16_bits(outf)), bf16_to_f64(ref), f"fused layer {l}")
        h = ref
    assert exempt <= 1
    assert nm.nvfp4_last_device_error() == 0
    # lm_head on the oracle's final hidden state
    V, H = c["V"], c["H"]
    logits = nm.lm_head_gemv(st.lm, to_dev_bf16(h), rms_eps=c["rms_eps"]).cpu().numpy()
    rows = np.unique(np.concatenate([np.arange(16), np.random.default_rng(2).integers(0, V, 512)]))
    host = gen.lm_head_master(c["seed"], V, H)
    g = np.float32(np.abs(gen.bf16_bits_to_f32(host)).max()) / np.float32(2688.0)
    cc, ss, _ = orc.quantize(host[rows], orc.GIVEN, g=float(g))
    hn = orc.rms_norm(h, c["rms_eps"])
    assert_close(logits[:, rows], orc.lm_head(orc.Mat(cc, ss, g), hn), "logits")


@pytest.mark.parametrize("cfg", [1, 2])
def test_stack_teacher_forced(nm, stack, cfg):
    """The benchmark's path: all 23 layers in one moe_stack_forward call; the
    oracle is teacher-forced on the GPU's own h_l of every layer."""
    from tests.test_gpu_stack import teacher_forced
    c0, st4 = stack
    c = configs.shape(cfg)
    T = c["T"]
    h0 = gen.hidden_bf16(T, c["H"], c["seed"], layer=configs.HIDDEN_LAYER, rho=c["rho"])
    hd = to_dev_bf16(h0)
    hout, idx, w = nm.moe_stack_forward(st4.layers, hd, c["K"], nm.W4A4, rms_eps=c["rms_eps"])
    torch.cuda.synchronize()
    assert nm.nvfp4_last_device_error() == 0
    OLs = [OracleLayer(c["seed"], l, c["H"], c["I"], c["S"], c["E"], c["bias"]) for l in range(c["layers"])]
    assert teacher_forced(nm, OLs, h0, hout, idx, w, c["K"], True, c["rms_eps"]) <= 1


def test_free_running_graph(nm, stack):
    """The timed step (CUDA graph: stack kernel + lm_head) is deterministic,
    equals a direct moe_stack_forward call bit for bit, and its first layer
    agrees with the per-layer call within tolerance."""
    from nvfp4_quantized_moe_sigmoid_gb300.model import MoEDecodeStack
    c0, st4 = stack
    c = configs.shape(1)
    st = MoEDecodeStack(c["layers"], c["E"], c["H"], c["I"], c["S"], c["K"], 1, w4a4=True, V=c["V"],
                        weights_from=st4, rms_eps=c["rms_eps"])
    st.make_workspace()
    assert st.path == "stack"
    h0 = gen.hidden_bf16(1, c["H"], c["seed"], layer=configs.HIDDEN_LAYER)
    st.h[0].copy_(to_dev_bf16(h0))
    st.capture()
    st.replay()
    torch.cuda.synchronize()
    first = st.h[1:].clone()
    st.replay()
    torch.cuda.synchronize()
    assert torch.equal(first.view(torch.int16), st.h[1:].view(torch.int16)), "replay not deterministic"
    assert torch.isfinite(st.logits).all()
    hd = to_dev_bf16(h0)
    hout, _, _ = nm.moe_stack_forward(st.layers, hd, c["K"], nm.W4A4, rms_eps=c["rms_eps"])
    torch.cuda.synchronize()
    assert torch.equal(hout.view(torch.int16), first.view(torch.int16))
    out, _, _ = nm.moe_layer_forward(st.layers[0], hd, c["K"], nm.W4A4, residual=hd, workspace=st.ws,
                                     rms_eps=c["rms_eps"])
    torch.cuda.synchronize()
    assert_close(bf16_to_f64(bf16_bits(out)), bf16_to_f64(bf16_bits(first[0])), "layer 0: layer call vs stack")
    assert nm.nvfp4_last_device_error() == 0


def test_concurrent_256_step_teacher_forced(nm, stack):
    """The 256-token concurrent step as the benchmark runs it (23 W4A4 layers
    on the grouped tensor-core path, then the lm_head GEMM), one free-running
    step on the GPU; the oracle, teacher-forced on the GPU's own h_l, checks
    the routing and h_{l+1} of 4 sampled tokens in every layer, and the
    logits of those tokens at sampled vocabulary rows."""
    from nvfp4_quantized_moe_sigmoid_gb300.model import MoEDecodeStack
    c0, st4 = stack
    c = configs.shape(4)
    T, L = c["T"], c["layers"]
    st = MoEDecodeStack(L, c["E"], c["H"], c["I"], c["S"], c["K"], T, w4a4=True, V=c["V"], weights_from=st4,
                        rms_eps=c["rms_eps"])
    st.make_workspace()
    assert st.path == "split"
    h0 = gen.hidden_bf16(T, c["H"], c["seed"], layer=configs.HIDDEN_LAYER, rho=c["rho"])
    st.h[0].copy_(to_dev_bf16(h0))
    st.step()
    torch.cuda.synchronize()
    assert nm.nvfp4_last_device_error() == 0
    hs = bf16_bits(st.h)  # [L + 1][T][H]
    idx, w = st.topk_idx.cpu().numpy(), st.topk_w.cpu().numpy()
    tok = np.array([0, 1, 131, 255])
    exempt = 0
    for l in range(L):
        OL = OracleLayer(c["seed"], l, c["H"], c["I"], c["S"], c["E"], c["bias"])
        ref, _, r = OL.forward(hs[l][tok], c["K"], True, True, rms_eps=c["rms_eps"])
        e = check_routing(idx[l][tok], w[l][tok], r, c["K"])
        exempt += e
        if e == 0:
            assert_close(bf16_to_f64(hs[l + 1][tok]), bf16_to_f64(ref), f"layer {l}")
    assert exempt <= 1
    V, H = c["V"], c["H"]
    rows = np.unique(np.concatenate([np.arange(16), np.random.default_rng(3).integers(0, V, 256)]))
    host = gen.lm_head_master(c["seed"], V, H)
    g = np.float32(np.abs(gen.bf16_bits_to_f32(host)).max()) / np.float32(2688.0)
    cc, ss, _ = orc.quantize(host[rows], orc.GIVEN, g=float(g))
    hn = orc.rms_norm(hs[L][tok], c["rms_eps"])
    logits = st.logits.cpu().numpy()[tok][:, rows]
    assert_close(logits, orc.lm_head(orc.Mat(cc, ss, g), hn), "logits")
