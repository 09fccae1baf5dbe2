"""moe_expert_forward (and the route + expert layer) on the GPU against the
oracle, elementwise within |err| <= 1e-2 + 2e-2 |ref|: small shapes with
several tiles and partial token groups, and the pages' full layer shape
(hidden 2688, 128 experts of 1856, shared 3712, top-6) at 1 and 4 tokens."""
import numpy as np
import pytest
import torch

from gen import configs, gen
from oracle.workload import OracleLayer
from tests.gpu_fixtures import dev_routing, device_layer, nm  # noqa: F401
from tests.helpers import assert_close, bf16_bits, bf16_to_f64, check_routing, to_dev_bf16

pytestmark = pytest.mark.gpu

SMALL = dict(E=16, H=256, I=128, S=192)


def run_layer(nm, L, OL, h, k, w4a4, residual, gpu_routing=False, rms_eps=0.0):
    hd = to_dev_bf16(h)
    r = OL.route(h, k, rms_eps)
    if gpu_routing:
        idx, w = nm.moe_route_topk(hd, L.router_w, L.router_b, k, rms_eps=rms_eps)
        torch.cuda.synchronize()
        check_routing(idx.cpu().numpy(), w.cpu().numpy(), r, k)
        assert np.array_equal(idx.cpu().numpy(), r["idx"]), "near-tie flip: layer output not comparable"
    else:
        idx, w = dev_routing(r)
    mode = nm.W4A4 if w4a4 else nm.W4A16
    ws = nm.make_workspace(L, h.shape[0], k, mode)
    out = nm.moe_expert_forward(L, hd, idx, w, mode, residual=hd if residual else None, workspace=ws,
                                rms_eps=rms_eps)
    torch.cuda.synchronize()
    assert nm.nvfp4_last_device_error() == 0
    ref, ref64, _ = OL.forward(h, k, w4a4, residual, routing=r, rms_eps=rms_eps)
    got = bf16_to_f64(bf16_bits(out))
    err = assert_close(got, bf16_to_f64(ref), "layer output")
    # the workspace counters are left zeroed: a second call gives the same bits
    out2 = nm.moe_expert_forward(L, hd, idx, w, mode, residual=hd if residual else None, workspace=ws,
                                 rms_eps=rms_eps)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    return err


@pytest.mark.parametrize("T", [1, 2, 3, 4])
@pytest.mark.parametrize("w4a4", [False, True])
@pytest.mark.parametrize("residual", [False, True])
def test_small_layer(nm, T, w4a4, residual):
    c = SMALL
    L = device_layer(nm, 7, 2, c["E"], c["H"], c["I"], c["S"], (-0.1, 0.1))
    OL = OracleLayer(7, 2, c["H"], c["I"], c["S"], c["E"], (-0.1, 0.1))
    h = gen.hidden_bf16(T, c["H"], 7, layer=2, rho=0.5)
    run_layer(nm, L, OL, h, 4, w4a4, residual)
    if residual:  # the pre-normed block: x = RMSNorm(3 h), residual 3 h
        h3 = gen.hidden_bf16(T, c["H"], 7, layer=2, rho=0.5)
        h3 = (gen.bf16_bits_to_f32(h3) * 3.0).astype(np.float32).view(np.uint32) >> 16
        run_layer(nm, L, OL, h3.astype(np.uint16), 4, w4a4, residual, gpu_routing=T == 1, rms_eps=1e-5)


def test_small_layer_odd_intermediate(nm):
    # I = 192: the 128-wide k chunks end in a half chunk on the down GEMV
    L = device_layer(nm, 8, 0, 8, 128, 192, 320, (-0.1, 0.1))
    OL = OracleLayer(8, 0, 128, 192, 320, 8, (-0.1, 0.1))
    h = gen.hidden_bf16(3, 128, 8, layer=0)
    run_layer(nm, L, OL, h, 3, True, True)
    run_layer(nm, L, OL, h, 3, False, False)


@pytest.fixture(scope="module")
def full_layer(nm):
    c = configs.shape(0)
    L = device_layer(nm, 0, 0, c["E"], c["H"], c["I"], c["S"], c["bias"])
    OL = OracleLayer(0, 0, c["H"], c["I"], c["S"], c["E"], c["bias"])
    return c, L, OL


def test_full_layer_w4a16_one_token(nm, full_layer):
    c, L, OL = full_layer
    h = gen.hidden_bf16(1, c["H"], 0, layer=configs.HIDDEN_LAYER)
    run_layer(nm, L, OL, h, c["K"], False, False, gpu_routing=True)


def test_full_layer_w4a4_one_token(nm, full_layer):
    c, L, OL = full_layer
    h = gen.hidden_bf16(1, c["H"], 0, layer=configs.HIDDEN_LAYER)
    run_layer(nm, L, OL, h, c["K"], True, True, gpu_routing=True)


def test_full_layer_w4a4_four_tokens(nm, full_layer):
    c, L, OL = full_layer
    h = gen.hidden_bf16(4, c["H"], 0, layer=configs.HIDDEN_LAYER, rho=0.5)
    run_layer(nm, L, OL, h, c["K"], True, True)


def test_full_layer_w4a4_prenorm(nm, full_layer):
    c, L, OL = full_layer
    h = gen.hidden_bf16(2, c["H"], 0, layer=9)
    h = ((gen.bf16_bits_to_f32(h) * 7.0).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    run_layer(nm, L, OL, h, c["K"], True, True, gpu_routing=True, rms_eps=1e-5)


def run_fused(nm, L, OL, h, k, w4a4, residual, rms_eps):
    hd = to_dev_bf16(h)
    mode = nm.W4A4 if w4a4 else nm.W4A16
    ws = nm.make_layer_workspace(L, h.shape[0], k, mode)
    outs = []
    for _ in range(2):  # the workspace counters are left zeroed: same bits again
        out, idx, w = nm.moe_layer_forward(L, hd, k, mode, residual=hd if residual else None, workspace=ws,
                                           rms_eps=rms_eps)
        torch.cuda.synchronize()
        outs.append(out)
    assert nm.nvfp4_last_device_error() == 0
    r = OL.route(h, k, rms_eps)
    check_routing(idx.cpu().numpy(), w.cpu().numpy(), r, k)
    assert np.array_equal(idx.cpu().numpy(), r["idx"]), "near-tie flip: layer output not comparable"
    ref, _, _ = OL.forward(h, k, w4a4, residual, routing=r, rms_eps=rms_eps)
    assert_close(bf16_to_f64(bf16_bits(outs[0])), bf16_to_f64(ref), "fused layer output")
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    # same result as the two-call path
    idx2, w2 = nm.moe_route_topk(hd, L.router_w, L.router_b, k, rms_eps=rms_eps)
    out2 = nm.moe_expert_forward(L, hd, idx2, w2, mode, residual=hd if residual else None, rms_eps=rms_eps)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx2)
    assert_close(bf16_to_f64(bf16_bits(out2)), bf16_to_f64(bf16_bits(outs[0])), "fused vs two-call")


@pytest.mark.parametrize("T", [1, 3, 4])
@pytest.mark.parametrize("w4a4,eps", [(False, 0.0), (True, 0.0), (True, 1e-5)])
def test_small_fused_layer(nm, T, w4a4, eps):
    c = SMALL
    L = device_layer(nm, 7, 2, c["E"], c["H"], c["I"], c["S"], (-0.1, 0.1))
    OL = OracleLayer(7, 2, c["H"], c["I"], c["S"], c["E"], (-0.1, 0.1))
    h = gen.hidden_bf16(T, c["H"], 7, layer=2, rho=0.5)
    run_fused(nm, L, OL, h, 4, w4a4, True, eps)


def test_full_fused_layer(nm, full_layer):
    c, L, OL = full_layer
    h = gen.hidden_bf16(1, c["H"], 0, layer=configs.HIDDEN_LAYER)
    run_fused(nm, L, OL, h, c["K"], False, False, 0.0)
    run_fused(nm, L, OL, h, c["K"], True, True, 1e-5)
    h4 = gen.hidden_bf16(4, c["H"], 0, layer=configs.HIDDEN_LAYER, rho=0.5)
    run_fused(nm, L, OL, h4, c["K"], True, True, 1e-5)


def test_full_layer_w4a16_stack_one_token(nm, full_layer):
    """The one-token W4A16 single-layer step as the benchmark times it: one
    moe_stack_forward call over one layer of the pages' shapes (no norm), the
    residual added; routing and output against the oracle."""
    c, L, OL = full_layer
    h = gen.hidden_bf16(1, c["H"], 0, layer=configs.HIDDEN_LAYER)
    hd = to_dev_bf16(h)
    ws = nm.make_stack_workspace([L], 1, c["K"], nm.W4A16)
    hout, idx, w = nm.moe_stack_forward([L], hd, c["K"], nm.W4A16, workspace=ws, rms_eps=c["rms_eps"])
    torch.cuda.synchronize()
    assert nm.nvfp4_last_device_error() == 0
    ref, _, r = OL.forward(h, c["K"], False, True, rms_eps=c["rms_eps"])
    assert check_routing(idx[0].cpu().numpy(), w[0].cpu().numpy(), r, c["K"]) == 0
    assert_close(bf16_to_f64(bf16_bits(hout[0])), bf16_to_f64(ref), "one-layer W4A16 stack")
