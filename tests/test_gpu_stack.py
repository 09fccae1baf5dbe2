"""moe_stack_forward (all layers of the residual chain in one persistent
kernel) against the oracle. The GPU runs the whole chain in one call; the
oracle is then teacher-forced on the GPU's own layer inputs: for every layer
l it is given the GPU's h_l and must agree with the GPU's routing of layer l
(bit-exact up to near-ties) and with the GPU's h_{l+1} (elementwise within
|err| <= 1e-2 + 2e-2 |ref|).

Small shapes (16 experts, hidden 256) leave most CTAs without a shared-expert
tile and exercise the empty cases of the work partition; the pages' full
shapes run in test_gpu_chain.py."""
import numpy as np
import pytest
import torch

from gen import gen
from oracle.workload import OracleLayer
from tests.gpu_fixtures import device_layer, nm  # noqa: F401
from tests.helpers import (assert_close, bf16_bits, bf16_to_f64, check_routing, colblock_loops,
                           colblock_vectorised, to_dev_bf16)

pytestmark = pytest.mark.gpu

SMALL = dict(E=16, H=256, I=128, S=192)
BIAS = (-0.1, 0.1)


def teacher_forced(nm, OLs, h0, hout, idx, w, k, w4a4, rms_eps):
    """Checks every layer of a GPU chain; returns the number of routing exemptions."""
    L = len(OLs)
    hs = [h0] + [bf16_bits(hout[l]) for l in range(L)]
    idx, w = idx.cpu().numpy(), w.cpu().numpy()
    exempt = 0
    for l in range(L):
        assert np.isfinite(bf16_to_f64(hs[l + 1])).all(), f"layer {l} output not finite"
        ref, _, r = OLs[l].forward(hs[l], k, w4a4, True, rms_eps=rms_eps)
        e = check_routing(idx[l], w[l], r, k)
        exempt += e
        if e == 0:
            assert_close(bf16_to_f64(hs[l + 1]), bf16_to_f64(ref), f"layer {l}")
    return exempt


@pytest.mark.parametrize("B,R,C", [(2, 64, 64), (1, 2688, 1856), (3, 256, 192)])
def test_colblock_layout(nm, B, R, C):
    rng = np.random.default_rng(B * 1000 + C)
    codes = rng.integers(0, 256, (B, R, C // 2), dtype=np.uint8)
    scales = rng.integers(0, 256, (B, R, C // 16), dtype=np.uint8)
    out = nm.nvfp4_colblock_layout(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda())
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    ref = colblock_vectorised(codes, scales)
    if B * R * C <= 2 * 64 * 64:
        np.testing.assert_array_equal(colblock_loops(codes, scales), ref)
    np.testing.assert_array_equal(got, ref)


@pytest.fixture(scope="module")
def small_stack(nm):
    c = SMALL
    layers = [device_layer(nm, 5, l, c["E"], c["H"], c["I"], c["S"], BIAS) for l in range(3)]
    OLs = [OracleLayer(5, l, c["H"], c["I"], c["S"], c["E"], BIAS) for l in range(3)]
    return layers, OLs


@pytest.mark.parametrize("T", [1, 2, 3, 4])
@pytest.mark.parametrize("w4a4", [False, True])
@pytest.mark.parametrize("eps", [0.0, 1e-5])
def test_small_stack(nm, small_stack, T, w4a4, eps):
    layers, OLs = small_stack
    k = 4
    mode = nm.W4A4 if w4a4 else nm.W4A16
    h0 = gen.hidden_bf16(T, SMALL["H"], 5, layer=9, rho=0.5)
    hd = to_dev_bf16(h0)
    ws = nm.make_stack_workspace(layers, T, k, mode)
    hout, idx, w = nm.moe_stack_forward(layers, hd, k, mode, workspace=ws, rms_eps=eps)
    torch.cuda.synchronize()
    assert nm.nvfp4_last_device_error() == 0
    exempt = teacher_forced(nm, OLs, h0, hout, idx, w, k, w4a4, eps)
    assert exempt <= 1
    # the counters were reset by the last CTA: the same workspace gives the same bits
    hout2, idx2, w2 = nm.moe_stack_forward(layers, hd, k, mode, workspace=ws, rms_eps=eps)
    torch.cuda.synchronize()
    assert torch.equal(hout.view(torch.int16), hout2.view(torch.int16))
    assert torch.equal(idx, idx2) and torch.equal(w, w2)


def test_single_layer_stack_matches_layer_call(nm, small_stack):
    """L = 1: the stack is one MoE layer; it agrees with moe_layer_forward to
    FP32 rounding (different summation orders) and routes identically."""
    layers, OLs = small_stack
    T, k = 2, 4
    h0 = gen.hidden_bf16(T, SMALL["H"], 5, layer=11, rho=0.5)
    hd = to_dev_bf16(h0)
    hout, idx, _ = nm.moe_stack_forward(layers[:1], hd, k, nm.W4A4, rms_eps=1e-5)
    out, idx1, _ = nm.moe_layer_forward(layers[0], hd, k, nm.W4A4, residual=hd, rms_eps=1e-5)
    torch.cuda.synchronize()
    assert torch.equal(idx[0], idx1)
    assert_close(bf16_to_f64(bf16_bits(hout[0])), bf16_to_f64(bf16_bits(out)), "stack vs layer call")


def test_stack_rejects_bad_shapes(nm, small_stack):
    layers, _ = small_stack
    hd = to_dev_bf16(gen.hidden_bf16(5, SMALL["H"], 5, layer=9))
    with pytest.raises(nm.NVFP4Error) as ei:  # 5 tokens: beyond the decode path
        nm.moe_stack_forward(layers, hd, 4, nm.W4A4, workspace=torch.zeros(1 << 20, dtype=torch.uint8,
                                                                             device="cuda"))
    assert ei.value.status == 2
    hd = to_dev_bf16(gen.hidden_bf16(1, SMALL["H"], 5, layer=9))
    with pytest.raises(nm.NVFP4Error) as ei:  # more layers than the launch holds
        nm.moe_stack_forward(layers * 11, hd, 4, nm.W4A4,
                             workspace=torch.zeros(1 << 20, dtype=torch.uint8, device="cuda"))
    assert ei.value.status == 2
    ws = nm.make_stack_workspace(layers, 1, 4, nm.W4A4)
    with pytest.raises(nm.NVFP4Error) as ei:  # workspace too small
        nm.moe_stack_forward(layers, hd, 4, nm.W4A4, workspace=ws[:ws.numel() // 2])
    assert ei.value.status == 4
    torch.cuda.synchronize()
    assert nm.nvfp4_last_device_error() == 0


def test_peer_wait_expiry_is_reported_and_recoverable(nm, small_stack):
    """A wait that runs out (a 1 ns limit on the waits for other CTAs' tagged
    words: no word is ever ready in time) ends the call early with
    NVFP4_ERR_TIMEOUT and leaves the context usable: after the workspace is
    re-initialised, the default limit gives the undisturbed result."""
    layers, _ = small_stack
    T, k, mode = 1, 4, nm.W4A4
    hd = to_dev_bf16(gen.hidden_bf16(T, SMALL["H"], 5, layer=13))
    ws = nm.make_stack_workspace(layers, T, k, mode)
    ref, ridx, _ = nm.moe_stack_forward(layers, hd, k, mode, workspace=ws, rms_eps=1e-5)
    torch.cuda.synchronize()
    assert nm.nvfp4_last_device_error() == 0
    try:
        nm.nvfp4_set_peer_wait_limit(1)
        nm.moe_stack_forward(layers, hd, k, mode, workspace=ws, rms_eps=1e-5)
        torch.cuda.synchronize()
        assert nm.nvfp4_last_device_error() == 6  # NVFP4_ERR_TIMEOUT
    finally:
        nm.nvfp4_set_peer_wait_limit(0)
    nm.moe_expert_forward_workspace_init(ws)
    out, idx, _ = nm.moe_stack_forward(layers, hd, k, mode, workspace=ws, rms_eps=1e-5)
    torch.cuda.synchronize()
    assert nm.nvfp4_last_device_error() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16)) and torch.equal(idx, ridx)
