"""The FP8 (E4M3) per-tensor W8A8 shared expert on the GPU against the
oracle: fp8_quantize bit for bit (codes and scales) on the pages' full-size
shared-expert matrices and on activation rows; moe_shared_fp8_forward
elementwise within |err| <= 1e-2 + 2e-2 |ref| at 1, 4 and 13 tokens (chunks
of 8 and a ragged tail), with and without the pre-norm and the residual; and
a full W4A4 layer whose shared expert is FP8 (the routed experts through
moe_expert_forward, the FP8 shared expert added by moe_shared_fp8_forward)."""
import numpy as np
import pytest
import torch

from gen import configs, fill, gen
from oracle import oracle as orc
from oracle.workload import OracleLayer
from tests.gpu_fixtures import dev_routing, device_layer, nm  # noqa: F401
from tests.helpers import assert_close, bf16_bits, bf16_to_f64, to_dev_bf16

pytestmark = pytest.mark.gpu


def gpu_fp8(nm, x, mode, g=None):
    xd = to_dev_bf16(x) if x.dtype == np.uint16 else torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    gs = None if g is None else torch.tensor([g], dtype=torch.float32, device="cuda")
    m = nm.fp8_quantize(xd, mode, global_scale=gs)
    torch.cuda.synchronize()
    return m.codes.cpu().numpy(), m.global_scale.cpu().numpy()


def same(nm, x, mode, g=None):
    q1, g1 = gpu_fp8(nm, x, mode, g)
    q0, g0 = orc.fp8_quantize(x, mode, g)
    assert np.array_equal(g1.view(np.uint32), g0.view(np.uint32)), "scale differs"
    assert np.array_equal(q1, q0), f"codes differ in {np.sum(q1 != q0)} places"


@pytest.fixture(scope="module")
def shared(nm):
    """The pages' shared expert (3712 x 2688 and 2688 x 3712) in FP8, on the
    device and in the oracle, from the same bf16 masters."""
    c = configs.shape(0)
    H, S = c["H"], c["S"]
    fb, _, _ = fill.fillers(c["seed"], c["bias"])
    up_m = torch.empty((S, H), dtype=torch.bfloat16, device="cuda")
    dn_m = torch.empty((H, S), dtype=torch.bfloat16, device="cuda")
    fb("sh_up", 0, 0, up_m)
    fb("sh_down", 0, 0, dn_m)
    up, dn = nm.fp8_quantize(up_m, nm.PER_TENSOR), nm.fp8_quantize(dn_m, nm.PER_TENSOR)
    wu, gu = orc.fp8_quantize(gen.sh_up_master(c["seed"], 0, S, H), orc.PER_TENSOR)
    wd, gd = orc.fp8_quantize(gen.sh_down_master(c["seed"], 0, H, S), orc.PER_TENSOR)
    torch.cuda.synchronize()
    assert np.array_equal(up.codes.cpu().numpy(), wu) and np.array_equal(dn.codes.cpu().numpy(), wd)
    assert up.global_scale.cpu().numpy()[0] == gu[0] and dn.global_scale.cpu().numpy()[0] == gd[0]
    return c, up, dn, (wu, gu[0], wd, gd[0])


def test_quantize_rows_tensor_and_given(nm):
    x = gen.hidden_bf16(9, 2688, 0, layer=4)
    same(nm, x, orc.PER_ROW)
    same(nm, x, orc.PER_TENSOR)
    f = (gen.normal_f32(6 * 96, 2, 8) * 3.0).astype(np.float32).reshape(6, 96)
    same(nm, f, orc.GIVEN, g=0.0017)  # includes values beyond 448 g: saturated
    z = np.zeros((3, 64), np.float32)
    z[1, 5] = -0.0
    z[2, 7] = 1e-30  # a tiny row: its own scale
    z[2, 8] = -1e-30
    same(nm, z, orc.PER_ROW)
    # every E4M3 midpoint and its neighbours, at a scale of 1
    v = np.array([orc.e4m3_value(b) for b in range(0x7F)], np.float64)
    mids = ((v[1:] + v[:-1]) / 2).astype(np.float32)
    pts = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    pts = np.concatenate([pts, -pts])
    pts = pts[: pts.size // 16 * 16].reshape(-1, 16)
    same(nm, pts, orc.GIVEN, g=1.0)


@pytest.mark.parametrize("T,eps,residual", [(1, 0.0, False), (4, 0.0, True), (13, 1e-5, True)])
def test_shared_expert_matches_oracle(nm, shared, T, eps, residual):
    c, up, dn, (wu, gu, wd, gd) = shared
    h = gen.hidden_bf16(T, c["H"], 0, layer=14, rho=0.3)
    if eps > 0:  # a pre-normed block sees a larger residual stream
        h = ((gen.bf16_bits_to_f32(h) * 5.0).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    hd = to_dev_bf16(h)
    res = gen.hidden_bf16(T, c["H"], 0, layer=15) if residual else None
    out = nm.moe_shared_fp8_forward(up, dn, hd, residual=to_dev_bf16(res) if residual else None, rms_eps=eps)
    torch.cuda.synchronize()
    assert nm.nvfp4_last_device_error() == 0
    x = orc.rms_norm(h, eps) if eps > 0 else h
    y, _ = orc.shared_fp8(x, wu, gu, wd, gd)
    if residual:
        y = y + bf16_to_f64(res)
    ref = bf16_to_f64(np.array([[orc.bf16_round(v) for v in row] for row in y], np.uint16))
    assert_close(bf16_to_f64(bf16_bits(out)), ref, "FP8 shared expert")


def test_layer_with_fp8_shared_expert(nm, shared):
    """The W4A4 card's precision recipe for one MoE layer: routed experts
    NVFP4 W4A4, shared expert FP8 W8A8. The routed experts run through
    moe_expert_forward with an all-zero NVFP4 shared expert (it adds exactly
    0); moe_shared_fp8_forward then adds the FP8 shared expert to their
    output."""
    c, up, dn, (wu, gu, wd, gd) = shared
    E, H, I, S, K = c["E"], c["H"], c["I"], c["S"], c["K"]
    L = device_layer(nm, 0, 0, E, H, I, S, c["bias"])
    zero = torch.zeros((S, H), dtype=torch.bfloat16, device="cuda")
    nm.nvfp4_quantize(zero, nm.PER_TENSOR, out=L.shared_up)
    nm.nvfp4_quantize(zero.view(H, S), nm.PER_TENSOR, out=L.shared_down)
    OL = OracleLayer(0, 0, H, I, S, E, c["bias"])
    OL.sh_up = orc.Mat.from_master(np.zeros((S, H), np.uint16))
    OL.sh_down = orc.Mat.from_master(np.zeros((H, S), np.uint16))
    T = 3
    h = gen.hidden_bf16(T, H, 0, layer=16, rho=0.4)
    hd = to_dev_bf16(h)
    r = OL.route(h, K)
    idx, w = dev_routing(r)
    routed = nm.moe_expert_forward(L, hd, idx, w, nm.W4A4, residual=hd)
    out = nm.moe_shared_fp8_forward(up, dn, hd, residual=routed)
    torch.cuda.synchronize()
    assert nm.nvfp4_last_device_error() == 0
    ref_routed, _, _ = OL.forward(h, K, True, True, routing=r)
    assert_close(bf16_to_f64(bf16_bits(routed)), bf16_to_f64(ref_routed), "routed experts")
    y, _ = orc.shared_fp8(h, wu, gu, wd, gd)
    # the oracle continues from the GPU's routed output (one bf16 rounding
    # each step, as the two calls make)
    y = y + bf16_to_f64(bf16_bits(routed))
    ref = bf16_to_f64(np.array([[orc.bf16_round(v) for v in row] for row in y], np.uint16))
    assert_close(bf16_to_f64(bf16_bits(out)), ref, "layer with the FP8 shared expert")
