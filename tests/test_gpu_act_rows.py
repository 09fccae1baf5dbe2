"""The NVFP4 activation rows the MoE kernels build in flight, read back from
the workspace (nvfp4_workspace_view) and compared bit for bit with the
oracle's quantiser applied to the same bf16 rows: the layer input (B operand
of the up GEMMs), the routed intermediate relu(up)^2 and the shared expert's
intermediate (B operands of the down GEMMs), all with a per-row global
amax / 2688 (W4A4: "Let's optimize Nemotron 3.5 Lightning - a worklog",
Step 3; the quantiser of "NVFP4 quantisation", Step 1).

The grouped tensor-core path keeps codes, scales and row globals; the
layer call's GEMV path keeps each element as the f16 product E2M1 value x
E4M3 scale (exact in f16), compared with the oracle's codes decoded the same
way. The intermediate rows are the kernels' own bf16 values, so the check
isolates the quantiser at every fused site; the layer outputs themselves are
checked against the oracle in test_gpu_moe.py."""
import numpy as np
import pytest
import torch

from gen import configs, gen
from oracle import oracle as orc
from tests.gpu_fixtures import device_layer, nm  # noqa: F401
from tests.helpers import to_dev_bf16

pytestmark = pytest.mark.gpu

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])
E4M3 = np.array([orc.e4m3_value(b) for b in range(256)])


@pytest.fixture(scope="module")
def layer(nm):
    c = configs.shape(0)
    L = device_layer(nm, 0, 0, c["E"], c["H"], c["I"], c["S"], c["bias"])
    return c, L


def rows_u8(ws, off, rows, pitch, width):
    a = ws[off:off + rows * pitch].reshape(rows, pitch)
    return np.ascontiguousarray(a[:, :width])


def view_rows(ws, v):
    """(values, scales or None, globals or None) of one region, on the host."""
    rows, cols = v["rows"], v["cols"]
    g = None
    if v["has_global"]:
        g = ws[v["global_offset"]:v["global_offset"] + 4 * rows].view(np.float32).copy()
    if v["format"] == 1:  # NVFP4 codes + E4M3 scales
        codes = rows_u8(ws, v["offset"], rows, v["pitch"], cols // 2)
        scales = rows_u8(ws, v["scales_offset"], rows, v["scales_pitch"], cols // 16)
        return codes, scales, g
    vals = rows_u8(ws, v["offset"], rows, v["pitch"], 2 * cols).view(np.uint16)
    return vals, None, g


def dequant_f16_bits(codes, scales):
    """E2M1 value x E4M3 scale per element as f16 bits (both exact in f16),
    with -0 taken as +0."""
    lo, hi = codes & 0xF, codes >> 4
    c = np.empty((codes.shape[0], codes.shape[1] * 2), np.uint8)
    c[:, 0::2], c[:, 1::2] = lo, hi
    v = E2M1[c] * np.repeat(E4M3[scales], 16, axis=1)
    v = v.astype(np.float16)
    v[v == 0] = 0.0
    return v.view(np.uint16)


def compare_quantised(ws, v, src_bf16, what):
    """src_bf16: the bf16 rows the kernel quantised. Returns mismatched rows."""
    got, gs, gg = view_rows(ws, v)
    codes, scales, g = orc.quantize(src_bf16, orc.PER_ROW)
    bad_g = gg.view(np.uint32) != g.view(np.uint32)
    if v["format"] == 1:
        bad = np.any(got != codes, axis=1) | np.any(gs != scales, axis=1) | bad_g
    else:
        f = got.copy()
        f[(f & 0x7FFF) == 0] = 0
        bad = np.any(f != dequant_f16_bits(codes, scales), axis=1) | bad_g
    n = int(bad.sum())
    assert n == 0, f"{what}: {n} of {len(bad)} rows differ from the oracle's quantiser (first {np.flatnonzero(bad)[:5]})"
    return n


@pytest.mark.parametrize("T", [5, 37])
def test_grouped_path_rows_bit_exact(nm, layer, T):
    c, L = layer
    K = c["K"]
    h = gen.hidden_bf16(T, c["H"], 0, layer=12, rho=0.5)
    hd = to_dev_bf16(h)
    idx, w = nm.moe_route_topk(hd, L.router_w, L.router_b, K)
    ws = nm.make_workspace(L, T, K, nm.W4A4)
    nm.moe_expert_forward(L, hd, idx, w, nm.W4A4, residual=hd, workspace=ws, rms_eps=0.0)
    torch.cuda.synchronize()
    assert nm.nvfp4_last_device_error() == 0
    wsh = ws.cpu().numpy()
    view = lambda r: nm.nvfp4_workspace_view(nm.CALL_EXPERT_FORWARD, L, T, K, nm.W4A4, r)
    assert view(nm.WS_ACT)["position_order"] == 1
    compare_quantised(wsh, view(nm.WS_X), h, "input rows")
    act, _, _ = view_rows(wsh, view(nm.WS_ACT))
    assert np.any(act != 0)
    compare_quantised(wsh, view(nm.WS_ACT_Q), act, "routed intermediate rows")
    act_sh, _, _ = view_rows(wsh, view(nm.WS_SH_ACT))
    compare_quantised(wsh, view(nm.WS_SH_ACT_Q), act_sh, "shared intermediate rows")


@pytest.mark.parametrize("T", [1, 4])
def test_layer_call_rows_bit_exact(nm, layer, T):
    c, L = layer
    K = c["K"]
    h = gen.hidden_bf16(T, c["H"], 0, layer=13, rho=0.5)
    hd = to_dev_bf16(h)
    ws = nm.make_layer_workspace(L, T, K, nm.W4A4)
    nm.moe_layer_forward(L, hd, K, nm.W4A4, residual=hd, workspace=ws, rms_eps=0.0)
    torch.cuda.synchronize()
    assert nm.nvfp4_last_device_error() == 0
    wsh = ws.cpu().numpy()
    view = lambda r: nm.nvfp4_workspace_view(nm.CALL_LAYER_FORWARD, L, T, K, nm.W4A4, r)
    compare_quantised(wsh, view(nm.WS_X), h, "input rows")
    act, _, _ = view_rows(wsh, view(nm.WS_ACT))
    assert np.any(act != 0)
    compare_quantised(wsh, view(nm.WS_ACT_Q), act, "routed intermediate rows")
    act_sh, _, _ = view_rows(wsh, view(nm.WS_SH_ACT))
    compare_quantised(wsh, view(nm.WS_SH_ACT_Q), act_sh, "shared intermediate rows")


def test_decode_path_keeps_only_bf16_rows(nm, layer):
    c, L = layer
    with pytest.raises(nm.NVFP4Error):
        nm.nvfp4_workspace_view(nm.CALL_EXPERT_FORWARD, L, 1, c["K"], nm.W4A4, nm.WS_X)
    v = nm.nvfp4_workspace_view(nm.CALL_EXPERT_FORWARD, L, 1, c["K"], nm.W4A4, nm.WS_ACT)
    assert v["format"] == nm.WS_BF16 and v["rows"] == c["K"]
