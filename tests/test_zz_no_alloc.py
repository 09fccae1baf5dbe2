"""moe_expert_forward_noalloc: the allocation-free variant of
moe_expert_forward, for hosts that hand an operator only its inputs and
outputs and do not let it allocate device memory. It runs the same kernels on
a fixed scratch array that keeps the previous call's contents, so it must give
bit-for-bit the result of moe_expert_forward with a fresh workspace on every
call, also when a call uses less of the array than the call before it.
Collected last so that a stop-at-first-failure run has already run every other
test; it also passes run alone in a fresh process."""
import ctypes

import pytest
import torch

from gen import gen
from tests.gpu_fixtures import device_layer, nm  # noqa: F401


def _noalloc(nm, L, h, idx, w, T, k, mode, eps):
    out = torch.empty_like(h)
    wc = L.c()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = nm.lib().moe_expert_forward_noalloc(ctypes.byref(wc), ctypes.c_void_p(h.data_ptr()),
                                             ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                             T, k, mode, eps, ctypes.c_void_p(h.data_ptr()),
                                             ctypes.c_void_p(out.data_ptr()), stream)
    assert st == 0, nm.nvfp4_status_string(st)
    return out


def _inputs(nm, L, T, H, k, eps, seed):
    from tests.helpers import to_dev_bf16
    h = to_dev_bf16(gen.hidden_bf16(T, H, seed, layer=1, rho=0.5))
    idx, w = nm.moe_route_topk(h, L.router_w, L.router_b, k, rms_eps=eps)
    return h, idx, w


@pytest.mark.gpu
@pytest.mark.parametrize("shape,T,mode,eps", [
    ((16, 256, 128, 192), 3, 1, 0.0),
    ((16, 256, 128, 192), 2, 0, 1e-5),
    ((128, 2688, 1856, 3712), 1, 1, 1e-5),
    ((128, 2688, 1856, 3712), 4, 1, 0.0),
])
def test_noalloc_matches_workspace_call(nm, shape, T, mode, eps):
    E, H, I, S = shape
    k = 4 if E == 16 else 6
    L = device_layer(nm, 3, 1, E, H, I, S, (-0.1, 0.1))
    h, idx, w = _inputs(nm, L, T, H, k, eps, 3)
    ref = nm.moe_expert_forward(L, h, idx, w, mode, residual=h, rms_eps=eps)
    outs = [_noalloc(nm, L, h, idx, w, T, k, mode, eps) for _ in range(2)]  # the scratch keeps its contents
    torch.cuda.synchronize()
    assert nm.nvfp4_last_device_error() == 0
    for out in outs:
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), "noalloc differs from the workspace call"


@pytest.mark.gpu
def test_noalloc_shrinking_calls_on_the_shared_scratch(nm):
    """T = 4, then 1, then 3 on the one scratch array: each call clears what it
    uses, so a larger call's leftovers (counters, partial rows) change nothing."""
    E, H, I, S, k, mode, eps = 128, 2688, 1856, 3712, 6, 1, 1e-5
    L = device_layer(nm, 5, 2, E, H, I, S, (-0.1, 0.1))
    for T in (4, 1, 3):
        h, idx, w = _inputs(nm, L, T, H, k, eps, 10 + T)
        ref = nm.moe_expert_forward(L, h, idx, w, mode, residual=h, rms_eps=eps)
        out = _noalloc(nm, L, h, idx, w, T, k, mode, eps)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"T={T}"
    assert nm.nvfp4_last_device_error() == 0


@pytest.mark.gpu
def test_noalloc_rejects_sizes_beyond_the_scratch(nm):
    # a wide hidden size makes the per-token partial rows alone exceed 1 MiB
    E, H, I, S, T, k = 1, 65536, 64, 64, 4, 1
    L = nm.MoELayer(E, H, I, S)
    assert nm.moe_expert_forward_workspace_size(L, T, k) > nm._abi.NOALLOC_SCRATCH_BYTES
    h = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    with pytest.raises(nm.NVFP4Error) as e:
        nm.moe_expert_forward_noalloc(L, h, idx, w, nm.W4A4)
    assert e.value.status == 4  # NVFP4_ERR_WORKSPACE, rejected before any launch


def test_noalloc_checks_the_layer_before_sizing():
    """A malformed layer gets the status moe_expert_forward gives it, not a
    workspace error from a size computed from bad fields (host checks only:
    nothing is launched)."""
    import __graft_entry__
    __graft_entry__.build()
    from nvfp4_quantized_moe_sigmoid_gb300 import _abi
    lib = _abi.load()
    wl = _abi.MoeLayerWeights()
    wl.num_experts, wl.hidden, wl.inter, wl.shared_inter = 8, 100, 64, 64  # hidden % 64 != 0
    for f in ("up_codes", "up_scales", "up_global", "down_codes", "down_scales", "down_global"):
        setattr(wl, f, 256)
    st = lib.moe_expert_forward_noalloc(ctypes.byref(wl), 256, 256, 256, 1, 1, 1, 0.0, None, 256, None)
    assert st == 2  # NVFP4_ERR_UNSUPPORTED_SHAPE, as moe_expert_forward
    wl.hidden = -64
    st = lib.moe_expert_forward_noalloc(ctypes.byref(wl), 256, 256, 256, 1, 1, 1, 0.0, None, 256, None)
    assert st == 1  # NVFP4_ERR_INVALID_ARG
