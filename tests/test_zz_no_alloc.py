"""moe_expert_forward_noalloc: the allocation-free variant of
moe_expert_forward, for hosts that hand an operator only its inputs and
outputs and do not let it allocate device memory. It must give the same
result as moe_expert_forward (within the parity tolerance of these tests) on
two consecutive calls, since its fixed scratch array keeps the previous
call's contents. Collected last so that a stop-at-first-failure run has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from gen import configs, gen
from tests.gpu_fixtures import device_layer, nm  # noqa: F401
from tests.helpers import assert_close, bf16_bits, bf16_to_f64, to_dev_bf16


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
    h = to_dev_bf16(gen.hidden_bf16(T, H, 3, layer=1, rho=0.5))
    idx, w = nm.moe_route_topk(h, L.router_w, L.router_b, k, rms_eps=eps)
    ref = nm.moe_expert_forward(L, h, idx, w, mode, residual=h, rms_eps=eps)
    lib = nm.lib()
    wc = L.c()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    outs = []
    for _ in range(2):  # the scratch keeps the previous call's contents
        out = torch.empty_like(h)
        st = lib.moe_expert_forward_noalloc(ctypes.byref(wc), ctypes.c_void_p(h.data_ptr()),
                                            ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                            T, k, mode, eps, ctypes.c_void_p(h.data_ptr()),
                                            ctypes.c_void_p(out.data_ptr()), stream)
        assert st == 0, nm.nvfp4_status_string(st)
        outs.append(out)
    torch.cuda.synchronize()
    assert nm.nvfp4_last_device_error() == 0
    r = bf16_to_f64(bf16_bits(ref))
    for out in outs:
        assert_close(bf16_to_f64(bf16_bits(out)), r, "noalloc vs workspace call")


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
