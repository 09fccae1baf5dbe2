"""GPU-side fixtures shared by the -m gpu tests: build + import the library,
and helpers that register synthetic weights on the device."""
import numpy as np
import pytest


@pytest.fixture(scope="session")
def nm():
    import __graft_entry__
    __graft_entry__.build()
    import torch
    torch.cuda.set_device(0)
    import nvfp4_quantized_moe_sigmoid_gb300 as nm
    return nm


def device_layer(nm, seed, layer, E, H, I, S, bias_range):
    """One MoE layer registered on the GPU from the device generator."""
    import torch
    from gen import fill
    fb, fr, fbias = fill.fillers(seed, bias_range)
    L = nm.MoELayer(E, H, I, S)
    fr(layer, L.router_w)
    fbias(layer, L.router_b)
    tmp = torch.empty(max(I, S) * H, dtype=torch.bfloat16, device="cuda")
    for e in range(E):
        m = tmp[:I * H].view(I, H)
        fb("up", layer, e, m)
        nm.nvfp4_quantize(m, nm.PER_TENSOR, out=L.expert_up(e))
        m = tmp[:H * I].view(H, I)
        fb("down", layer, e, m)
        nm.nvfp4_quantize(m, nm.PER_TENSOR, out=L.expert_down(e))
    m = tmp[:S * H].view(S, H)
    fb("sh_up", layer, 0, m)
    nm.nvfp4_quantize(m, nm.PER_TENSOR, out=L.shared_up)
    m = tmp[:H * S].view(H, S)
    fb("sh_down", layer, 0, m)
    nm.nvfp4_quantize(m, nm.PER_TENSOR, out=L.shared_down)
    torch.cuda.synchronize()
    return L


def dev_routing(orc_r):
    import torch
    idx = torch.from_numpy(np.ascontiguousarray(orc_r["idx"], np.int32)).cuda()
    w = torch.from_numpy(np.ascontiguousarray(orc_r["w"], np.float32)).cuda()
    return idx, w
