"""The library in a second CUDA context of the same device (cuCtxCreate):
moe_expert_forward_noalloc, whose scratch array is a device symbol, and the
decode kernels, whose shared-memory limit is raised per module, must both be
looked up again there. The call in the new context (all buffers allocated
and copied with the driver API: torch's memory belongs to the primary
context) must give the bits the primary context gave, and the primary
context must still work after the second one is destroyed."""
import ctypes

import numpy as np
import pytest
import torch

from gen import gen
from oracle.workload import OracleLayer
from tests.gpu_fixtures import dev_routing, device_layer, nm  # noqa: F401
from tests.helpers import to_dev_bf16

pytestmark = pytest.mark.gpu

SHAPE = dict(E=8, H=2688, I=1856, S=3712)  # the pages' expert shapes; ring > 48 KB of shared memory


def driver():
    cu = ctypes.CDLL("libcuda.so.1")
    cu.cuCtxCreate_v4.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p, ctypes.c_uint, ctypes.c_int]
    cu.cuCtxDestroy_v2.argtypes = [ctypes.c_void_p]
    cu.cuMemAlloc_v2.argtypes = [ctypes.POINTER(ctypes.c_uint64), ctypes.c_size_t]
    cu.cuMemFree_v2.argtypes = [ctypes.c_uint64]
    cu.cuMemcpyHtoD_v2.argtypes = [ctypes.c_uint64, ctypes.c_void_p, ctypes.c_size_t]
    cu.cuMemcpyDtoH_v2.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_size_t]
    cu.cuCtxSynchronize.argtypes = []
    cu.cuDeviceGet.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.c_int]
    return cu


def ok(r):
    assert r == 0, f"CUDA driver call returned {r}"


def test_noalloc_call_in_a_second_context(nm):
    from nvfp4_quantized_moe_sigmoid_gb300 import _abi
    c = SHAPE
    T, k = 2, 6
    L = device_layer(nm, 9, 0, c["E"], c["H"], c["I"], c["S"], (-0.1, 0.1))
    OL = OracleLayer(9, 0, c["H"], c["I"], c["S"], c["E"], (-0.1, 0.1))
    h = gen.hidden_bf16(T, c["H"], 9, layer=5)
    idx, w = dev_routing(OL.route(h, k))
    hd = to_dev_bf16(h)
    ref = nm.moe_expert_forward_noalloc(L, hd, idx, w, nm.W4A4)
    torch.cuda.synchronize()
    ref = ref.view(torch.int16).cpu().numpy()
    # every buffer the call reads, as host copies
    host = {
        "up_codes": L.up_codes, "up_scales": L.up_scales, "up_global": L.up_global,
        "down_codes": L.down_codes, "down_scales": L.down_scales, "down_global": L.down_global,
        "su_codes": L.shared_up.codes, "su_scales": L.shared_up.scales, "su_global": L.shared_up.global_scale,
        "sd_codes": L.shared_down.codes, "sd_scales": L.shared_down.scales, "sd_global": L.shared_down.global_scale,
        "hidden": hd, "idx": idx, "w": w,
    }
    host = {n: (t.view(torch.int16) if t.dtype == torch.bfloat16 else t).contiguous().cpu().numpy()
            for n, t in host.items()}
    torch.cuda.synchronize()

    cu = driver()
    dev = ctypes.c_int()
    ok(cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()))
    ctx = ctypes.c_void_p()
    ok(cu.cuCtxCreate_v4(ctypes.byref(ctx), None, 0, dev.value))  # now current on this thread
    ptrs = {}
    try:
        for n, a in host.items():
            p = ctypes.c_uint64()
            ok(cu.cuMemAlloc_v2(ctypes.byref(p), a.nbytes))
            ok(cu.cuMemcpyHtoD_v2(p.value, a.ctypes.data, a.nbytes))
            ptrs[n] = p.value
        out = ctypes.c_uint64()
        ok(cu.cuMemAlloc_v2(ctypes.byref(out), ref.nbytes))
        ptrs["out"] = out.value
        su = _abi.NVFP4Matrix(ptrs["su_codes"], ptrs["su_scales"], ptrs["su_global"], c["S"], c["H"])
        sd = _abi.NVFP4Matrix(ptrs["sd_codes"], ptrs["sd_scales"], ptrs["sd_global"], c["H"], c["S"])
        lw = _abi.MoeLayerWeights(c["E"], c["H"], c["I"], c["S"], ptrs["up_codes"], ptrs["up_scales"],
                                  ptrs["up_global"], ptrs["down_codes"], ptrs["down_scales"], ptrs["down_global"],
                                  su, sd)
        lib = _abi.load()
        st = lib.moe_expert_forward_noalloc(ctypes.byref(lw), ctypes.c_void_p(ptrs["hidden"]),
                                            ctypes.c_void_p(ptrs["idx"]), ctypes.c_void_p(ptrs["w"]), T, k, nm.W4A4,
                                            0.0, None, ctypes.c_void_p(ptrs["out"]), None)
        assert st == 0, f"status {st} in the second context"
        ok(cu.cuCtxSynchronize())
        assert lib.nvfp4_last_device_error(None) == 0
        got = np.empty_like(ref)
        ok(cu.cuMemcpyDtoH_v2(got.ctypes.data, ptrs["out"], got.nbytes))
        assert np.array_equal(got, ref), f"{np.sum(got != ref)} outputs differ from the primary context's"
    finally:
        for p in ptrs.values():
            cu.cuMemFree_v2(p)
        ok(cu.cuCtxDestroy_v2(ctx))  # pops it: the primary context is current again
    again = nm.moe_expert_forward_noalloc(L, hd, idx, w, nm.W4A4)
    torch.cuda.synchronize()
    assert np.array_equal(again.view(torch.int16).cpu().numpy(), ref)
