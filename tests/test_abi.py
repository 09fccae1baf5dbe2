"""The C-ABI library loads and exports every symbol include/nvfp4moe.h
declares; host-side argument checks reject bad calls before any launch (no
GPU is needed for these)."""
import ctypes
import os

import pytest

from tests.helpers import header_functions

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def abi():
    import __graft_entry__
    __graft_entry__.build()
    from nvfp4_quantized_moe_sigmoid_gb300 import _abi
    return _abi


def test_header_lists_the_boundary():
    names = header_functions()
    for n in ["nvfp4_quantize", "moe_route_topk", "moe_expert_forward", "lm_head_gemv",
              "moe_expert_forward_workspace_size", "nvfp4_status_string",
              "nvfp4_last_device_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(abi):
    lib = ctypes.CDLL(abi.LIB_PATH)
    for n in header_functions():
        assert hasattr(lib, n), f"missing export {n}"
    assert set(header_functions()) <= set(abi.EXPORTS)


def test_status_strings(abi):
    L = abi.load()
    assert L.nvfp4_status_string(0) == b"ok"
    assert L.nvfp4_status_string(6) == b"device wait timed out"
    assert L.nvfp4_status_string(99) == b"unknown status"


def test_host_validation_rejects_bad_arguments(abi):
    L = abi.load()
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: calls are rejected first
    odd = ctypes.c_void_p(0x10001)
    # nvfp4_quantize: null global, bad cols, bad mode, misaligned input
    assert L.nvfp4_quantize(fake, 1, 4, 32, 0, null, fake, fake, null) == 1
    assert L.nvfp4_quantize(fake, 1, 4, 24, 0, fake, fake, fake, null) == 2
    assert L.nvfp4_quantize(fake, 1, 4, 32, 7, fake, fake, fake, null) == 1
    assert L.nvfp4_quantize(odd, 1, 4, 32, 0, fake, fake, fake, null) == 3
    # moe_route_topk: k > E, H % 16, E > 256, misaligned hidden
    assert L.moe_route_topk(fake, fake, fake, 1, 64, 8, 9, 0.0, fake, fake, null) == 1
    assert L.moe_route_topk(fake, fake, fake, 1, 72, 8, 2, 0.0, fake, fake, null) == 2
    assert L.moe_route_topk(fake, fake, fake, 1, 64, 300, 2, 0.0, fake, fake, null) == 2
    assert L.moe_route_topk(odd, fake, fake, 1, 64, 8, 2, 0.0, fake, fake, null) == 3
    assert L.moe_route_topk(null, fake, fake, 1, 64, 8, 2, 0.0, fake, fake, null) == 1
    # lm_head_gemv
    m = abi.NVFP4Matrix(0x10000, 0x10000, 0x10000, 100, 2688)
    assert L.lm_head_gemv(ctypes.byref(m), fake, 1, 0.0, fake, null) == 2
    m = abi.NVFP4Matrix(0x10000, 0x10000, 0x10000, 128, 2688)
    assert L.lm_head_gemv(ctypes.byref(m), odd, 1, 0.0, fake, null) == 3
    assert L.lm_head_gemv(ctypes.byref(m), fake, 0, 0.0, fake, null) == 1
    # moe_expert_forward: shapes, workspace size, null weights
    sh_up = abi.NVFP4Matrix(0x10000, 0x10000, 0x10000, 3712, 2688)
    sh_dn = abi.NVFP4Matrix(0x10000, 0x10000, 0x10000, 2688, 3712)
    w = abi.MoeLayerWeights(128, 2688, 1856, 3712, 0x10000, 0x10000, 0x10000, 0x10000, 0x10000,
                            0x10000, sh_up, sh_dn)
    need = L.moe_expert_forward_workspace_size(ctypes.byref(w), 1, 6, 1)
    assert need > 0
    assert L.moe_expert_forward(ctypes.byref(w), fake, fake, fake, 1, 6, 1, 0.0, null, ctypes.c_void_p(0x20000),
                                ctypes.c_void_p(0x30000), need - 1, null) == 4
    assert L.moe_expert_forward(ctypes.byref(w), fake, fake, fake, 1, 6, 5, 0.0, null, ctypes.c_void_p(0x20000),
                                ctypes.c_void_p(0x30000), need, null) == 1
    bad = abi.MoeLayerWeights(128, 2688, 1850, 3712, 0x10000, 0x10000, 0x10000, 0x10000, 0x10000,
                              0x10000, sh_up, sh_dn)
    assert L.moe_expert_forward(ctypes.byref(bad), fake, fake, fake, 1, 6, 1, 0.0, null, fake, fake, need,
                                null) == 2
    # widths that are multiples of 16 but not of 64 (I = 1840): moe_expert_forward takes them (the
    # generic kernels, any token count, the decode workspace), the fused layer call does not
    sh_up16 = abi.NVFP4Matrix(0x10000, 0x10000, 0x10000, 3712, 2688)
    w16 = abi.MoeLayerWeights(128, 2688, 1840, 3712, 0x10000, 0x10000, 0x10000, 0x10000, 0x10000,
                              0x10000, sh_up16, sh_dn)
    need16 = L.moe_expert_forward_workspace_size(ctypes.byref(w16), 8, 6, 1)
    assert need16 >= 8 * 6 * 1840 * 2 + 8 * 6 * 2688 * 4
    assert L.moe_expert_forward(ctypes.byref(w16), fake, fake, fake, 8, 6, 1, 0.0, null, ctypes.c_void_p(0x20000),
                                ctypes.c_void_p(0x30000), need16 - 1, null) == 4
    assert L.moe_layer_forward(ctypes.byref(w16), fake, fake, fake, 1, 6, 1, 0.0, null, fake, fake, fake,
                               ctypes.c_void_p(0x30000), need16, null) == 2
    nul = abi.MoeLayerWeights(128, 2688, 1856, 3712, 0, 0x10000, 0x10000, 0x10000, 0x10000, 0x10000,
                              sh_up, sh_dn)
    assert L.moe_expert_forward(ctypes.byref(nul), fake, fake, fake, 1, 6, 1, 0.0, null, fake, fake, need,
                                null) == 1
    # nvfp4_colblock_layout: null input, rows % 32, cols % 16, misaligned out
    assert L.nvfp4_colblock_layout(null, fake, 1, 64, 32, fake, null) == 1
    assert L.nvfp4_colblock_layout(fake, fake, 1, 48, 32, fake, null) == 2
    assert L.nvfp4_colblock_layout(fake, fake, 1, 64, 24, fake, null) == 2
    assert L.nvfp4_colblock_layout(fake, fake, 1, 64, 32, odd, null) == 3
    assert L.nvfp4_colblock_layout(fake, fake, 0, 64, 32, fake, null) == 1


def test_workspace_size_grows_with_tokens(abi):
    L = abi.load()
    sh_up = abi.NVFP4Matrix(1, 1, 1, 3712, 2688)
    sh_dn = abi.NVFP4Matrix(1, 1, 1, 2688, 3712)
    w = abi.MoeLayerWeights(128, 2688, 1856, 3712, 1, 1, 1, 1, 1, 1, sh_up, sh_dn)
    a = L.moe_expert_forward_workspace_size(ctypes.byref(w), 1, 6, 1)
    b = L.moe_expert_forward_workspace_size(ctypes.byref(w), 4, 6, 1)
    assert b > a > 6 * 1856 * 2


def test_package_fails_loudly_without_library(abi, tmp_path):
    with pytest.raises(ImportError):
        abi.load.__wrapped__ if False else None
        from nvfp4_quantized_moe_sigmoid_gb300 import _abi as a2
        saved = a2._lib
        a2._lib = None
        try:
            a2.load(str(tmp_path / "missing.so"))
        finally:
            a2._lib = saved


def test_colblock_references_agree():
    """The vectorised column-block reference equals the byte-by-byte statement
    of the layout in include/nvfp4moe.h (the GPU test compares the kernel with
    the vectorised one at the full shapes)."""
    import numpy as np
    from tests.helpers import colblock_loops, colblock_vectorised
    rng = np.random.default_rng(7)
    for B, R, C in [(2, 64, 64), (1, 96, 48), (3, 32, 16)]:
        codes = rng.integers(0, 256, (B, R, C // 2), dtype=np.uint8)
        scales = rng.integers(0, 256, (B, R, C // 16), dtype=np.uint8)
        a = colblock_loops(codes, scales)
        assert a.shape == (B, C // 16, 9 * R)
        np.testing.assert_array_equal(a, colblock_vectorised(codes, scales))
        # every input byte lands exactly once
        assert sorted(a.reshape(-1).tolist()) == sorted(codes.reshape(-1).tolist() + scales.reshape(-1).tolist())


def test_workspace_view_of_the_layer_call(abi):
    """nvfp4_workspace_view (host arithmetic only): the regions of a
    moe_layer_forward workspace lie inside it, do not overlap, and the
    quantised regions of a W4A16 call are refused."""
    L = abi.load()
    sh_up = abi.NVFP4Matrix(0x10000, 0x10000, 0x10000, 3712, 2688)
    sh_dn = abi.NVFP4Matrix(0x10000, 0x10000, 0x10000, 2688, 3712)
    w = abi.MoeLayerWeights(128, 2688, 1856, 3712, 0x10000, 0x10000, 0x10000, 0x10000, 0x10000,
                            0x10000, sh_up, sh_dn)
    for T in (1, 4):
        total = L.moe_layer_forward_workspace_size(ctypes.byref(w), T, 6, 1)
        spans = []
        for region, (rows, cols) in enumerate([(T, 2688), (6 * T, 1856), (6 * T, 1856), (T, 3712), (T, 3712)]):
            v = abi.WsView()
            assert L.nvfp4_workspace_view(1, ctypes.byref(w), T, 6, 1, region, ctypes.byref(v)) == 0
            assert (v.rows, v.cols, v.pitch) == (rows, cols, 2 * cols)
            assert v.format == (0 if region in (1, 3) else 2) and v.has_global == (region not in (1, 3))
            spans.append((v.offset, v.offset + rows * v.pitch))
            if v.has_global:
                spans.append((v.global_offset, v.global_offset + 4 * rows))
        spans.sort()
        assert spans[-1][1] <= total
        assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:])), spans
        v = abi.WsView()
        assert L.nvfp4_workspace_view(1, ctypes.byref(w), T, 6, 0, 0, ctypes.byref(v)) == 2
        assert L.nvfp4_workspace_view(1, ctypes.byref(w), T, 6, 0, 1, ctypes.byref(v)) == 0
    v = abi.WsView()
    assert L.nvfp4_workspace_view(1, ctypes.byref(w), 5, 6, 1, 0, ctypes.byref(v)) == 2
    assert L.nvfp4_workspace_view(2, ctypes.byref(w), 1, 6, 1, 0, ctypes.byref(v)) == 1
    assert L.nvfp4_workspace_view(1, ctypes.byref(w), 1, 6, 1, 5, ctypes.byref(v)) == 1
    assert L.nvfp4_workspace_view(1, ctypes.byref(w), 1, 6, 1, 0, None) == 1
