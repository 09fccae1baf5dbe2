"""Python binding of libnvfp4moe.so: the NVFP4 sigmoid-routed MoE decode path
and the NVFP4 weight-only lm_head as sm_103a CUDA kernels.

The functions below carry the C-ABI names of include/nvfp4moe.h and only
marshal arguments: torch CUDA tensors provide device memory and the current
stream, every step of the computation runs in the library's kernels. There is
no CPU or PyTorch fallback; importing this package without the built library
raises ImportError.
"""
import ctypes

import torch

from . import _abi

__all__ = ["NVFP4Matrix", "MoELayer", "NVFP4Error", "nvfp4_quantize", "moe_route_topk",
           "moe_expert_forward_workspace_size", "moe_expert_forward_workspace_init",
           "moe_expert_forward", "moe_expert_forward_noalloc", "moe_layer_forward",
           "moe_layer_forward_workspace_size", "moe_stack_forward", "moe_stack_forward_workspace_size",
           "make_stack_workspace", "nvfp4_colblock_layout", "moe_permute", "lm_head_gemv", "lm_head_forward",
           "make_lm_head_workspace",
           "nvfp4_status_string", "nvfp4_last_device_error", "nvfp4_workspace_view",
           "FP8Matrix", "fp8_quantize", "moe_shared_fp8_workspace_size", "moe_shared_fp8_forward",
           "W4A16", "W4A4", "PER_TENSOR", "PER_ROW", "GIVEN", "lib"]

W4A16, W4A4 = 0, 1
PER_TENSOR, PER_ROW, GIVEN = 0, 1, 2

_L = _abi.load()


def lib():
    return _L


class NVFP4Error(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {_abi.STATUS.get(status, status)} "
                         f"({_L.nvfp4_status_string(status).decode()})")


def _check(status, what):
    if status != 0:
        raise NVFP4Error(status, what)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def nvfp4_status_string(status: int) -> str:
    return _L.nvfp4_status_string(int(status)).decode()


def nvfp4_last_device_error(stream=None) -> int:
    return _L.nvfp4_last_device_error(_stream(stream))


def nvfp4_set_decode_max_tokens(t=4):
    """moe_expert_forward runs up to t tokens (0..4) on the decode GEMV kernels,
    more on the grouped path."""
    _check(_L.nvfp4_set_decode_max_tokens(int(t)), "nvfp4_set_decode_max_tokens")


def nvfp4_set_peer_wait_limit(ns=0):
    """Limit (ns) of the stack kernel's waits on other CTAs; 0 restores 1 s."""
    _check(_L.nvfp4_set_peer_wait_limit(int(ns)), "nvfp4_set_peer_wait_limit")


def nvfp4_fp4_mma_peak(n=256, chains=1, iters=20000, stream=None) -> float:
    """Dense FP4 tensor-pipe throughput of this GPU in TFLOP/s (block-scaled
    tcgen05 MMAs, M = 128, N = n, K = 64, on every SM)."""
    out = ctypes.c_double(0.0)
    _check(_L.nvfp4_fp4_mma_peak(n, chains, iters, ctypes.byref(out), _stream(stream)), "nvfp4_fp4_mma_peak")
    return out.value


class NVFP4Matrix:
    """An NVFP4 matrix [n][k] in the canonical layout (device tensors)."""

    def __init__(self, codes, scales, global_scale):
        self.codes, self.scales, self.global_scale = codes, scales, global_scale
        self.n, self.k = codes.shape[-2], codes.shape[-1] * 2

    @staticmethod
    def empty(n, k, device="cuda"):
        return NVFP4Matrix(torch.empty((n, k // 2), dtype=torch.uint8, device=device),
                           torch.empty((n, k // 16), dtype=torch.uint8, device=device),
                           torch.empty(1, dtype=torch.float32, device=device))

    def c(self):
        return _abi.NVFP4Matrix(self.codes.data_ptr(), self.scales.data_ptr(),
                                self.global_scale.data_ptr(), self.n, self.k)

    def nbytes(self):
        return self.codes.numel() + self.scales.numel()


class FP8Matrix:
    """An FP8 (E4M3) matrix [n][k] with one FP32 scale (device tensors)."""

    def __init__(self, codes, global_scale):
        self.codes, self.global_scale = codes, global_scale
        self.n, self.k = codes.shape[-2], codes.shape[-1]

    @staticmethod
    def empty(n, k, device="cuda"):
        return FP8Matrix(torch.empty((n, k), dtype=torch.uint8, device=device),
                         torch.empty(1, dtype=torch.float32, device=device))

    def c(self):
        return _abi.FP8Matrix(self.codes.data_ptr(), self.global_scale.data_ptr(), self.n, self.k)


class MoELayer:
    """Device weights of one MoE layer: router (fp32 gate + fp32 bias), stacked
    routed experts (NVFP4 up [E][I][H], down [E][H][I]) and one shared expert."""

    def __init__(self, E, H, I, S, device="cuda"):
        self.E, self.H, self.I, self.S = E, H, I, S
        u8 = dict(dtype=torch.uint8, device=device)
        self.router_w = torch.empty((E, H), dtype=torch.float32, device=device)
        self.router_b = torch.empty(E, dtype=torch.float32, device=device)
        self.up_codes = torch.empty((E, I, H // 2), **u8)
        self.up_scales = torch.empty((E, I, H // 16), **u8)
        self.up_global = torch.empty(E, dtype=torch.float32, device=device)
        self.down_codes = torch.empty((E, H, I // 2), **u8)
        self.down_scales = torch.empty((E, H, I // 16), **u8)
        self.down_global = torch.empty(E, dtype=torch.float32, device=device)
        self.shared_up = NVFP4Matrix.empty(S, H, device)
        self.shared_down = NVFP4Matrix.empty(H, S, device)
        # column-block copies of the down weights for moe_stack_forward,
        # made on first use from the weights at that time (stack_layout)
        self.down_cb = None
        self.shared_down_cb = None
        self._c = None

    def expert_up(self, e):
        return NVFP4Matrix(self.up_codes[e], self.up_scales[e], self.up_global[e:e + 1])

    def expert_down(self, e):
        return NVFP4Matrix(self.down_codes[e], self.down_scales[e], self.down_global[e:e + 1])

    def stack_layout(self, stream=None):
        """(Re)writes the column-block copies of the down weights that
        moe_stack_forward reads; call again after changing the down weights."""
        E, H, I, S = self.E, self.H, self.I, self.S
        if self.down_cb is None:
            self.down_cb = torch.empty((E, I // 16, 9 * H), dtype=torch.uint8, device=self.down_codes.device)
            self.shared_down_cb = torch.empty((S // 16, 9 * H), dtype=torch.uint8, device=self.down_codes.device)
        nvfp4_colblock_layout(self.down_codes, self.down_scales, out=self.down_cb, stream=stream)
        nvfp4_colblock_layout(self.shared_down.codes, self.shared_down.scales, out=self.shared_down_cb,
                              stream=stream)

    def c(self):
        if self._c is None:
            self._c = _abi.MoeLayerWeights(
                self.E, self.H, self.I, self.S,
                self.up_codes.data_ptr(), self.up_scales.data_ptr(), self.up_global.data_ptr(),
                self.down_codes.data_ptr(), self.down_scales.data_ptr(), self.down_global.data_ptr(),
                self.shared_up.c(), self.shared_down.c())
        return self._c


# ------------------------------------------------------------------ calls
def nvfp4_quantize(x, mode=PER_TENSOR, out: NVFP4Matrix = None, global_scale=None, stream=None):
    """Quantise x [rows][cols] (bf16 or float32, CUDA) to NVFP4. PER_ROW gives
    one global per row. Returns an NVFP4Matrix (global_scale [1] or [rows])."""
    x = x.contiguous()
    rows, cols = x.shape
    if out is None:
        out = NVFP4Matrix.empty(rows, cols, x.device)
        if mode == PER_ROW:
            out.global_scale = torch.empty(rows, dtype=torch.float32, device=x.device)
    if mode == GIVEN:
        out.global_scale.copy_(global_scale)
    st = _L.nvfp4_quantize(_ptr(x), int(x.dtype == torch.bfloat16), rows, cols, mode,
                           _ptr(out.global_scale), _ptr(out.codes), _ptr(out.scales), _stream(stream))
    _check(st, "nvfp4_quantize")
    return out


def fp8_quantize(x, mode=PER_TENSOR, out: FP8Matrix = None, global_scale=None, stream=None):
    """Quantise x [rows][cols] (bf16 or float32, CUDA) to E4M3 with one scale
    (PER_TENSOR, GIVEN) or one per row (PER_ROW). Returns an FP8Matrix."""
    x = x.contiguous()
    rows, cols = x.shape
    if out is None:
        out = FP8Matrix.empty(rows, cols, x.device)
        if mode == PER_ROW:
            out.global_scale = torch.empty(rows, dtype=torch.float32, device=x.device)
    if mode == GIVEN:
        out.global_scale.copy_(global_scale)
    st = _L.fp8_quantize(_ptr(x), int(x.dtype == torch.bfloat16), rows, cols, mode, _ptr(out.global_scale),
                         _ptr(out.codes), _stream(stream))
    _check(st, "fp8_quantize")
    return out


def moe_shared_fp8_workspace_size(up: FP8Matrix, T) -> int:
    u = up.c()
    return int(_L.moe_shared_fp8_workspace_size(ctypes.byref(u), T))


def moe_shared_fp8_forward(up: FP8Matrix, down: FP8Matrix, hidden, residual=None, out=None, workspace=None,
                           rms_eps=0.0, stream=None):
    """The FP8 W8A8 shared expert: out = bf16(down . bf16(relu(up . x)^2) +
    residual) with per-token E4M3 activations."""
    T = hidden.shape[0]
    if out is None:
        out = torch.empty_like(hidden)
    if workspace is None:
        workspace = torch.empty(moe_shared_fp8_workspace_size(up, T), dtype=torch.uint8, device=hidden.device)
    u, d = up.c(), down.c()
    st = _L.moe_shared_fp8_forward(ctypes.byref(u), ctypes.byref(d), _ptr(hidden), T, float(rms_eps), _ptr(residual),
                                   _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "moe_shared_fp8_forward")
    return out


def moe_route_topk(hidden, router_w, bias, k, topk_idx=None, topk_w=None, rms_eps=0.0, stream=None):
    T, H = hidden.shape
    E = router_w.shape[0]
    if topk_idx is None:
        topk_idx = torch.empty((T, k), dtype=torch.int32, device=hidden.device)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=hidden.device)
    st = _L.moe_route_topk(_ptr(hidden), _ptr(router_w), _ptr(bias), T, H, E, k, float(rms_eps),
                           _ptr(topk_idx), _ptr(topk_w), _stream(stream))
    _check(st, "moe_route_topk")
    return topk_idx, topk_w


def moe_expert_forward_workspace_size(layer: MoELayer, T, k, mode=W4A4) -> int:
    w = layer.c()
    return int(_L.moe_expert_forward_workspace_size(ctypes.byref(w), T, k, mode))


def moe_expert_forward_workspace_init(workspace, stream=None):
    _check(_L.moe_expert_forward_workspace_init(_ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_expert_forward_workspace_init")


WS_X, WS_ACT, WS_ACT_Q, WS_SH_ACT, WS_SH_ACT_Q = 0, 1, 2, 3, 4
WS_BF16, WS_CODES, WS_F16_DEQUANT = 0, 1, 2
CALL_EXPERT_FORWARD, CALL_LAYER_FORWARD = 0, 1


def nvfp4_workspace_view(call, layer: MoELayer, T, k, mode, region) -> dict:
    """Where region `region` (WS_*) of a moe_expert_forward (call 0) or
    moe_layer_forward (call 1) workspace lies: the fields of nvfp4_ws_view."""
    w = layer.c()
    v = _abi.WsView()
    _check(_L.nvfp4_workspace_view(call, ctypes.byref(w), T, k, mode, region, ctypes.byref(v)),
           "nvfp4_workspace_view")
    return {f: getattr(v, f) for f, _ in _abi.WsView._fields_}


def make_workspace(layer: MoELayer, T, k, mode=W4A4, stream=None):
    n = moe_expert_forward_workspace_size(layer, T, k, mode)
    ws = torch.empty(n, dtype=torch.uint8, device=layer.up_codes.device)
    moe_expert_forward_workspace_init(ws, stream)
    return ws


def moe_expert_forward(layer: MoELayer, hidden, topk_idx, topk_w, mode=W4A4, residual=None,
                       out=None, workspace=None, rms_eps=0.0, stream=None):
    T = hidden.shape[0]
    k = topk_idx.shape[1]
    if out is None:
        out = torch.empty_like(hidden)
    if workspace is None:
        workspace = make_workspace(layer, T, k, mode, stream)
    w = layer.c()
    st = _L.moe_expert_forward(ctypes.byref(w), _ptr(hidden), _ptr(topk_idx), _ptr(topk_w), T, k,
                               mode, float(rms_eps), _ptr(residual), _ptr(out), _ptr(workspace),
                               workspace.numel(), _stream(stream))
    _check(st, "moe_expert_forward")
    return out


def moe_layer_forward_workspace_size(layer: MoELayer, T, k, mode=W4A4) -> int:
    w = layer.c()
    return int(_L.moe_layer_forward_workspace_size(ctypes.byref(w), T, k, mode))


def make_layer_workspace(layer: MoELayer, T, k, mode=W4A4, stream=None):
    n = max(moe_layer_forward_workspace_size(layer, T, k, mode),
            moe_expert_forward_workspace_size(layer, T, k, mode))
    ws = torch.empty(n, dtype=torch.uint8, device=layer.up_codes.device)
    moe_expert_forward_workspace_init(ws, stream)
    return ws


def moe_layer_forward(layer: MoELayer, hidden, k, mode=W4A4, residual=None, out=None, topk_idx=None,
                      topk_w=None, workspace=None, rms_eps=0.0, stream=None):
    """Router + experts + shared expert + combine of one layer (1..4 tokens);
    returns (out, topk_idx, topk_w)."""
    T = hidden.shape[0]
    if out is None:
        out = torch.empty_like(hidden)
    if topk_idx is None:
        topk_idx = torch.empty((T, k), dtype=torch.int32, device=hidden.device)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=hidden.device)
    if workspace is None:
        workspace = make_layer_workspace(layer, T, k, mode, stream)
    w = layer.c()
    st = _L.moe_layer_forward(ctypes.byref(w), _ptr(layer.router_w), _ptr(layer.router_b), _ptr(hidden), T, k,
                              mode, float(rms_eps), _ptr(residual), _ptr(out), _ptr(topk_idx), _ptr(topk_w),
                              _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "moe_layer_forward")
    return out, topk_idx, topk_w


def nvfp4_colblock_layout(codes, scales, out=None, stream=None):
    """Column-block copy of NVFP4 matrices codes [..][rows][cols/2], scales
    [..][rows][cols/16] (uint8, CUDA): out [batch][cols/16][9 rows] uint8."""
    rows, half = codes.shape[-2], codes.shape[-1]
    cols = 2 * half
    batch = codes.numel() // (rows * half)
    if out is None:
        out = torch.empty((batch, cols // 16, 9 * rows), dtype=torch.uint8, device=codes.device)
    st = _L.nvfp4_colblock_layout(_ptr(codes.contiguous()), _ptr(scales.contiguous()), batch, rows, cols,
                                  _ptr(out), _stream(stream))
    _check(st, "nvfp4_colblock_layout")
    return out


def _stack_layers(layers):
    """ctypes array of moe_stack_layer for a list of MoELayer; makes each
    layer's column-block down weights on first use."""
    arr = (_abi.MoeStackLayer * len(layers))()
    for i, Lw in enumerate(layers):
        if Lw.down_cb is None:
            Lw.stack_layout()
        arr[i] = _abi.MoeStackLayer(Lw.c(), Lw.router_w.data_ptr(), Lw.router_b.data_ptr(), Lw.down_cb.data_ptr(),
                                    Lw.shared_down_cb.data_ptr())
    return arr


def moe_stack_forward_workspace_size(layers, T, k, mode=W4A4) -> int:
    arr = _stack_layers(layers)
    return int(_L.moe_stack_forward_workspace_size(arr, len(layers), T, k, mode))


def make_stack_workspace(layers, T, k, mode=W4A4, stream=None):
    n = moe_stack_forward_workspace_size(layers, T, k, mode)
    if n == 0:
        raise NVFP4Error(2, "moe_stack_forward_workspace_size")
    ws = torch.empty(n, dtype=torch.uint8, device=layers[0].up_codes.device)
    moe_expert_forward_workspace_init(ws, stream)
    return ws


def moe_stack_forward(layers, hidden, k, mode=W4A4, hidden_out=None, topk_idx=None, topk_w=None,
                      workspace=None, rms_eps=0.0, stream=None, c_layers=None):
    """L layers of the pre-norm residual chain h_{l+1} = h_l + moe_l(norm(h_l))
    in one persistent kernel (1..4 tokens). Returns (hidden_out [L][T][H],
    topk_idx [L][T][k], topk_w [L][T][k]); hidden_out[l] is h_{l+1}.
    c_layers: a cached _stack_layers(layers) array, to skip rebuilding it."""
    L = len(layers)
    T, H = hidden.shape
    dev = hidden.device
    if hidden_out is None:
        hidden_out = torch.empty((L, T, H), dtype=hidden.dtype, device=dev)
    if topk_idx is None:
        topk_idx = torch.empty((L, T, k), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((L, T, k), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = make_stack_workspace(layers, T, k, mode, stream)
    arr = c_layers if c_layers is not None else _stack_layers(layers)
    st = _L.moe_stack_forward(arr, L, _ptr(hidden), T, k, mode, float(rms_eps), _ptr(hidden_out),
                              _ptr(topk_idx), _ptr(topk_w), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "moe_stack_forward")
    return hidden_out, topk_idx, topk_w


def moe_permute(topk_idx, num_experts, with_tiles=False, stream=None):
    """Pairs (t, j) grouped by expert, stable: returns (offsets [E+1],
    perm [T*k], inv [T*k]) and, with with_tiles, the 64-position tile
    offsets [E+1]."""
    T, k = topk_idx.shape
    dev = topk_idx.device
    offsets = torch.empty(num_experts + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    inv = torch.empty(T * k, dtype=torch.int32, device=dev)
    tiles = torch.empty(num_experts + 1, dtype=torch.int32, device=dev) if with_tiles else None
    st = _L.moe_permute(_ptr(topk_idx.contiguous()), T, k, num_experts, _ptr(offsets), _ptr(perm), _ptr(inv),
                        _ptr(tiles), _stream(stream))
    _check(st, "moe_permute")
    return (offsets, perm, inv, tiles) if with_tiles else (offsets, perm, inv)


def moe_expert_forward_noalloc(layer: MoELayer, hidden, topk_idx, topk_w, mode=W4A4, residual=None,
                               out=None, rms_eps=0.0, stream=None):
    """moe_expert_forward without a workspace argument, for callers that cannot
    allocate: the library's fixed device scratch array (1 MiB per GPU) is used
    instead; calls that overlap on the GPU race on it."""
    T = hidden.shape[0]
    k = topk_idx.shape[1]
    if out is None:
        out = torch.empty_like(hidden)
    w = layer.c()
    st = _L.moe_expert_forward_noalloc(ctypes.byref(w), _ptr(hidden), _ptr(topk_idx), _ptr(topk_w), T, k,
                                       mode, float(rms_eps), _ptr(residual), _ptr(out), _stream(stream))
    _check(st, "moe_expert_forward_noalloc")
    return out


def lm_head_gemv(w: NVFP4Matrix, hidden, logits=None, rms_eps=0.0, stream=None):
    T = hidden.shape[0]
    if logits is None:
        logits = torch.empty((T, w.n), dtype=torch.float32, device=hidden.device)
    m = w.c()
    st = _L.lm_head_gemv(ctypes.byref(m), _ptr(hidden), T, float(rms_eps), _ptr(logits), _stream(stream))
    _check(st, "lm_head_gemv")
    return logits


def make_lm_head_workspace(w: NVFP4Matrix, T):
    n = int(_L.lm_head_forward_workspace_size(ctypes.byref(w.c()), T))
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=w.codes.device)


def lm_head_forward(w: NVFP4Matrix, hidden, logits=None, workspace=None, rms_eps=0.0, stream=None):
    """lm_head_gemv for any token count (dense GEMM above 8 tokens)."""
    T = hidden.shape[0]
    if logits is None:
        logits = torch.empty((T, w.n), dtype=torch.float32, device=hidden.device)
    if workspace is None:
        workspace = make_lm_head_workspace(w, T)
    m = w.c()
    st = _L.lm_head_forward(ctypes.byref(m), _ptr(hidden), T, float(rms_eps), _ptr(logits), _ptr(workspace),
                            workspace.numel(), _stream(stream))
    _check(st, "lm_head_forward")
    return logits
