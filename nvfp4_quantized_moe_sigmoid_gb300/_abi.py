"""ctypes view of include/nvfp4moe.h. Loading fails loudly if the CUDA
library has not been built: there is no fallback implementation."""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# NVFP4MOE_LIB may name another build of the same library (the phase-trace
# variant, libnvfp4moe_trace.so); by default the in-tree libnvfp4moe.so.
LIB_PATH = os.environ.get("NVFP4MOE_LIB") or os.path.join(HERE, "libnvfp4moe.so")

P = ctypes.c_void_p
I32, I64 = ctypes.c_int32, ctypes.c_int64

EXPORTS = ["nvfp4_quantize", "moe_route_topk", "moe_expert_forward_workspace_size",
           "moe_expert_forward_workspace_init", "moe_expert_forward", "moe_expert_forward_noalloc",
           "moe_layer_forward", "moe_layer_forward_workspace_size",
           "moe_stack_forward", "moe_stack_forward_workspace_size", "moe_permute",
           "lm_head_gemv", "lm_head_forward", "lm_head_forward_workspace_size",
           "nvfp4_colblock_layout", "nvfp4_status_string", "nvfp4_last_device_error",
           "nvfp4_fp4_mma_peak", "nvfp4_set_peer_wait_limit", "nvfp4_set_decode_max_tokens",
           "nvfp4_workspace_view", "fp8_quantize", "moe_shared_fp8_workspace_size",
           "moe_shared_fp8_forward"]

NOALLOC_SCRATCH_BYTES = 1 << 20  # NVFP4MOE_NOALLOC_SCRATCH_BYTES
STACK_MAX_LAYERS = 32  # NVFP4MOE_STACK_MAX_LAYERS

STATUS = {0: "NVFP4_OK", 1: "NVFP4_ERR_INVALID_ARG", 2: "NVFP4_ERR_UNSUPPORTED_SHAPE",
          3: "NVFP4_ERR_MISALIGNED", 4: "NVFP4_ERR_WORKSPACE", 5: "NVFP4_ERR_CUDA",
          6: "NVFP4_ERR_TIMEOUT"}


class NVFP4Matrix(ctypes.Structure):
    _fields_ = [("codes", P), ("scales", P), ("global_scale", P), ("n", I64), ("k", I64)]


class MoeLayerWeights(ctypes.Structure):
    _fields_ = [("num_experts", I32), ("hidden", I32), ("inter", I32), ("shared_inter", I32),
                ("up_codes", P), ("up_scales", P), ("up_global", P),
                ("down_codes", P), ("down_scales", P), ("down_global", P),
                ("shared_up", NVFP4Matrix), ("shared_down", NVFP4Matrix)]


class FP8Matrix(ctypes.Structure):
    _fields_ = [("codes", P), ("global_scale", P), ("n", I64), ("k", I64)]


class WsView(ctypes.Structure):
    _fields_ = [("offset", ctypes.c_uint64), ("rows", I64), ("cols", I64), ("pitch", I64),
                ("scales_offset", ctypes.c_uint64), ("scales_pitch", I64), ("global_offset", ctypes.c_uint64),
                ("format", I32), ("has_global", I32), ("position_order", I32), ("reserved", I32)]


class MoeStackLayer(ctypes.Structure):
    _fields_ = [("moe", MoeLayerWeights), ("router_w", P), ("router_bias", P),
                ("down_colblock", P), ("shared_down_colblock", P)]


_lib = None


def load(path: str = LIB_PATH):
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libnvfp4moe.so is not built ({path}); run "
                          "nvfp4_quantized_moe_sigmoid_gb300.build.build() first")
    L = ctypes.CDLL(path)
    L.nvfp4_quantize.argtypes = [P, ctypes.c_int, I64, I64, ctypes.c_int, P, P, P, P]
    L.nvfp4_quantize.restype = ctypes.c_int
    L.moe_route_topk.argtypes = [P, P, P, I32, I32, I32, I32, ctypes.c_float, P, P, P]
    L.moe_route_topk.restype = ctypes.c_int
    L.moe_expert_forward_workspace_size.argtypes = [ctypes.POINTER(MoeLayerWeights), I32, I32,
                                                    ctypes.c_int]
    L.moe_expert_forward_workspace_size.restype = ctypes.c_size_t
    L.moe_expert_forward_workspace_init.argtypes = [P, ctypes.c_size_t, P]
    L.moe_expert_forward_workspace_init.restype = ctypes.c_int
    L.moe_expert_forward.argtypes = [ctypes.POINTER(MoeLayerWeights), P, P, P, I32, I32,
                                     ctypes.c_int, ctypes.c_float, P, P, P, ctypes.c_size_t, P]
    L.moe_expert_forward.restype = ctypes.c_int
    L.moe_layer_forward_workspace_size.argtypes = [ctypes.POINTER(MoeLayerWeights), I32, I32, ctypes.c_int]
    L.moe_layer_forward_workspace_size.restype = ctypes.c_size_t
    L.moe_layer_forward.argtypes = [ctypes.POINTER(MoeLayerWeights), P, P, P, I32, I32, ctypes.c_int,
                                    ctypes.c_float, P, P, P, P, P, ctypes.c_size_t, P]
    L.moe_layer_forward.restype = ctypes.c_int
    L.moe_stack_forward_workspace_size.argtypes = [ctypes.POINTER(MoeStackLayer), I32, I32, I32, ctypes.c_int]
    L.moe_stack_forward_workspace_size.restype = ctypes.c_size_t
    L.moe_stack_forward.argtypes = [ctypes.POINTER(MoeStackLayer), I32, P, I32, I32, ctypes.c_int, ctypes.c_float,
                                    P, P, P, P, ctypes.c_size_t, P]
    L.moe_stack_forward.restype = ctypes.c_int
    L.nvfp4_colblock_layout.argtypes = [P, P, I64, I64, I64, P, P]
    L.nvfp4_colblock_layout.restype = ctypes.c_int
    L.moe_permute.argtypes = [P, I32, I32, I32, P, P, P, P, P]
    L.moe_permute.restype = ctypes.c_int
    L.moe_expert_forward_noalloc.argtypes = [ctypes.POINTER(MoeLayerWeights), P, P, P, I32, I32,
                                             ctypes.c_int, ctypes.c_float, P, P, P]
    L.moe_expert_forward_noalloc.restype = ctypes.c_int
    L.lm_head_gemv.argtypes = [ctypes.POINTER(NVFP4Matrix), P, I32, ctypes.c_float, P, P]
    L.lm_head_gemv.restype = ctypes.c_int
    L.lm_head_forward_workspace_size.argtypes = [ctypes.POINTER(NVFP4Matrix), I32]
    L.lm_head_forward_workspace_size.restype = ctypes.c_size_t
    L.lm_head_forward.argtypes = [ctypes.POINTER(NVFP4Matrix), P, I32, ctypes.c_float, P, P, ctypes.c_size_t, P]
    L.lm_head_forward.restype = ctypes.c_int
    L.nvfp4_status_string.argtypes = [ctypes.c_int]
    L.nvfp4_status_string.restype = ctypes.c_char_p
    L.nvfp4_last_device_error.argtypes = [P]
    L.nvfp4_last_device_error.restype = ctypes.c_int
    L.nvfp4_fp4_mma_peak.argtypes = [I32, I32, I32, ctypes.POINTER(ctypes.c_double), P]
    L.nvfp4_fp4_mma_peak.restype = ctypes.c_int
    L.nvfp4_set_peer_wait_limit.argtypes = [ctypes.c_uint64]
    L.nvfp4_set_peer_wait_limit.restype = ctypes.c_int
    L.nvfp4_set_decode_max_tokens.argtypes = [I32]
    L.nvfp4_set_decode_max_tokens.restype = ctypes.c_int
    L.nvfp4_workspace_view.argtypes = [I32, ctypes.POINTER(MoeLayerWeights), I32, I32, ctypes.c_int, I32,
                                       ctypes.POINTER(WsView)]
    L.nvfp4_workspace_view.restype = ctypes.c_int
    L.fp8_quantize.argtypes = [P, ctypes.c_int, I64, I64, ctypes.c_int, P, P, P]
    L.fp8_quantize.restype = ctypes.c_int
    L.moe_shared_fp8_workspace_size.argtypes = [ctypes.POINTER(FP8Matrix), I32]
    L.moe_shared_fp8_workspace_size.restype = ctypes.c_size_t
    L.moe_shared_fp8_forward.argtypes = [ctypes.POINTER(FP8Matrix), ctypes.POINTER(FP8Matrix), P, I32, ctypes.c_float,
                                         P, P, P, ctypes.c_size_t, P]
    L.moe_shared_fp8_forward.restype = ctypes.c_int
    _lib = L
    return L
