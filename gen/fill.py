"""Device fillers that put the synthetic workload's tensors straight into
CUDA tensors (same values as the host fills in gen.py)."""
import torch

from . import gen

_KIND = {"up": gen.KIND_UP, "down": gen.KIND_DOWN, "sh_up": gen.KIND_SH_UP,
         "sh_down": gen.KIND_SH_DOWN, "lm_head": gen.KIND_LM_HEAD}


def fillers(seed, bias_range):
    def fill_bf16(kind, layer, index, t):
        gen.dev_normal_bf16(t, seed, gen.tensor_id(_KIND[kind], layer, index), gen.WEIGHT_SIGMA)

    def fill_router(layer, t):
        tmp = torch.empty(t.numel(), dtype=torch.bfloat16, device=t.device)
        gen.dev_normal_bf16_as_f32(t, tmp, seed, gen.tensor_id(gen.KIND_ROUTER_W, layer, 0),
                                   gen.WEIGHT_SIGMA)

    def fill_bias(layer, t):
        gen.dev_uniform_f32(t, seed, gen.tensor_id(gen.KIND_ROUTER_B, layer, 0), *bias_range)

    return fill_bf16, fill_router, fill_bias


def hidden(t, seed, layer=0, rho=0.0, t0=0):
    gen.dev_hidden_bf16(t, seed, layer=layer, rho=rho, t0=t0)
