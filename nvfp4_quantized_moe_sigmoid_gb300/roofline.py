"""Algorithmic byte and FLOP model of the hot path (what a perfect kernel must
move or compute), used to turn measured times into roofline fractions.

Per unit (NVFP4 = 0.5625 byte per element: half a byte of E2M1 code plus one
E4M3 byte per 16 elements; the fp32 per-tensor globals are counted too):
  routed expert, up + down   2 * I * H * 0.5625
  shared expert, up + down   2 * S * H * 0.5625
  router                     E * H * 4 + E * 4       (fp32 gate + fp32 bias)
  lm_head                    V * H * 0.5625
  activations                bf16 h in (route + experts + residual), bf16 out,
                             fp32 logits out
Weights of an expert chosen by several tokens of a step are read once
(unique experts are counted per layer).
"""


def nvfp4_bytes(n, k):
    return n * (k // 2) + n * (k // 16) + 4


def expert_bytes(H, I):
    return nvfp4_bytes(I, H) + nvfp4_bytes(H, I)


def shared_bytes(H, S):
    return nvfp4_bytes(S, H) + nvfp4_bytes(H, S)


def router_bytes(E, H):
    return E * H * 4 + E * 4


def layer_bytes(T, unique, E, H, I, S, k):
    """Bytes one MoE layer must move for T tokens with `unique` distinct experts."""
    act = T * H * 2 * 3 + T * H * 2 + T * k * 8  # h (router, experts, residual), out, topk
    return router_bytes(E, H) + unique * expert_bytes(H, I) + shared_bytes(H, S) + act


def expert_call_bytes(T, unique, H, I, S, k):
    """Bytes of one moe_expert_forward call (no router)."""
    return unique * expert_bytes(H, I) + shared_bytes(H, S) + T * H * 2 * 3 + T * k * 8


def lm_head_bytes(T, V, H):
    return nvfp4_bytes(V, H) + T * H * 2 + T * V * 4


def step_bytes(T, uniques, E, H, I, S, k, V=None):
    b = sum(layer_bytes(T, u, E, H, I, S, k) for u in uniques)
    if V:
        b += lm_head_bytes(T, V, H)
    return b


def moe_fp4_flops(T, L, H, I, S, k):
    """FP4 tensor-core flops of the expert GEMMs of L MoE layers (W4A4): the
    routed experts' up and down for T k (token, choice) pairs and the shared
    expert's for T tokens."""
    return L * (2 * T * k * 2 * I * H + 2 * T * 2 * S * H)


def step_flops(T, L, E, H, I, S, k, V=None):
    f = L * (2 * T * E * H + 2 * T * k * 2 * I * H + 2 * T * 2 * S * H)
    if V:
        f += 2 * T * V * H
    return f


# ---- the pages' own byte arithmetic ("Let's optimize Nemotron 3.5 Lightning -
# a worklog", Step 4; the W4A4 card's precision table), which the model above
# refines (it also counts the block scales and globals)
def bf16_weight_bytes(n, k):
    """Dense bf16 matrix [n][k]."""
    return n * k * 2


def fp4_code_bytes(n, k):
    """E2M1 codes of an [n][k] NVFP4 matrix alone (the pages' "176 MB")."""
    return n * k // 2


def lm_head_quant_saving(V, H, bw_bytes_per_s):
    """Reads saved per decode step by storing the lm_head [V][H] as NVFP4
    codes instead of bf16, and the time they take at bw_bytes_per_s:
    (bf16 bytes, NVFP4 code bytes, saved bytes, saved seconds)."""
    b16, b4 = bf16_weight_bytes(V, H), fp4_code_bytes(V, H)
    return b16, b4, b16 - b4, (b16 - b4) / bw_bytes_per_s


def routed_expert_tensors(L, E):
    """NVFP4 routed-expert weight tensors of L MoE layers: up_proj and
    down_proj of each of the E experts (no gate_proj)."""
    return L * E * 2

