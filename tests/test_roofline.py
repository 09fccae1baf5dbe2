"""Pins of the byte model that turns measured times into roofline fractions
(nvfp4_quantized_moe_sigmoid_gb300/roofline.py), against the pages' own
arithmetic and the NVFP4 format definition."""
from nvfp4_quantized_moe_sigmoid_gb300 import roofline as rf

H, I, S, E, V, L = 2688, 1856, 3712, 128, 131072, 23


def test_lm_head_saving_matches_worklog_step4():
    # "704 MB in BF16 -> 176 MB in NVFP4 saves 528 MB of reads per step,
    # ~330 us at 1.60 TB/s" (131,072 x 2,688 = 352M parameters)
    b16, b4, saved, secs = rf.lm_head_quant_saving(V, H, 1.60e12)
    assert V * H == 352_321_536
    assert round(b16 / 1e6) == 705 and int(b16 / 1e6) == 704
    assert round(b4 / 1e6) == 176
    assert round(saved / 1e6) == 528
    assert round(secs * 1e6) == 330


def test_routed_tensor_count_matches_w4a4_card():
    # routed MoE experts {up,down}_proj, NVFP4 W4A4: 5888 tensors over 23 MoE layers of 128 experts
    assert rf.routed_expert_tensors(L, E) == 5888


def test_nvfp4_bytes_per_element():
    # E2M1 code: 4 bits; E4M3 scale: 8 bits per 16 elements; one fp32 global
    for n, k in [(1, 16), (I, H), (H, I), (V, H)]:
        assert rf.nvfp4_bytes(n, k) == n * k * 0.5625 + 4
    assert rf.nvfp4_bytes(V, H) - 4 == rf.fp4_code_bytes(V, H) * 9 // 8


def test_layer_bytes_is_the_sum_of_its_parts():
    routed = rf.nvfp4_bytes(I, H) + rf.nvfp4_bytes(H, I)
    shared = rf.nvfp4_bytes(S, H) + rf.nvfp4_bytes(H, S)
    router = E * H * 4 + E * 4
    assert routed == 5_612_552 and shared == 11_225_096 and router == 1_376_768
    act = 1 * H * 2 * 4 + 1 * 6 * 8
    assert rf.layer_bytes(1, 6, E, H, I, S, 6) == router + 6 * routed + shared + act
    # two tokens that share every expert move the weights once
    assert rf.layer_bytes(2, 6, E, H, I, S, 6) - rf.layer_bytes(1, 6, E, H, I, S, 6) == H * 2 * 4 + 6 * 8
    step = rf.step_bytes(1, [6] * L, E, H, I, S, 6, V)
    assert step == L * rf.layer_bytes(1, 6, E, H, I, S, 6) + rf.nvfp4_bytes(V, H) + H * 2 + V * 4
