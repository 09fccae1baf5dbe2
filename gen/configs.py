"""The five workloads of the hot path, as plain data (shapes, token counts,
seeds, distributions). No arithmetic of the method lives here.

Shapes follow the pages: hidden 2688, 128 routed experts with top-6 and a
1856-wide intermediate, one shared expert, 23 MoE layers, vocabulary 131072
(worklog Step 0 and Step 4; W4A16 model card "What was changed" and
"Checkpoint layout"; DGX Spark post "The setup"). The shared expert is 3712
wide.
"""
H, I, S, E, K, V, L = 2688, 1856, 3712, 128, 6, 131072, 23

# rms_eps: the chained configs normalise each block's input (pre-norm) and
# the lm_head input; a single layer on an N(0, 1) input is fed as is.
RMS_EPS = 1e-5
CONFIGS = {
    0: dict(name="decode_1tok_1layer_w4a16", T=1, layers=1, w4a4=False, lm_head=False,
            bias=(-0.1, 0.1), rho=0.0, seed=0, rms_eps=0.0),
    1: dict(name="decode_1tok_23layer_w4a4_lmhead", T=1, layers=L, w4a4=True, lm_head=True,
            bias=(-0.1, 0.1), rho=0.0, seed=0, rms_eps=RMS_EPS),
    2: dict(name="verify_4tok_23layer_w4a4_lmhead", T=4, layers=L, w4a4=True, lm_head=True,
            bias=(-0.1, 0.1), rho=0.5, seed=0, rms_eps=RMS_EPS),
    3: dict(name="prefill_1024tok_1layer_w4a4", T=1024, layers=1, w4a4=True, lm_head=False,
            bias=(-0.5, 0.5), rho=0.0, seed=0, rms_eps=0.0),
    4: dict(name="concurrent_256tok_23layer_w4a4_lmhead", T=256, layers=L, w4a4=True,
            lm_head=True, bias=(-0.1, 0.1), rho=0.0, seed=0, rms_eps=RMS_EPS),
}

# the hidden states entering layer 0 are drawn under this layer id; a
# stand-alone lm_head input N(0,1) under LM_INPUT_LAYER
HIDDEN_LAYER = 0
LM_INPUT_LAYER = 200


def shape(cfg):
    c = dict(CONFIGS[cfg]) if isinstance(cfg, int) else dict(cfg)
    c.update(H=H, I=I, S=S, E=E, K=K, V=V)
    return c

# The model's MTP head (worklog Step 5 and Step 6) has its own 128-expert MoE
# of the same shapes; its tensors are drawn under this layer id. It drafts
# SPEC_K tokens per step, and the main model verifies SPEC_K + 1 positions.
DRAFTER_LAYER = 100
SPEC_K = 3

