"""A stack of NVFP4 MoE layers plus the NVFP4 lm_head, resident in HBM, and the
decode step that runs them through the C ABI:

    for each layer l:  idx, w = moe_route_topk(norm(h_l))
                       h_{l+1} = h_l + moe_expert_forward(norm(h_l), idx, w)
    logits = lm_head_forward(norm(h_L))   (lm_head_gemv up to 8 tokens)

where norm is the unit-weight RMS norm each block of the pre-norm model
applies to its input (fused into the kernels; rms_eps = 0 disables it).
With 1..4 tokens all layers run as one moe_stack_forward call (path
"stack"); "layer" runs one moe_layer_forward per layer and "split" the
two calls above per layer.

("Let's optimize Nemotron 3.5 Lightning - a worklog": a decode step streams
the active experts of every MoE layer and the lm_head; the chain keeps only
the MoE layers and their residual adds.) Weights are registered once with
nvfp4_quantize from bf16 masters supplied by the caller.
"""
import torch

from . import (MoELayer, NVFP4Matrix, PER_TENSOR, W4A4, W4A16, _stack_layers, lm_head_forward,
               make_layer_workspace, make_lm_head_workspace, make_stack_workspace, moe_expert_forward,
               moe_layer_forward, moe_route_topk, moe_stack_forward, nvfp4_quantize)


def register_layer(Lw: MoELayer, layer_id, fill_bf16, fill_router, fill_bias):
    """Fills one MoE layer's router and quantises its bf16 master weights
    (drawn under layer_id) to NVFP4 on the device."""
    E, H, I, S = Lw.E, Lw.H, Lw.I, Lw.S
    tmp = torch.empty(max(I * H, S * H), dtype=torch.bfloat16, device=Lw.up_codes.device)
    fill_router(layer_id, Lw.router_w)
    fill_bias(layer_id, Lw.router_b)
    for e in range(E):
        m = tmp[:I * H].view(I, H)
        fill_bf16("up", layer_id, e, m)
        nvfp4_quantize(m, PER_TENSOR, out=Lw.expert_up(e))
        m = tmp[:H * I].view(H, I)
        fill_bf16("down", layer_id, e, m)
        nvfp4_quantize(m, PER_TENSOR, out=Lw.expert_down(e))
    m = tmp[:S * H].view(S, H)
    fill_bf16("sh_up", layer_id, 0, m)
    nvfp4_quantize(m, PER_TENSOR, out=Lw.shared_up)
    m = tmp[:H * S].view(H, S)
    fill_bf16("sh_down", layer_id, 0, m)
    nvfp4_quantize(m, PER_TENSOR, out=Lw.shared_down)
    Lw.down_cb = None  # column-block copies are made again from these weights on first use
    del tmp


class MoEDecodeStack:
    def __init__(self, layers, E, H, I, S, k, T, w4a4=True, V=None, device="cuda",
                 weights_from=None, rms_eps=1e-5):
        """weights_from: another stack whose registered weights this one shares."""
        self.L, self.E, self.H, self.I, self.S, self.k, self.T = layers, E, H, I, S, k, T
        self.rms_eps = rms_eps
        self.V = V
        self.mode = W4A4 if w4a4 else W4A16
        self.device = device
        if weights_from is not None:
            self.layers, self.lm = weights_from.layers, weights_from.lm
        else:
            self.layers = [MoELayer(E, H, I, S, device) for _ in range(layers)]
            self.lm = NVFP4Matrix.empty(V, H, device) if V else None
        self.h = torch.zeros((layers + 1, T, H), dtype=torch.bfloat16, device=device)
        self.topk_idx = torch.zeros((layers, T, k), dtype=torch.int32, device=device)
        self.topk_w = torch.zeros((layers, T, k), dtype=torch.float32, device=device)
        self.logits = torch.zeros((T, V), dtype=torch.float32, device=device) if V else None
        self.ws = None
        self.stack_ws = None
        self.c_layers = None
        self.graph = None
        self.path = "stack" if T <= 4 else "split"

    # ------------------------------------------------------------ weights
    def register(self, fill_bf16, fill_router, fill_bias):
        """fill_bf16(kind, layer, index, t) writes a bf16 master into t;
        fill_router(layer, t) / fill_bias(layer, t) write the fp32 router."""
        H = self.H
        for l, Lw in enumerate(self.layers):
            register_layer(Lw, l, fill_bf16, fill_router, fill_bias)
        if self.lm is not None:
            full = torch.empty((self.V, H), dtype=torch.bfloat16, device=self.device)
            fill_bf16("lm_head", 0, 0, full)
            nvfp4_quantize(full, PER_TENSOR, out=self.lm)
            del full
        self.make_workspace()

    def make_workspace(self):
        self.ws = make_layer_workspace(self.layers[0], self.T, self.k, self.mode)
        if self.lm is not None:
            self.lm_ws = make_lm_head_workspace(self.lm, self.T)
        if self.T <= 4:
            for Lw in self.layers:  # the column-block down weights, from the weights just registered
                Lw.stack_layout()
            self.stack_ws = make_stack_workspace(self.layers, self.T, self.k, self.mode)
            self.c_layers = _stack_layers(self.layers)

    # ------------------------------------------------------------ the step
    def step(self, stream=None):
        """One decode step on self.h[0] -> self.h[L] (and logits)."""
        if self.path == "stack":
            moe_stack_forward(self.layers, self.h[0], self.k, self.mode, hidden_out=self.h[1:],
                              topk_idx=self.topk_idx, topk_w=self.topk_w, workspace=self.stack_ws,
                              rms_eps=self.rms_eps, stream=stream, c_layers=self.c_layers)
        for l, Lw in enumerate(self.layers if self.path != "stack" else []):
            if self.path == "layer":
                moe_layer_forward(Lw, self.h[l], self.k, self.mode, residual=self.h[l], out=self.h[l + 1],
                                  topk_idx=self.topk_idx[l], topk_w=self.topk_w[l], workspace=self.ws,
                                  rms_eps=self.rms_eps, stream=stream)
                continue
            moe_route_topk(self.h[l], Lw.router_w, Lw.router_b, self.k, self.topk_idx[l],
                           self.topk_w[l], rms_eps=self.rms_eps, stream=stream)
            moe_expert_forward(Lw, self.h[l], self.topk_idx[l], self.topk_w[l], self.mode,
                               residual=self.h[l], out=self.h[l + 1], workspace=self.ws,
                               rms_eps=self.rms_eps, stream=stream)
        if self.lm is not None:
            lm_head_forward(self.lm, self.h[self.L], self.logits, workspace=self.lm_ws, rms_eps=self.rms_eps,
                            stream=stream)

    def capture(self):
        """Capture one step in a CUDA graph (after one eager step)."""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.step()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.step()
        torch.cuda.synchronize()
        return self.graph

    def replay(self):
        self.graph.replay()

    # ------------------------------------------------------------ bytes
    def unique_experts(self):
        """Per layer, the number of distinct experts selected this step."""
        idx = self.topk_idx.view(self.L, -1).cpu()
        return [int(torch.unique(idx[l]).numel()) for l in range(self.L)]


def graph_sizes_not_multiple(sizes, k):
    """The CUDA-graph batch sizes that a speculative step with k drafts cannot
    replay: every step verifies k + 1 positions per sequence, so only
    multiples of k + 1 match a step's shape ("cudagraph_capture_sizes must be
    multiples of k+1" in the W4A4 card's serving notes; a size that matches
    none falls back to an uncaptured step)."""
    return [s for s in sizes if s % (k + 1)]


class SpecDecodeStep:
    """One self-speculative decode step ("Let's optimize Nemotron 3.5
    Lightning - a worklog", Step 5 and Step 6): the model's MTP head drafts k
    tokens one pass at a time, then the main stack verifies k + 1 positions
    in one pass.

    Only the hot path is modelled. A draft pass is the drafter's own NVFP4
    MoE layer (128 experts, the same kernels, its own weights) on one token,
    then the lm_head over it; the verify pass is the main stack's MoE layers
    on k + 1 tokens, then the lm_head over them. The attention, embedding and
    sampling steps in between are not on this path: a draft pass here takes
    the previous pass's output as its input.

    main: a MoEDecodeStack with T = k + 1 (the verify pass); drafter: a
    registered MoELayer of the main stack's shapes."""

    def __init__(self, main: MoEDecodeStack, drafter: MoELayer, k: int):
        if main.T != k + 1:
            raise ValueError(f"the verify pass takes k + 1 = {k + 1} tokens, the stack has {main.T}")
        if graph_sizes_not_multiple([main.T], k):
            raise ValueError("verify batch is not a multiple of k + 1")
        self.main, self.drafter, self.k = main, drafter, k
        dev = main.device
        H = main.H
        self.hd = torch.zeros((k + 1, 1, H), dtype=torch.bfloat16, device=dev)  # draft pass inputs / outputs
        self.d_idx = torch.zeros((k, 1, 1, main.k), dtype=torch.int32, device=dev)
        self.d_w = torch.zeros((k, 1, 1, main.k), dtype=torch.float32, device=dev)
        self.d_logits = (torch.zeros((k, 1, main.V), dtype=torch.float32, device=dev) if main.V else None)
        self.d_layers = [drafter]
        self.d_ws = make_stack_workspace(self.d_layers, 1, main.k, main.mode)
        self.d_c = _stack_layers(self.d_layers)
        self.d_lm_ws = make_lm_head_workspace(main.lm, 1) if main.lm is not None else None
        self.graph = None

    def step(self, stream=None):
        m = self.main
        for d in range(self.k):
            moe_stack_forward(self.d_layers, self.hd[d], m.k, m.mode, hidden_out=self.hd[d + 1:d + 2],
                              topk_idx=self.d_idx[d], topk_w=self.d_w[d], workspace=self.d_ws,
                              rms_eps=m.rms_eps, stream=stream, c_layers=self.d_c)
            if m.lm is not None:
                lm_head_forward(m.lm, self.hd[d + 1], self.d_logits[d], workspace=self.d_lm_ws,
                                rms_eps=m.rms_eps, stream=stream)
        m.step(stream)

    def capture(self):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.step()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.step()
        torch.cuda.synchronize()
        return self.graph

