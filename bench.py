"""Benchmark of the NVFP4 MoE decode hot path on GB300.

Default workload (the headline): one batch-1 decode step through 23 W4A4
NVFP4 MoE layers (hidden 2688, 128 experts of 1856, top-6 sigmoid router with
correction bias, shared expert 3712, residual chain) and the NVFP4 weight-only
lm_head 131072 x 2688 -> fp32 logits. Weights are synthetic (seeded bf16
N(0, 0.02) masters quantised on the device), inputs are synthetic N(0, 1).

The step is captured once as a CUDA graph and replayed: one persistent
cooperative kernel runs all 23 MoE layers (moe_stack_forward), then the
lm_head kernel. Every step streams ~1.26 GB of weights, ten times the 129 MB
L2, so no step finds its inputs in L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl reference]

--impl reference times the CPU oracle (the plain reference implementation of
the same computation) on the host cores on a bounded sample of the workload.
One JSON line is printed by rank 0.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "batch-1 NVFP4 MoE+lm_head decode µs/token and HBM GB/s (% of GB300 peak)"
UNIT = "us/token"
NOMINAL_HBM_GBS = 8000.0


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), "measured"
    return 6800.0, "fallback"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=1)
    ap.add_argument("--layers", type=int, default=0,
                    help="run only this many MoE layers of the config (small cases for ncu captures); 0 = all")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="time only the chosen config (by default the headline run also times configs 0, 2, 3, 4)")
    ap.add_argument("--sweep", action="store_true",
                    help="one MoE layer across token counts on each path (decode GEMV, stack, grouped tcgen05): "
                         "prints the crossover table instead of the JSON line")
    ap.add_argument("--trace", action="store_true",
                    help="per-phase timeline of the stack kernel (1-4 token configs) from the phase-trace build "
                         "of the library; prints a table instead of the JSON line")
    return ap.parse_args()


# ------------------------------------------------------------------ dist
# N > 1: one process per GPU, each an independent replica of the step (the
# path does not shard on one GPU's worth of work: no data-path collective);
# the process group carries only the timing barrier and the max over ranks.
def dist_init(backend=None):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group(backend or os.environ.get("NVFP4MOE_DIST_BACKEND", "nccl"))
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_us_per_token(ms_slowest_rank, steps, T, ws):
    """µs per token of the whole job: ws replicas each ran T tokens per step,
    timed by the slowest rank."""
    return ms_slowest_rank / steps * 1e3 / (T * ws)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def physical_gpu_index(local_rank):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local_rank < len(ids) and ids[local_rank].isdigit():
            return int(ids[local_rank])
    return local_rank


# ------------------------------------------------------------------ oracle timing
class OracleRun:
    """The CPU oracle on the same workload: the first n_layers MoE layers of
    the chain (route + experts + shared + combine) and 1/lm_den of the
    lm_head rows. Weights are generated and quantised once, outside the
    timed part; run() returns the time scaled to a full step (exactly the
    step when n_layers is all of them and lm_den is 1), in microseconds per
    token, and the seconds it took."""

    def __init__(self, cfg_id, n_layers, lm_den):
        from gen import configs, gen
        from oracle import oracle as orc
        from oracle.workload import OracleLayer

        self.orc = orc
        self.c = c = configs.shape(cfg_id)
        self.h0 = gen.hidden_bf16(c["T"], c["H"], c["seed"], layer=configs.HIDDEN_LAYER, rho=c["rho"])
        self.nl = min(n_layers, c["layers"])
        self.layers = []
        h = self.h0
        for l in range(self.nl):
            OL = OracleLayer(c["seed"], l, c["H"], c["I"], c["S"], c["E"], c["bias"])
            h, _, _ = OL.forward(h, c["K"], c["w4a4"], True, rms_eps=c["rms_eps"])
            self.layers.append(OL)
        self.rows = 0
        if c["lm_head"]:
            self.rows = c["V"] // lm_den
            master = gen.lm_head_master(c["seed"], c["V"], c["H"], 0, self.rows)
            cc, ss, gg = orc.quantize(master, orc.PER_TENSOR)
            self.W = orc.Mat(cc, ss, gg[0])
        self.full = self.nl == c["layers"] and (not c["lm_head"] or self.rows == c["V"])
        if self.full:
            self.desc = (f"the full step: {c['layers']} MoE layers (route+experts+shared+combine)"
                         + (f" and all {c['V']} lm_head rows" if c["lm_head"] else "") + f" at T={c['T']}")
        else:
            self.desc = (f"{self.nl} of {c['layers']} MoE layers (route+experts+shared+combine)"
                         + (f" and {self.rows} of {c['V']} lm_head rows" if c["lm_head"] else "")
                         + f" at T={c['T']}, scaled to a full step")

    def run(self, threads):
        c, orc = self.c, self.orc
        orc.set_threads(threads)
        h = self.h0
        t0 = time.perf_counter()
        eps = c["rms_eps"]
        for OL in self.layers:
            x = orc.rms_norm(h, eps) if eps > 0 else h
            r = orc.route(x, OL.Wg, OL.bias, c["K"])
            h, _ = orc.moe_layer(x, r["idx"], r["w"], OL.up, OL.down, OL.sh_up, OL.sh_down,
                                 c["w4a4"], h, c["E"])
        t_layers = time.perf_counter() - t0
        t_lm = 0.0
        if self.rows:
            t0 = time.perf_counter()
            orc.lm_head(self.W, orc.rms_norm(h, eps) if eps > 0 else h)
            t_lm = time.perf_counter() - t0
        per_step = t_layers / self.nl * c["layers"] + (t_lm * c["V"] / self.rows if self.rows else 0)
        return per_step / c["T"] * 1e6, t_layers + t_lm


def config_dict(c, ws):
    """The workload as both arms name it."""
    return {"workload": c["name"], "T": c["T"], "layers": c["layers"], "hidden": c["H"], "experts": c["E"],
            "top_k": c["K"], "inter": c["I"], "shared_inter": c["S"],
            "vocab": c["V"] if c["lm_head"] else None, "mode": "W4A4" if c["w4a4"] else "W4A16",
            "parallelism": "replicas" if ws > 1 else "single",
            "l2": "inputs larger than L2: each step streams the step's weights (>= 46 MB per layer) once; "
                  "the decode step streams 1.26 GB vs 129 MB of L2"}


def run_reference(args, ws, rank):
    """The reference arm: the CPU oracle (the plain, slow reference of the same
    computation) on the full workload of the config, on the host cores."""
    if rank != 0:
        return
    threads = len(os.sched_getaffinity(0))
    run = OracleRun(args.config, 10 ** 6, 1)
    vals, secs = [], []
    for i in range(args.warmup + args.steps):
        v, t = run.run(threads)
        if i >= args.warmup:
            vals.append(v)
            secs.append(t)
    value = statistics.median(vals)
    c = run.c
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.median(secs) * 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(c, ws),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": run.desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def launches_per_step(st, T, L, lm_head):
    """Kernels of the library one step launches (memsets not counted)."""
    if st.path == "stack":
        n = 1
    elif T <= 4:
        n = 3 * L  # router, up, down
    else:
        n = 8 * L  # router, permute, token rows, up, 2 x intermediate rows, down, combine
    if lm_head:
        n += (T + 7) // 8 if T <= 8 else 2
    return n


# DRAM bytes (read + write) per W4A4 layer of k_moe_stack at one token, from
# one ncu capture of the current kernel (2 layers: 92.696576 MB read +
# 2.381056 MB written, halved). None whenever the kernel has changed since
# its last capture (traffic is then reported as null).
STACK_T1_W4A4_DRAM_BYTES_PER_LAYER = 47538816


def graph_of(fn, reps):
    """A CUDA graph of `reps` back-to-back calls of fn (captured after one
    eager call): replaying it times the calls' kernels without launch gaps."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    torch.cuda.synchronize()
    return g


def time_graph(g, iters, warm=2):
    import torch
    for _ in range(warm):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()
    e0.record(stream)
    for _ in range(iters):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


def measure_other_config(cfg_id, base, nm, rf, peak, fp4_peak, iters=10):
    """One more configuration on the weights already registered for the
    headline (the configs share seed-0 weights; the prefill config has its
    own router bias): µs/token, algorithmic GB/s and their fraction of the
    measured HBM copy peak, from a graph of one step replayed `iters` times."""
    import copy
    import torch
    from gen import configs, fill
    from nvfp4_quantized_moe_sigmoid_gb300.model import MoEDecodeStack

    c = dict(configs.shape(cfg_id))
    T, L, E, H, I, S, K, V = c["T"], c["layers"], c["E"], c["H"], c["I"], c["S"], c["K"], c["V"]
    st = MoEDecodeStack(L, E, H, I, S, K, T, w4a4=c["w4a4"], V=V if c["lm_head"] else None,
                        rms_eps=c["rms_eps"], weights_from=base)
    st.layers = base.layers[:L]
    st.lm = base.lm if c["lm_head"] else None
    if tuple(c["bias"]) != tuple(configs.shape(1)["bias"]):
        st.layers = [copy.copy(Lw) for Lw in st.layers]
        _, _, fbias = fill.fillers(c["seed"], c["bias"])
        for l, Lw in enumerate(st.layers):
            Lw.router_b = torch.empty_like(Lw.router_b)
            Lw._c = None
            fbias(l, Lw.router_b)
    st.make_workspace()
    fill.hidden(st.h[0], c["seed"], layer=configs.HIDDEN_LAYER, rho=c["rho"])
    torch.cuda.synchronize()
    g = st.capture()
    ms = time_graph(g, iters, warm=3)
    uniques = st.unique_experts()
    assert nm.nvfp4_last_device_error() == 0
    b = rf.step_bytes(T, uniques, E, H, I, S, K, V if c["lm_head"] else None)
    gbs = b / (ms * 1e-3) / 1e9
    out = {"workload": c["name"], "path": st.path, "T": T, "layers": L, "mode": "W4A4" if c["w4a4"] else "W4A16",
           "ms_per_step": ms, "us_per_token": ms * 1e3 / T, "step_bytes": b, "gbs": gbs, "frac_of_measured_hbm": gbs / peak,
           "unique_experts_mean": sum(uniques) / len(uniques)}
    if st.path != "stack" and c["w4a4"]:
        # the grouped expert GEMMs run on the FP4 tensor pipe: their flops
        # against this GPU's measured dense FP4 throughput
        fl = rf.moe_fp4_flops(T, L, H, I, S, K)
        out["fp4_moe_flops"] = fl
        out["fp4_tflops_over_step"] = fl / (ms * 1e-3) / 1e12
        out["fp4_frac_of_measured_peak"] = out["fp4_tflops_over_step"] / fp4_peak if fp4_peak else None
    del st, g
    torch.cuda.empty_cache()
    return out


def measure_spec_step(base, nm, rf, peak, iters=10):
    """One self-speculative step with the MTP drafter (worklog Step 5 and
    Step 6): k = 3 draft passes (the drafter's own 128-expert NVFP4 MoE layer
    at one token, then the lm_head) and the verify pass (the 23 main layers
    and the lm_head over k + 1 tokens), on the headline's weights and a
    drafter layer of its own."""
    import torch
    from gen import configs, fill
    from nvfp4_quantized_moe_sigmoid_gb300.model import MoEDecodeStack, SpecDecodeStep, register_layer

    c = dict(configs.shape(2))
    K = configs.SPEC_K
    main = MoEDecodeStack(c["layers"], c["E"], c["H"], c["I"], c["S"], c["K"], K + 1, w4a4=True, V=c["V"],
                          rms_eps=c["rms_eps"], weights_from=base)
    main.make_workspace()
    fill.hidden(main.h[0], c["seed"], layer=configs.HIDDEN_LAYER, rho=c["rho"])
    d = nm.MoELayer(c["E"], c["H"], c["I"], c["S"])
    register_layer(d, configs.DRAFTER_LAYER, *fill.fillers(c["seed"], c["bias"]))
    step = SpecDecodeStep(main, d, K)
    fill.hidden(step.hd[0], c["seed"], layer=configs.DRAFTER_LAYER)
    torch.cuda.synchronize()
    g = step.capture()
    ms = time_graph(g, iters, warm=3)
    assert nm.nvfp4_last_device_error() == 0
    uniques = main.unique_experts()
    b = (rf.step_bytes(K + 1, uniques, c["E"], c["H"], c["I"], c["S"], c["K"], c["V"])
         + K * (rf.layer_bytes(1, c["K"], c["E"], c["H"], c["I"], c["S"], c["K"]) + rf.lm_head_bytes(1, c["V"], c["H"])))
    out = {"workload": "spec_decode_k3_step: %d drafter passes (1 MoE layer + lm_head, 1 token) + verify "
                       "(%d layers + lm_head, %d tokens)" % (K, c["layers"], K + 1),
           "ms_per_step": ms, "us_per_verified_position": ms * 1e3 / (K + 1), "step_bytes": b,
           "gbs": b / (ms * 1e-3) / 1e9, "frac_of_measured_hbm": b / (ms * 1e-3) / 1e9 / peak,
           "context": "at the pages' ~2.8 accepted tokens per step (real text, RTX PRO 6000) this step would "
                      "give %.1f us per accepted token" % (ms * 1e3 / 2.8)}
    del step, main, g
    torch.cuda.empty_cache()
    return out


def measure_shared_fp8(nm, peak, iters=10):
    """The FP8 W8A8 shared expert (the W4A4 card's precision for the shared
    experts) at 1 and 4 tokens: moe_shared_fp8_forward on the pages' shared
    expert (3712 x 2688 up, 2688 x 3712 down, E4M3, per-tensor scales) with
    the residual add, timed in a graph of 5 back-to-back calls."""
    import torch
    from gen import configs, fill

    c = configs.shape(1)
    H, S = c["H"], c["S"]
    fb, _, _ = fill.fillers(c["seed"], c["bias"])
    up_m = torch.empty((S, H), dtype=torch.bfloat16, device="cuda")
    dn_m = torch.empty((H, S), dtype=torch.bfloat16, device="cuda")
    fb("sh_up", 0, 0, up_m)
    fb("sh_down", 0, 0, dn_m)
    up, dn = nm.fp8_quantize(up_m, nm.PER_TENSOR), nm.fp8_quantize(dn_m, nm.PER_TENSOR)
    del up_m, dn_m
    # 8 copies (160 MB, more than L2): the back-to-back calls of a graph each
    # stream their own copy
    copies = [(nm.FP8Matrix(up.codes.clone(), up.global_scale), nm.FP8Matrix(dn.codes.clone(), dn.global_scale))
              for _ in range(8)]
    out = {}
    for T in (1, 4):
        h = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        fill.hidden(h, c["seed"], layer=configs.HIDDEN_LAYER)
        o = torch.empty_like(h)
        ws_ = torch.empty(nm.moe_shared_fp8_workspace_size(up, T), dtype=torch.uint8, device="cuda")
        turn = iter(range(1 << 30))

        def call():
            u, d = copies[next(turn) % len(copies)]
            nm.moe_shared_fp8_forward(u, d, h, residual=h, out=o, workspace=ws_, rms_eps=c["rms_eps"])

        g = graph_of(call, 5)
        us = time_graph(g, iters) / 5 * 1e3
        del g
        assert nm.nvfp4_last_device_error() == 0
        b = 2 * S * H + 8 + T * H * 2 * 3
        out["%d_tokens" % T] = {"us": us, "bytes": b, "gbs": b / (us * 1e-6) / 1e9,
                                "frac_of_measured_hbm": b / (us * 1e-6) / 1e9 / peak}
    out["workload"] = ("FP8 W8A8 shared expert (moe_shared_fp8_forward: E4M3 up %d x %d and down %d x %d, "
                       "per-token E4M3 activations, RMS norm, residual add; each call on its own copy of "
                       "the weights, 8 copies > L2)" % (S, H, H, S))
    return out


# ------------------------------------------------------------------ GPU arm
def run_ours(args, ws, rank, local):
    import torch

    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_quantized_moe_sigmoid_gb300 as nm
    from nvfp4_quantized_moe_sigmoid_gb300 import roofline as rf
    from nvfp4_quantized_moe_sigmoid_gb300.model import MoEDecodeStack
    from gen import configs, fill

    c = dict(configs.shape(args.config))
    if args.layers > 0 and args.layers < c["layers"]:
        c["layers"] = args.layers
        c["name"] = "%s_first%dlayers" % (c["name"], args.layers)  # a profiling case, not the benchmark
    T, L, E, H, I, S, K, V = c["T"], c["layers"], c["E"], c["H"], c["I"], c["S"], c["K"], c["V"]
    st = MoEDecodeStack(L, E, H, I, S, K, T, w4a4=c["w4a4"], V=V if c["lm_head"] else None,
                        rms_eps=c["rms_eps"])
    st.register(*fill.fillers(c["seed"], c["bias"]))
    fill.hidden(st.h[0], c["seed"], layer=configs.HIDDEN_LAYER, rho=c["rho"])
    h0 = st.h[0].clone()
    torch.cuda.synchronize()
    st.capture()
    stream = torch.cuda.current_stream()

    # warm-up
    for _ in range(args.warmup):
        st.replay()
    torch.cuda.synchronize()
    uniques = st.unique_experts()
    assert nm.nvfp4_last_device_error() == 0

    # timed region: K graph replays between events on the replay stream
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(physical_gpu_index(local)) as clk:
        barrier(ws)
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(args.steps):
            st.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), ws)
    ms_step = ms_total / args.steps
    us_token = whole_job_us_per_token(ms_total, args.steps, T, ws)
    step_b = rf.step_bytes(T, uniques, E, H, I, S, K, V if c["lm_head"] else None)
    peak, peak_kind = measured_peaks()
    gbs_step = step_b / (ms_step * 1e-3) / 1e9

    # the dominant call timed inside a graph: REPS back-to-back calls on the
    # launching stream, replayed; its average is the kernel's time per launch
    # without launch gaps (each call streams its weights from HBM again)
    REPS = 5
    if st.path == "stack":
        dom = graph_of(lambda: nm.moe_stack_forward(st.layers, st.h[0], K, st.mode, hidden_out=st.h[1:],
                                                    topk_idx=st.topk_idx, topk_w=st.topk_w,
                                                    workspace=st.stack_ws, rms_eps=st.rms_eps,
                                                    c_layers=st.c_layers), REPS)
        call_b = sum(rf.layer_bytes(T, u, E, H, I, S, K) for u in uniques)
        kname = "k_moe_stack (moe_stack_forward: all %d MoE layers in one launch)" % L
    else:
        def split_layers():
            for l, Lw in enumerate(st.layers):
                nm.moe_route_topk(st.h[l], Lw.router_w, Lw.router_b, K, st.topk_idx[l], st.topk_w[l],
                                  rms_eps=st.rms_eps)
                nm.moe_expert_forward(Lw, st.h[l], st.topk_idx[l], st.topk_w[l], st.mode, residual=st.h[l],
                                      out=st.h[l + 1], workspace=st.ws, rms_eps=st.rms_eps)
        dom = graph_of(split_layers, 1)
        call_b = sum(rf.layer_bytes(T, u, E, H, I, S, K) for u in uniques)
        kname = "the MoE layers (router + grouped expert kernels, %d layers)" % L
    dom_ms = time_graph(dom, 6) / (REPS if st.path == "stack" else 1)
    del dom
    traffic = None
    if st.path == "stack" and T == 1 and c["w4a4"] and STACK_T1_W4A4_DRAM_BYTES_PER_LAYER is not None:
        traffic = STACK_T1_W4A4_DRAM_BYTES_PER_LAYER * L
    roof = {"bound": "hbm", "kernel": kname,
            "achieved": call_b / (dom_ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
            "frac": None, "traffic": traffic, "algorithmic_bytes": call_b,
            "avg_launch_us": dom_ms * 1e3, "peak_kind": peak_kind,
            "timing": "CUDA events around graph replays of %d back-to-back launches" % REPS}
    roof["frac"] = roof["achieved"] / peak
    extra = {}
    if c["lm_head"]:
        lmg = graph_of(lambda: nm.lm_head_forward(st.lm, st.h[L], st.logits, workspace=st.lm_ws,
                                                  rms_eps=st.rms_eps), REPS)
        lmm = time_graph(lmg, 6) / REPS
        del lmg
        lb = rf.lm_head_bytes(T, V, H)
        extra["lm_head"] = {"avg_us": lmm * 1e3, "achieved_gbs": lb / (lmm * 1e-3) / 1e9,
                            "frac": lb / (lmm * 1e-3) / 1e9 / peak}

    # end to end through the API: pinned host input -> step -> pinned host logits
    e2e = None
    if not args.no_e2e:
        h_host = h0.cpu().pin_memory()
        out_dev = st.logits if c["lm_head"] else st.h[L]
        out_host = torch.empty(out_dev.shape, dtype=out_dev.dtype).pin_memory()
        for _ in range(3):
            st.h[0].copy_(h_host, non_blocking=True)
            st.replay()
            out_host.copy_(out_dev, non_blocking=True)
        torch.cuda.synchronize()
        barrier(ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record(stream)
        for _ in range(args.steps):
            st.h[0].copy_(h_host, non_blocking=True)
            st.replay()
            out_host.copy_(out_dev, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        barrier(ws)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws) / args.steps
        e2e = {"value": e2e_ms * 1e3 / (T * ws), "unit": UNIT,
               "h2d_bytes_per_step": h_host.numel() * h_host.element_size(),
               "d2h_bytes_per_step": out_host.numel() * out_host.element_size(),
               "wall_us_per_step": wall / args.steps * 1e6}

    # the other configurations, on the same weights (parity cases elsewhere;
    # reported here so that every number comes from this run)
    others = None
    fp4 = None
    if rank == 0 and not args.no_other_configs and args.layers == 0 and args.config == 1:
        # the dense FP4 tensor-pipe peak of this GPU (block-scaled tcgen05 MMAs on every SM)
        fp4 = {"tflops": max(nm.nvfp4_fp4_mma_peak(n, 1, 20000) for n in (128, 256)),
               "kind": "measured: nvfp4_fp4_mma_peak, tcgen05.mma kind::mxf4nvf4 M=128 K=64, N=128 and 256, "
                       "best of the two"}
        others = {}
        st.graph = None
        for oc in (0, 2, 3, 4):
            others[configs.shape(oc)["name"]] = measure_other_config(oc, st, nm, rf, peak, fp4["tflops"])
        others["spec_decode_k3_step"] = measure_spec_step(st, nm, rf, peak)
        others["shared_expert_fp8"] = measure_shared_fp8(nm, peak)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        threads = len(os.sched_getaffinity(0))
        full = OracleRun(args.config, 10 ** 6, 1)
        v_all, secs_all = full.run(threads)
        sample = OracleRun(args.config, 2, 16)
        v_one, secs_one = sample.run(1)
        cpu = {"value": v_all, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": full.desc,
               "seconds": secs_all,
               "single_thread": {"value": v_one, "unit": UNIT, "cores": 1, "sample": sample.desc,
                                 "seconds": secs_one}}

    if rank == 0:
        line = {"metric": METRIC, "value": us_token, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": False,
                "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4(e2m1,e4m3)->f16 mma, f32 acc",
                "data": "synthetic",
                "config": dict(config_dict(c, ws), graph="one CUDA graph per step", path=st.path),
                "step_gbs": gbs_step, "step_frac_of_measured_hbm": gbs_step / peak,
                "step_frac_of_8tbs": gbs_step / NOMINAL_HBM_GBS, "step_bytes": step_b,
                "unique_experts_per_layer": uniques,
                "roofline": roof, "cpu_baseline": cpu, "clocks": clk.summary(), "e2e": e2e,
                "gpu_launches": args.steps * launches_per_step(st, T, L, c["lm_head"]),
                "other_configs": others, "fp4_peak": fp4, **extra}
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ phase trace
TRACE_EVENTS = ["layer start", "h_l read (tagged words)", "router logits posted", "producer's plan free",
                "plan written", "up tiles done", "row amax final, down operands", "down units done",
                "all partials read", "rows of h_l+1 written", "producer: first item", "producer: last item",
                "producer: plan seen"]


def run_trace(args, local):
    """Runs the config's decode step with the phase-trace build of the library
    and prints, per phase boundary of the stack kernel, the median over layers
    of the median and the maximum over CTAs of its time after the first CTA
    saw h_l final, plus the layer period."""
    import importlib.util
    import numpy as np

    spec = importlib.util.spec_from_file_location(
        "_nvfp4moe_build", os.path.join(ROOT, "nvfp4_quantized_moe_sigmoid_gb300", "build.py"))
    pb = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(pb)
    os.environ["NVFP4MOE_LIB"] = pb.build_trace()
    import torch

    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build()
    import ctypes
    import nvfp4_quantized_moe_sigmoid_gb300 as nm
    from nvfp4_quantized_moe_sigmoid_gb300 import _abi
    from nvfp4_quantized_moe_sigmoid_gb300.model import MoEDecodeStack
    from gen import configs, fill

    assert _abi.LIB_PATH == pb.TRACE_LIB
    c = dict(configs.shape(args.config))
    if args.layers > 0:
        c["layers"] = min(c["layers"], args.layers)
    T, L = c["T"], c["layers"]
    if T > 4:
        return run_trace_tc(args, local, c)
    st = MoEDecodeStack(L, c["E"], c["H"], c["I"], c["S"], c["K"], T, w4a4=c["w4a4"],
                        V=c["V"] if c["lm_head"] else None, rms_eps=c["rms_eps"])
    st.register(*fill.fillers(c["seed"], c["bias"]))
    fill.hidden(st.h[0], c["seed"], layer=configs.HIDDEN_LAYER, rho=c["rho"])
    for _ in range(max(3, args.warmup)):
        st.step()
    torch.cuda.synchronize()
    st.step()
    n = 256 * 32 * 16
    buf = np.zeros(n, dtype=np.uint64)
    lib = nm._L
    lib.nvfp4moe_stack_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    lib.nvfp4moe_stack_trace_read.restype = ctypes.c_int
    assert lib.nvfp4moe_stack_trace_read(buf.ctypes.data, buf.nbytes) == 0
    assert nm.nvfp4_last_device_error() == 0
    G = torch.cuda.get_device_properties(local).multi_processor_count
    tr = buf.reshape(256, 32, 16)[:G, :L, :].astype(np.float64)
    ref = tr[:, :, 1].min(axis=0)  # first CTA to see h_l final, per layer
    rows = []
    first = 1 if L > 1 else 0
    for ev, name in enumerate(TRACE_EVENTS):
        med, mx = [], []
        for l in range(first, L):
            v = tr[:, l, ev]
            v = v[v > 0]
            if v.size == 0:
                continue
            d = (v - ref[l]) / 1e3
            med.append(np.median(d))
            mx.append(np.max(d))
        if med:
            rows.append((name, float(np.median(med)), float(np.median(mx))))
    period = np.diff(ref) / 1e3
    print(f"phase trace: {c['name']}, {L} layers, T={T}, {G} CTAs; times in us after the first CTA saw h_l final "
          f"(median over layers {first}..{L - 1})")
    print(f"{'event':34s} {'median CTA':>11s} {'last CTA':>10s}")
    for name, a, b in rows:
        print(f"{name:34s} {a:11.2f} {b:10.2f}")
    if period.size:
        print(f"layer period: median {np.median(period):.2f} us, min {period.min():.2f}, max {period.max():.2f}")


TC_TRACE_MHZ = 2070.0  # the SM clock under load (clocks sampled by the benchmark)
TC_TRACE_KERNELS = ["grouped up GEMM (k_grouped_tc, last layer)", "grouped down GEMM (k_grouped_tc, last layer)",
                    "lm_head GEMM (k_lm_head_tc, last chunk)"]


def run_trace_tc(args, local, c):
    """The stage trace of the tensor-core kernels (trace build): for CTAs
    0..3 of the last launch of each, the medians over pipeline stages of the
    hand-off intervals, and the per-item times."""
    import ctypes
    import numpy as np
    import torch
    import nvfp4_quantized_moe_sigmoid_gb300 as nm
    from nvfp4_quantized_moe_sigmoid_gb300.model import MoEDecodeStack
    from gen import configs, fill

    T, L = c["T"], c["layers"]
    st = MoEDecodeStack(L, c["E"], c["H"], c["I"], c["S"], c["K"], T, w4a4=c["w4a4"],
                        V=c["V"] if c["lm_head"] else None, rms_eps=c["rms_eps"])
    st.register(*fill.fillers(c["seed"], c["bias"]))
    fill.hidden(st.h[0], c["seed"], layer=configs.HIDDEN_LAYER, rho=c["rho"])
    lib = nm._L
    lib.nvfp4moe_tc_trace_read.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t]
    lib.nvfp4moe_tc_trace_read.restype = ctypes.c_int
    buf = np.zeros(4 * 11 * 1024, dtype=np.uint64)
    for _ in range(max(3, args.warmup)):
        st.step()
    torch.cuda.synchronize()
    for k in range(3):  # clears what the warm-up left
        assert lib.nvfp4moe_tc_trace_read(k, buf.ctypes.data, buf.nbytes) == 0
    st.step()
    torch.cuda.synchronize()
    assert nm.nvfp4_last_device_error() == 0
    print(f"stage trace: {c['name']}, {L} layers, T={T}; per kernel, CTAs 0-3, medians over stages (us)")
    for k, name in enumerate(TC_TRACE_KERNELS):
        assert lib.nvfp4moe_tc_trace_read(k, buf.ctypes.data, buf.nbytes) == 0
        tr = buf.reshape(4, 11, 1024).astype(np.float64) / TC_TRACE_MHZ  # SM clocks -> us
        if not (tr[:, 4] > 0).any():
            continue
        # an entry not written by this launch is 0 (the read clears)
        print(f"-- {name}")
        for cta in range(4):
            t = tr[cta]
            ns = int((t[4] > 0).sum())
            ni = int((t[5] > 0).sum())
            if ns < 2:
                continue
            t0 = t[0][0]
            g = np.arange(ns)
            mma = t[4][:ns]
            span = mma[-1] - t0
            med = lambda x: float(np.median(x)) if len(x) else float("nan")
            print(f"   CTA {cta}: {ns} stages, {ni} items, span {span:.1f}; MMA-issue interval {med(np.diff(mma)):.3f}"
                  f" (mean {np.mean(np.diff(mma)):.3f}); producer space wait {med(t[1][:ns] - t[0][:ns]):.3f};"
                  f" copies landed after issue {med(t[2][:ns] - t[1][:ns]):.3f}; operands prepared {med(t[3][:ns] - t[2][:ns]):.3f};"
                  f" MMA issue after prepared {med(mma - t[3][:ns]):.3f}; issue-to-MMA lead {med(mma - t[1][:ns]):.3f}")
            if ni > 1:
                it, e0, e1 = t[5][:ni], t[6][:ni], t[7][:ni]
                print(f"          item period {med(np.diff(it)):.2f}, epilogue {med(e1 - e0):.2f},"
                      f" epilogue start after item start {med(e0 - it):.2f}")
            print(f"          producer: space free {med(t[8][:ns] - t[0][:ns]):.3f}, tensor copies issued"
                  f" {med(t[9][:ns] - t[8][:ns]):.3f}, scale copies issued {med(t[10][:ns] - t[9][:ns]):.3f},"
                  f" arrive {med(t[1][:ns] - t[10][:ns]):.3f}, next stage {med(t[0][1:ns] - t[1][:ns - 1]):.3f}")
            if cta == 0:
                rel = lambda x: " ".join(f"{v - t0:6.2f}" for v in x[:12])
                print(f"          first stages, producer issued: {rel(t[1])}")
                print(f"                        landed:          {rel(t[2])}")
                print(f"                        MMA issued:      {rel(mma)}")


# ------------------------------------------------------------------ concurrency sweep
SWEEP_T = [1, 2, 3, 4, 5, 8, 16, 32, 64, 128, 256, 512, 1024]


def run_sweep(args, local):
    """One W4A4 MoE layer at the pages' shapes (layer 0 of the seed-0
    weights, router bias U(-0.1, 0.1)) across token counts, on every path the
    library has for it: the decode GEMV kernels and the one-layer stack kernel
    (up to 4 tokens) and the grouped tensor-core path (any count; forced at
    1..4 with nvfp4_set_decode_max_tokens(0)). Each number is one route +
    experts + combine pass timed in a graph of 5 back-to-back passes. Prints
    a table: the measured crossover of the backend choice."""
    import torch

    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_quantized_moe_sigmoid_gb300 as nm
    from nvfp4_quantized_moe_sigmoid_gb300 import roofline as rf
    from nvfp4_quantized_moe_sigmoid_gb300.model import register_layer
    from gen import configs, fill

    c = configs.shape(1)
    E, H, I, S, K = c["E"], c["H"], c["I"], c["S"], c["K"]
    L0 = nm.MoELayer(E, H, I, S)
    register_layer(L0, 0, *fill.fillers(c["seed"], c["bias"]))
    torch.cuda.synchronize()
    peak, _ = measured_peaks()
    rows = []
    for T in SWEEP_T:
        h = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        fill.hidden(h, c["seed"], layer=configs.HIDDEN_LAYER)
        out = torch.empty_like(h)
        idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
        w = torch.empty((T, K), dtype=torch.float32, device="cuda")
        res = {}
        for path in ("decode", "stack", "grouped"):
            if path != "grouped" and T > 4:
                continue
            nm.nvfp4_set_decode_max_tokens(4 if path == "decode" else 0)
            if path == "stack":
                ws_ = nm.make_stack_workspace([L0], T, K, nm.W4A4)
                hout = torch.empty((1, T, H), dtype=torch.bfloat16, device="cuda")
                sidx = torch.empty((1, T, K), dtype=torch.int32, device="cuda")
                sw = torch.empty((1, T, K), dtype=torch.float32, device="cuda")
                fn = (lambda: nm.moe_stack_forward([L0], h, K, nm.W4A4, hidden_out=hout, topk_idx=sidx,
                                                   topk_w=sw, workspace=ws_, rms_eps=c["rms_eps"]))
            else:
                ws_ = nm.make_workspace(L0, T, K, nm.W4A4)
                fn = (lambda: (nm.moe_route_topk(h, L0.router_w, L0.router_b, K, idx, w, rms_eps=c["rms_eps"]),
                               nm.moe_expert_forward(L0, h, idx, w, nm.W4A4, residual=h, out=out, workspace=ws_,
                                                     rms_eps=c["rms_eps"])))
            g = graph_of(fn, 5)
            ms = time_graph(g, 4) / 5
            del g
            assert nm.nvfp4_last_device_error() == 0
            res[path] = ms * 1e3
        nm.nvfp4_set_decode_max_tokens(4)
        u = int(torch.unique(idx if "decode" in res or "grouped" in res else sidx).numel())
        b = rf.layer_bytes(T, u, E, H, I, S, K)
        rows.append((T, u, res, b))
    print("concurrency sweep: one W4A4 MoE layer (hidden %d, %d experts of %d, top-%d, shared %d), "
          "us per layer (us per token)" % (H, E, I, K, S))
    print("| T | unique experts | decode GEMV | stack (1 layer) | grouped tcgen05 | best | best GB/s (frac of %.0f) |" % peak)
    print("|---|---|---|---|---|---|---|")
    for T, u, res, b in rows:
        cell = lambda p: ("%.1f (%.2f)" % (res[p], res[p] / T)) if p in res else "-"
        best = min(res, key=res.get)
        gbs = b / (res[best] * 1e-6) / 1e9
        print("| %d | %d | %s | %s | %s | %s | %.0f (%.2f) |" % (T, u, cell("decode"), cell("stack"), cell("grouped"),
                                                          best, gbs, gbs / peak))


def main():
    args = parse()
    ws, rank, local = dist_init()
    if args.sweep:
        run_sweep(args, local)
        return
    if args.trace:
        run_trace(args, local)
        return
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
