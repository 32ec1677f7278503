#!/usr/bin/env python3
"""Benchmark of the quantized mul_mat hot path (decode GEMV and prefill GEMM) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl syn|reference]

A step is one decode pass over the seven projections of one Llama-1B-shaped layer
(q, k, v, o, gate, up: Q4_K; down: Q6_K; d = 2048, ffn = 8192, one token) through one
syn_mul_mat_batch call: one launch converts the seven activations, one decode launch streams
every weight once (the same step as seven syn_mul_mat calls is reported too).  The timed steps
are captured 16 to a CUDA graph, as a model's decode captures its layers in one graph; the
same step with one graph per step is reported as graph_per_step_value.  Weights are
~N(0, 0.02) quantized with syn_quantize, activations ~N(0, 1), both synthetic.  Steps
rotate over enough weight copies (>= 4x the L2 size) that every step reads its weights
from HBM.  The printed value is weight GB/s: algorithmic bytes (weights + fp32 inputs +
fp32 outputs) per step x steps / time.  A second object reports the prefill GEMM
(Llama-8B FFN up/down, Q4_K, 512 tokens) in TFLOP/s.

--impl reference times the CPU oracle (the plain scalar C implementation the tests
compare against) on the host cores, on a bounded sample of the same workload.
Under torchrun (N > 1) every rank runs its own replica (no collective on the data path:
the decode products of different layers/requests are independent).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized mul_mat weight GB/s (decode GEMV) and TFLOP/s (prefill), % roofline"
WORKLOAD = "llama1b_layer_decode_q4_k_m"
STEPS_PER_GRAPH = 16


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for nm, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------------------

def build_weights(torch, syn, workloads, synth, mats, wl_id, n_copies):
    """Quantized weights on the device: copy 0 from the seeded fp32 weights, copies 1..
    are byte copies (they only defeat the L2)."""
    base = []
    for i, m in enumerate(mats):
        w32 = torch.from_numpy(synth.weight(wl_id, i, m.n_out, m.n_in)).cuda()
        base.append(syn.quantize(m.wtype, w32))
        del w32
    copies = [base]
    for _ in range(1, n_copies):
        copies.append([b.clone() for b in base])
    return copies


def recorded_traffic(summary: str, source: str):
    """DRAM bytes per launch from an ncu summary under profiles/, or None when the kernel
    source has changed since the counters were taken (the summary records its sha256)."""
    import hashlib
    import re
    try:
        text = open(os.path.join(ROOT, "profiles", summary)).read()
        src = open(os.path.join(ROOT, source), "rb").read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch: (\d+) \(source: (\S+) sha256 prefix ([0-9a-f]+)\)", text)
    if not m or m.group(2) != source or not hashlib.sha256(src).hexdigest().startswith(m.group(3)):
        return None
    return int(m.group(1))


def max_over_ranks(t: float, dist, device: str = "cuda") -> float:
    """The largest of the ranks' elapsed times (every rank gets it): a whole-job figure is the
    work of all ranks over the time of the slowest one."""
    if dist is None:
        return t
    import torch
    tt = torch.tensor([t], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def time_graphs(torch, graphs, steps, stream, tail=None):
    """Seconds for `steps` replays (cycling over graphs), plus one replay of `tail`."""
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(steps):
        graphs[i % len(graphs)].replay()
    if tail is not None:
        tail.replay()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / 1e3


def gpu_arm(args, rank, world, dist):
    import torch

    from gguf_block_quantized_gb300 import syn, synth, workloads

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dev = torch.cuda.current_device()
    props = torch.cuda.get_device_properties(dev)
    l2 = props.L2_cache_size
    hbm_peak, tc_peak, tc_sustained, peak_src = load_peaks()
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)

    # ---------------- decode: Llama-1B layer set, one token ----------------
    mats = workloads.LLAMA1B_LAYER
    n_tok = 1
    set_bytes = sum(m.weight_bytes for m in mats)
    n_copies = max(2, -(-4 * l2 // set_bytes))
    W = build_weights(torch, syn, workloads, synth, mats, 2, n_copies)
    X = [torch.from_numpy(synth.activations(2, i, n_tok, m.n_in)).cuda() for i, m in enumerate(mats)]
    Y = [torch.empty((n_tok, m.n_out), device="cuda") for m in mats]
    alg_bytes = sum(workloads.gemv_bytes(m, n_tok) for m in mats)

    def items(c):
        return [(m.wtype, W[c][i], m.n_out, m.n_in, X[i], Y[i]) for i, m in enumerate(mats)]

    def step(c):  # the layer's seven products in one grouped call (one decode launch)
        syn.mul_mat_batch(items(c), n_tok, stream=stream)

    def step_single(c):  # the same products, one syn_mul_mat call (one launch) each
        for i, m in enumerate(mats):
            syn.mul_mat(m.wtype, W[c][i], m.n_out, m.n_in, X[i], Y=Y[i], stream=stream)

    for c in range(n_copies):  # initialise library state outside capture
        step(c)
        step_single(c)
    torch.cuda.synchronize()
    # the timed steps: STEPS_PER_GRAPH consecutive steps per CUDA graph (as a model's decode
    # captures its layers in one graph), each step reading another weight copy
    l0 = syn.launch_count()
    graphs = []
    for c0 in range(n_copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in range(STEPS_PER_GRAPH):
                step((c0 * STEPS_PER_GRAPH + r) % n_copies)
        graphs.append(g)
    launches_per_step = (syn.launch_count() - l0) // (n_copies * STEPS_PER_GRAPH)
    rem = args.steps % STEPS_PER_GRAPH
    rem_graph = None
    if rem:
        rem_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(rem_graph, stream=stream):
            for r in range(rem):
                step(r % n_copies)
    per_step = []  # one graph per step (the launch of each graph not hidden)
    for c in range(n_copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(c)
        per_step.append(g)
    singles = []
    for c in range(n_copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step_single(c)
        singles.append(g)
    for i in range(args.warmup):  # W warm-up steps (whole graphs, at least W steps)
        if i % STEPS_PER_GRAPH == 0:
            graphs[(i // STEPS_PER_GRAPH) % n_copies].replay()
    for g in per_step:
        g.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()

    def timed_steps():  # exactly args.steps steps
        return time_graphs(torch, graphs, args.steps // STEPS_PER_GRAPH, stream, tail=rem_graph)

    with ClockSampler(dev) as clk:
        t = timed_steps()
        # keep the sampler alive for a few samples even when the region is short
        extra = 0
        while len(clk.lines) < 5 and extra < 40:
            timed_steps()
            extra += 1
    t = max_over_ranks(t, dist)
    value = alg_bytes * args.steps * world / t / 1e9
    ms_per_step = t / args.steps * 1e3
    n_ps = max(100, args.steps // 4)
    t_ps = time_graphs(torch, per_step, n_ps, stream) / n_ps
    per_step_value = alg_bytes / t_ps / 1e9
    for i in range(3):
        singles[i % n_copies].replay()
    t_single = time_graphs(torch, singles, max(100, args.steps // 4), stream) / max(100, args.steps // 4)
    single_value = alg_bytes / t_single / 1e9

    # the dominant kernel: the grouped decode launch, timed alone in graphs of 20
    reps = 20
    gs = []
    for c0 in range(min(n_copies, 4)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in range(reps):
                step((c0 * reps + r) % n_copies)
        gs.append(g)
    for g in gs:
        g.replay()
    k_time = time_graphs(torch, gs, 40, stream) / (40 * reps)
    achieved = alg_bytes / k_time / 1e9
    # each matrix alone (single launches), for reference
    per_mat = []
    for i, m in enumerate(mats):
        gs = []
        for c0 in range(min(n_copies, 4)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for r in range(reps):
                    c = (c0 * reps + r) % n_copies
                    syn.mul_mat(m.wtype, W[c][i], m.n_out, m.n_in, X[i], Y=Y[i], stream=stream)
            gs.append(g)
        for g in gs:
            g.replay()
        tm = time_graphs(torch, gs, 40, stream) / (40 * reps)
        per_mat.append((m, tm))

    # ---------------- e2e through the public API, host buffers ----------------
    # the layer's seven inputs packed in one pinned host buffer (and the outputs in another):
    # one host-to-device copy, the grouped call, one device-to-host copy, a synchronize
    x_off = [0]
    for m in mats:
        x_off.append(x_off[-1] + n_tok * m.n_in)
    y_off = [0]
    for m in mats:
        y_off.append(y_off[-1] + n_tok * m.n_out)
    xh = torch.empty(x_off[-1]).pin_memory()
    for i, m in enumerate(mats):
        xh[x_off[i]:x_off[i + 1]] = torch.from_numpy(synth.activations(2, i, n_tok, m.n_in)).reshape(-1)
    yh = torch.empty(y_off[-1]).pin_memory()
    xd_all = torch.empty_like(xh, device="cuda")
    yd_all = torch.empty(y_off[-1], device="cuda")
    xd = [xd_all[x_off[i]:x_off[i + 1]].view(n_tok, m.n_in) for i, m in enumerate(mats)]
    yd = [yd_all[y_off[i]:y_off[i + 1]].view(n_tok, m.n_out) for i, m in enumerate(mats)]
    e2e_steps = max(50, min(args.steps, 2000))
    h2d = xh.numel() * 4
    d2h = yh.numel() * 4

    # one prepared host-staged grouped call per weight copy (syn_mul_mat_batch_staged: the
    # host-to-device copy of the packed inputs, the products, the device-to-host copy of the
    # packed outputs); its arguments are marshalled once, as a decode loop would hold them
    batches = [syn.prepare_batch([(m.wtype, W[c][i], m.n_out, m.n_in, xd[i], yd[i]) for i, m in enumerate(mats)],
                                 n_tok, stream=stream, staged=(xh, xd_all, yd_all, yh)) for c in range(n_copies)]

    def e2e_step(c):
        batches[c]()
        stream.synchronize()

    for c in range(3):
        e2e_step(c)
    s0 = time.perf_counter()
    for k in range(e2e_steps):
        e2e_step(k % n_copies)
    e2e_t = max_over_ranks(time.perf_counter() - s0, dist)
    e2e_value = alg_bytes * e2e_steps * world / e2e_t / 1e9
    # the same step captured in a CUDA graph (copies and launches), one replay + a synchronize
    # per step, as a decode loop would run it
    e2e_graphs = []
    for c in range(n_copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            batches[c]()
        e2e_graphs.append(g)
    for c in range(3):
        e2e_graphs[c % n_copies].replay()
        stream.synchronize()
    s0 = time.perf_counter()
    for k in range(e2e_steps):
        e2e_graphs[k % n_copies].replay()
        stream.synchronize()
    e2e_graph_value = alg_bytes * e2e_steps * world / max_over_ranks(time.perf_counter() - s0, dist) / 1e9

    # ---------------- prefill: Llama-8B FFN up/down, Q4_K, 512 tokens ----------------
    pre = workloads.LLAMA8B_FFN
    p_tok = 512
    PW = [syn.quantize(m.wtype, torch.from_numpy(synth.weight(4, i, m.n_out, m.n_in)).cuda()) for i, m in enumerate(pre)]
    PX = [torch.from_numpy(synth.activations(4, i, p_tok, m.n_in)).cuda() for i, m in enumerate(pre)]
    PY = [torch.empty((p_tok, m.n_out), device="cuda") for m in pre]
    syn.syn_reserve(max(m.n_in for m in pre), p_tok, stream.cuda_stream)
    for i, m in enumerate(pre):
        syn.mul_mat(m.wtype, PW[i], m.n_out, m.n_in, PX[i], Y=PY[i], stream=stream)
    pre_res = []
    for i, m in enumerate(pre):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            syn.mul_mat(m.wtype, PW[i], m.n_out, m.n_in, PX[i], Y=PY[i], stream=stream)
        for _ in range(3):
            g.replay()
        n_it = 50
        tm = time_graphs(torch, [g], n_it, stream) / n_it
        flops = workloads.gemm_flops(m, p_tok)
        pre_res.append({"matrix": m.name, "shape": [m.n_out, m.n_in], "n_tok": p_tok, "ms": tm * 1e3,
                        "tflops": flops / tm / 1e12})
    pre_flops = sum(workloads.gemm_flops(m, p_tok) for m in pre)
    pre_time = sum(r["ms"] for r in pre_res) / 1e3
    pre_tflops = pre_flops / pre_time / 1e12

    configs = other_configs(torch, syn, synth, workloads, stream, l2, hbm_peak, tc_peak, args.quick)

    clocks = clk.summary()
    out = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "q4_k/q6_k weights x q8_k activations, int32 block dots (dp4a), fp32 accumulate",
        "data": "synthetic: weights ~N(0,0.02) quantized by syn_quantize, activations ~N(0,1)",
        "config": {"workload": WORKLOAD, "matrices": [[m.name, workloads.TYPE_NAMES[m.wtype], m.n_out, m.n_in]
                                                       for m in mats],
                   "n_tok": n_tok, "parallelism": f"replicas x{world}",
                   "l2": f"rotating {n_copies} weight copies ({n_copies * set_bytes / 1e6:.0f} MB >= 4x L2 "
                         f"{l2 / 1e6:.0f} MB)", "cuda_graphs": f"{STEPS_PER_GRAPH} steps per graph",
                   "api": "syn_mul_mat_batch (one conversion + one decode launch per step)"},
        "roofline": {"bound": "hbm", "kernel": "k_act_decode + k_gemv<1>: the conversion launch and the "
                                               "grouped decode launch of the 7 matrices",
                     "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "peak_source": peak_src,
                     "traffic": recorded_traffic("k_gemv_llama1b_layer.md", "gguf_block_quantized_gb300/csrc/gemv.cu"),
                     "traffic_note": "dram__bytes_read+write of k_gemv from one ncu capture (profiles/); "
                                     "achieved/launch_us cover the conversion + decode launch pair",
                     "launch_us": round(k_time * 1e6, 3),
                     "single_launch_us": {m.name: round(tm * 1e6, 3) for m, tm in per_mat}},
        "graph_per_step_value": {"value": round(per_step_value, 2), "unit": "GB/s",
                                 "note": "the same step, one CUDA graph launch per step"},
        "single_call_value": {"value": round(single_value, 2), "unit": "GB/s",
                              "note": "same step as 7 separate syn_mul_mat calls (7 launches)"},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "note": "one syn_mul_mat_batch_staged call per step (host-to-device copy of the 7 packed inputs from pinned memory, the grouped products, device-to-host copy of the packed outputs), then a stream synchronize"},
        "e2e_cuda_graph": {"value": round(e2e_graph_value, 2), "unit": "GB/s",
                           "note": "the e2e step (copy in, grouped call, copy out) captured in a CUDA graph; "
                                   "one replay and a stream synchronize per step"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "prefill": {"workload": "llama8b_ffn_q4_k_prefill_512", "value": round(pre_tflops, 1), "unit": "TFLOP/s",
                    "roofline": {"bound": "tensor", "kernel": "k_gemm (tcgen05 kind::f16) + k_act_half",
                                 "achieved": round(pre_tflops, 1), "peak": tc_peak, "unit": "TFLOP/s",
                                 "frac": round(pre_tflops / tc_peak, 4), "peak_source": peak_src,
                                 "note": "fp16 operands; bf16 measured peak used (same nominal rate)"},
                    "matrices": pre_res},
        "configs": configs,
    }
    return out


def time_calls(torch, stream, fn, n_variants, reps, trials=5):
    """Median time of one fn(c) call (c cycles over n_variants) in graphs of `reps` calls."""
    for c in range(n_variants):
        fn(c)
    torch.cuda.synchronize()
    gs = []
    for g0 in range(min(4, n_variants)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in range(reps):
                fn((g0 * reps + r) % n_variants)
        gs.append(g)
    for g in gs:
        g.replay()
    ts = []
    for _ in range(trials):
        ts.append(time_graphs(torch, gs, len(gs), stream) / (len(gs) * reps))
    return sorted(ts)[len(ts) // 2]


def other_configs(torch, syn, synth, workloads, stream, l2, hbm_peak, tc_peak, quick):
    """The workloads besides the headline one: Q8_0 2048x2048 and the Q6_K lm_head as decode
    products (rotating copies >= 4x L2), and the Llama-8B Q4_K_M weight sweep (every
    projection of 32 layers + lm_head) as decode at 1 token and as prefill at 2048 tokens.
    The sweep's 4.6 GB of weights are drawn on the device (torch's Philox generator, seeds
    5000 + i) and quantized with syn_quantize; numpy on the host would take minutes."""
    out = {}

    def gemv_cfg(name, mats, wl_id, n_tok):
        set_bytes = sum(m.weight_bytes for m in mats)
        n_cop = max(2, -(-4 * l2 // set_bytes))
        W = build_weights(torch, syn, workloads, synth, mats, wl_id, n_cop)
        X = [torch.from_numpy(synth.activations(wl_id, i, n_tok, m.n_in)).cuda() for i, m in enumerate(mats)]
        Y = [torch.empty((n_tok, m.n_out), device="cuda") for m in mats]

        def fn(c):
            for i, m in enumerate(mats):
                syn.mul_mat(m.wtype, W[c][i], m.n_out, m.n_in, X[i], Y=Y[i], stream=stream)
        t = time_calls(torch, stream, fn, n_cop, 20)
        alg = sum(workloads.gemv_bytes(m, n_tok) for m in mats)
        out[name] = {"value": round(alg / t / 1e9, 1), "unit": "GB/s", "frac": round(alg / t / 1e9 / hbm_peak, 4),
                     "us": round(t * 1e6, 3), "n_tok": n_tok, "alg_bytes": alg}
        del W

    gemv_cfg("q8_0_2048x2048_decode", workloads.Q8_0_SQUARE, 1, 1)
    gemv_cfg("q6_k_lm_head_decode_1tok", workloads.LM_HEAD_1B, 3, 1)
    gemv_cfg("q6_k_lm_head_decode_4tok", workloads.LM_HEAD_1B, 3, 4)
    # the 32-weight formats Q4_0 / Q5_0 and F16 weights on the Llama-8B FFN up shape
    for wt, nm in ((workloads.Q4_0, "q4_0"), (workloads.Q5_0, "q5_0"), (workloads.F16, "f16")):
        gemv_cfg(f"{nm}_14336x4096_decode", [workloads.Matrix("ffn_up", wt, 14336, 4096)],
                 8 if wt == workloads.F16 else 6, 1)
        m = workloads.Matrix("ffn_up", wt, 14336, 4096)
        wl = 8 if wt == workloads.F16 else 7
        Wp = syn.quantize(wt, torch.from_numpy(synth.weight(wl, 0, m.n_out, m.n_in)).cuda())
        Xp = torch.from_numpy(synth.activations(wl, 0, 512, m.n_in)).cuda()
        Yp = torch.empty((512, m.n_out), device="cuda")
        syn.syn_reserve(m.n_in, 512, stream.cuda_stream)
        t = time_calls(torch, stream, lambda c: syn.mul_mat(wt, Wp, m.n_out, m.n_in, Xp, Y=Yp, stream=stream), 1, 4)
        fl = workloads.gemm_flops(m, 512)
        out[f"{nm}_14336x4096_prefill_512tok"] = {"value": round(fl / t / 1e12, 1), "unit": "TFLOP/s",
                                                  "frac": round(fl / t / 1e12 / tc_peak, 4), "us": round(t * 1e6, 2)}
        del Wp, Xp, Yp
    torch.cuda.empty_cache()

    # deterministic mode (every product on the decode kernels, no split rows): the layer step
    # and a 512-token prefill of the Llama-8B FFN up shape (Q4_K)
    mats = workloads.LLAMA1B_LAYER
    n_cop = max(2, -(-4 * l2 // sum(m.weight_bytes for m in mats)))
    W = build_weights(torch, syn, workloads, synth, mats, 2, n_cop)
    X = [torch.from_numpy(synth.activations(2, i, 1, m.n_in)).cuda() for i, m in enumerate(mats)]
    Y = [torch.empty((1, m.n_out), device="cuda") for m in mats]
    m8 = workloads.Matrix("ffn_up", workloads.Q4_K, 14336, 4096)
    Wp = syn.quantize(m8.wtype, torch.from_numpy(synth.weight(4, 0, m8.n_out, m8.n_in)).cuda())
    Xp = torch.from_numpy(synth.activations(4, 0, 512, m8.n_in)).cuda()
    Yp = torch.empty((512, m8.n_out), device="cuda")
    prev = syn.set_deterministic(True)
    try:
        t = time_calls(torch, stream, lambda c: syn.mul_mat_batch(
            [(m.wtype, W[c][i], m.n_out, m.n_in, X[i], Y[i]) for i, m in enumerate(mats)], 1, stream=stream), n_cop, 16)
        alg = sum(workloads.gemv_bytes(m, 1) for m in mats)
        out["deterministic_llama1b_layer_decode"] = {"value": round(alg / t / 1e9, 1), "unit": "GB/s",
                                                     "frac": round(alg / t / 1e9 / hbm_peak, 4),
                                                     "us": round(t * 1e6, 3)}
        t = time_calls(torch, stream, lambda c: syn.mul_mat(m8.wtype, Wp, m8.n_out, m8.n_in, Xp, Y=Yp, stream=stream),
                       1, 2, trials=3)
        fl = workloads.gemm_flops(m8, 512)
        out["deterministic_q4_k_14336x4096_prefill_512tok"] = {
            "value": round(fl / t / 1e12, 1), "unit": "TFLOP/s", "frac": round(fl / t / 1e12 / tc_peak, 4),
            "us": round(t * 1e6, 2), "note": "decode kernels, 64 groups of 8 tokens: weights read 64 times"}
    finally:
        syn.set_deterministic(prev)
    del W, X, Y, Wp, Xp, Yp
    torch.cuda.empty_cache()

    # GGUF: the layer's seven weight tensors written to a synthetic file, opened (mmap and
    # structure checks) and copied to the device with syn_gguf_upload (page cache warm)
    import tempfile
    mats = workloads.LLAMA1B_LAYER
    code = {workloads.Q4_K: syn.GGML_Q4_K, workloads.Q6_K: syn.GGML_Q6_K}
    with tempfile.TemporaryDirectory() as td:
        path = os.path.join(td, "layer.gguf")
        w = syn.GGUFWriter(path)
        w.kv_string("general.architecture", b"llama")
        for i, m in enumerate(mats):
            q = syn.quantize(m.wtype, torch.from_numpy(synth.weight(2, i, m.n_out, m.n_in)).cuda()).cpu().numpy()
            w.add_tensor(f"blk.0.{m.name}.weight", code[m.wtype], [m.n_in, m.n_out], q)
        w.finish()
        dst = [torch.empty(m.weight_bytes, dtype=torch.uint8, device="cuda") for m in mats]
        times = []
        for _ in range(4):
            t0 = time.perf_counter()
            r = syn.GGUFReader(path)
            t1 = time.perf_counter()
            for i, m in enumerate(mats):
                syn.check(syn.syn_gguf_upload(r.h, i, dst[i].data_ptr(), m.weight_bytes, stream.cuda_stream))
            stream.synchronize()
            t2 = time.perf_counter()
            r.close()
            times.append((t1 - t0, t2 - t1))
        o = sorted(t[0] for t in times[1:])[1]
        u = sorted(t[1] for t in times[1:])[1]
        wsum = sum(m.weight_bytes for m in mats)
        out["gguf_llama1b_layer_open_upload"] = {"value": round(wsum / u / 1e9, 2), "unit": "GB/s",
                                                 "open_us": round(o * 1e6, 1), "upload_ms": round(u * 1e3, 3),
                                                 "bytes": wsum, "note": "host mmap -> device, one copy per tensor"}
        del dst
    if quick:
        return out

    # Llama-8B Q4_K_M sweep
    mats = workloads.llama8b_q4_k_m()
    gen = torch.Generator(device="cuda")
    W = []
    for i, m in enumerate(mats):
        gen.manual_seed(5000 + i)
        w32 = torch.randn((m.n_out, m.n_in), generator=gen, device="cuda") * 0.02
        W.append(syn.quantize(m.wtype, w32))
        del w32
    torch.cuda.empty_cache()
    dims = sorted({m.n_in for m in mats})
    layers = [mats[7 * k:7 * k + 7] for k in range(len(mats) // 7)]
    head = mats[-1]
    wsum = sum(m.weight_bytes for m in mats)

    def inputs(n_tok, seed):
        gen.manual_seed(seed)
        return {d: torch.randn((n_tok, d), generator=gen, device="cuda") for d in dims}

    # decode: one syn_mul_mat_batch per layer (its seven projections) + the lm_head
    X1 = inputs(1, 4999)
    Y1 = [torch.empty((1, m.n_out), device="cuda") for m in mats]

    def token(_c):
        for k, lay in enumerate(layers):
            syn.mul_mat_batch([(m.wtype, W[7 * k + i], m.n_out, m.n_in, X1[m.n_in], Y1[7 * k + i])
                               for i, m in enumerate(lay)], 1, stream=stream)
        syn.mul_mat(head.wtype, W[-1], head.n_out, head.n_in, X1[head.n_in], Y=Y1[-1], stream=stream)
    t = time_calls(torch, stream, token, 1, 1)
    alg = sum(workloads.gemv_bytes(m, 1) for m in mats)
    out["llama8b_q4_k_m_decode_1tok"] = {"value": round(alg / t / 1e9, 1), "unit": "GB/s",
                                         "frac": round(alg / t / 1e9 / hbm_peak, 4), "ms_per_token": round(t * 1e3, 4),
                                         "weight_bytes": wsum, "matrices": len(mats),
                                         "api": "syn_mul_mat_batch per layer + syn_mul_mat for the lm_head"}
    del X1, Y1
    # prefill at 2048 tokens, called as a model calls it: per layer q/k/v in one grouped call on
    # the attention input, o on its own input, gate/up in one grouped call on the FFN input,
    # down on its own input; then the lm_head (a grouped call converts a shared input once)
    p_tok = 2048
    gen.manual_seed(4998)
    d_model, d_ffn = layers[0][0].n_in, layers[0][6].n_in
    XA, XO, XF = (torch.randn((p_tok, d_model), generator=gen, device="cuda") for _ in range(3))
    XD = torch.randn((p_tok, d_ffn), generator=gen, device="cuda")
    YP = [torch.empty((p_tok, m.n_out), device="cuda") for m in layers[0]]
    YH = torch.empty((p_tok, head.n_out), device="cuda")
    syn.syn_reserve(max(dims), p_tok, stream.cuda_stream)

    def prefill(_c):
        for k, lay in enumerate(layers):
            w = W[7 * k:7 * k + 7]
            syn.mul_mat_batch([(lay[i].wtype, w[i], lay[i].n_out, lay[i].n_in, XA, YP[i]) for i in range(3)], p_tok,
                              stream=stream)
            syn.mul_mat(lay[3].wtype, w[3], lay[3].n_out, lay[3].n_in, XO, Y=YP[3], stream=stream)
            syn.mul_mat_batch([(lay[i].wtype, w[i], lay[i].n_out, lay[i].n_in, XF, YP[i]) for i in (4, 5)], p_tok,
                              stream=stream)
            syn.mul_mat(lay[6].wtype, w[6], lay[6].n_out, lay[6].n_in, XD, Y=YP[6], stream=stream)
        syn.mul_mat(head.wtype, W[-1], head.n_out, head.n_in, XF, Y=YH, stream=stream)
    t = time_calls(torch, stream, prefill, 1, 1, trials=3)
    fl = sum(workloads.gemm_flops(m, p_tok) for m in mats)
    out["llama8b_q4_k_m_prefill_2048tok"] = {"value": round(fl / t / 1e12, 1), "unit": "TFLOP/s",
                                             "frac": round(fl / t / 1e12 / tc_peak, 4), "ms": round(t * 1e3, 3),
                                             "flops": fl, "matrices": len(mats),
                                             "api": "per layer syn_mul_mat_batch(q, k, v), syn_mul_mat(o), "
                                                    "syn_mul_mat_batch(gate, up), syn_mul_mat(down); syn_mul_mat(lm_head)"}
    del W, XA, XO, XF, XD, YP, YH
    torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline)
# ----------------------------------------------------------------------------------------

def oracle_arm(budget_s: float, max_steps: int | None = None):
    import numpy as np

    import oracle
    from gguf_block_quantized_gb300 import synth, workloads

    mats = workloads.LLAMA1B_LAYER
    cores = os.cpu_count() or 1
    Wq = [oracle.quantize(m.wtype, synth.weight(2, i, m.n_out, m.n_in)) for i, m in enumerate(mats)]
    X = [synth.activations(2, i, 1, m.n_in) for i, m in enumerate(mats)]
    alg = sum(workloads.gemv_bytes(m, 1) for m in mats)
    done, t0 = 0, time.perf_counter()
    while True:
        for i, m in enumerate(mats):
            oracle.mul_mat(m.wtype, Wq[i], m.n_out, m.n_in, X[i], n_threads=cores)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_steps and done >= max_steps):
            break
    return {"value": round(alg * done / el / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} passes over the 7 Llama-1B layer matrices (n_tok=1), {el:.1f} s, "
                      f"row-split over {cores} threads"}, done, el


def oracle_configs(budget_s: float = 4.0):
    """The oracle (CPU, this machine's cores) on every benchmark configuration: single thread
    on the decode configurations, row-split over all cores on the 512-token prefill, and on a
    sampled subset of the Llama-8B sweep (64 rows x 16 tokens of each distinct matrix shape,
    extrapolated to the whole sweep by the number of multiply-adds).  Each measurement runs
    for about budget_s seconds.  Weights are blocks of the real formats; their values do not
    change the oracle's speed, so a matrix is one quantized 128-row slice repeated."""
    import numpy as np

    import oracle
    from gguf_block_quantized_gb300 import synth, workloads

    cores = os.cpu_count() or 1

    def weights(m, seed):
        rows = min(128, m.n_out)
        q = oracle.quantize(m.wtype, synth.normal(seed, (rows, m.n_in), 0.02))
        return np.ascontiguousarray(np.tile(q, (-(-m.n_out // rows), 1))[:m.n_out])

    def timed(fn):
        n, t0 = 0, time.perf_counter()
        while True:
            fn()
            n += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                return el / n

    out = {"cores": cores}
    for name, mats, n_tok, threads in (("q8_0_2048x2048_decode", workloads.Q8_0_SQUARE, 1, 1),
                                       ("llama1b_layer_decode", workloads.LLAMA1B_LAYER, 1, 1),
                                       ("q6_k_lm_head_decode_1tok", workloads.LM_HEAD_1B, 1, 1),
                                       ("q6_k_lm_head_decode_4tok", workloads.LM_HEAD_1B, 4, 1)):
        Ws = [weights(m, 900 + i) for i, m in enumerate(mats)]
        Xs = [synth.normal(950 + i, (n_tok, m.n_in)) for i, m in enumerate(mats)]
        t = timed(lambda: [oracle.mul_mat(m.wtype, Ws[i], m.n_out, m.n_in, Xs[i], n_threads=threads)
                           for i, m in enumerate(mats)])
        alg = sum(workloads.gemv_bytes(m, n_tok) for m in mats)
        out[name] = {"value": round(alg / t / 1e9, 4), "unit": "GB/s", "threads": threads, "s_per_pass": round(t, 4)}
    # 512-token prefill of the FFN up matrix, rows split over all cores
    m = workloads.LLAMA8B_FFN[0]
    W = weights(m, 960)
    X = synth.normal(961, (512, m.n_in))
    t = timed(lambda: oracle.mul_mat(m.wtype, W, m.n_out, m.n_in, X, n_threads=cores))
    out["q4_k_14336x4096_prefill_512tok"] = {"value": round(workloads.gemm_flops(m, 512) / t / 1e12, 5),
                                             "unit": "TFLOP/s", "threads": cores, "s_per_pass": round(t, 3)}
    # the Llama-8B sweep: sampled entries of each distinct shape, extrapolated
    mats = workloads.llama8b_q4_k_m()
    shapes = {}
    for mm in mats:
        shapes[(mm.wtype, mm.n_out, mm.n_in)] = shapes.get((mm.wtype, mm.n_out, mm.n_in), 0) + 1
    rng = np.random.default_rng(962)
    for n_tok, key in ((1, "llama8b_q4_k_m_decode_1tok"), (2048, "llama8b_q4_k_m_prefill_2048tok")):
        t_all, macs_all = 0.0, 0
        for (wt, n_out, n_in), count in shapes.items():
            mm = workloads.Matrix("s", wt, n_out, n_in)
            W = weights(mm, 963)
            X = synth.normal(964, (n_tok, n_in))
            rows = np.sort(rng.choice(n_out, 64, replace=False))
            toks = np.sort(rng.choice(n_tok, min(16, n_tok), replace=False))
            t = timed(lambda: oracle.mul_mat_sampled(wt, W, n_out, n_in, X, rows, toks)) if budget_s > 0 else 0.0
            frac = (rows.size * toks.size) / (n_out * n_tok)  # sampled share of the outputs
            t_all += count * t / frac
            macs_all += count * n_out * n_in * n_tok
        if n_tok == 1:
            alg = sum(workloads.gemv_bytes(mm, 1) for mm in mats)
            out[key] = {"value": round(alg / t_all / 1e9, 4), "unit": "GB/s", "threads": 1,
                        "note": "extrapolated from 64 sampled rows of each distinct shape"}
        else:
            out[key] = {"value": round(2 * macs_all / t_all / 1e12, 6), "unit": "TFLOP/s", "threads": 1,
                        "note": "extrapolated from 64 rows x 16 tokens of each distinct shape"}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="syn", choices=["syn", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--quick", action="store_true", help="skip the Llama-8B weight sweep")
    ap.add_argument("--oracle-configs", action="store_true",
                    help="time the CPU oracle on every configuration (no GPU work) and print one JSON line")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.oracle_configs:
        if rank == 0:
            print(json.dumps({"oracle_configs": oracle_configs(budget_s=args.cpu_budget / 2)}), flush=True)
        return

    if args.impl == "reference":
        if rank != 0:
            return
        cb, done, el = oracle_arm(budget_s=max(5.0, min(60.0, args.cpu_budget)))
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / done * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32 block dots, fp64 sum",
            "data": "synthetic", "config": {"workload": WORKLOAD, "n_tok": 1},
            "cpu_baseline": cb, "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                                        "d2h_bytes_per_step": 0}}), flush=True)
        return

    dist = None
    if world > 1:
        import torch
        import torch.distributed as td
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        td.init_process_group("nccl")
        dist = td
    out = gpu_arm(args, rank, world, dist)
    if rank == 0:
        cb, _, _ = oracle_arm(budget_s=args.cpu_budget)
        out["cpu_baseline"] = cb
        print(json.dumps(out), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
