#!/usr/bin/env python3
"""Benchmark of the quantized mul_mat hot path (decode GEMV and prefill GEMM) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl syn|reference] [--quick]

A step is one decode token through every projection of a Llama-8B-shaped model in the
Q4_K_M mix (32 layers, d = 4096, ffn = 14336, 32q/8kv heads of 128: q, k, v, o, gate, up
Q4_K; v and down Q6_K in 16 of the 32 layers; a Q6_K lm_head over a 128256-token
vocabulary): 225 matrices, 4.6 GB of weights, one syn_mul_mat_batch call per layer (one
conversion launch and one decode launch stream the layer's seven matrices) and one
syn_mul_mat for the lm_head.  Each step is one replay of a CUDA graph holding the token's
33 calls, as a model's decode captures its layers; the 4.6 GB of weights a step reads are
far larger than the L2, so every step streams them from HBM.  The printed value is weight
GB/s: algorithmic bytes (weights + fp32 inputs + fp32 outputs of every product) per step
x steps / time.  Weights are ~N(0, 0.02) drawn by the seeded generator the parity tests
use and quantized with syn_quantize; activations ~N(0, 1).

The `prefill` object is the same sweep at 2048 tokens in TFLOP/s, each layer called as a
model calls it (q/k/v grouped on one input, o, gate/up grouped on one input, down).  The
`configs` object holds the other workloads (Q8_0 2048x2048; a Llama-1B layer; the Q6_K
lm_head at 1 and 4 tokens; the Llama-8B FFN pair at 512 tokens; Q4_0/Q5_0/F16;
deterministic mode; GGUF upload).

--impl reference times the CPU oracle (the plain scalar C implementation the tests
compare against) on the host cores, on the same sweep (each distinct matrix shape's weights
one quantized 256-row chunk of the seeded rows, repeated to the full size: the oracle's
speed does not depend on the values), one pass per step; the same passes, timed for about
10 s before any GPU work, are the GPU arm's cpu_baseline.  Under torchrun (N > 1) every rank runs its own replica (no
collective on the data path: the decode products of different requests are independent).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized mul_mat weight GB/s (decode GEMV) and TFLOP/s (prefill), % roofline"
WORKLOAD = "llama8b_q4_k_m_decode_sweep"
SWEEP_WL = 5            # synth workload id of the Llama-8B sweep (weights and activations)
PREFILL_TOK = 2048


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


def recorded_traffic(key: str, field: str = "bytes_per_launch"):
    """DRAM bytes of a kernel from profiles/traffic.json (one ncu capture): per launch, or for
    the prefill the sum over one layer's launches (field), or None when any source the kernel
    is built from has changed since the counters were taken (the record holds the sha256 of
    those sources, concatenated in the listed order)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
            rec = json.load(fh)[key]
        h = hashlib.sha256()
        for src in rec["sources"]:
            with open(os.path.join(ROOT, src), "rb") as fh:
                h.update(fh.read())
    except (OSError, KeyError, ValueError):
        return None
    return int(rec[field]) if h.hexdigest() == rec["sha256"] else None


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


def capture(torch, stream, fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def sweep_config(world: int):
    from gguf_block_quantized_gb300 import workloads
    mats = workloads.llama8b_q4_k_m()
    return {"workload": WORKLOAD, "model_shape": "Llama-8B (32 layers, d=4096, ffn=14336, 32q/8kv heads of 128, "
                                                 "vocab 128256)",
            "quant_mix": "Q4_K_M: Q4_K, with attn_v/ffn_down Q6_K in 16 layers; Q6_K lm_head",
            "matrices": len(mats), "weight_bytes": sum(m.weight_bytes for m in mats), "n_tok": 1,
            "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2: every step streams 4.6 GB of weights",
            "cuda_graphs": "one token (32 grouped layer calls + the lm_head call) per graph replay",
            "api": "syn_mul_mat_batch per layer (7 products: one conversion + one decode launch), "
                   "syn_mul_mat for the lm_head"}


# ----------------------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------------------

def quantized_weights(torch, syn, synth, mats, wl_id):
    """Every matrix of `mats` drawn from synth (the seeded generator the parity tests use) and
    quantized on the device; the next matrix is drawn on the host while this one uploads."""
    out = []
    with ThreadPoolExecutor(1) as ex:
        nxt = ex.submit(synth.weight, wl_id, 0, mats[0].n_out, mats[0].n_in)
        for i, m in enumerate(mats):
            w = nxt.result()
            if i + 1 < len(mats):
                nxt = ex.submit(synth.weight, wl_id, i + 1, mats[i + 1].n_out, mats[i + 1].n_in)
            w32 = torch.from_numpy(w).cuda()
            out.append(syn.quantize(m.wtype, w32))
            del w32, w
    torch.cuda.synchronize()
    return out


def gpu_arm(args, rank, world, dist):
    import torch

    from gguf_block_quantized_gb300 import syn, synth, workloads

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dev = torch.cuda.current_device()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    hbm_peak, tc_peak, tc_sustained, peak_src = load_peaks()
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)

    # ---------------- the Llama-8B Q4_K_M sweep: weights ----------------
    mats = workloads.llama8b_q4_k_m()
    layers = [mats[7 * k:7 * k + 7] for k in range(len(mats) // 7)]
    head = mats[-1]
    W = quantized_weights(torch, syn, synth, mats, SWEEP_WL)
    d_model, d_ffn = layers[0][0].n_in, layers[0][6].n_in
    # the activations of a layer: q/k/v read XA, o reads XO, gate/up read XF, down reads XD
    # (one packed device buffer, so that the end-to-end step copies them in with one copy)
    in_sizes = [d_model, d_model, d_model, d_ffn]
    x_host = [synth.activations(SWEEP_WL, j, 1, n) for j, n in enumerate(in_sizes)]
    xh = torch.empty(sum(in_sizes), dtype=torch.float32).pin_memory()
    offs = [0]
    for j, n in enumerate(in_sizes):
        xh[offs[-1]:offs[-1] + n] = torch.from_numpy(x_host[j]).reshape(-1)
        offs.append(offs[-1] + n)
    xd_all = xh.cuda()
    XA, XO, XF, XD = (xd_all[offs[j]:offs[j + 1]].view(1, n) for j, n in enumerate(in_sizes))
    src = [XA, XA, XA, XO, XF, XF, XD]
    Y1 = [torch.empty((1, m.n_out), device="cuda") for m in mats]

    def layer_items(k):
        return [(m.wtype, W[7 * k + i], m.n_out, m.n_in, src[i], Y1[7 * k + i]) for i, m in enumerate(layers[k])]

    prepared = [syn.prepare_batch(layer_items(k), 1, stream=stream) for k in range(len(layers))]

    def run_layers():
        for p in prepared:
            p()

    def run_head():
        syn.mul_mat(head.wtype, W[-1], head.n_out, head.n_in, XF, Y=Y1[-1], stream=stream)

    def token():
        run_layers()
        run_head()

    alg_bytes = sum(workloads.gemv_bytes(m, 1) for m in mats)
    layer_bytes = sum(workloads.gemv_bytes(m, 1) for m in mats[:-1])
    token()  # library state (partitions, workspace) set up outside capture
    torch.cuda.synchronize()
    l0 = syn.launch_count()
    g_token = capture(torch, stream, token)
    launches_per_step = syn.launch_count() - l0
    g_layers = capture(torch, stream, run_layers)
    g_head = capture(torch, stream, lambda: [run_head() for _ in range(8)])
    for _ in range(args.warmup):
        g_token.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()

    def timed_steps():  # exactly args.steps steps
        return time_graphs(torch, [g_token], args.steps, stream)

    with ClockSampler(dev) as clk:
        t = timed_steps()
        extra = 0  # keep the sampler alive for a few samples even when the region is short
        while len(clk.lines) < 5 and extra < 200:
            timed_steps()
            extra += 1
    t = max_over_ranks(t, dist)
    value = alg_bytes * args.steps * world / t / 1e9
    ms_per_step = t / args.steps * 1e3
    assert syn.device_status() == syn.OK

    # the dominant kernel: k_gemv, launched per layer behind its conversion launch; the 32
    # layer calls replayed alone, their mean duration is one launch pair's
    for _ in range(2):
        g_layers.replay()
    n_rep = max(5, min(50, args.steps))
    t_layers = time_graphs(torch, [g_layers], n_rep, stream) / (n_rep * len(layers))
    achieved = layer_bytes / len(layers) / t_layers / 1e9
    g_head.replay()
    t_head = time_graphs(torch, [g_head], 4, stream) / 32
    head_value = workloads.gemv_bytes(head, 1) / t_head / 1e9

    # ---------------- e2e: the public API, host buffers ----------------
    # every step copies the token's inputs in from pinned memory (the first layer's call,
    # syn_mul_mat_batch_staged), runs the 32 layers, and copies the logits out (the lm_head
    # as a staged call), then synchronizes
    yh = torch.empty(head.n_out, dtype=torch.float32).pin_memory()
    empty_h = torch.empty(0, dtype=torch.float32).pin_memory()
    empty_d = torch.empty(0, dtype=torch.float32, device="cuda")
    stage_in = syn.prepare_batch(layer_items(0), 1, stream=stream, staged=(xh, xd_all, empty_d, empty_h))
    stage_out = syn.prepare_batch([(head.wtype, W[-1], head.n_out, head.n_in, XF, Y1[-1])], 1, stream=stream,
                                  staged=(empty_h, empty_d, Y1[-1].view(-1), yh))

    def e2e_step():
        stage_in()
        for p in prepared[1:]:
            p()
        stage_out()
        stream.synchronize()

    for _ in range(3):
        e2e_step()
    e2e_steps = max(20, min(args.steps, 200))
    s0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_t = max_over_ranks(time.perf_counter() - s0, dist)
    e2e_value = alg_bytes * e2e_steps * world / e2e_t / 1e9
    del g_token, g_layers, g_head

    # ---------------- prefill: the same sweep at 2048 tokens ----------------
    p_tok = PREFILL_TOK
    PA, PO, PF, PD = (torch.from_numpy(synth.activations(SWEEP_WL, 10 + j, p_tok, n)).cuda()
                      for j, n in enumerate(in_sizes))
    YP = [torch.empty((p_tok, m.n_out), device="cuda") for m in layers[0]]
    YH = torch.empty((p_tok, head.n_out), device="cuda")
    syn.syn_reserve(d_ffn, p_tok, stream.cuda_stream)

    def prefill_layers():
        for k, lay in enumerate(layers):
            w = W[7 * k:7 * k + 7]
            syn.mul_mat_batch([(lay[i].wtype, w[i], lay[i].n_out, lay[i].n_in, PA, YP[i]) for i in range(3)], p_tok,
                              stream=stream)
            syn.mul_mat(lay[3].wtype, w[3], lay[3].n_out, lay[3].n_in, PO, Y=YP[3], stream=stream)
            syn.mul_mat_batch([(lay[i].wtype, w[i], lay[i].n_out, lay[i].n_in, PF, YP[i]) for i in (4, 5)], p_tok,
                              stream=stream)
            syn.mul_mat(lay[6].wtype, w[6], lay[6].n_out, lay[6].n_in, PD, Y=YP[6], stream=stream)

    def prefill_head():
        syn.mul_mat(head.wtype, W[-1], head.n_out, head.n_in, PF, Y=YH, stream=stream)

    prefill_layers()
    prefill_head()
    torch.cuda.synchronize()
    gp_layers = capture(torch, stream, prefill_layers)
    gp_head = capture(torch, stream, prefill_head)
    gp_layers.replay()
    gp_head.replay()
    tl, th = [], []
    for _ in range(3):
        tl.append(time_graphs(torch, [gp_layers], 1, stream))
        th.append(time_graphs(torch, [gp_head], 1, stream))
    t_pl, t_ph = statistics.median(tl), statistics.median(th)
    p_flops = sum(workloads.gemm_flops(m, p_tok) for m in mats)
    pl_flops = sum(workloads.gemm_flops(m, p_tok) for m in mats[:-1])
    p_value = p_flops / (t_pl + t_ph) / 1e12
    p_layer = pl_flops / t_pl / 1e12
    assert syn.device_status() == syn.OK
    del gp_layers, gp_head, PA, PO, PF, PD, YP, YH, W, Y1, prepared, stage_in, stage_out, src, XA, XO, XF, XD
    torch.cuda.empty_cache()

    configs = other_configs(torch, syn, synth, workloads, stream, l2, hbm_peak, tc_peak, args.quick)

    clocks = clk.summary()
    return {
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
        "data": "synthetic: weights ~N(0,0.02) from the seeded generator of the parity tests, quantized by "
                "syn_quantize; activations ~N(0,1)",
        "config": sweep_config(world),
        "frac_of_peak": round(value / hbm_peak, 4),
        "roofline": {"bound": "hbm", "kernel": "k_act_decode + k_gemv<1>: one layer's conversion launch and grouped "
                                               "decode launch (7 matrices); mean over the 32 layers",
                     "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "peak_source": peak_src,
                     "traffic": recorded_traffic("k_gemv/llama8b_layer"),
                     "traffic_note": "dram__bytes_read+write per k_gemv launch, mean of a Q6_K-v/down layer and a "
                                     "Q4_K layer, from one ncu capture (profiles/traffic.json); null when the "
                                     "kernel's sources changed since",
                     "alg_bytes_per_launch": round(layer_bytes / len(layers)),
                     "launch_us": round(t_layers * 1e6, 3),
                     "lm_head": {"us": round(t_head * 1e6, 3), "value": round(head_value, 1),
                                 "frac": round(head_value / hbm_peak, 4)}},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": xh.numel() * 4,
                "d2h_bytes_per_step": yh.numel() * 4, "steps": e2e_steps,
                "note": "per token: syn_mul_mat_batch_staged for layer 0 (host-to-device copy of the layer inputs "
                        "from pinned memory, then its products), syn_mul_mat_batch for layers 1-31, "
                        "syn_mul_mat_batch_staged for the lm_head (device-to-host copy of the logits), a stream "
                        "synchronize"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "prefill": {"workload": "llama8b_q4_k_m_prefill_sweep_2048tok", "value": round(p_value, 1),
                    "unit": "TFLOP/s", "frac": round(p_value / tc_peak, 4), "ms": round((t_pl + t_ph) * 1e3, 3),
                    "flops": p_flops,
                    "api": "per layer syn_mul_mat_batch(q, k, v), syn_mul_mat(o), syn_mul_mat_batch(gate, up), "
                           "syn_mul_mat(down); syn_mul_mat(lm_head)",
                    "roofline": {"bound": "tensor", "kernel": "k_act_half + k_deq_half (fp16 weight expansion, "
                                                              "at 2048 tokens the Q6_K products) + "
                                                              "k_gemm (tcgen05 kind::f16): the calls of one layer, "
                                                              "mean over the 32 layers",
                                 "achieved": round(p_layer, 1), "peak": tc_peak, "unit": "TFLOP/s",
                                 "frac": round(p_layer / tc_peak, 4), "peak_source": peak_src,
                                 "traffic": recorded_traffic("k_gemm/llama8b_prefill_layer", "bytes_per_layer"),
                                 "traffic_note": "dram__bytes_read+write of one layer's seven k_gemm launches (a "
                                                 "Q6_K-v/down layer at 2048 tokens), from one ncu capture "
                                                 "(profiles/traffic.json); null when the kernel's sources changed "
                                                 "since",
                                 "launch_us": round(t_pl / len(layers) * 1e6, 2),
                                 "lm_head_us": round(t_ph * 1e6, 1),
                                 "note": "fp16 operands; the bf16 measured peak is the denominator (same nominal rate)"}},
        "configs": configs,
    }


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


def build_copies(torch, syn, synth, mats, wl_id, n_copies):
    """Quantized weights on the device: copy 0 from the seeded fp32 weights, copies 1..
    are byte copies (they only defeat the L2)."""
    base = [syn.quantize(m.wtype, torch.from_numpy(synth.weight(wl_id, i, m.n_out, m.n_in)).cuda())
            for i, m in enumerate(mats)]
    return [base] + [[b.clone() for b in base] for _ in range(1, n_copies)]


def other_configs(torch, syn, synth, workloads, stream, l2, hbm_peak, tc_peak, quick):
    """The workloads besides the headline sweep, each timed in CUDA graphs: decode products
    rotate over weight copies >= 4x the L2 so that every call reads HBM."""
    out = {}

    def gemv_cfg(name, mats, wl_id, n_tok, grouped=False):
        set_bytes = sum(m.weight_bytes for m in mats)
        n_cop = max(2, -(-4 * l2 // set_bytes))
        W = build_copies(torch, syn, synth, mats, wl_id, n_cop)
        X = [torch.from_numpy(synth.activations(wl_id, i, n_tok, m.n_in)).cuda() for i, m in enumerate(mats)]
        Y = [torch.empty((n_tok, m.n_out), device="cuda") for m in mats]

        def fn(c):
            if grouped:
                syn.mul_mat_batch([(m.wtype, W[c][i], m.n_out, m.n_in, X[i], Y[i]) for i, m in enumerate(mats)],
                                  n_tok, stream=stream)
            else:
                for i, m in enumerate(mats):
                    syn.mul_mat(m.wtype, W[c][i], m.n_out, m.n_in, X[i], Y=Y[i], stream=stream)
        t = time_calls(torch, stream, fn, n_cop, 20)
        alg = sum(workloads.gemv_bytes(m, n_tok) for m in mats)
        out[name] = {"value": round(alg / t / 1e9, 1), "unit": "GB/s", "frac": round(alg / t / 1e9 / hbm_peak, 4),
                     "us": round(t * 1e6, 3), "n_tok": n_tok, "alg_bytes": alg}
        del W, X, Y

    gemv_cfg("q8_0_2048x2048_decode", workloads.Q8_0_SQUARE, 1, 1)
    gemv_cfg("llama1b_layer_decode_grouped", workloads.LLAMA1B_LAYER, 2, 1, grouped=True)
    out["llama1b_layer_decode_grouped"]["api"] = "one syn_mul_mat_batch call (one conversion + one decode launch)"
    gemv_cfg("q6_k_lm_head_decode_1tok", workloads.LM_HEAD_1B, 3, 1)
    gemv_cfg("q6_k_lm_head_decode_4tok", workloads.LM_HEAD_1B, 3, 4)

    # the Llama-8B FFN pair at 512 tokens (prefill)
    pre = workloads.LLAMA8B_FFN
    PW = [syn.quantize(m.wtype, torch.from_numpy(synth.weight(4, i, m.n_out, m.n_in)).cuda()) for i, m in enumerate(pre)]
    PX = [torch.from_numpy(synth.activations(4, i, 512, m.n_in)).cuda() for i, m in enumerate(pre)]
    PY = [torch.empty((512, m.n_out), device="cuda") for m in pre]
    syn.syn_reserve(max(m.n_in for m in pre), 512, stream.cuda_stream)
    res, t_sum = [], 0.0
    for i, m in enumerate(pre):
        t = time_calls(torch, stream, lambda c: syn.mul_mat(m.wtype, PW[i], m.n_out, m.n_in, PX[i], Y=PY[i],
                                                             stream=stream), 1, 10)
        t_sum += t
        res.append({"matrix": m.name, "shape": [m.n_out, m.n_in], "us": round(t * 1e6, 2),
                    "tflops": round(workloads.gemm_flops(m, 512) / t / 1e12, 1)})
    fl = sum(workloads.gemm_flops(m, 512) for m in pre)
    out["llama8b_ffn_q4_k_prefill_512tok"] = {"value": round(fl / t_sum / 1e12, 1), "unit": "TFLOP/s",
                                              "frac": round(fl / t_sum / 1e12 / tc_peak, 4), "matrices": res}
    del PW, PX, PY
    torch.cuda.empty_cache()
    if quick:
        return out

    # the 32-weight formats Q4_0 / Q5_0 and F16 weights on the Llama-8B FFN up shape
    for wt, nm in ((workloads.Q4_0, "q4_0"), (workloads.Q5_0, "q5_0"), (workloads.F16, "f16")):
        m = workloads.Matrix("ffn_up", wt, 14336, 4096)
        gemv_cfg(f"{nm}_14336x4096_decode", [m], 8 if wt == workloads.F16 else 6, 1)
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

    # deterministic mode (every product on the decode kernels, no split rows): the Llama-1B
    # layer step and a 512-token prefill of the Llama-8B FFN up shape (Q4_K)
    mats = workloads.LLAMA1B_LAYER
    n_cop = max(2, -(-4 * l2 // sum(m.weight_bytes for m in mats)))
    W = build_copies(torch, syn, synth, mats, 2, n_cop)
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

    # GGUF: the Llama-1B layer's seven weight tensors written to a synthetic file, opened
    # (mmap and structure checks) and copied to the device with syn_gguf_upload (page cache warm)
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
    return out


# ----------------------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline)
# ----------------------------------------------------------------------------------------

def oracle_sample():
    """The oracle's inputs for the sweep.  Quantizing all 4.1e9 weights on the host with the
    oracle would take minutes, and its speed does not depend on the weight values, so each
    distinct (format, shape) gets one quantized 256-row chunk of the seeded weights (the
    rows the GPU arm draws for the first matrix of that shape), repeated to the full row
    count.  One pass is every one of the 225 products, rows split over all host cores.
    Returns (one pass, algorithmic bytes of a pass, cores)."""
    import numpy as np

    import oracle
    from gguf_block_quantized_gb300 import synth, workloads

    mats = workloads.llama8b_q4_k_m()
    cores = os.cpu_count() or 1
    tiles = {}
    for i, m in enumerate(mats):
        key = (m.wtype, m.n_out, m.n_in)
        if key not in tiles:
            q = oracle.quantize(m.wtype, synth.weight_rows(SWEEP_WL, i, m.n_in, 0, m.n_out))
            tiles[key] = np.ascontiguousarray(np.tile(q, (-(-m.n_out // q.shape[0]), 1))[:m.n_out])
    d_model, d_ffn = mats[0].n_in, mats[6].n_in
    xs = [synth.activations(SWEEP_WL, j, 1, n) for j, n in enumerate([d_model, d_model, d_model, d_ffn])]
    src = [xs[0], xs[0], xs[0], xs[1], xs[2], xs[2], xs[3]]
    X = [src[i % 7] if i < len(mats) - 1 else xs[2] for i in range(len(mats))]

    def one_pass():
        for i, m in enumerate(mats):
            oracle.mul_mat(m.wtype, tiles[(m.wtype, m.n_out, m.n_in)], m.n_out, m.n_in, X[i], n_threads=cores)

    return one_pass, sum(workloads.gemv_bytes(m, 1) for m in mats), cores


def oracle_timed(n_steps=None, budget_s=None, warmup=1):
    one_pass, alg, cores = oracle_sample()
    for _ in range(warmup):
        one_pass()
    done, t0 = 0, time.perf_counter()
    while True:
        one_pass()
        done += 1
        el = time.perf_counter() - t0
        if (n_steps is not None and done >= n_steps) or (budget_s is not None and el >= budget_s):
            break
    return {"value": round(alg * done / el / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} passes over all 225 Llama-8B Q4_K_M products (n_tok=1; each distinct shape's "
                      f"weights one 256-row chunk of the seeded rows, repeated), {el:.1f} s, rows split over "
                      f"{cores} threads"}, done, el


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="syn", choices=["syn", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--quick", action="store_true", help="skip the 32-weight, F16, deterministic and GGUF configs")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        cb, done, el = oracle_timed(n_steps=args.steps, warmup=args.warmup)
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / done * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32 block dots, fp64 sum",
            "data": "synthetic", "config": sweep_config(1),
            "cpu_baseline": cb, "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                                        "d2h_bytes_per_step": 0}}), flush=True)
        return

    # the oracle baseline first, before this process touches the GPU (N = 1 only)
    cb = oracle_timed(budget_s=args.cpu_budget)[0] if world == 1 else None
    dist = None
    if world > 1:
        import torch
        import torch.distributed as td
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        td.init_process_group("nccl")
        dist = td
    out = gpu_arm(args, rank, world, dist)
    if rank == 0:
        if cb is not None:
            out["cpu_baseline"] = cb
        print(json.dumps(out), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
