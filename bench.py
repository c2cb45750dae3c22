#!/usr/bin/env python
"""Throughput of the quantized-expert MoE layer forward pass on GB300.

One step = one pass of the whole hot path (routing, permutation, gate/up GEMM with fused
dequantization and SiLU*up, down GEMM with fused weighted combine) through every layer of a
48-layer stack with distinct seeded weights (the 30B-A3B shape: 128 experts, hidden 2048,
intermediate 768, top-8), on one batch of synthetic tokens.  Layers are independent: each
consumes the same activations with its own router logits.

Default workload: NVFP4 W4A4 (dynamic NVFP4 activations), 16,384 tokens x 48 layers with
Zipf(1.1)-skewed routing -- the largest single-GPU configuration.  Prints one JSON line.
--config 1 is FP8 block-128x128 W8A16 decode (T = 16, with the T = 1 and 4 sweep points).
  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--tokens T] [--impl ours|reference]
Multi-GPU (torchrun): every rank runs its own replica on its own tokens (weak scaling, no
collective on the data path; one all-reduce of the elapsed time only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s per format; HBM GB/s & tensor-pipe util vs GB300 peak"
FMT_ID = {"fp8": 1, "int4": 2, "nvfp4_w4a16": 3, "nvfp4_w4a4": 4, "bf16": 5, "fp8_w8a8": 6}
# dense tensor rate of each format's MMA operands relative to bf16 (nominal GB300 figures:
# bf16 2.25, fp8 4.5, fp4 13.5 PFLOP/s); W8A16 / W4A16 run bf16 operands after dequantization
TENSOR_RATIO = {"fp8": 1.0, "int4": 1.0, "nvfp4_w4a16": 1.0, "nvfp4_w4a4": 13.5 / 2.25, "bf16": 1.0,
                "fp8_w8a8": 4.5 / 2.25}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", type=int, default=4, choices=[1, 2, 3, 4, 5, 6, 7, 8])
    p.add_argument("--tokens", type=int, default=None, help="tokens per step (default: the config's largest)")
    p.add_argument("--layers", type=int, default=None, help="layers per step (default 48)")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-sweep", action="store_true")
    p.add_argument("--no-graph", action="store_true", help="launch layer by layer instead of replaying a CUDA graph")
    return p.parse_args()


def workload(args):
    c = dict(synth.CONFIGS[args.config])
    c["T"] = args.tokens if args.tokens is not None else max(c["T"])
    c["L"] = args.layers if args.layers is not None else c["layers"]
    return c


def format_mix(c):
    """The format, or for a mixed stack each format with its layer count."""
    fm = synth.layer_formats(c, c["L"])
    kinds = list(dict.fromkeys(fm))
    return kinds[0] if len(kinds) == 1 else " + ".join(f"{f} x{fm.count(f)}" for f in kinds)


def describe(c):
    return (f"{c['name']}: {format_mix(c)} experts, T={c['T']} tokens x {c['L']} layers, hidden {c['H']}, "
            f"intermediate {c['I']}, {c['E']} experts, top-{c['k']}"
            + (f", Zipf({c['zipf']}) routing skew" if c["zipf"] else ", N(0,1) logits")
            + (", static activation scales calibrated on the batch" if c.get("static_act") else ""))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------------------------------
# Replicas across ranks (weak scaling: every rank runs the whole layer stack on its own tokens)
# ------------------------------------------------------------------------------------------
def rank_seed(seed, rank):
    """Seed of a rank's synthetic tokens and weights: every replica draws its own batch."""
    return seed + 7919 * rank


def max_over_ranks(value, device, world):
    """The largest value over all ranks (the job is as slow as its slowest replica)."""
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, T, L, seconds_per_step):
    """Whole-job throughput: every rank's T tokens through L layers per step."""
    return world * T * L / seconds_per_step


def per_expert_bytes(fmt, H, I):
    import nvfp4_expert_gemms_gb300 as M

    d = M.moe_packed_size(fmt, 1, H, I)
    gu = int(d.size[M.MOE_T_GU_A]) + int(d.size[M.MOE_T_GU_B]) + int(d.size[M.MOE_T_GU_GS])
    dn = int(d.size[M.MOE_T_D_A]) + int(d.size[M.MOE_T_D_B]) + int(d.size[M.MOE_T_D_GS])
    return gu, dn


def source_digest(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(fmt, T):
    """Per-launch DRAM traffic of the gate/up kernel from the committed ncu summary, when it was
    captured on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for ln in open(path):
        ln = ln.split("#")[0].split()
        if len(ln) == 5 and ln[0] == fmt and int(ln[1]) == T:
            srcs = ln[3].split(",")
            try:
                if source_digest(srcs) == ln[4]:
                    return float(ln[2])
            except FileNotFoundError:
                return None
    return None


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.file,
                                         stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for ln in f:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) == 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------------------------
# CPU oracle timing (test infrastructure: only this leg of the bench loads oracle/)
# ------------------------------------------------------------------------------------------
class OracleSample:
    """A bounded sample of the workload for timing the oracle as it stands on host cores:
    `layers` layers with their own weights (only the routed experts are drawn and packed, and
    that set-up is untimed), all T tokens when T <= 64, else a seeded subset of 64 tokens per
    layer (tokens are independent, so a subset is the same computation at a smaller size)."""

    def __init__(self, c, seed, layers=2):
        import oracle

        oracle.build()
        self.oracle = oracle
        self.c = c
        T, H, I, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
        self.x = synth.gen_x(T, H, seed)
        self.n_tok = T if T <= 64 else 64
        self.items = []
        fmts = synth.layer_formats(c, c["L"])
        first = [fmts.index(f) for f in dict.fromkeys(fmts)]  # one layer of each format, then the next ones
        order = first + [l for l in range(c["L"]) if l not in first]
        for layer in order[:min(layers, c["L"])]:
            fid = FMT_ID[fmts[layer]]
            lg = synth.gen_logits(T, E, seed, layer, zipf_alpha=c["zipf"])
            toks = None if self.n_tok == T else np.sort(
                np.random.default_rng([seed, layer]).choice(T, size=self.n_tok, replace=False)).astype(np.int32)
            idx, _ = oracle.route(lg if toks is None else lg[toks], k)
            experts = np.unique(idx)
            wgu, wd = synth.gen_expert_weights(E, H, I, seed, layer, experts=experts)
            self.items.append((fid, lg, toks, oracle.pack_experts(fid, wgu, wd, experts=experts)))
        self.desc = (f"{len(self.items)} layer(s) x {self.n_tok} of {T} tokens of the same workload "
                     f"(only routed experts drawn; packing untimed)")

    def run(self, min_seconds=0.0, nthreads=None):
        """Oracle forward over the sample (repeated until min_seconds) on nthreads host threads
        (default: all); returns (tokens/s, seconds)."""
        nthreads = self.cores() if nthreads is None else nthreads
        spent, tokens = 0.0, 0
        act_gs = None
        if self.c.get("static_act"):  # x's scale from the batch, h's a fixed calibrated-range stand-in
            amax = float(np.abs(synth.bf16_bits_to_f32(self.x)).max())
            act_gs = np.array([np.float32(2688.0) / np.float32(amax), np.float32(2688.0)], np.float32)
        while True:
            for fid, lg, toks, packed in self.items:
                t0 = time.perf_counter()
                self.oracle.moe_layer(fid, self.x, lg, packed, self.c["k"], tokens=toks, act_gs=act_gs,
                                      nthreads=nthreads)
                spent += time.perf_counter() - t0
                tokens += self.n_tok
            if spent >= min_seconds:
                return tokens / spent, spent

    def cores(self):
        if not hasattr(self, "_cores"):  # read once: a single-threaded run lowers the OpenMP default
            self._cores = self.oracle.max_threads()
        return self._cores


def cpu_model():
    """The host CPU's model name (x86 'model name', Arm implementer/part), or the machine type."""
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        return platform.machine()
    for key in ("model name", "Model name", "Hardware"):
        for ln in info:
            if ln.split(":")[0].strip() == key:
                return ln.split(":", 1)[1].strip()
    parts = {ln.split(":")[0].strip(): ln.split(":", 1)[1].strip() for ln in info if ":" in ln}
    if "CPU implementer" in parts:
        return f"{platform.machine()} implementer {parts['CPU implementer']} part {parts.get('CPU part', '?')}"
    return platform.machine()


# ------------------------------------------------------------------------------------------
# Our arm
# ------------------------------------------------------------------------------------------
def run_ours(args, c, rank, world, local_rank):
    import torch

    import nvfp4_expert_gemms_gb300 as M

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    fmt, T, H, I, E, k, L = c["fmt"], c["T"], c["H"], c["I"], c["E"], c["k"], c["L"]
    fmts = synth.layer_formats(c, L)  # fmt throughout, or a mixed stack
    seed = rank_seed(args.seed, rank)
    layers = []
    for l in range(L):
        wgu, wd = synth.gen_expert_weights_device(E, H, I, seed, l, dev)
        layers.append(M.MoELayer(fmts[l], wgu, wd))
        del wgu, wd
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    x = torch.from_numpy(synth.gen_x(T, H, seed).view(np.int16)).to(dev).view(torch.bfloat16)
    lg_host = np.stack([synth.gen_logits(T, E, seed, l, zipf_alpha=c["zipf"]) for l in range(L)])
    lg = torch.from_numpy(lg_host).to(dev)
    outs = torch.empty((L, T, H), dtype=torch.bfloat16, device=dev)
    first_of = {f: layers[fmts.index(f)].desc for f in dict.fromkeys(fmts)}

    def ws_bytes(Ts, host_io=False):  # one workspace serves every layer: the largest format's size
        size = M.moe_workspace_size_host_io if host_io else M.moe_workspace_size
        return max(size(d, Ts, k) for d in first_of.values())

    ws = torch.empty(ws_bytes(T), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    # distinct routed experts per layer: the unit of algorithmic weight bytes
    D = [int(torch.unique(torch.topk(lg[l], k, dim=-1).indices).numel()) for l in range(L)]
    peb = {f: per_expert_bytes(f, H, I) for f in first_of}  # (gate/up, down) packed bytes per expert
    x_b, lg_b, out_b = T * H * 2, T * E * 4, T * H * 2
    layer_bytes = [D[l] * sum(peb[fmts[l]]) + x_b + lg_b + out_b for l in range(L)]
    gu_bytes = [D[l] * peb[fmts[l]][0] + x_b for l in range(L)]
    main_layers = [l for l in range(L) if fmts[l] == fmt]  # the roofline's kernel: the config's format
    flops_layer = 2.0 * T * k * (H * 2 * I + I * H)
    gu_flops = 2.0 * T * k * H * 2 * I

    # gate/up launch times are sampled on every 8th layer: an event between two kernels is a
    # graph node that also cuts the programmatic (overlapped) launch edge, so the other layers
    # run without events
    sampled = [l for l in main_layers if l % 8 == min(7, L - 1)] or [main_layers[-1]]

    act = None
    if c.get("static_act"):  # static activation scales, calibrated per layer on this batch (untimed)
        act = torch.stack([M.moe_calibrate_act_scales(x, lg[l], layers[l].desc, layers[l].packed, k, ws)
                           for l in range(L)])
        torch.cuda.synchronize()

    def forward(l, xx, lgl, out_l, wsp):
        if act is None:
            M.moe_layer_forward(xx, lgl, layers[l].desc, layers[l].packed, k, out_l, wsp)
        else:
            M.moe_layer_forward_static_act(xx, lgl, layers[l].desc, layers[l].packed, k, act[l], out_l, wsp)

    def step(timed_events=None):
        for l in range(L):
            if timed_events is not None and l in timed_events:
                M.moe_time_next_step(0, *timed_events[l][:2])
                M.moe_time_next_step(1, *timed_events[l][2:])
            forward(l, x, lg[l], outs[l], ws)

    def as_runner(fn):
        """The step as a CUDA graph (captured after an eager warm-up call) or as eager launches.
        Returns (run, kernels per step)."""
        fn()  # eager call: one-time set-up (function attributes) happens outside any capture
        torch.cuda.synchronize()
        n0 = M.moe_kernel_launch_count()
        if args.no_graph:
            fn()
            torch.cuda.synchronize()
            return fn, M.moe_kernel_launch_count() - n0
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g.replay, M.moe_kernel_launch_count() - n0

    ev = {l: tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for l in sampled}
    for evs in ev.values():  # torch creates the CUDA event on first record; the library re-records it
        for e_ in evs:
            e_.record()
    run, launches_per_step = as_runner(lambda: step(ev))
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    assert M.moe_get_device_error(ws) == 0, "device error flag set during warm-up"

    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = getattr(torch.cuda.get_device_properties(local_rank), "uuid", None)
    clocks = Clocks(f"GPU-{uuid}" if uuid is not None else local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    t_start.record()
    step_ev[0].record()
    for s in range(args.steps):
        run()
        step_ev[s + 1].record()
    t_stop.record()
    torch.cuda.synchronize()
    n_launch = launches_per_step * args.steps
    clk = clocks.stop()
    assert M.moe_get_device_error(ws) == 0, "device error flag set during the timed steps"
    if world > 1:
        torch.distributed.barrier()
    ms_total = t_start.elapsed_time(t_stop)
    gu_ms = [ev[l][0].elapsed_time(ev[l][1]) for l in sampled]  # the last timed step's sampled launches
    dn_ms = [ev[l][2].elapsed_time(ev[l][3]) for l in sampled]
    per_step = sorted(step_ev[i].elapsed_time(step_ev[i + 1]) for i in range(args.steps))

    def pct(q):
        return per_step[min(len(per_step) - 1, int(round(q * (len(per_step) - 1))))]
    ms_total = max_over_ranks(ms_total, dev, world)
    ms_step = ms_total / args.steps
    value = job_tokens_per_s(world, T, L, ms_step / 1e3)

    peaks, peak_src = load_peaks()
    gu_avg_s = statistics.mean(gu_ms) / 1e3
    hbm_bound = c["fmt"] in ("fp8", "int4") or T <= 256
    if hbm_bound:
        achieved = statistics.mean(gu_bytes[l] for l in sampled) / gu_avg_s / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4)}
    else:
        peak = peaks["bf16_tflops_sustained"] * TENSOR_RATIO[fmt]
        achieved = gu_flops / gu_avg_s / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4)}
    traffic = recorded_traffic(fmt + ("_static" if c.get("static_act") else ""), T)  # recorded per launch at the
    # 48-layer mean; rescaled to the sampled layers
    if traffic is not None:
        traffic = round(traffic * statistics.mean(gu_bytes[l] for l in sampled) /
                        statistics.mean(gu_bytes[l] for l in main_layers))
    roof.update({"traffic": traffic, "kernel": "grouped gate/up GEMM",
                 "launch_ms": round(gu_avg_s * 1e3, 4), "peak_source": peak_src,
                 "step_fraction": round(gu_avg_s * 1e3 * L / ms_step, 3), "sampled_layers": len(sampled),
                 "down_launch_ms": round(statistics.mean(dn_ms), 4)})
    layer_s = ms_step / 1e3 / L
    bound_s = sum(max(layer_bytes[l] / (peaks["hbm_gbs"] * 1e9),
                      flops_layer / (peaks["bf16_tflops_sustained"] * TENSOR_RATIO[fmts[l]] * 1e12)) for l in range(L))
    whole = {"hbm_gbs": round(statistics.mean(layer_bytes) / layer_s / 1e9, 1),
             "tflops": round(flops_layer / layer_s / 1e12, 2),
             "roofline_frac": round(bound_s / (ms_step / 1e3), 4),
             "distinct_experts_per_layer": round(statistics.mean(D), 1)}

    # end to end through the host-buffer entry point: inputs copied in, results copied out
    ws_io = torch.empty(ws_bytes(T, host_io=True), dtype=torch.uint8, device=dev)
    x_h = torch.from_numpy(synth.gen_x(T, H, seed).view(np.int16)).view(torch.bfloat16).pin_memory()
    lg_h = torch.from_numpy(lg_host).pin_memory()
    out_h = torch.empty((L, T, H), dtype=torch.bfloat16).pin_memory()

    x_d = torch.empty_like(x)
    lg_d = torch.empty_like(lg[0])

    def step_host():
        for l in range(L):
            if act is None:
                M.moe_layer_forward_host(x_h, lg_h[l], layers[l].desc, layers[l].packed, k, out_h[l], ws_io)
            else:  # the static entry has device I/O: the same copies, issued around it
                x_d.copy_(x_h, non_blocking=True)
                lg_d.copy_(lg_h[l], non_blocking=True)
                forward(l, x_d, lg_d, outs[l], ws_io)
                out_h[l].copy_(outs[l], non_blocking=True)

    run_host, _ = as_runner(step_host)
    for _ in range(args.warmup):
        run_host()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run_host()
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / args.steps
    e2e = {"value": round(job_tokens_per_s(world, T, L, max_over_ranks(e2e_s, dev, world)), 1), "unit": "tokens/s",
           "h2d_bytes_per_step": L * (x_b + lg_b), "d2h_bytes_per_step": L * out_b,
           "api": ("moe_layer_forward_host (pinned host buffers)" if act is None else
                   "moe_layer_forward_static_act between copies from / to pinned host buffers")
                  + ("" if args.no_graph else ", CUDA graph")}

    sweep = None
    if not args.no_sweep and rank == 0 and len(synth.CONFIGS[args.config]["T"]) > 1:
        sweep = {}
        for Ts in synth.CONFIGS[args.config]["T"]:
            if Ts == T:
                sweep[str(Ts)] = round(value / world, 1)
                continue
            xs = x[:Ts].contiguous()
            lgs = [lg[l, :Ts].contiguous() for l in range(L)]
            wss = torch.empty(ws_bytes(Ts), dtype=torch.uint8, device=dev)
            run_s, _ = as_runner(lambda: [forward(l, xs, lgs[l], outs[l, :Ts], wss) for l in range(L)])
            for _ in range(2):
                run_s()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(3):
                run_s()
            b.record()
            torch.cuda.synchronize()
            sweep[str(Ts)] = round(Ts * L / (a.elapsed_time(b) / 3 / 1e3), 1)

    step_stats = {"median": round(statistics.median(per_step), 4), "p10": round(pct(0.1), 4),
                  "p90": round(pct(0.9), 4)}
    return {"value": value, "ms_per_step": ms_step, "roofline": roof, "layer": whole, "e2e": e2e,
            "gpu_launches": int(n_launch), "clocks": clk, "sweep": sweep, "step_ms": step_stats}


def main():
    args = parse_args()
    c = workload(args)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    base = {"metric": METRIC, "unit": "tokens/s", "n_gpus": max(world, args.gpus if world == 1 else world),
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "data": "synthetic (seeded draws of the synth module: bf16 N(0,1) activations, N(0,0.02) weights, N(0,1) logits)",
            "config": {"workload": describe(c), "format": format_mix(c), "tokens": c["T"], "layers": c["L"],
                       "hidden": c["H"], "intermediate": c["I"], "experts": c["E"], "top_k": c["k"],
                       "l2": "inputs larger than L2: each step streams the distinct weights of all layers",
                       "parallelism": f"replicas x{world}",
                       "launch": "eager" if args.no_graph else "CUDA graph of the whole step (replayed)"}}

    if args.impl == "reference":
        if rank != 0:
            return
        smp = OracleSample(c, args.seed)
        smp.cores()
        for _ in range(args.warmup):
            smp.run()
        vals = []
        t0 = time.perf_counter()
        for _ in range(args.steps):
            vals.append(smp.run()[0])
        wall = time.perf_counter() - t0
        v = statistics.mean(vals)
        line = dict(base, impl="reference", value=round(v, 3), ms_per_step=round(1e3 * c["T"] * c["L"] / v, 3),
                    dtype="f64", n_gpus=1,
                    cpu_baseline={"value": round(v, 3), "unit": "tokens/s", "cores": smp.cores(), "kind": "oracle",
                                  "sample": smp.desc, "cpu_model": cpu_model(), "nproc": os.cpu_count()},
                    e2e={"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                         "d2h_bytes_per_step": 0},
                    sampled_seconds=round(wall, 2), sampled_seconds_per_step=round(wall / max(args.steps, 1), 3),
                    note=(f"CPU oracle timed on the host cores; each step is the bounded sample above "
                          f"({wall:.1f} s wall for {args.steps} steps); ms_per_step extrapolates to the full step"))
        print(json.dumps(line))
        return

    import torch

    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    r = run_ours(args, c, rank, world, local_rank)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        smp = OracleSample(c, args.seed)
        cores = smp.cores()
        v, spent = smp.run(min_seconds=10.0, nthreads=cores)  # OpenMP over tokens on every core
        v1, spent1 = smp.run(min_seconds=5.0, nthreads=1)  # and on one core
        cpu = {"value": round(v, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": smp.desc,
               "seconds": round(spent, 1), "cpu_model": cpu_model(), "nproc": os.cpu_count(),
               "single_thread": {"value": round(v1, 3), "cores": 1, "seconds": round(spent1, 1)}}
    if rank == 0:
        dtype = {"fp8": ("f32 (e4m3 weight x two-term e4m3 split of the bf16 activations; exact except"
                         " elements under ~1/1800 of their row maximum)"), "int4": "f32", "nvfp4_w4a16": "f32",
                 "nvfp4_w4a4": "f32", "bf16": "f32 (bf16 products)", "fp8_w8a8": "f32 (e4m3 x e4m3 products)"}[c["fmt"]]
        line = dict(base, value=round(r["value"], 1), ms_per_step=round(r["ms_per_step"], 4), dtype=dtype,
                    roofline=r["roofline"], cpu_baseline=cpu, e2e=r["e2e"], gpu_launches=r["gpu_launches"],
                    clocks=r["clocks"], layer=r["layer"], step_ms=r["step_ms"])
        if r["sweep"]:
            line["sweep_tokens_per_s"] = r["sweep"]
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
