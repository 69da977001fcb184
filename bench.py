#!/usr/bin/env python
"""Benchmark of the NVFP4 routed-MoE layer (moe_forward) on GB300.

Metric: MoE-layer tokens/s (token-layers per second for stacked workloads), with the dominant
kernel's roofline fraction (HBM GB/s for the decode and batched-decode workloads, 16-bit tensor
TFLOP/s for the prefill workloads) against the measured peaks, the CPU oracle timed beside it,
and an end-to-end number through host buffers.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload all|decode|batched|prefill|long|tiny]
    python bench.py --impl reference ...      # the CPU oracle as the reference arm

The default (--workload all) measures the four benchmark workloads in one run and prints ONE
JSON line: the long cold prefill (4 layers x T = 32768, Zipf routing) is the headline (its
value, roofline, e2e and CPU baseline are the line's own keys), and `workloads` holds the same
fields for the decode/verify sweep, the batched decode and the prefill chunk.

One step = one pass of the whole layer over one batch of every layer of the workload (decode:
four layers with T = 1, 2, 4, 8; long: four layers of T = 32768).  Inputs are synthetic
(seeded, see synth/), weights random-init NVFP4, resident in HBM before timing.  Each step uses
the next of P distinct input batches, so the experts touched change from step to step; every
layer's weights (907 MB each) exceed L2.  The steps are replayed as CUDA graphs.  N > 1 runs N
independent replicas (one per GPU, no collective on the data path); value = all ranks' tokens /
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s"
UNIT = "tokens/s"
HEADLINE = "long"                       # the workload of the line's own keys under --workload all
SUBWORKLOADS = ("decode", "batched", "prefill")
DTYPE = ("nvfp4 weights (e2m1 x e4m3 per 16 x fp32 scale2) x bf16 activations; "
         "f16 x f16 tensor-core products (exact for both operands), fp32 accumulate")


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=None)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="all", choices=["all"] + list(synth.WORKLOADS))
    p.add_argument("--pool", type=int, default=None, help="distinct input batches cycled through")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--warmup-seconds", type=float, default=1.0,
                   help="keep warming up (whole steps) at least this long, for steady clocks")
    p.add_argument("--fp8", action="store_true", help="with --one-forward: the FP8-activation arm")
    p.add_argument("--one-forward", type=int, default=None, metavar="LAYER",
                   help="profiling aid: build layer LAYER of the workload, run four forwards, exit "
                        "(no timing, no JSON line)")
    return p.parse_args()


DEFAULTS = {  # steps, warmup, pool
    "tiny": (2000, 50, 16), "decode": (2000, 50, 16), "batched": (500, 20, 8),
    "prefill": (50, 5, 4), "long": (8, 3, 2),
}


def workload_entries(name):
    """(T, seed) of every layer one step runs."""
    w = synth.WORKLOADS[name]
    if w.layers > 1:
        return [(w.Ts[0], synth.layer_seed(w, w.seeds[0], l)) for l in range(w.layers)]
    return list(zip(w.Ts, w.seeds))


def describe(name):
    """The workload, as both arms state it in `config`."""
    w = synth.WORKLOADS[name]
    return {"workload": w.description, "T": list(w.Ts), "H": w.H, "E": w.E, "k": w.k, "I": w.I,
            "shared_expert": True, "layers_per_step": len(workload_entries(name)),
            "seeds": [s for _, s in workload_entries(name)], "logit_bias": w.logit_bias,
            "outlier_frac": w.outlier_frac, "weights": "NVFP4 (e2m1 x e4m3/16 x fp32 scale2)"}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm": float(d["hbm_gbs"]), "bf16": float(d["bf16_tflops"]),
                "bf16_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


def slowest_rank_ms(elapsed_ms, dist=None, device="cpu"):
    """The job's time: the largest of the ranks' times (a MAX all-reduce over the process group),
    or the value itself on one rank."""
    if dist is None:
        return float(elapsed_ms)
    tt = torch.tensor([float(elapsed_ms)], device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def replica_throughput(world, steps, tokens_per_step, max_ms):
    """Whole-job tokens/s of `world` independent replicas: every rank's tokens over the slowest
    rank's time."""
    return world * steps * tokens_per_step / (max_ms / 1e3)


def stored_traffic(workload, kernel, src_files):
    """DRAM bytes per launch from the committed ncu summary, or None when absent or when the
    kernel's source changed since the capture."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    h = hashlib.sha256()
    for f in src_files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    sha = h.hexdigest()[:16]
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == workload and parts[1] == kernel:
            return float(parts[2]) if parts[3] == sha else None
    return None


class ClockSampler:
    """nvidia-smi clock/throttle samples of this process's GPU while running."""
    Q = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.uuid = str(getattr(torch.cuda.get_device_properties(device), "uuid", "")).lower()
        self.proc = None
        self.out = ""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            if self.uuid and self.uuid.replace("gpu-", "") not in f[0].lower():
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[4:8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- oracle legs

def oracle_prepare(name, gen_device):
    """The oracle's inputs for one token of every layer of the workload (its first input batch):
    x, logits and the oracle-quantized weights of the groups that token uses (set-up, untimed)."""
    import concurrent.futures as cf

    import oracle
    w = synth.WORKLOADS[name]
    prepared = []
    for T, seed in workload_entries(name):
        shape = w.shape(T)
        x = synth.activations(T, w.H, seed, 0, w.outlier_frac, device=gen_device).cpu()
        lg = synth.router_logits(T, w.E, seed, 0, w.logit_bias, device=gen_device).cpu()
        ids, _ = oracle.route(lg, w.k)
        groups = sorted(set(ids[0].tolist()) | {w.E})
        G = w.E + 1
        packs = []
        for proj, (N, K) in (("gate_up", (2 * w.I, w.H)), ("down", (w.H, w.I))):
            P_ = np.zeros((G, N, K // 2), np.uint8)
            S_ = np.zeros((G, N, K // 16), np.uint8)
            Z_ = np.zeros((G,), np.float32)

            def one(g):
                return g, oracle.quantize(synth.projection_weights(shape, seed, 0, proj, [g], device=gen_device).cpu().numpy())
            with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
                for g, (p, s, z) in ex.map(one, groups):
                    P_[g], S_[g], Z_[g] = p[0], s[0], z[0]
            packs.append((P_, S_, Z_))
        prepared.append((x, lg, packs[0], packs[1]))

    def run_once():
        for x, lg, gu, dn in prepared:
            oracle.moe_forward(x, lg, gu, dn, w.k, tokens=[0])
        return len(prepared)
    return run_once


def oracle_sample(name, gen_device, budget_s=8.0, max_reps=8):
    """Time the CPU oracle on one token of every layer of the workload, repeated within a
    bounded budget."""
    run_once = oracle_prepare(name, gen_device)
    run_once()  # warm
    t0 = time.perf_counter()
    toks, reps = 0, 0
    while reps < max_reps and (reps == 0 or time.perf_counter() - t0 < budget_s):
        toks += run_once()
        reps += 1
    dt = time.perf_counter() - t0
    return {"value": toks / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{toks} tokens: token 0 of each of the {toks // reps} layer(s) of the workload, "
                      f"{reps} repetition(s); fp64 C++ oracle with std::thread over its work items"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return 0
    name = HEADLINE if args.workload == "all" else args.workload
    steps = args.steps if args.steps is not None else 20
    warmup = args.warmup if args.warmup is not None else 3
    gen = "cuda" if torch.cuda.is_available() else "cpu"
    run_once = oracle_prepare(name, gen)
    for _ in range(warmup):
        run_once()
    t0 = time.perf_counter()
    toks = 0
    for _ in range(steps):
        toks += run_once()
    dt = time.perf_counter() - t0
    value = toks / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": warmup, "ms_per_step": 1e3 * dt / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": describe(name),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"each step: token 0 of each of the {len(workload_entries(name))} "
                                       "layer(s) of the workload through the fp64 oracle"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- our arm

def build_layer(moe, w, T, seed, pool, device):
    shape = w.shape(T)
    ms = moe.Shape(T=T, H=w.H, I=w.I, E=w.E, k=w.k, has_shared=1)
    G = w.E + 1
    weights = []
    for proj, (N, K) in (("gate_up", (2 * w.I, w.H)), ("down", (w.H, w.I))):
        packed = torch.empty(G, N, K // 2, dtype=torch.uint8, device=device)
        scales = torch.empty(G, N, K // 16, dtype=torch.uint8, device=device)
        scale2 = torch.empty(G, dtype=torch.float32, device=device)
        for g0 in range(0, G, 32):
            gs = list(range(g0, min(G, g0 + 32)))
            q = moe.quantize_nvfp4(synth.projection_weights(shape, seed, 0, proj, gs, device=device))
            packed[g0:g0 + len(gs)], scales[g0:g0 + len(gs)], scale2[g0:g0 + len(gs)] = q.packed, q.scales, q.scale2
        weights.append(moe.NVFP4Weights(packed, scales, scale2))
    xs = [synth.activations(T, w.H, seed, p, w.outlier_frac, device=device) for p in range(pool)]
    lgs = [synth.router_logits(T, w.E, seed, p, w.logit_bias, device=device) for p in range(pool)]
    ws = moe.workspace(ms, device=device)
    out = torch.empty(T, w.H, dtype=torch.bfloat16, device=device)
    # distinct routed experts of every input batch, from the library's own route/permute
    uniq = []
    for p in range(pool):
        ids, _ = moe.route_topk(lgs[p], ms)
        counts, *_ = moe.permute(ids, ms, ws)
        uniq.append(int((counts > 0).sum().item()))
    return dict(T=T, ms=ms, gu=weights[0], dn=weights[1], xs=xs, lgs=lgs, ws=ws, out=out, uniq=uniq)


def launches_per_forward(arm, T):
    """Kernels one moe_forward launches: arm 0 one; arm 1 route+permute, gate_up, down+combine;
    arm 2 route+permute (one cooperative kernel; up to 64 tokens the top-k, then permutation and
    gather in one kernel) and the expert-ordered f16 copy of x, gate_up, the f16 copy of h, down,
    combine; arm 3 route+permute, gate_up, down, combine."""
    return {0: 1, 1: 3, 2: 6, 3: 4}[arm]


def measure(moe, name, steps, warmup, pool, device, dist, world, warmup_seconds, cpu_baseline):
    """Time `steps` steps of workload `name` and return its part of the JSON line."""
    w = synth.WORKLOADS[name]
    layers = [build_layer(moe, w, T, seed, pool, device) for T, seed in workload_entries(name)]
    tokens_per_step = sum(L["T"] for L in layers)
    arms = [moe.forward_arm(L["ms"]) for L in layers]
    launches = sum(launches_per_forward(a, L["T"]) for a, L in zip(arms, layers))
    stream = torch.cuda.Stream(device)

    # events[p][layer]: the 5 stage events of one profiled step on input batch p
    events = [[[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in layers] for _ in range(pool)]
    with torch.cuda.stream(stream):   # torch creates an event's handle on its first record
        for ev in (e for p in events for L_ in p for e in L_):
            ev.record(stream)
    stream.synchronize()
    with torch.cuda.stream(stream):
        for p in range(pool):  # one eager pass per batch before capture
            for L in layers:
                moe.forward(L["xs"][p], L["lgs"][p], L["gu"], L["dn"], L["ms"], L["ws"], out=L["out"])
    stream.synchronize()
    bad = [moe.device_status(L["ws"]) for L in layers]
    if any(bad):
        raise RuntimeError(f"{name}: device status after the first pass: {bad}")
    # plain graphs (the timed steps) and profiled graphs (event nodes at the stage boundaries,
    # about 2 us each, so they stay out of the timed value; they give the per-stage times)
    graphs, pgraphs = [], []
    for p in range(pool):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for L in layers:
                moe.forward(L["xs"][p], L["lgs"][p], L["gu"], L["dn"], L["ms"], L["ws"], out=L["out"])
        graphs.append(g)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for li, L in enumerate(layers):
                moe.forward_profiled(L["xs"][p], L["lgs"][p], L["gu"], L["dn"], L["ms"], L["ws"], L["out"],
                                     events[p][li])
        pgraphs.append(g)

    H, I, E, k = w.H, w.I, w.E, w.k
    gu_expert = 2 * I * H // 2 + 2 * I * H // 16 + 4
    dn_expert = H * I // 2 + H * I // 16 + 4
    acc = dict(stage=[[0.0] * 4 for _ in layers], gu_bytes=0.0, dn_bytes=0.0, gu_flops=0.0, fwd_bytes=0.0,
               fwd_flops=0.0)

    def collect(p):
        evs = events[p]
        evs[-1][4].synchronize()
        for li, L in enumerate(layers):
            e = evs[li]
            for s in range(4):
                acc["stage"][li][s] += e[s].elapsed_time(e[s + 1])

    def work(p):
        for L in layers:
            T, U = L["T"], L["uniq"][p] + 1
            S = T * k
            acc["gu_bytes"] += U * gu_expert + T * H * 2 + (S + T) * I * 2
            acc["dn_bytes"] += U * dn_expert + (S + T) * I * 2 + T * H * 2 + S * 8
            acc["gu_flops"] += 2.0 * (2 * I) * H * (S + T)
            acc["fwd_flops"] += 2.0 * 3 * I * H * (S + T)
            acc["fwd_bytes"] += U * (gu_expert + dn_expert) + T * H * 2 + T * E * 4 + T * H * 2

    with ClockSampler(device) as clk:
        with torch.cuda.stream(stream):
            t_w = time.perf_counter()
            i = 0
            while i < warmup or time.perf_counter() - t_w < warmup_seconds:
                for p in range(pool):
                    graphs[p].replay()
                    pgraphs[p].replay()
                i += pool
            stream.synchronize()
            if dist:
                dist.barrier()
            stream.synchronize()
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for i in range(steps):
                graphs[i % pool].replay()
            t1.record(stream)
            t1.synchronize()
            if dist:
                dist.barrier()
            # stage times: the same steps again, profiled
            for i in range(steps):
                p = i % pool
                pgraphs[p].replay()
                work(p)
                collect(p)
        stream.synchronize()
    max_ms = slowest_rank_ms(t0.elapsed_time(t1), dist, device)
    ms_per_step = max_ms / steps
    value = replica_throughput(world, steps, tokens_per_step, max_ms)
    n_launch = steps * len(layers)
    tot_stage = [sum(acc["stage"][li][s] for li in range(len(layers))) for s in range(4)]
    pk = peaks()
    src = "quantized_moe_expert_nvfp4_gb300/csrc/"
    # HBM-bound workloads stream the selected experts' weights; the prefill workloads are
    # contractions (tensor-bound).  The dominant kernel: the whole-layer kernel of the one-launch
    # decode arm (timed by the plain graphs: per launch = the step's time / layers), else the
    # stage with the largest time (event-timed in the profiled pass).
    hbm_bound = name in ("decode", "batched", "tiny")
    long_step = ms_per_step * steps > 50.0
    if all(a == 0 for a in arms):
        t_launch_ms = ms_per_step / len(layers)
        alg = acc["fwd_bytes"] / n_launch
        kname, kfile = "decode_fused_kernel", ["decode_fused.cu", "topk.cuh", "internal.cuh", "mma_frag.cuh"]
        roofline = {"bound": "hbm", "achieved": alg / (t_launch_ms / 1e3) / 1e9, "peak": pk["hbm"], "unit": "GB/s",
                    "kernel": kname + " (the whole layer: route, gate_up, down, combine)",
                    "algorithmic_bytes_per_launch": alg, "avg_launch_us": 1e3 * t_launch_ms,
                    "timing": "plain CUDA graphs, the step's time divided by its launches"}
    elif hbm_bound:
        dom = 1 if tot_stage[1] >= tot_stage[2] else 2
        t_launch_ms = tot_stage[dom] / n_launch
        alg = (acc["gu_bytes"] if dom == 1 else acc["dn_bytes"]) / n_launch
        kname = f"grouped_gemm_tc_kernel<{'gate_up' if dom == 1 else 'down'}>" if all(a == 2 for a in arms) \
            else ("grouped_simt_kernel<gate_up>" if dom == 1 else "down_combine_gemv_kernel")
        kfile = ["gemm_tc.cu", "internal.cuh", "mma_frag.cuh"] if all(a == 2 for a in arms) else ["grouped_simt.cu"]
        roofline = {"bound": "hbm", "achieved": alg / (t_launch_ms / 1e3) / 1e9, "peak": pk["hbm"], "unit": "GB/s",
                    "kernel": kname, "algorithmic_bytes_per_launch": alg, "avg_launch_us": 1e3 * t_launch_ms,
                    "timing": "CUDA events around the kernel on its stream (profiled replay of the timed steps)"}
    else:
        t_launch_ms = tot_stage[1] / n_launch
        alg = acc["gu_flops"] / n_launch
        kname = "grouped_gemm_tc_kernel<gate_up>" if all(a == 2 for a in arms) else "grouped_simt_kernel<gate_up>"
        kfile = ["gemm_tc.cu", "internal.cuh", "mma_frag.cuh"]
        peak = pk["bf16_sustained"] if long_step else pk["bf16"]
        roofline = {"bound": "tensor", "achieved": alg / (t_launch_ms / 1e3) / 1e12, "peak": peak,
                    "unit": "TFLOP/s", "kernel": kname, "algorithmic_flops_per_launch": alg,
                    "avg_launch_us": 1e3 * t_launch_ms,
                    "timing": "CUDA events around the kernel on its stream (profiled replay of the timed steps)"}
    roofline["frac"] = roofline["achieved"] / roofline["peak"]
    roofline["peak_source"] = pk["source"] + (" (sustained)" if roofline["bound"] == "tensor" and long_step else
                                              " (burst)" if roofline["bound"] == "tensor" else "")
    roofline["traffic"] = stored_traffic(name, kname, [src + f for f in kfile])
    # the whole layer against the same roofline, from the plain timing
    if roofline["bound"] == "hbm":
        layer_ach = acc["fwd_bytes"] / steps / (ms_per_step / 1e3) / 1e9
        layer = {"achieved": layer_ach, "unit": "GB/s", "frac": layer_ach / pk["hbm"],
                 "algorithmic_bytes_per_step": acc["fwd_bytes"] / steps}
    else:
        layer_ach = acc["fwd_flops"] / steps / (ms_per_step / 1e3) / 1e12
        layer = {"achieved": layer_ach, "unit": "TFLOP/s", "frac": layer_ach / roofline["peak"],
                 "algorithmic_flops_per_step": acc["fwd_flops"] / steps}

    # the layer from x alone: the router GEMM (NVFP4 router weights) in front of the same layer,
    # timed the same way, and the router GEMM by itself
    for L in layers:
        L["rw"] = moe.quantize_nvfp4(synth.router_weights(w.shape(L["T"]), 17, device=device))
        L["rlog"] = torch.empty(L["T"], E, dtype=torch.float32, device=device)
    rgraphs, rogs = [], []
    for p in range(pool):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for L in layers:
                moe.forward_routed(L["xs"][p], L["rw"], L["gu"], L["dn"], L["ms"], L["ws"], out=L["out"])
        rgraphs.append(g)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for L in layers:
                moe.router_logits(L["xs"][p], L["rw"], L["ms"], L["ws"], logits=L["rlog"])
        rogs.append(g)
    with torch.cuda.stream(stream):
        for gs in (rgraphs, rogs):
            for p in range(pool):
                gs[p].replay()
        stream.synchronize()
        r0, r1, r2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        r0.record(stream)
        for i in range(steps):
            rgraphs[i % pool].replay()
        r1.record(stream)
        for i in range(steps):
            rogs[i % pool].replay()
        r2.record(stream)
        r2.synchronize()
    routed_ms = slowest_rank_ms(r0.elapsed_time(r1), dist, device) / steps
    router_ms = slowest_rank_ms(r1.elapsed_time(r2), dist, device) / steps
    with_router = {"value": replica_throughput(world, 1, tokens_per_step, routed_ms), "unit": UNIT,
                   "ms_per_step": routed_ms, "router_us_per_layer": 1e3 * router_ms / len(layers),
                   "what": "moe_forward_routed: logits = x . deq(W_r)^T (NVFP4 router, E x H) computed in front of "
                           "the same layer, timed like the headline steps; router_us_per_layer: the router GEMM alone"}
    del rgraphs, rogs

    # the FP8-activation arm (its own numerics: e4m3 weights re-quantized once, e4m3 activation
    # rows with fp32 scales), timed the same way on the same inputs
    fp8_arm = None
    if all(a == 2 for a in arms) and not hbm_bound:
        for L in layers:
            L["gu8"], L["dn8"] = moe.prepare_fp8(L["gu"]), moe.prepare_fp8(L["dn"])
        fgraphs = []
        for p in range(pool):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for L in layers:
                    moe.forward_fp8(L["xs"][p], L["lgs"][p], L["gu8"], L["dn8"], L["ms"], L["ws"], out=L["out"])
            fgraphs.append(g)
        with torch.cuda.stream(stream):
            for p in range(pool):
                fgraphs[p].replay()
            stream.synchronize()
            f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            f0.record(stream)
            for i in range(steps):
                fgraphs[i % pool].replay()
            f1.record(stream)
            f1.synchronize()
        fp8_ms = slowest_rank_ms(f0.elapsed_time(f1), dist, device) / steps
        fp8_peak = 2.0 * roofline["peak"]
        fl = acc["fwd_flops"] / steps
        fp8_arm = {"value": replica_throughput(world, 1, tokens_per_step, fp8_ms), "unit": UNIT,
                   "ms_per_step": fp8_ms,
                   "layer_roofline": {"bound": "tensor", "achieved": fl / (fp8_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                                      "peak": fp8_peak, "frac": fl / (fp8_ms / 1e3) / 1e12 / fp8_peak,
                                      "peak_source": roofline["peak_source"] + " x 2 (nominal fp8 / bf16 ratio)"},
                   "numerics": "e4m3 x e4m3 tcgen05 (kind::f8f6f4): weights re-quantized to e4m3 per row at load, "
                               "x and h rows quantized to e4m3 with one fp32 scale each, fp32 accumulation and epilogue",
                   "what": "moe_forward_fp8 on the same inputs, timed like the headline steps"}
        for L in layers:
            del L["gu8"], L["dn8"]
        del fgraphs

    # the per-expert register arm inside the tcgen05 grouped GEMMs (expert groups of at most 8
    # token rows on mma.sync in the same launch), timed the same way; the headline steps keep the
    # library default (every item on tcgen05)
    register_arm = None
    if all(a == 2 for a in arms):
        share = []
        for L in layers:
            ids = torch.topk(L["lgs"][0], w.k, dim=1).indices.reshape(-1)
            cnt = torch.bincount(ids, minlength=E).tolist() + ([L["T"]] if w.shape(L["T"]).has_shared else [])
            tile = 64 if L["T"] <= moe.DECODE_MAX_T else 128
            rows = [min(c - i, tile) for c in cnt for i in range(0, c, tile)]
            share.append(sum(r <= 8 for r in rows) / max(len(rows), 1))
        moe.set_narrow_rows(8)
        try:
            ngraphs = []
            for p in range(pool):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for L in layers:
                        moe.forward(L["xs"][p], L["lgs"][p], L["gu"], L["dn"], L["ms"], L["ws"], out=L["out"])
                ngraphs.append(g)
        finally:
            moe.set_narrow_rows(-1)
        with torch.cuda.stream(stream):
            for p in range(pool):
                ngraphs[p].replay()
            stream.synchronize()
            n0, n1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            n0.record(stream)
            for i in range(steps):
                ngraphs[i % pool].replay()
            n1.record(stream)
            n1.synchronize()
        nar_ms = slowest_rank_ms(n0.elapsed_time(n1), dist, device) / steps
        register_arm = {"value": replica_throughput(world, 1, tokens_per_step, nar_ms), "unit": UNIT,
                        "ms_per_step": nar_ms, "narrow_rows": 8,
                        "narrow_item_share": [round(x, 3) for x in share],
                        "what": "moe_forward with moe_set_narrow_rows(8): work items of at most 8 token rows run on "
                                "the dequant warps' mma.sync register arm inside the same tcgen05 launch, timed like "
                                "the headline steps (the headline keeps every item on tcgen05)"}
        del ngraphs

    # end to end through host buffers: every step copies its inputs in from pinned host memory,
    # runs the C-ABI calls and copies the results back to pinned memory, all inside the timed
    # region.  When a step moves more than 64 MB (the long prefill) every layer call copies its x
    # and logits in and its output out on their own streams (the copies in of call n+1 and out of
    # call n-1 overlap call n; device buffers double-buffered per layer); otherwise the whole step's
    # inputs (every layer's x and logits, back to back in one pinned buffer) move in one copy and
    # its outputs in one copy, on their own streams: the copy in of step n+1 and the copy out of
    # step n-1 overlap step n's calls (device buffers double-buffered per step), with fewer host
    # calls per step than the per-layer form (a 64-token layer's calls take microseconds).
    e2e_steps = min(steps, 200)
    step_bytes = sum(L["T"] * (2 * H * 2 + E * 4) for L in layers)
    overlap = step_bytes > (64 << 20)   # per-layer copies
    if overlap:
        hx = [[L["xs"][p].cpu().pin_memory() for p in range(pool)] for L in layers]
        hl = [[L["lgs"][p].cpu().pin_memory() for p in range(pool)] for L in layers]
        ho = [[torch.empty(L["T"], H, dtype=torch.bfloat16).pin_memory() for _ in range(2)] for L in layers]
        dx = [[torch.empty_like(L["xs"][0]) for _ in range(2)] for L in layers]
        dl = [[torch.empty_like(L["lgs"][0]) for _ in range(2)] for L in layers]
        do = [[torch.empty_like(L["out"]) for _ in range(2)] for L in layers]
    else:
        # one pinned buffer per pooled batch: every layer's x, then its logits, back to back
        xb = [L["T"] * H * 2 for L in layers]
        lb = [L["T"] * E * 4 for L in layers]
        ob = [L["T"] * H * 2 for L in layers]
        in_off = [sum(xb[:i]) + sum(lb[:i]) for i in range(len(layers))]
        out_off = [sum(ob[:i]) for i in range(len(layers))]
        hin = []
        for p in range(pool):
            buf = torch.empty(sum(xb) + sum(lb), dtype=torch.uint8).pin_memory()
            for li, L in enumerate(layers):
                buf[in_off[li]:in_off[li] + xb[li]].copy_(L["xs"][p].cpu().view(torch.uint8).reshape(-1))
                buf[in_off[li] + xb[li]:in_off[li] + xb[li] + lb[li]].copy_(L["lgs"][p].cpu().view(torch.uint8).reshape(-1))
            hin.append(buf)
        hout = [torch.empty(sum(ob), dtype=torch.uint8).pin_memory() for _ in range(2)]
        din = [torch.empty(sum(xb) + sum(lb), dtype=torch.uint8, device=device) for _ in range(2)]
        dout = [torch.empty(sum(ob), dtype=torch.uint8, device=device) for _ in range(2)]
        dviews = [[(din[b][in_off[li]:in_off[li] + xb[li]].view(torch.bfloat16).view(L["T"], H),
                    din[b][in_off[li] + xb[li]:in_off[li] + xb[li] + lb[li]].view(torch.float32).view(L["T"], E),
                    dout[b][out_off[li]:out_off[li] + ob[li]].view(torch.bfloat16).view(L["T"], H))
                   for li, L in enumerate(layers)] for b in range(2)]
    h2d_s, d2h_s = torch.cuda.Stream(device), torch.cuda.Stream(device)
    in_ready = [[torch.cuda.Event() for _ in range(2)] for _ in layers]
    done = [[torch.cuda.Event() for _ in range(2)] for _ in layers]
    out_read = [[torch.cuda.Event() for _ in range(2)] for _ in layers]

    def e2e_step(i):
        p, b = i % pool, i % 2
        if not overlap:
            with torch.cuda.stream(h2d_s):
                h2d_s.wait_event(done[0][b])          # the step two back has read these inputs
                din[b].copy_(hin[p], non_blocking=True)
                in_ready[0][b].record(h2d_s)
            with torch.cuda.stream(stream):
                stream.wait_event(in_ready[0][b])
                stream.wait_event(out_read[0][b])     # its outputs have been copied out
                for (x, lg, out), L in zip(dviews[b], layers):
                    moe.forward(x, lg, L["gu"], L["dn"], L["ms"], L["ws"], out=out)
                done[0][b].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(done[0][b])
                hout[b].copy_(dout[b], non_blocking=True)
                out_read[0][b].record(d2h_s)
            return
        for li, L in enumerate(layers):
            with torch.cuda.stream(h2d_s):
                if overlap:
                    h2d_s.wait_event(done[li][b])      # the call two steps back has read these buffers
                dx[li][b].copy_(hx[li][p], non_blocking=True)
                dl[li][b].copy_(hl[li][p], non_blocking=True)
                if overlap:
                    in_ready[li][b].record(h2d_s)
            with torch.cuda.stream(stream):
                if overlap:
                    stream.wait_event(in_ready[li][b])
                    stream.wait_event(out_read[li][b])  # its output buffer has been copied out
                moe.forward(dx[li][b], dl[li][b], L["gu"], L["dn"], L["ms"], L["ws"], out=do[li][b])
                if overlap:
                    done[li][b].record(stream)
            with torch.cuda.stream(d2h_s):
                if overlap:
                    d2h_s.wait_event(done[li][b])
                ho[li][b].copy_(do[li][b], non_blocking=True)
                if overlap:
                    out_read[li][b].record(d2h_s)

    for i in range(2):   # untimed: the buffers' first use
        e2e_step(i)
    torch.cuda.synchronize(device)
    if dist:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(h2d_s)
    for i in range(e2e_steps):
        e2e_step(i)
    d2h_s.wait_stream(stream)
    d2h_s.wait_stream(h2d_s)
    e1.record(d2h_s)
    e1.synchronize()
    e2e_ms = slowest_rank_ms(e0.elapsed_time(e1), dist, device)
    h2d = sum(L["T"] * H * 2 + L["T"] * E * 4 for L in layers)
    d2h = sum(L["T"] * H * 2 for L in layers)
    e2e = {"value": replica_throughput(world, e2e_steps, tokens_per_step, e2e_ms), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "method": ("moe_forward per layer call with pinned-host x/logits copied in and the output copied out "
                      "every call; copies on their own streams overlap the neighbouring calls' compute" if overlap else
                      "moe_forward per layer call; every step's inputs (every layer's x and logits) copied in from "
                      "pinned host memory in one copy and its outputs copied out in one copy, on their own streams, "
                      "overlapping the neighbouring steps' calls")}
    torch.cuda.synchronize(device)

    status = [moe.device_status(L["ws"]) for L in layers]
    if any(status):
        raise RuntimeError(f"{name}: device status {status}")
    stage_names = (["whole layer (one launch)", "-", "-", "-"] if all(a == 0 for a in arms)
                   else ["route+permute+x gather", "gate_up GEMM", "h conversion+down GEMM", "combine"]
                   if all(a == 2 for a in arms) else ["route+permute", "gate_up", "down", "combine"])
    res = {"value": value, "unit": UNIT, "steps": steps, "warmup": warmup, "ms_per_step": ms_per_step,
           "config": describe(name), "roofline": roofline, "layer_roofline": layer, "e2e": e2e,
           "with_router": with_router,
           "fp8_arm": fp8_arm,
           "register_arm": register_arm,
           "gpu_launches": steps * launches, "clocks": clk.summary(),
           "arm": sorted({moe.ARM_NAMES[a] for a in arms}),
           "method": {"l2": "inputs larger than L2: every layer's NVFP4 weights (907 MB) resident, a fresh input "
                            f"batch each step ({pool} batches cycled), experts differ per step",
                      "cuda_graphs": True, "timed": "CUDA events on the launching stream around the plain graphs"},
           "stages_us_per_forward": {f"layer {li} (T={L['T']})": {stage_names[s]: round(1e3 * acc["stage"][li][s] / steps, 2)
                                                                   for s in range(4) if stage_names[s] != "-"}
                                     for li, L in enumerate(layers)},
           "distinct_experts_mean": [float(np.mean(L["uniq"])) for L in layers]}
    if cpu_baseline:
        res["cpu_baseline"] = oracle_sample(name, device)
    del layers, graphs, pgraphs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def run_ours(args):
    import quantized_moe_expert_nvfp4_gb300 as moe
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    moe.load()
    head = HEADLINE if args.workload == "all" else args.workload
    if args.one_forward is not None:   # for ncu: -s 3 -c 1 on the arm's kernel selects the fourth forward
        w = synth.WORKLOADS[head]
        T, seed = workload_entries(head)[args.one_forward]
        L = build_layer(moe, w, T, seed, 1, device)
        if args.fp8:
            gu8, dn8 = moe.prepare_fp8(L["gu"]), moe.prepare_fp8(L["dn"])
        for _ in range(4):
            if args.fp8:
                moe.forward_fp8(L["xs"][0], L["lgs"][0], gu8, dn8, L["ms"], L["ws"], out=L["out"])
            else:
                moe.forward(L["xs"][0], L["lgs"][0], L["gu"], L["dn"], L["ms"], L["ws"], out=L["out"])
        torch.cuda.synchronize()
        if moe.device_status(L["ws"]) != 0:
            raise RuntimeError(f"device status {moe.device_status(L['ws'])}")
        print(f"one forward: {head} layer {args.one_forward} (T={T}), arm {moe.forward_arm(L['ms'])}")
        return 0
    cpu = world == 1 and not args.no_cpu_baseline and rank == 0

    def run(name, steps_arg):
        d_steps, d_warm, d_pool = DEFAULTS[name]
        steps = steps_arg if steps_arg is not None else d_steps
        warmup = max(3, args.warmup if args.warmup is not None else d_warm)
        return measure(moe, name, steps, warmup, args.pool or d_pool, device, dist, world,
                       args.warmup_seconds, cpu)

    subs = {}
    if args.workload == "all":
        for name in SUBWORKLOADS:   # each with its own default step count (reported in its entry)
            subs[name] = run(name, None)
    main = run(head, args.steps)
    if rank == 0:
        line = {"metric": METRIC, "value": main["value"], "unit": UNIT, "n_gpus": world, "steps": main["steps"],
                "warmup": main["warmup"], "ms_per_step": main["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": DTYPE, "data": "synthetic",
                "config": main["config"], "roofline": main["roofline"], "e2e": main["e2e"],
                "gpu_launches": main["gpu_launches"], "clocks": main["clocks"],
                "parallelism": f"replicas x{world}"}
        for key in ("cpu_baseline", "layer_roofline", "with_router", "fp8_arm", "register_arm", "arm", "method", "stages_us_per_forward",
                    "distinct_experts_mean"):
            if key in main:
                line[key] = main[key]
        if subs:
            line["workloads"] = subs
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
