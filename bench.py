#!/usr/bin/env python
"""Throughput of the latent MoE layer on B300: one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole layer (router, top-k, permutation, W_in,
expert SwiGLU, weighted group reduce, W_out, combine) over one batch of
synthetic seeded tokens of the named workload (default: the Edge0-shaped
layer at a decode / speculative-verify batch of 8 tokens). Weights are
rotated over several device copies so that no step finds its weights in L2.
value = tokens/s over the device-timed region (CUDA events, max over ranks);
e2e = the same through lmoe_layer_forward_host (pinned host buffers, copies
in the timed region). --impl reference times the CPU oracle instead.
Multi-GPU: independent replicas (no collective), one process per GPU.
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

METRIC = "MoE-layer tokens/s at decode batch 8 and 16K prefill; % HBM / tensor roofline"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="decode_t8")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--copies", type=int, default=0, help="device weight copies rotated across steps (0: auto)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="decode_t8 only: skip the 16K-prefill sub-record")
    ap.add_argument("--passes", type=int, default=0,
                    help="for profilers: build one weight copy of --workload, run N plain forwards, no timing")
    ap.add_argument("--sweep", action="store_true",
                    help="decode / speculative-verify sweep: one JSON line per batch T = 1..16 of the Edge0 layer")
    return ap.parse_args()


# ------------------------------------------------------------- distributed

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def dist_init(world, use_cuda):
    if world <= 1:
        return None
    import torch.distributed as dist
    dist.init_process_group(backend="nccl" if use_cuda else "gloo")
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, v: float, device=None) -> float:
    if dist is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.th.join(timeout=2)
        sm = [float(r[0]) for r in self.rows if len(r) >= 8 and r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if len(r) >= 8 and r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in self.rows:
            if len(r) >= 8:
                for n, v in zip(names, r[4:8]):
                    if v.lower() == "active":
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------- roofline bits

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6400.0), d.get("bf16_tflops", 1800.0), d.get("bf16_tflops_sustained", 1400.0), "measured"
    return 6400.0, 1800.0, 1400.0, "fallback"


def stage_bytes(sh, T, idx):
    """Algorithmic HBM bytes of each decode-path kernel for one pass: every
    weight byte the routing needs, read once (int4 + bf16 scales = 9/16 byte
    per weight), plus activations in and out."""
    import numpy as np
    epg = sh.E // sh.G
    experts = np.unique(idx.reshape(-1))
    groups = np.unique(experts // epg)
    wq = 0.5 + 2.0 / 32  # bytes per int4 weight including its scale
    b = {}
    b["route"] = 4 * sh.d * sh.E + 2 * T * sh.d + (4 * sh.E if sh.has_bias else 0)
    b["win"] = len(groups) * sh.L * sh.d * wq + 2 * T * sh.d
    b["gateup"] = len(experts) * 2 * sh.f * sh.L * wq
    b["down"] = len(experts) * sh.L * sh.f * wq
    b["wout"] = len(groups) * sh.d * sh.L * wq + 2 * T * sh.d
    b["decode_fused"] = sum(b.values())
    if sh.lora_rank:
        # the LoRA matrices of the routed groups; around the single-kernel pass
        # the branch runs in its own kernels (lora_p: A_in, lora_hl: B_in,
        # lora_q: A_out, lora_out: B_out), in the multi-kernel sequence
        # lora_p / lora_q and the B matrices beside W_in / W_out
        r = sh.lora_rank
        b["lora_p"] = len(groups) * sh.d * r * 2
        b["lora_hl"] = len(groups) * r * sh.L * 2
        b["lora_q"] = len(groups) * sh.L * r * 2
        b["lora_out"] = len(groups) * r * sh.d * 2 + 2 * T * sh.d
        b["win_lora"] = len(groups) * r * sh.L * 2
        b["wout_lora"] = len(groups) * r * sh.d * 2
    return b


def step_bytes(sb):
    """Algorithmic bytes of one pass from stage_bytes: the layer's own stages
    plus, with LoRA, the branch's matrices counted once."""
    base = sum(sb[n] for n in ("route", "win", "gateup", "down", "wout"))
    if "lora_hl" in sb:
        base += sb["lora_p"] + sb["lora_hl"] + sb["lora_q"] + sb["wout_lora"]
    return base


def stage_flops(sh, T, idx):
    """Algorithmic flops of each prefill-path kernel (the group-factored
    minimum: W_in and W_out once per distinct (group, token), the router in
    fp32-equivalent multiply-adds)."""
    import numpy as np
    epg = sh.E // sh.G
    rows = int(sum(len(np.unique(np.nonzero((idx // epg == g).any(axis=1))[0])) for g in range(sh.G)))
    f = {}
    f["route"] = 2.0 * T * sh.d * sh.E
    f["win"] = 2.0 * sh.d * sh.L * rows
    f["gateup"] = 2.0 * 2 * sh.L * sh.f * T * sh.k
    f["down"] = 2.0 * sh.f * sh.L * T * sh.k
    f["wout"] = 2.0 * sh.L * sh.d * rows
    if sh.lora_rank:
        # Recover-LoRA: P = x . A_in for every (group, token) that uses the
        # group, Q = Z . A_out, and the rank-r K blocks of W_in and W_out
        r = sh.lora_rank
        f["lora_p"] = 2.0 * sh.d * r * rows
        f["lora_q"] = 2.0 * sh.L * r * rows
        f["win"] += 2.0 * r * sh.L * rows
        f["wout"] += 2.0 * r * sh.d * rows
    f["permute"] = 0.0
    f["zreduce"] = 0.0
    f["dequant"] = 0.0
    f["tsort"] = 0.0
    return f, rows


def source_sha(files) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def read_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of a kernel on a workload, from the committed ncu
    summary table profiles/traffic.txt, if the sources the counters were taken
    on are unchanged; else None. Table rows: kernel, workload, bytes per
    launch, comma-separated source files, sha256 prefix of those sources."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    for line in open(p):
        f = line.split("#", 1)[0].split()
        if len(f) != 5 or f[0] != kernel or f[1] != workload:
            continue
        try:
            if source_sha(f[3].split(",")) != f[4]:
                return None
            return float(f[2])
        except OSError:
            return None
    return None


# ------------------------------------------------------------------ oracle

def oracle_tokens_per_s(name: str, budget_s: float = 12.0, tokens=None):
    import lmoe_synth as S
    import oracle as O
    sh, T, W, x = S.make_workload(name)
    Ly = O.Layer(sh, W)
    sel = x if tokens is None else x[tokens]
    n = 0
    t0 = time.perf_counter()
    reps = 0
    while True:
        O.layer_forward(Ly, sel)
        n += sel.shape[0]
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return n / dt, reps, sel.shape[0]


def run_reference(args):
    rank, local, world = dist_env()
    if rank != 0:
        return
    import lmoe_synth as S
    import oracle as O
    stacks = {**S.STACK_WORKLOADS, **{n: v[:4] for n, v in S.STAGED_STACK_WORKLOADS.items()}}
    if args.workload in stacks:  # one token through one layer per step; value over the whole stack
        sh, nl, T, xseed = stacks[args.workload]
        Ly = O.Layer(sh, S.make_stack_layer(sh, 0))
        x = S.make_x(1, sh.d, xseed)
        for _ in range(max(args.warmup, 0)):
            O.layer_forward(Ly, x)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            O.layer_forward(Ly, x)
        dt = time.perf_counter() - t0
        value = args.steps / dt / nl
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * dt / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": args.workload, "layers": nl, "T": T},
                "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                 "sample": f"one token through one of the {nl} layers per step"},
                "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    sh, T, W, x = S.make_workload(args.workload)
    Ly = O.Layer(sh, W)
    for i in range(max(args.warmup, 0)):
        O.layer_forward(Ly, x[i % T:i % T + 1])
    t0 = time.perf_counter()
    for i in range(args.steps):
        O.layer_forward(Ly, x[i % T:i % T + 1])
    dt = time.perf_counter() - t0
    value = args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": args.workload, "tokens_per_step": 1, "T": T},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"one token of {args.workload} per step (full layer, literal per-assignment form)"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------- ours

def measure_layer(args, workload, local, dev, dist, world, steps, warmup, copies=0, cpu_baseline=True):
    """One workload of the single-layer path: device-timed K graph replays,
    per-kernel event timing, roofline of the dominant kernel, e2e through the
    host-buffer entry point. Returns the JSON fields of its line."""
    import numpy as np
    import torch

    import lmoe_synth as S
    from sparse_latent_moe_lmoe_b300 import LatentMoE, capi
    from sparse_latent_moe_lmoe_b300.layer import to_device

    sh, T, W, x = S.make_workload(workload)
    if copies <= 0:  # enough distinct weight copies that a step never finds its weights in L2
        copies = 8 if T <= 16 else 2
    base = {n: to_device(W.get(n), dev) for n in capi.WEIGHT_FIELDS}
    wcopies = [base] + [{n: (None if t is None else t.clone()) for n, t in base.items()} for _ in range(copies - 1)]
    layers = [LatentMoE(sh, c, device=local) for c in wcopies]
    xt = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    y = torch.empty_like(xt)
    stream = torch.cuda.current_stream()
    for m in layers:
        m.workspace(T, host_staging=True)
    idx, _, _ = layers[0].route(xt)
    idx_np = idx.cpu().numpy()
    sb = stage_bytes(sh, T, idx_np)
    n_kernels = capi.lmoe_stage_name(layers[0].h, T, 0)[1]
    prefill = capi.lmoe_stage_name(layers[0].h, T, 1)[0] == "permute"

    # one CUDA graph per weight copy: a replay launches the whole layer
    for i, m in enumerate(layers):
        m.forward(xt, out=y)
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    graphs = []
    for m in layers:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            m.forward(xt, out=y)
        graphs.append(g)
    torch.cuda.synchronize()

    def step(i):
        graphs[i % len(graphs)].replay()

    for i in range(max(warmup, 3)):
        step(i)
    torch.cuda.synchronize()

    # ---- clocks: sampled over >= 1 s of identical replays that ends with the
    # timed region (a timed region of a few ms is shorter than one sample)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    t_end = time.perf_counter() + 1.0
    n_window = 0
    while time.perf_counter() < t_end:
        for _ in range(50):
            step(n_window)
            n_window += 1
        torch.cuda.synchronize()

    # ---- timed region: K steps, device time
    barrier(dist)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    ms = e0.elapsed_time(e1)
    ck = clocks.stop()
    if ck is not None:
        ck["window"] = f"{n_window} untimed replays (>= 1 s) immediately before the {steps} timed steps"
    ms = max_over_ranks(dist, ms, dev)
    value = world * T * steps / (ms / 1000.0)

    # ---- per-kernel durations: the same graphs with an event pair captured
    # around every kernel launch (on the launching stream), replayed; each
    # kernel's time is the median over the replays
    import ctypes
    names = [capi.lmoe_stage_name(layers[0].h, T, i)[0] for i in range(n_kernels)]
    samples = {n: [] for n in names}
    pgraphs = []
    for m in layers:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_kernels)]
        for e in ev:  # torch creates the CUDA event on first record
            e.record(stream)
        torch.cuda.synchronize()
        arr = (ctypes.c_void_p * (2 * n_kernels))(*[e.cuda_event for e in ev])
        capi.lmoe_set_stage_events(m.h, arr, n_kernels)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            m.forward(xt, out=y)
        capi.lmoe_set_stage_events(m.h, None, 0)
        pgraphs.append((g, ev))
    torch.cuda.synchronize()
    n_rep = max(steps, 50)
    try:
        for i in range(n_rep):
            g, ev = pgraphs[i % len(pgraphs)]
            g.replay()
            torch.cuda.synchronize()
            for j, n in enumerate(names):
                samples[n].append(ev[2 * j].elapsed_time(ev[2 * j + 1]))
        stage_timing = f"graph replay, event pair around each kernel, median of {n_rep} replays"
    except Exception:  # event nodes not timeable here: time stream launches instead
        samples = {n: [] for n in names}
        for i in range(n_rep):
            m = layers[i % len(layers)]
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_kernels)]
            for e in ev:
                e.record(stream)
            arr = (ctypes.c_void_p * (2 * n_kernels))(*[e.cuda_event for e in ev])
            capi.lmoe_set_stage_events(m.h, arr, n_kernels)
            m.forward(xt, out=y)
            capi.lmoe_set_stage_events(m.h, None, 0)
            torch.cuda.synchronize()
            for j, n in enumerate(names):
                samples[n].append(ev[2 * j].elapsed_time(ev[2 * j + 1]))
        stage_timing = f"stream launches, event pair around each kernel, median of {n_rep} launches"
    # per stage: the median over replays of one launch, times its launches per step
    per = {n: statistics.median(v) * names.count(n) for n, v in samples.items()}
    dom = max(per, key=per.get)
    hbm, bf16, bf16s, peak_src = measured_peaks()
    step_s = ms / steps * 1e-3
    if prefill:
        sf, rows = stage_flops(sh, T, idx_np)
        achieved = sf.get(dom, 0.0) / (per[dom] * 1e-3) / 1e12
        total = sum(sf.values())
        # each kernel is timed on its own and the whole step lasts milliseconds:
        # the burst peak is the denominator; the sustained one is given beside it
        roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": bf16, "unit": "TFLOP/s",
                    "frac": achieved / bf16, "traffic": read_traffic(dom, workload),
                    "peak_source": peak_src + " bf16 burst (dense cuBLAS GEMM)",
                    "frac_of_sustained_peak": achieved / bf16s, "sustained_peak": bf16s,
                    "flops_per_launch": sf.get(dom, 0.0), "timing": stage_timing,
                    "step": {"flops": total, "achieved": total / step_s / 1e12,
                             "frac": total / step_s / 1e12 / bf16,
                             "frac_of_sustained_peak": total / step_s / 1e12 / bf16s,
                             "group_token_rows": rows}}
    else:
        achieved = sb.get(dom, 0.0) / (per[dom] * 1e-3) / 1e9
        total_bytes = step_bytes(sb)
        roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                    "frac": achieved / hbm, "traffic": read_traffic(dom, workload), "peak_source": peak_src,
                    "bytes_per_launch": sb.get(dom, 0.0), "timing": stage_timing,
                    "step": {"bytes": total_bytes, "achieved": total_bytes / step_s / 1e9,
                             "frac": total_bytes / step_s / 1e9 / hbm}}

    # ---- e2e through the host-buffer entry point
    xh = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    # warm-up: every rotating handle once (each keeps its call as a CUDA graph), at least 3 calls
    for i in range(max(3, len(layers))):
        layers[i % len(layers)].forward_host(xh, yh)
    barrier(dist)
    t0 = time.perf_counter()
    for i in range(steps):
        layers[i % len(layers)].forward_host(xh, yh)
    t1 = time.perf_counter()
    e2e_s = max_over_ranks(dist, t1 - t0, dev)
    e2e = {"value": world * T * steps / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": T * sh.d * 2,
           "d2h_bytes_per_step": T * sh.d * 2}
    line = {"value": value, "unit": "tokens/s", "ms_per_step": ms / steps,
            "config": {"workload": workload, "T": T, "d": sh.d, "E": sh.E, "G": sh.G, "k": sh.k, "L": sh.L,
                       "f": sh.f, "lora_rank": sh.lora_rank, "parallelism": f"replicas x{world}",
                       "l2": f"{copies} rotating device weight copies (> L2)",
                       "distinct_experts": int(len(np.unique(idx_np))),
                       "active_groups": int(len(np.unique(idx_np // (sh.E // sh.G))))},
            "roofline": roofline, "stages_us": {n: 1000 * v for n, v in per.items()},
            "e2e": e2e, "gpu_launches": capi.lmoe_launch_count(layers[0].h, T) * steps, "clocks": ck}
    rank = dist_env()[0]
    if cpu_baseline and rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, reps, n = oracle_tokens_per_s(workload)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                "sample": f"all {n} tokens of {workload}, full layer, repeated {reps}x"}
    for m in layers:
        m.close()
    del layers, wcopies, base, graphs, pgraphs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return line


def run_ours(args):
    import torch

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = dist_init(world, True)
    main = measure_layer(args, args.workload, local, dev, dist, world, args.steps, args.warmup, args.copies)
    line = {"metric": METRIC, "value": main.pop("value"), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": main.pop("ms_per_step"), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": ("nvfp4" if args.workload.endswith("_nvfp4") else "int4")
            + " weights, fp16 tensor-core operands, fp32 accumulate",
            "data": "synthetic"}
    line.update(main)
    # the metric's second half: the 16K-token prefill, in the same run
    if args.workload == "decode_t8" and not args.no_prefill:
        pf = measure_layer(args, "prefill_t16384_zipf", local, dev, dist, world, args.steps, args.warmup, 0,
                           cpu_baseline=False)
        line["prefill"] = pf
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ------------------------------------------------------------------- stack

def run_stack(args):
    """A stack of layers (x_{l+1} = bf16(x_l + bf16(layer_l(x_l)))), each
    layer with its own weights (13 GB for 48 Edge0 layers, far beyond L2, so
    no rotation is needed). A step is one pass of T tokens through all
    layers; value = T / step time."""
    import numpy as np
    import torch

    import lmoe_synth as S
    from sparse_latent_moe_lmoe_b300 import LatentMoE, LatentMoEStack, capi

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = dist_init(world, True)
    sh, nl, T, xseed = S.STACK_WORKLOADS[args.workload]
    t0 = time.perf_counter()
    layers = []
    for l in range(nl):
        W = S.make_stack_layer(sh, l)
        layers.append(LatentMoE(sh, W, device=local))
        del W
    gen_s = time.perf_counter() - t0
    stack = LatentMoEStack(layers)
    x = S.make_x(T, sh.d, xseed)
    xt = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    y = torch.empty_like(xt)
    stack.workspace(T)
    # the algorithmic work of this input, layer by layer on the stack's own chain
    decode = T <= 16
    total_bytes = total_flops = 0.0
    int4_bytes = 0.0
    cur = xt
    for m in layers:
        idx, _, _ = m.route(cur)
        idx_np = idx.cpu().numpy()
        sb = stage_bytes(sh, T, idx_np)
        total_bytes += step_bytes(sb)
        int4_bytes += sum(v for n, v in sb.items() if n in ("win", "gateup", "down", "wout")) - 4 * T * sh.d
        sf, _ = stage_flops(sh, T, idx_np)
        total_flops += sum(sf.values())
        yl = m.forward(cur)
        cur = (cur.float() + yl.float()).to(torch.bfloat16)
    per_layer = capi.lmoe_launch_count(layers[0].h, T)
    stack.forward(xt, out=y)
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        stack.forward(xt, out=y)
    torch.cuda.synchronize()
    for _ in range(max(args.warmup, 3)):
        g.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(dist)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    ms = max_over_ranks(dist, e0.elapsed_time(e1), dev)
    ck = clocks.stop()
    step_s = ms / args.steps / 1000.0
    value = world * T / step_s
    hbm, bf16, bf16s, peak_src = measured_peaks()
    if decode:
        achieved = total_bytes / step_s / 1e9
        roofline = {"bound": "hbm", "kernel": "stack", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                    "frac": achieved / hbm, "traffic": None, "peak_source": peak_src,
                    "bytes_per_launch": total_bytes, "timing": "graph replay of the whole stack"}
    else:
        achieved = total_flops / step_s / 1e12
        roofline = {"bound": "tensor", "kernel": "stack", "achieved": achieved, "peak": bf16s, "unit": "TFLOP/s",
                    "frac": achieved / bf16s, "traffic": None,
                    "peak_source": peak_src + " bf16 sustained (the stack runs for tens of ms back to back)",
                    "frac_of_burst_peak": achieved / bf16,
                    "flops_per_launch": total_flops, "timing": "graph replay of the whole stack"}
    # end to end: pinned host x in, y out, every step
    xh = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    xd = torch.empty_like(xt)
    for _ in range(2):
        xd.copy_(xh, non_blocking=True)
        stack.forward(xd, out=y)
        yh.copy_(y, non_blocking=True)
    torch.cuda.synchronize()
    n_e2e = max(1, min(args.steps, 20))
    ta = time.perf_counter()
    for _ in range(n_e2e):
        xd.copy_(xh, non_blocking=True)
        stack.forward(xd, out=y)
        yh.copy_(y, non_blocking=True)
        torch.cuda.synchronize()
    e2e_s = max_over_ranks(dist, time.perf_counter() - ta, dev) / n_e2e
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int4 weights, fp16 tensor-core operands, fp32 accumulate",
            "data": "synthetic",
            "config": {"workload": args.workload, "layers": nl, "T": T, "d": sh.d, "E": sh.E, "G": sh.G, "k": sh.k,
                       "L": sh.L, "f": sh.f, "parallelism": f"replicas x{world}",
                       "l2": f"{nl} layers of distinct weights ({nl * 272.6 / 1000:.1f} GB > L2)",
                       "weight_generation_s": round(gen_s, 1)},
            "int4_bytes_per_token": int4_bytes / T, "weight_bytes_per_token": total_bytes / T,
            "roofline": roofline,
            "e2e": {"value": world * T / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": T * sh.d * 2,
                    "d2h_bytes_per_step": T * sh.d * 2},
            "gpu_launches": nl * (per_layer + 1) * args.steps, "clocks": ck}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle as O
        Ly = O.Layer(sh, S.make_stack_layer(sh, 0))
        xt1 = x[:1]
        tb = time.perf_counter()
        cur1 = xt1
        for _ in range(nl):  # the oracle's cost does not depend on the weights: layer 0's reused
            y1, _, _, _ = O.layer_forward(Ly, cur1)
            cur1 = O.residual(cur1, y1)
        cs = time.perf_counter() - tb
        line["cpu_baseline"] = {"value": 1.0 / cs, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                "sample": f"one token through {nl} oracle layer evaluations (layer-0 weights reused)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_staged_stack(args):
    """A stack whose expert weights stay in page-locked host memory, with a
    fixed number of GPU slots per layer: every step routes new tokens, each
    layer stages its routed experts that hold no slot, and the next layer's
    prerouter stages its predicted experts on a second stream meanwhile. One
    CUDA graph per input (the slot tables live on the device and carry over
    from step to step). value = T / step time; the line adds the staging
    counters and the bytes moved over the host link per token."""
    import numpy as np
    import torch

    import lmoe_synth as S
    from sparse_latent_moe_lmoe_b300 import LatentMoE, LatentMoEStack, capi

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = dist_init(world, True)
    sh, nl, T, xseed, slots = S.STAGED_STACK_WORKLOADS[args.workload]
    t0 = time.perf_counter()
    layers = []
    for l in range(nl):
        W = S.make_stack_layer(sh, l)
        layers.append(LatentMoE(sh, W, device=local, flags=capi.FLAG_STAGED_EXPERTS, expert_slots=slots,
                                expert_weights_on_host=True))
        del W
    gen_s = time.perf_counter() - t0
    stack = LatentMoEStack(layers)
    stack.workspace(T)
    n_in = max(args.steps, 1) + max(args.warmup, 3)
    xs = [torch.from_numpy(S.make_x(T, sh.d, 5000 + i).view(np.int16)).to(dev).view(torch.bfloat16)
          for i in range(n_in)]
    y = torch.empty_like(xs[0])
    stack.forward(xs[0], out=y)
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    graphs = []
    for xi in xs:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            stack.forward(xi, out=y)
        graphs.append(g)
    torch.cuda.synchronize()
    nw = max(args.warmup, 3)
    for g in graphs[:nw]:
        g.replay()
    torch.cuda.synchronize()
    before = [m.stage_stats() for m in layers]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(dist)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for g in graphs[nw:nw + args.steps]:
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    ms = max_over_ranks(dist, e0.elapsed_time(e1), dev)
    ck = clocks.stop()
    after = [m.stage_stats() for m in layers]
    d = {k: sum(a[k] - b[k] for a, b in zip(after, before)) for k in after[0]}
    step_s = ms / args.steps / 1000.0
    value = world * T / step_s
    tok = T * args.steps
    staging = {"slots_per_layer": slots, "experts_per_layer": sh.E, "routed_per_token": d["routed"] / tok,
               "hit_rate": d["hits"] / max(d["routed"], 1), "on_demand_per_token": d["staged_on_demand"] / tok,
               "prefetched_per_token": d["prefetched"] / tok, "host_bytes_per_token": d["bytes_copied"] / tok,
               "host_link_gbs": d["bytes_copied"] / (ms / 1000.0) / 1e9,
               "predictor": "the next layer's own router on the current layer's input (a stand-in for a trained head)"}
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": nw, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int4 weights, fp16 tensor-core operands, fp32 accumulate",
            "data": "synthetic",
            "config": {"workload": args.workload, "layers": nl, "T": T, "d": sh.d, "E": sh.E, "G": sh.G, "k": sh.k,
                       "L": sh.L, "f": sh.f, "parallelism": f"replicas x{world}",
                       "inputs": "new tokens every step (one graph per input)",
                       "weight_generation_s": round(gen_s, 1)},
            "staging": staging, "roofline": None, "e2e": None,
            "gpu_launches": nl * (capi.lmoe_launch_count(layers[0].h, T) + 1 + 3) * args.steps, "clocks": ck}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_passes(args):
    """N plain forwards of one weight copy of the workload (the call a bench
    step makes, without graphs or timing): a short, self-contained program
    for ncu captures."""
    import numpy as np
    import torch

    import lmoe_synth as S
    from sparse_latent_moe_lmoe_b300 import LatentMoE

    sh, T, W, x = S.make_workload(args.workload)
    m = LatentMoE(sh, W, device=0)
    xt = torch.from_numpy(x.view(np.int16)).to(torch.device("cuda", 0)).view(torch.bfloat16)
    for _ in range(args.passes):
        m.forward(xt)
    torch.cuda.synchronize()
    m.check()
    print(json.dumps({"passes": args.passes, "workload": args.workload, "ok": True}), flush=True)


def run_sweep(args):
    """Tokens/s and HBM roofline fraction of the decode path at T = 1..16
    (speculative decoding verifies several candidate tokens per weight read):
    one JSON line per T, device time of K graph replays over 8 rotating weight
    copies, the same input recipe as decode_t8 (x drawn for each T)."""
    import numpy as np
    import torch

    import lmoe_synth as S
    from sparse_latent_moe_lmoe_b300 import LatentMoE, capi
    from sparse_latent_moe_lmoe_b300.layer import to_device

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sh, _, W, _ = S.make_workload("decode_t8")
    base = {n: to_device(W.get(n), dev) for n in capi.WEIGHT_FIELDS}
    copies = [base] + [{n: (None if t is None else t.clone()) for n, t in base.items()} for _ in range(7)]
    layers = [LatentMoE(sh, c, device=local) for c in copies]
    hbm = measured_peaks()[0]
    stream = torch.cuda.current_stream()
    cap = torch.cuda.Stream()
    for T in range(1, 17):
        x = S.make_x(T, sh.d, 100 + T)
        xt = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
        y = torch.empty_like(xt)
        for m in layers:
            m.forward(xt, out=y)
        idx, _, _ = layers[0].route(xt)
        sb = stage_bytes(sh, T, idx.cpu().numpy())
        total = step_bytes(sb)
        torch.cuda.synchronize()
        graphs = []
        for m in layers:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                m.forward(xt, out=y)
            graphs.append(g)
        for i in range(max(args.warmup, 3)):
            graphs[i % 8].replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            graphs[i % 8].replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        line = {"mode": "sweep", "workload": f"Edge0 layer, decode T={T}", "T": T, "tokens_per_s": T / (ms * 1e-3),
                "us_per_step": 1000 * ms, "bytes_per_step": total, "achieved_gbs": total / (ms * 1e-3) / 1e9,
                "hbm_frac": total / (ms * 1e-3) / 1e9 / hbm, "distinct_experts": int(len(np.unique(idx.cpu().numpy()))),
                "kernel": capi.lmoe_stage_name(layers[0].h, T, 0)[0], "steps": args.steps}
        if rank == 0:
            print(json.dumps(line), flush=True)
        del graphs


def main():
    args = parse()
    import lmoe_synth as S
    if args.impl == "reference":
        run_reference(args)
    elif args.passes > 0:
        run_passes(args)
    elif args.sweep:
        run_sweep(args)
    elif args.workload in S.STACK_WORKLOADS:
        run_stack(args)
    elif args.workload in S.STAGED_STACK_WORKLOADS:
        run_staged_stack(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
