#!/usr/bin/env python
"""Benchmark of the quantized MoE decode layer step on GB300.

Metric: decode tokens/s per MoE layer step (one token through one layer),
and the expert GEMVs' HBM GB/s against the measured peak.

Default workload (one GPU): the single-token decode layer -- dim 4096, inter
2048, 384 routed experts (Q2_K gate/up, Q3_K down, all resident in one HBM
arena), top 6, bf16 router and bf16 shared expert -- stacked as 8 independent
layers captured in one CUDA graph. A step is one replay: one token through the
8 layers (865 MB of distinct weights, far above the 129 MB L2, so nothing is
served from L2 between steps); the steps take 64 distinct tokens in turn, so
the picks change from step to step. value = token-layer steps per second over
all ranks.

Other workloads (--workload): batch8 (the same layers at m = 8 tokens),
decode_kq (the default workload with a K-quant shared expert: Q2_K w1/w3,
Q3_K w2), chain40 (40 stacked layers, one token, one replay = one 40-layer
decode step; tokens/s), prefill (512 tokens through one layer on the tensor-core arm,
correction bias ~U(-1, 1); tokens/s).

--impl reference times the CPU oracle (oracle/, plain C, f64) on the same
workload and metric: each step one token through one layer, on the host cores.

Multi-GPU: replicas only (the decode step does not shard here); under
torchrun every rank runs its own replica, the time is the max over ranks and
value = all ranks' units / that time.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_HBM_GBS = 6800.0

WORKLOADS = {
    # name: (m, layers per step, metric, unit)
    "decode": (1, 8, "decode tokens/s per MoE layer step (1 GB300)", "token-layer steps/s"),
    "batch8": (8, 8, "decode tokens/s per MoE layer step (1 GB300), m=8", "token-layer steps/s"),
    "decode_kq": (1, 8, "decode tokens/s per MoE layer step (1 GB300), K-quant shared expert", "token-layer steps/s"),
    "chain40": (1, 40, "decode tokens/s, 40-layer MoE decode step (1 GB300)", "tokens/s"),
    # the batched (prefill) arm: 512 tokens through one layer, expert load
    # skewed by a correction bias ~U(-1, 1)
    "prefill": (512, 1, "prefill tokens/s through one MoE layer, 512 tokens (1 GB300)", "tokens/s"),
}


NX = 64  # distinct tokens the timed steps rotate through


def decode_cfg(m, n_routed=384):
    import moe_decode_quantized_gb300 as moe
    return moe.Config(dim=4096, inter=2048, n_routed=n_routed, topk=6, norm_topk_prob=True, max_tokens=m,
                      gate_temp=1.0, route_scale=2.5, swiglu_limit=7.0)


# ------------------------------------------------------------------ distributed helpers

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def aggregate(units: float, seconds: float, world: int):
    """(total units over ranks, max seconds over ranks) -- replicas: no data-path collective."""
    if world <= 1:
        return units, seconds
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    s = torch.tensor([seconds], dtype=torch.float64, device=dev)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    dist.all_reduce(s, op=dist.ReduceOp.MAX)
    return float(u.item()), float(s.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) while the GPU works."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.lines = []
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        out, _ = self.p.communicate(timeout=10)
        rows = []
        for line in out.splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 8:
                continue
            try:
                rows.append((float(f[0]), float(f[1]), f[4:8]))
            except ValueError:
                continue
        if not rows:
            return None
        smax = max(r[1] for r in rows)
        busy = [r for r in rows if r[0] >= 0.5 * smax] or rows
        sm = sorted(r[0] for r in busy)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i, v in enumerate(r[2]) if v.lower().startswith("active")})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": smax, "reasons": reasons, "samples": len(busy)}


# ------------------------------------------------------------------ bytes (algorithmic)

def algorithmic_bytes(cfg, m, ne, shared_kquant=False):
    """Bytes one layer step must move, per kernel (router, gate/up, down)."""
    dim, inter, n, k = cfg.dim, cfg.inter, cfg.n_routed, cfg.topk
    q2 = inter * (dim // 256) * 84
    q3 = dim * (inter // 256) * 110
    router = n * dim * 2 + m * dim * 2 + m * n * 4
    # gate/up: routed Q2_K gate+up, the whole shared expert (bf16 W1, W3, W2,
    # or Q2_K W1, W3 and Q3_K W2), x; writes g, u, h, gs, us, hs (bf16, or f32
    # to be quantised to q8_1 for the Q3_K W2) and sd
    shared = 2 * q2 + q3 if shared_kquant else 3 * inter * dim * 2
    gateup = 2 * ne * q2 + shared + m * dim * 2 + 3 * m * k * inter * 4 \
        + m * inter * (4 + 4 + (4 if shared_kquant else 2)) + m * dim * 4
    # down: routed Q3_K down, h of the plan; writes down rows; reads sd and the
    # residual, writes acc, the residual and x_next
    down = ne * q3 + m * k * inter * 4 + m * k * dim * 4 + m * dim * (4 + 4 + 4 + 4 + 2)
    return router, gateup, down


def kernel_hash():
    """Hash of the kernel sources with comments and blank lines removed, so
    that the committed ncu counts stay valid across comment-only edits (no
    string literal in these sources holds a comment marker)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "moe_decode_quantized_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")) and f != "moe_synth.cu":
            src = open(os.path.join(csrc, f), encoding="utf-8").read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            src = re.sub(r"//[^\n]*", "", src)
            code = "\n".join(line.rstrip() for line in src.splitlines() if line.strip())
            h.update(code.encode())
    return h.hexdigest()[:16]


def measured_traffic(kernel):
    """Per-launch DRAM bytes of one kernel ("router", "gateup", "down") from the
    committed ncu summary, or None when it has none or the kernels changed since."""
    try:
        t = json.load(open(TRAFFIC))
    except (OSError, ValueError):
        return None
    return t.get(f"{kernel}_dram_bytes_per_launch") if t.get("kernel_hash") == kernel_hash() else None


def hbm_peak():
    try:
        return float(json.load(open(PEAKS))["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ CPU oracle (baseline leg)

def oracle_sample(cfg, m, budget_s, seed=1000, max_steps=10 ** 9, warmup=0, bias_range=(-0.1, 0.1),
                  shared_kquant=False):
    """The oracle as it stands, on host cores: one layer step per iteration over
    the same synthetic decode layer. Returns (steps, seconds, threads, sample text)."""
    import numpy as np
    import oracle
    from moe_decode_quantized_gb300 import synth

    threads = os.cpu_count() or 1
    shp = synth.LayerShape(cfg.dim, cfg.inter, cfg.n_routed)
    oc = oracle.cfg(cfg.dim, cfg.inter, cfg.n_routed, cfg.topk, cfg.norm_topk_prob, cfg.gate_temp,
                    cfg.route_scale, cfg.swiglu_limit)
    router = synth.router_bf16(seed, 0, cfg.n_routed, cfg.dim)
    bias = synth.bias_f32(seed, 0, cfg.n_routed, *bias_range)
    if shared_kquant:
        img = np.frombuffer(synth.expert_bytes(seed, 0, synth.SHARED_KQ_INDEX, shp), np.uint8)
        shared = (img[shp.gate_off:shp.gate_off + shp.gate_bytes], img[shp.up_off:shp.up_off + shp.up_bytes],
                  img[shp.down_off:shp.down_off + shp.down_bytes])
    else:
        shared = synth.shared_bf16(seed, 0, cfg.dim, cfg.inter)
    cache = {}
    done, spent, i = 0, 0.0, 0
    while done < max_steps and (spent < budget_s or done == 0):
        x = synth.x_bf16(seed, i, m, cfg.dim)
        picks, _, _, _ = oracle.route(oc, oracle.router_logits(x, router), bias)
        experts = {}
        for e in np.unique(picks):
            e = int(e)
            if e not in cache:
                if len(cache) > 64:
                    cache.pop(next(iter(cache)))
                cache[e] = synth.expert_bytes(seed, 0, e, shp)
            experts[e] = cache[e]
        t0 = time.perf_counter()
        oracle.layer(oc, x, router, bias, experts, (shp.gate_off, shp.up_off, shp.down_off), shared,
                     threads=threads, shared_kquant=shared_kquant)
        dt = time.perf_counter() - t0
        i += 1
        if i <= warmup:
            continue
        spent += dt
        done += 1
    sample = (f"{done} layer steps of {m} tokens through the decode layer (dim {cfg.dim}, inter {cfg.inter}, "
              f"{cfg.n_routed}x{cfg.topk}, {'K-quant' if shared_kquant else 'bf16'} shared expert, bias U{bias_range}), "
              f"oracle.layer timed, {threads} threads")
    return done, spent, threads, sample


# ------------------------------------------------------------------ our arm

def run_ours(args):
    import numpy as np
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    from moe_decode_quantized_gb300 import build as mbuild
    mbuild.build()
    import moe_decode_quantized_gb300 as moe
    from moe_decode_quantized_gb300.workload import Workload, x_tensor

    m, L, metric, unit = WORKLOADS[args.workload]
    if args.layers:
        L = args.layers
    cfg = decode_cfg(m, args.experts)
    kq = args.workload == "decode_kq"
    wl = Workload(cfg, n_layers=L, seed=rank, shared=True, shared_kquant=kq)
    layers = [wl.layer(l) for l in range(L)]
    x_a = x_tensor(rank, 0, m, cfg.dim)
    x_b = torch.empty_like(x_a)
    residual = torch.zeros((m, cfg.dim), dtype=torch.float32, device="cuda")
    hw = moe.header_words(cfg, m)
    headers = torch.zeros(L * hw, dtype=torch.int32, device="cuda")
    graph = moe.Graph(cfg, layers, wl.arena, m, x_a, x_b, residual, headers, wl.ws)
    stream = torch.cuda.current_stream()
    # the steps rotate through NX distinct tokens held on the device: step i
    # copies token i % NX into the graph's input and zeroes the residual before
    # the replay (the synthetic layers carry no normalisation, so a residual
    # carried from step to step would grow without bound), so routing and the
    # picked slots vary from step to step
    xs = torch.stack([x_tensor(rank, 1000 + i, m, cfg.dim) for i in range(NX)])
    it = [0]

    def step():
        x_a.copy_(xs[it[0] % NX])
        it[0] += 1
        residual.zero_()
        graph.launch()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak:  # clocks settle under load
        for _ in range(50):
            step()
        torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    ms = ev0.elapsed_time(ev1)
    status = moe.read_status(wl.ws)
    if status:
        raise RuntimeError(f"workspace status {status:#x} after the timed region")
    # decode / batch8: token-layer steps; chain40: tokens through the whole stack
    units_local = float(args.steps * m * (1 if args.workload == "chain40" else L))
    units, secs = aggregate(units_local, ms / 1e3, world)
    value = units / secs

    # distinct experts per layer step (for the algorithmic bytes): from the headers
    h = headers.cpu().numpy()
    po = m * (1 + 3 * cfg.topk)
    ne_list = [int(h[l * hw + po]) for l in range(L)]
    ne = float(np.mean(ne_list))

    # e2e: the same replays through the host-buffer C-ABI call (pinned buffers,
    # H2D of the token's x and residual, D2H of x, residual and the headers),
    # the tokens rotating through the same NX rows, here in host memory
    xhs = xs.cpu().pin_memory()
    rh = torch.zeros_like(residual, device="cpu").pin_memory()
    xo = torch.empty_like(xhs[0]).pin_memory()
    ro = torch.empty_like(rh).pin_memory()
    hh = torch.zeros(L * hw, dtype=torch.int32).pin_memory()
    for i in range(max(1, args.warmup)):
        graph.launch_host(xhs[i % NX], rh, xo, ro, hh)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(stream)
    for i in range(args.steps):
        graph.launch_host(xhs[i % NX], rh, xo, ro, hh)
    e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier(world)
    e_units, e_secs = aggregate(units_local, max(e0.elapsed_time(e1) / 1e3, wall), world)
    h2d = xo.numel() * xo.element_size() + rh.numel() * rh.element_size()
    d2h = h2d + hh.numel() * 4

    # per-kernel durations (router+select, gate/up, down) with CUDA events on the
    # launching stream, kernels not overlapped, layers rotating (cold L2)
    xp = x_tensor(rank, 7, m, cfg.dim)
    xq = torch.empty_like(xp)
    rp = torch.zeros_like(residual)
    hp = torch.zeros(hw, dtype=torch.int32, device="cuda")
    reps = max(2, min(16, args.steps // L + 1))
    kms = []
    xp0 = xp.clone()
    for r in range(reps + 1):
        xp.copy_(xp0)  # a new token each round through the layers
        rp.zero_()
        for l in range(L):
            t = moe.layer_step_profiled(cfg, layers[l], wl.arena, xp, rp, xq, hp, m, wl.ws)
            xp, xq = xq, xp
            if r > 0:
                kms.append(t)
    kms = np.array(kms, np.float64)
    k_ms = kms.mean(axis=0)
    b_router, b_gateup, b_down = algorithmic_bytes(cfg, m, ne, kq)
    peak, peak_kind = hbm_peak()
    # the roofline of the kernel with the largest measured time
    names = ["router", "gateup", "down"]
    dom = int(np.argmax(k_ms))
    b_dom = (b_router, b_gateup, b_down)[dom]
    achieved = b_dom / (k_ms[dom] * 1e-3) / 1e9
    expert_gbs = (b_gateup + b_down) / ((k_ms[1] + k_ms[2]) * 1e-3) / 1e9

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        n, spent, thr, sample = oracle_sample(cfg, m, args.cpu_budget, shared_kquant=kq)
        cu = n * m / spent
        if args.workload == "chain40":
            cu = cu / L
        cpu = {"value": cu, "unit": unit, "cores": thr, "kind": "oracle", "sample": sample}

    if rank == 0:
        layer_bytes = b_router + b_gateup + b_down
        sh_text = "Q2_K/Q3_K shared expert" if kq else "bf16 shared expert"
        out = {
            "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "q2_k/q3_k x q8_1 int8 dot (dp4a) + bf16, f32 accumulate",
            "data": "synthetic (seeded SplitMix64: random Q2_K/Q3_K blocks, bf16 ~N(0,0.02) router"
                    + (", random Q2_K/Q3_K shared expert" if kq else " and shared expert") + ", x ~N(0,1))",
            "config": {
                "workload": f"{args.workload}: MoE decode layer dim 4096, inter 2048, {cfg.n_routed} routed experts top 6 "
                            f"(Q2_K gate/up, Q3_K down), bf16 router + {sh_text}, m={m}",
                "layers_per_step": L, "tokens_per_layer_step": m, "graph": "CUDA graph, PDL-chained kernels",
                "token": f"{NX} distinct tokens in turn: step i copies token i % {NX} (resident on the device) "
                         "into the graph's input and zeroes the residual inside the timed region (two copies a step)",
                "l2": f"inputs larger than L2: {L} distinct layers, {L * layer_bytes / 1e6:.0f} MB per step",
                "parallelism": f"replicas x{world}",
                "distinct_experts_per_layer_step": ne,
                "us_per_layer_step": ms * 1e3 / (args.steps * L),
                "layer_step_algorithmic_bytes": layer_bytes,
                "layer_step_roofline_frac_of_measured": (layer_bytes / (ms * 1e-3 / (args.steps * L)) / 1e9) / peak,
            },
            "roofline": {"bound": "hbm", "kernel": f"moe_{names[dom]}_kernel", "achieved": achieved, "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                         # the committed DRAM counts are per launch of the one-token step
                         # with the bf16 shared expert
                         "traffic": measured_traffic(names[dom]) if m == 1 and not kq else None,
                         "algorithmic_bytes": b_dom,
                         "avg_launch_us": k_ms[dom] * 1e3,
                         "timing": "per-kernel CUDA events on the launching stream, kernels launched one at a "
                                   "time over the workload's layers after the timed region"},
            "kernels_us": {"router_select": k_ms[0] * 1e3, "gateup": k_ms[1] * 1e3, "down": k_ms[2] * 1e3},
            "expert_gemv_gbs": expert_gbs, "expert_gemv_frac": expert_gbs / peak,
            "e2e": {"value": e_units / e_secs, "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps * L * 3,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(out))
    graph.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------ the prefill arm

PREFILL_BIAS = (-1.0, 1.0)
PREFILL_STAGES = ["router", "select_plan", "xhat_gather", "gate", "up", "swiglu_q8", "down", "shared", "finish"]


def run_prefill(args):
    import numpy as np
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    from moe_decode_quantized_gb300 import build as mbuild
    mbuild.build()
    import moe_decode_quantized_gb300 as moe
    from moe_decode_quantized_gb300.workload import Workload, x_tensor

    m, _, metric, unit = WORKLOADS["prefill"]
    cfg = decode_cfg(1, args.experts)
    wl = Workload(cfg, n_layers=1, seed=rank, shared=True, bias_range=PREFILL_BIAS)
    nb = 4  # distinct batches the steps take in turn
    xs = torch.stack([x_tensor(rank, 3000 + i, m, cfg.dim) for i in range(nb)])
    res = torch.zeros((m, cfg.dim), dtype=torch.float32, device="cuda")
    xn = torch.empty_like(xs[0])
    picks = torch.zeros((m, cfg.topk), dtype=torch.int32, device="cuda")
    weights = torch.zeros((m, cfg.topk), dtype=torch.float32, device="cuda")
    ws = torch.empty(moe.prefill_workspace_bytes(cfg, m), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    it = [0]

    def step():
        res.zero_()
        moe.prefill_step(cfg, wl.layer(0), wl.arena, cfg.n_routed, xs[it[0] % nb], res, xn, picks, weights, m, ws)
        it[0] += 1

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak:
        for _ in range(10):
            step()
        torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    ms = ev0.elapsed_time(ev1)
    if moe.prefill_status(cfg, m, ws):
        raise RuntimeError("prefill status set after the timed region")
    units, secs = aggregate(float(args.steps * m), ms / 1e3, world)

    # stages with CUDA events on the launching stream, the batches in turn
    st = np.mean([moe.prefill_step_profiled(cfg, wl.layer(0), wl.arena, cfg.n_routed, xs[i % nb], res, xn,
                                            picks, weights, m, ws) for i in range(2 * nb)], axis=0)
    used = len(np.unique(picks.cpu().numpy()))
    dim, inter, P = cfg.dim, cfg.inter, m * cfg.topk
    q2 = inter * (dim // 256) * 84
    q3 = dim * (inter // 256) * 110
    # algorithmic bytes and flops of the three routed GEMMs: the picked
    # experts' blocks once, the group rows (fp16 hi + lo for gate / up) once,
    # the outputs once; flops of the products the layer defines
    gemm_bytes = {"gate": used * q2 + P * dim * 4 + P * inter * 4, "up": used * q2 + P * dim * 4 + P * inter * 4,
                  "down": used * q3 + P * inter * 2 + P * dim * 4}
    gemm_flops = {"gate": 2.0 * P * inter * dim, "up": 2.0 * P * inter * dim, "down": 2.0 * P * dim * inter}
    idx = {n: i for i, n in enumerate(PREFILL_STAGES)}
    st = [float(v) for v in st]
    dom = max(gemm_bytes, key=lambda n: st[idx[n]])
    dur = st[idx[dom]] * 1e-3
    peak, peak_kind = hbm_peak()
    achieved = gemm_bytes[dom] / dur / 1e9
    try:
        bf16_peak = float(json.load(open(PEAKS))["bf16_tflops"])
    except (OSError, ValueError, KeyError):
        bf16_peak = 1900.0

    # e2e: x from pinned host memory in, the residual back, every step
    xh = xs.cpu().pin_memory()
    rh = torch.empty_like(res, device="cpu").pin_memory()
    xd = torch.empty_like(xs[0])
    for i in range(max(1, args.warmup)):
        xd.copy_(xh[i % nb], non_blocking=True)
        res.zero_()
        moe.prefill_step(cfg, wl.layer(0), wl.arena, cfg.n_routed, xd, res, xn, picks, weights, m, ws)
        rh.copy_(res, non_blocking=True)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(stream)
    for i in range(args.steps):
        xd.copy_(xh[i % nb], non_blocking=True)
        res.zero_()
        moe.prefill_step(cfg, wl.layer(0), wl.arena, cfg.n_routed, xd, res, xn, picks, weights, m, ws)
        rh.copy_(res, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier(world)
    e_units, e_secs = aggregate(float(args.steps * m), max(e0.elapsed_time(e1) / 1e3, wall), world)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        n, spent, thr, sample = oracle_sample(cfg, 4, args.cpu_budget, bias_range=PREFILL_BIAS)
        cpu = {"value": n * 4 / spent, "unit": unit, "cores": thr, "kind": "oracle", "sample": sample}

    if rank == 0:
        out = {
            "metric": metric, "value": units / secs, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16 router / shared GEMMs; routed Q2_K / Q3_K dequantised to fp16 (gate / up as hi + lo "
                     "pairs), f32 accumulate in TMEM",
            "data": "synthetic (seeded SplitMix64: random Q2_K/Q3_K blocks, bf16 ~N(0,0.02) router and shared "
                    "expert, x ~N(0,1), correction bias ~U(-1,1))",
            "config": {
                "workload": f"prefill: {m} tokens through one MoE layer (dim 4096, inter 2048, {cfg.n_routed} "
                            "routed experts top 6, Q2_K gate/up, Q3_K down, bf16 router + bf16 shared expert)",
                "tokens_per_step": m, "batches": f"{nb} distinct batches in turn",
                "experts_read_per_step": used,
                "l2": f"inputs larger than L2: {used} experts' blocks ({used * (2 * q2 + q3) / 1e6:.0f} MB) "
                      "plus the 50 MB shared expert per step",
                "parallelism": f"replicas x{world}",
                "stages_us": {n: float(v * 1e3) for n, v in zip(PREFILL_STAGES, st)},
            },
            "roofline": {"bound": "hbm", "kernel": f"moe_tc_gemm ({dom})", "achieved": achieved, "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak, "traffic": None,
                         "algorithmic_bytes": gemm_bytes[dom], "avg_launch_us": dur * 1e6,
                         "tensor_tflops": gemm_flops[dom] / dur / 1e12,
                         "tensor_frac_of_bf16_peak": gemm_flops[dom] / dur / 1e12 / bf16_peak,
                         "timing": "CUDA events between the prefill stages on the launching stream"},
            "e2e": {"value": e_units / e_secs, "unit": unit, "h2d_bytes_per_step": m * cfg.dim * 2,
                    "d2h_bytes_per_step": m * cfg.dim * 4},
            "gpu_launches": args.steps * 17,  # router, scores, top-k, plan, x_hat, 2 gathers, gate, up, SwiGLU, down, 3 shared GEMMs, its SwiGLU, finish
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------ reference arm (the oracle)

REF_CAP_S = 120.0  # seconds of oracle time at most (the timed steps stop there)

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return  # under torchrun only rank 0 runs the CPU reference
    m, L, metric, unit = WORKLOADS[args.workload]
    cfg = decode_cfg(m)
    bias = (-0.1, 0.1)
    if args.workload == "prefill":  # each step a bounded sample: 4 of the 512 tokens
        m, bias = 4, PREFILL_BIAS
    # K steps after W warm-up steps, unless the oracle's time passes REF_CAP_S
    # first: "steps" is the number timed
    n, spent, thr, sample = oracle_sample(cfg, m, budget_s=REF_CAP_S, max_steps=args.steps,
                                          warmup=args.warmup, bias_range=bias,
                                          shared_kquant=args.workload == "decode_kq")
    value = n * m / spent
    if args.workload == "chain40":
        value = value / (args.layers or L)
    out = {
        "impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": world,
        "steps": n, "steps_requested": args.steps, "warmup": args.warmup, "ms_per_step": spent * 1e3 / max(1, n),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same seeded generator as the GPU arm)",
        "config": {"workload": f"{args.workload}: the CPU oracle, one layer step per step, m={m}",
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": unit, "cores": thr, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decode")
    ap.add_argument("--layers", type=int, default=0, help="layers per step (default: the workload's)")
    ap.add_argument("--experts", type=int, default=384, help="routed experts per layer (384; fewer only for profiling)")
    ap.add_argument("--soak", type=float, default=1.0, help="seconds of untimed load before timing")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "prefill":
        run_prefill(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
