"""Benchmark of the batched routed-MoE FFN layer on GB300.

One step = one pass of the whole layer (router + softmax/top-k + Q8_1 of x,
CSR bucketing, grouped gate/up/down experts, combine) over one batch of N
synthetic tokens of the OLMoE-shaped layer (N=2048, D=2048, E=64, top_k=8,
F=1024, norm_topk_prob off).  Metric: MoE-FFN prefill tokens/s per layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timing: W untimed warm-up steps, then K steps between a barrier and a
device synchronise on both sides; every step is bracketed by CUDA events on
the launching stream with events between the stages, and the L2 is flushed
(a 512 MB write) between steps outside the events.  Under torchrun each rank
runs its own token batch (replicas, weak scaling) and rank 0 prints the line
with the maximum time over ranks.  With one GPU the line also carries
`configs`: the layer's other workloads (tiny, decode batches of 1/4/8 tokens
with Q8_0 and of 8 tokens with Q4_K weights, the Qwen3-MoE-shaped layer with a
shared expert, the Zipf-skewed long prefill, the OLMoE layer with Q4_K and with
Q3_K experts), each timed the same way after the headline, with its tokens/s,
layer roofline fraction, dominant kernel's fraction and stage times.
--impl reference times the CPU oracle on the host cores on a bounded sample of
the same workload.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mixture_experts_ffn_top_gb300.workloads import QK, Q8_0_BYTES, WORKLOADS, make_hidden, make_inputs, row_bytes  # noqa: E402,F401

METRIC = "MoE-FFN prefill tokens/s/layer, OLMoE shape N=2048; % of int8 tensor peak"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "olmoe"
L2_FLUSH_BYTES = 512 << 20
STAGE_STEPS = 50  # steps of the per-stage breakdown (moe_ffn_prefill_timed)
SMALL_BATCH = 8  # batches the library routes in one launch on the matvec path
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def rank_hidden(wl, hidden0: np.ndarray, rank: int, world: int) -> np.ndarray:
    """The token batch a rank processes: the workload's own batch on a single GPU, an
    independent seeded batch of the same shape per rank when several replicas run."""
    return hidden0 if world == 1 else make_hidden(wl, seed_offset=rank)


def max_over_ranks(x: float, device) -> float:
    """Largest value over the ranks of the default process group (x itself when alone)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, tokens_per_rank: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every rank's batch, over the slowest rank's step time."""
    return world * tokens_per_rank / (ms_per_step / 1e3)


def bind_near_gpu(ops):
    """Move this thread onto the CPUs of the host NUMA node closest to the current GPU (the node
    the device reports), so host memory it allocates and first touches is local to the GPU's
    host link.  Returns (node or None, the previous CPU set or None)."""
    try:
        node = ops.moe_device_host_numa_node()
        with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
            spec = f.read().strip()
    except (OSError, RuntimeError, ValueError):
        return None, None
    if node < 0 or not spec:
        return None, None
    cpus = set()
    for part in spec.split(","):
        lo, _, hi = part.partition("-")
        cpus.update(range(int(lo), int(hi or lo) + 1))
    before = os.sched_getaffinity(0)
    mine = cpus & before
    if not mine:
        return node, None
    os.sched_setaffinity(0, mine)
    return node, before


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def algorithmic_work(wl, topk_idx: np.ndarray | None):
    """Algorithmic bytes and int8 ops of one layer pass: touched experts' weights (in their block
    format, Q8_0 or Q4_K), hidden read once, routerW, (shared expert weights and gate), output written
    once; ops = 2 * MACs."""
    N, D, E, F, Fs, k = wl.N, wl.D, wl.E, wl.F, wl.Fs, wl.top_k
    per_expert = 3 * F * row_bytes(wl.wfmt, D)
    touched = E if topk_idx is None else int(np.unique(topk_idx).size)
    wbytes = touched * per_expert + (3 * Fs * row_bytes(wl.wfmt, D) if Fs else 0)
    bytes_ = wbytes + N * D * 4 + E * D * 4 + (D * 4 if Fs else 0) + N * D * 4
    ops = 2 * N * k * 3 * F * D + (2 * N * 3 * Fs * D if Fs else 0)
    ops_gate_up = 2 * N * k * 2 * F * D + (2 * N * 2 * Fs * D if Fs else 0)  # the gate/up launch alone
    return dict(bytes=bytes_, weight_bytes=wbytes, touched_experts=touched, int8_ops=ops,
                int8_ops_gate_up=ops_gate_up)


class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons) during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def wait_first(self, timeout_s: float = 3.0):
        """Block until nvidia-smi has produced its first sample (it takes a while to start)."""
        t0 = time.perf_counter()
        while self.proc is not None and not self.lines and time.perf_counter() - t0 < timeout_s:
            time.sleep(0.01)

    def stop(self, t_begin: float, t_end: float):
        """Samples taken inside [t_begin, t_end]; for a window shorter than the sampling period,
        the last sample before it and the first after it."""
        if self.proc is None:
            return None
        time.sleep(0.05)  # let one more sample land after the window
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        return clock_summary(self.lines, t_begin, t_end)


def clock_summary(lines, t_begin: float, t_end: float):
    """Median SM clock, max clock and throttle reasons of the (time, csv line) samples taken inside
    [t_begin, t_end]; when none fell inside (a window shorter than the sampling period), the last
    sample before it and the first after it."""
    inside = [ln for t, ln in lines if t_begin <= t <= t_end]
    n_inside = len(inside)
    if not inside:
        inside = [ln for t, ln in lines if t < t_begin][-1:] + [ln for t, ln in lines if t > t_end][:1]
    sm, mx, reasons = [], 0.0, set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for ln in inside:
        parts = [p.strip() for p in ln.split(",")]
        if len(parts) < 8:
            continue
        try:
            sm.append(float(parts[0]))
            mx = max(mx, float(parts[1]))
        except ValueError:
            continue
        for n, v in zip(names, parts[4:8]):
            if v.lower() == "active":
                reasons.add(n)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
            "samples_in_window": n_inside}


def cpu_baseline(wl, inp, sample_tokens: int, min_seconds: float = 10.0, max_passes: int = 20):
    """The oracle, as it stands, on the first `sample_tokens` tokens of the workload (host cores),
    whole layer per pass, repeated until about `min_seconds` of CPU work (bounded by max_passes)."""
    import oracle

    oracle.build()
    sample_tokens = max(1, min(sample_tokens, wl.N))
    sub = dict(inp)
    sub["hidden"] = np.ascontiguousarray(inp["hidden"][:sample_tokens])
    passes, t0 = 0, time.perf_counter()
    while True:
        oracle.moe_ffn_inputs(sub, wl.top_k, wl.norm_topk_prob, keep=False)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or passes >= max_passes:
            break
    return dict(value=passes * sample_tokens / dt, unit=UNIT, cores=oracle.num_threads(), kind="oracle",
                sample=f"{passes} pass(es) over the first {sample_tokens} of {wl.N} tokens of the {wl.name} "
                       f"layer ({wl.describe()}), whole layer per pass, {dt:.2f} s wall")


def run_reference(args, rank, world):
    """--impl reference: the CPU oracle timed on the host cores (rank 0 only)."""
    if rank != 0:
        return
    wl = WORKLOADS[args.workload]
    inp = make_inputs(wl)
    sample = args.ref_tokens
    times = []
    import oracle

    oracle.build()
    for i in range(args.warmup + args.steps):
        sub = dict(inp)
        sub["hidden"] = np.ascontiguousarray(inp["hidden"][:sample])
        t0 = time.perf_counter()
        oracle.moe_ffn_inputs(sub, wl.top_k, wl.norm_topk_prob, keep=False)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    value = sample / (ms / 1e3)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "i8", "data": "synthetic",
            "config": {"workload": f"{wl.name}: {wl.describe()}", "sample_tokens": sample},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"first {sample} of {wl.N} tokens per step, whole layer"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


CONFIG_WORKLOADS = ["tiny", "decode_n1", "decode_n4", "decode_n8", "decode_n8_q4k", "qwen3moe_shared", "skewed",
                    "olmoe_q4k", "olmoe_q3k"]


def resolve_path(ops, w, wl, path):
    """The expert path a moe_ffn_prefill call takes (the library's auto rule)."""
    if path != ops.MOE_PATH_AUTO:
        return path
    tensor = ops.moe_weights_tensor_path(w) and wl.N >= 64 and (wl.N * wl.top_k) // wl.E >= 8
    return ops.MOE_PATH_TENSOR if tensor else ops.MOE_PATH_MATVEC


def router_launches(wl):
    """Launches of the routing of a batch of more than SMALL_BATCH tokens: one on the tensor cores
    (E a multiple of 8, 8 <= E <= 256), else the SIMT logits and softmax."""
    return 1 if (wl.E % 8 == 0 and 8 <= wl.E <= 256) else 2


def launches_per_step(ops, wl, resolved_path):
    experts = 2 * (2 if wl.Fs else 1)  # matvec: gate/up and down, routed (and shared)
    if resolved_path == ops.MOE_PATH_TENSOR:
        return router_launches(wl) + 1 + 3 + 1  # router, bucketing(+plan), gather, gate/up, down, combine
    if wl.N <= SMALL_BATCH:
        return 1 + experts + 1  # routing in one launch, the expert matvecs, combine
    return router_launches(wl) + 1 + experts + 1


def measure(ops, wl, inp, hidden, steps, warmup, path, device, flush, peaks, world=1):
    """One workload's layer: plain moe_ffn_prefill steps between two events (L2 flushed before
    each), then the stage-timed variant; throughput, roofline fractions and stage times."""
    import torch

    layer = ops.MoeLayer.from_numpy(inp, device=device, top_k=wl.top_k, max_tokens=wl.N)
    w, ws, stream = layer.w, layer.ws, torch.cuda.current_stream()
    out = torch.empty((wl.N, wl.D), dtype=torch.float32, device=device)

    def step(ev=None):
        if ev is None:
            ops.moe_ffn_prefill(w, hidden, layer.routerW, layer.shexp_gate, wl.top_k, wl.norm_topk_prob, ws,
                                out=out, path=path)
        else:
            ops.moe_ffn_prefill_timed(w, hidden, layer.routerW, layer.shexp_gate, wl.top_k, wl.norm_topk_prob, ws,
                                      ev, out=out, path=path)

    for _ in range(warmup):
        step()
        flush.fill_(1)
    torch.cuda.synchronize()
    if layer.status():
        raise RuntimeError(f"{wl.name}: device status set during warm-up")
    resolved = resolve_path(ops, w, wl, path)
    topk_idx = layer.views(wl.N)["topk_idx"].cpu().numpy()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for i in range(steps):
        flush.fill_(1)  # before the step's events: every step starts with a cold L2
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    if layer.status():
        raise RuntimeError(f"{wl.name}: device status set during the timed steps")
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    n_stage = min(steps, STAGE_STEPS)
    sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(n_stage)]
    for i in range(n_stage):
        flush.fill_(1)
        step(sevs[i])
    torch.cuda.synchronize()
    if layer.status():
        raise RuntimeError(f"{wl.name}: device status set during the stage-timed steps")
    stage_ms = {s: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in sevs) for j, s in enumerate(ops.PREFILL_STAGES)}
    work = algorithmic_work(wl, topk_idx)
    exp_ms = stage_ms["gate_up"] + stage_ms["down"]
    if resolved == ops.MOE_PATH_TENSOR:
        gu_ms = stage_ms["gate_up"]
        tflops = work["int8_ops_gate_up"] / (gu_ms / 1e3) / 1e12
        peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
        roof = {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                "kernel": "grouped_gemm_kernel gate/up launch (tcgen05 kind::f16 on exact fp16 integers)"}
    else:
        gbs = work["weight_bytes"] / (exp_ms / 1e3) / 1e9
        peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
        roof = {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                "kernel": "grouped expert matvec: gate/up + down launches (dp4a)"}
    layer_roof_s = max(work["int8_ops"] / (peaks.get("bf16_tflops", 1900.0) * 1e12),
                       work["bytes"] / (peaks.get("hbm_gbs", 6800.0) * 1e9))
    res = dict(layer=layer, out=out, step=step, ms=ms, t_wall=t_wall, value=job_throughput(world, wl.N, ms),
               stage_ms=stage_ms, stage_step_ms=statistics.mean(e[0].elapsed_time(e[6]) for e in sevs),
               work=work, roofline=roof, layer_roof_s=layer_roof_s, resolved=resolved, n_stage=n_stage,
               launches=launches_per_step(ops, wl, resolved))
    return res


def config_entry(ops, wl, r):
    """The per-workload record of the bench line."""
    return {"workload": f"{wl.name}: {wl.describe()}", "tokens_per_s": r["value"], "ms_per_step": r["ms"],
            "expert_path": {1: "matvec", 2: "tensor"}[r["resolved"]],
            "layer_roofline_us": r["layer_roof_s"] * 1e6, "layer_roofline_frac": r["layer_roof_s"] / (r["ms"] / 1e3),
            "dominant_kernel": {k: r["roofline"][k] for k in ("kernel", "bound", "achieved", "peak", "unit", "frac")},
            "stage_ms": r["stage_ms"], "algorithmic": r["work"]}


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from mixture_experts_ffn_top_gb300 import ops

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    peaks, peak_src = load_peaks()
    wl = WORKLOADS[args.workload]
    inp = make_inputs(wl)
    inp["hidden"] = rank_hidden(wl, inp["hidden"], rank, world)  # each rank its own token batch
    hidden = torch.from_numpy(inp["hidden"]).to(device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    path = args.path
    stream = torch.cuda.current_stream()
    N, D, k = wl.N, wl.D, wl.top_k

    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    gpu_index = int(vis[local_rank]) if len(vis) > local_rank and vis[local_rank].strip().isdigit() else local_rank
    clocks = ClockSampler(gpu_index)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    clocks.wait_first()
    t_clk0 = time.perf_counter()
    # the headline workload: its timed steps lie inside the clock sampler's window
    head = measure(ops, wl, inp, hidden, args.steps, args.warmup, path, device, flush, peaks, world)
    t_clk1 = time.perf_counter()
    if world > 1:
        dist.barrier()
    clk = clocks.stop(t_clk0, t_clk1)
    ms = max_over_ranks(head["ms"], device)
    value = job_throughput(world, N, ms)
    layer, w, ws = head["layer"], head["layer"].w, head["layer"].ws
    routerW, shg = layer.routerW, layer.shexp_gate
    stage_ms = head["stage_ms"]
    roofline = dict(head["roofline"], peak_source=peak_src,
                    traffic=measured_traffic("gate_up", wl.name) if head["resolved"] == ops.MOE_PATH_TENSOR
                    else TRAFFIC.get(("experts", head["resolved"])))
    head_path, head_work, layer_roof_s = head["resolved"], head["work"], head["layer_roof_s"]
    head_launches, n_stage = head["launches"], head["n_stage"]

    # e2e: the public host-buffer call (moe_ffn_prefill_host) on pinned host memory; the hidden rows
    # come in and the output rows go out over the host link inside the timed region (the router
    # reads them and the combine writes them in place)
    numa_node, cpus0 = bind_near_gpu(ops)  # pinned pages land on the node of the allocating CPU
    h_host = torch.from_numpy(inp["hidden"]).pin_memory()
    o_host = torch.empty((N, D), dtype=torch.float32).pin_memory()
    o_host.zero_()
    if cpus0 is not None:
        os.sched_setaffinity(0, cpus0)

    def e2e_step():
        ops.moe_ffn_prefill_host(w, h_host, routerW, shg, k, wl.norm_topk_prob, ws, o_host, path=path)

    def timed(fn, n):
        out = []
        for _ in range(n):
            flush.fill_(1)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            out.append(e0.elapsed_time(e1))
        return statistics.mean(out)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e2e_mean = max_over_ranks(timed(e2e_step, args.steps), device)
    if layer.status():
        raise RuntimeError("device status set during the e2e steps")

    # the same layer with the residual add fused into its combine (out = residual + FFN(hidden))
    residual = torch.randn((N, D), dtype=torch.float32, device=device, generator=None)
    res_out = torch.empty_like(residual)

    def res_step():
        ops.moe_ffn_prefill_residual(w, hidden, routerW, shg, residual, k, wl.norm_topk_prob, ws, out=res_out,
                                     path=path)

    for _ in range(max(1, args.warmup)):
        res_step()
    res_mean = max_over_ranks(timed(res_step, args.steps), device)
    if layer.status():
        raise RuntimeError("device status set during the residual steps")

    # ... and with the next layer's RMSNorm of that output fused in as well (a second output row)
    gamma = torch.ones(D, dtype=torch.float32, device=device)
    normed = torch.empty_like(residual)

    def norm_step():
        ops.moe_ffn_prefill_residual_rmsnorm(w, hidden, routerW, shg, residual, gamma, 1e-6, k, wl.norm_topk_prob, ws,
                                             out=res_out, normed=normed, path=path)

    for _ in range(max(1, args.warmup)):
        norm_step()
    norm_mean = max_over_ranks(timed(norm_step, args.steps), device)
    if layer.status():
        raise RuntimeError("device status set during the residual + norm steps")

    # two chained layers (hidden <- hidden + FFN_l(hidden), l = 0, 1): the stack entry point, whose
    # second router starts behind the first layer's combine, against two separate residual calls
    from dataclasses import replace as _replace

    inp2 = make_inputs(_replace(wl, seed=wl.seed + 100))
    layer2 = ops.MoeLayer.from_numpy(inp2, device=device, top_k=k, max_tokens=N)
    hs = hidden.clone()

    def stack_step():
        hs.copy_(hidden)
        ops.moe_ffn_prefill_stack([w, layer2.w], [routerW, layer2.routerW], [shg, layer2.shexp_gate], hs, k,
                                  wl.norm_topk_prob, ws, path=path)

    h_a, h_b = hidden.clone(), torch.empty_like(hidden)

    def two_calls_step():
        h_a.copy_(hidden)
        ops.moe_ffn_prefill_residual(w, h_a, routerW, shg, h_a, k, wl.norm_topk_prob, ws, out=h_b, path=path)
        ops.moe_ffn_prefill_residual(layer2.w, h_b, layer2.routerW, layer2.shexp_gate, h_b, k, wl.norm_topk_prob, ws,
                                     out=h_a, path=path)

    for _ in range(max(1, args.warmup)):
        stack_step()
        two_calls_step()
    stack_ms = max_over_ranks(timed(stack_step, args.steps), device)
    two_ms = max_over_ranks(timed(two_calls_step, args.steps), device)
    torch.cuda.synchronize()
    if not torch.equal(hs, h_a):
        raise RuntimeError("the layer stack and two separate calls disagree")

    # the same two layers pre-normed (normed = RMSNorm_0(h); h += FFN_l(normed); the next norm fused
    # into each combine, a final norm after the last layer)
    gam = [gamma, gamma, gamma]
    nrm = torch.empty_like(hidden)

    def stack_norm_step():
        hs.copy_(hidden)
        ops.moe_ffn_prefill_stack_rmsnorm([w, layer2.w], [routerW, layer2.routerW], [shg, layer2.shexp_gate], gam,
                                          1e-6, hs, k, wl.norm_topk_prob, ws, normed=nrm, path=path)

    for _ in range(max(1, args.warmup)):
        stack_norm_step()
    stack_norm_ms = max_over_ranks(timed(stack_norm_step, args.steps), device)
    del layer2
    del head, layer, w, ws, routerW, shg
    torch.cuda.empty_cache()

    # the other workloads, one after another on this GPU, each at the same steps/warm-up
    configs = {}
    if world == 1 and not args.no_configs:
        for name in CONFIG_WORKLOADS:
            if name == wl.name:
                continue
            cwl = WORKLOADS[name]
            cinp = make_inputs(cwl)
            r = measure(ops, cwl, cinp, torch.from_numpy(cinp["hidden"]).to(device), args.steps, args.warmup, path,
                        device, flush, peaks)
            configs[name] = config_entry(ops, cwl, r)
            del r
            torch.cuda.empty_cache()

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "i8", "data": "synthetic",
        "config": {"workload": f"{wl.name}: {wl.describe()}", "tokens_per_rank": N,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "expert_path": {1: "matvec", 2: "tensor"}[head_path],
                   "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MB write); expert weights exceed L2",
                   "step": "one moe_ffn_prefill call between two events; stage times from "
                           f"moe_ffn_prefill_timed over {n_stage} further steps"},
        "stage_ms": stage_ms,
        "layer_roofline_us": layer_roof_s * 1e6,
        "layer_roofline_frac": layer_roof_s / (ms / 1e3),
        "algorithmic": head_work,
        "roofline": roofline,
        "e2e": {"value": job_throughput(world, N, e2e_mean), "unit": UNIT, "h2d_bytes_per_step": N * D * 4,
                "d2h_bytes_per_step": N * D * 4, "ms_per_step": e2e_mean,
                "api": "moe_ffn_prefill_host on pinned host buffers (read and written in place over the host link)",
                "host_numa_node": numa_node},
        "with_residual": {"value": job_throughput(world, N, res_mean), "unit": UNIT, "ms_per_step": res_mean,
                          "api": "moe_ffn_prefill_residual (residual add fused into the combine)"},
        "with_residual_rmsnorm": {"value": job_throughput(world, N, norm_mean), "unit": UNIT, "ms_per_step": norm_mean,
                                  "api": "moe_ffn_prefill_residual_rmsnorm (residual add and the next layer's "
                                         "RMSNorm fused into the combine)"},
        "layer_stack": {"layers": 2, "ms_per_step": stack_ms, "ms_two_separate_calls": two_ms,
                        "tokens_per_s_per_layer": job_throughput(world, 2 * N, stack_ms),
                        "api": "moe_ffn_prefill_stack (second router launched behind the first combine; "
                               "the step includes one hidden-size device copy, as do the separate calls)"},
        "layer_stack_rmsnorm": {"layers": 2, "ms_per_step": stack_norm_ms,
                                "tokens_per_s_per_layer": job_throughput(world, 2 * N, stack_norm_ms),
                                "api": "moe_ffn_prefill_stack_rmsnorm (an input norm before each layer, the later "
                                       "ones and a final one fused into the combines; one hidden-size copy)"},
        "gpu_launches": head_launches * args.steps,
        "clocks": clk,
        "configs": configs,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, inp, args.cpu_tokens)
    print(json.dumps(line), flush=True)


# ncu dram__bytes_read.sum + dram__bytes_write.sum per launch of the dominant kernel, keyed by
# (stage, workload), with the sha256 prefix of the kernel source the counters were taken on
# (profiles/launches_olmoe_layer.md); reported only while the source is unchanged.
TRAFFIC = {("gate_up", "olmoe"): (674.3e6, "mixture_experts_ffn_top_gb300/csrc/expert_gemm.cu",
                                  "031c18b8eae26e1d")}


def measured_traffic(stage, workload):
    entry = TRAFFIC.get((stage, workload))
    if entry is None:
        return None
    nbytes, src, digest = entry
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), src)
    try:
        with open(path, "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:16] != digest:
                return None
    except OSError:
        return None
    return nbytes


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--path", type=int, default=0, help="0 auto, 1 matvec, 2 tensor")
    ap.add_argument("--cpu-tokens", type=int, default=2048, help="oracle sample (tokens per pass) for cpu_baseline")
    ap.add_argument("--ref-tokens", type=int, default=64, help="oracle sample per step for --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="time the headline workload only")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
