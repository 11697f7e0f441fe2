#!/usr/bin/env python
"""Benchmark of the FP8 FFN sublayer stack on GB300.

One step = one graph replay of the whole stack (steps A1..A4 for every layer)
over one batch of M tokens, inputs resident in HBM.  Prints one JSON line:
tokens/s of the whole job, microseconds per layer, an end-to-end figure
through the C ABI with host buffers, the roofline of the dominant kernel,
the clocks seen during the timed region, and the CPU oracle's throughput.

  python bench.py [--config vla_action_expert] [--steps K] [--warmup W]
  python bench.py --impl reference ...   # the CPU oracle as the reference arm

Multi-GPU (torchrun, one rank per GPU): replicas only -- every rank runs the
same workload on its own GPU; timing is barrier-bracketed and the slowest
rank's time counts.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import synthetic  # noqa: E402

DEFAULT_CONFIG = "vla_action_expert"
L2_FLUSH_BYTES = 2 * 129 * 1024 * 1024
WARM_L2 = False  # --warm-l2: no flush between timed steps (a diagnostic, not the bench line)
VARIANTS = {"plain": "RMSNorm weight", "fold": "norm weight folded into W_gate/W_up (Pi0)",
            "ada": "AdaRMSNorm, one modulation row per token (Pi0.5)"}
CLOCK_FIELDS = ["timestamp", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
STEP_NAMES = ["norm_quant", "gemm_gate_up_act", "gemm_down"]
KERNEL_SOURCES = {"norm_quant": ["k_elementwise.cu", "frt_ptx.cuh"],
                  "gemm_gate_up_act": ["k_gemm_tc.cuh", "k_gemm_fp8.cu", "frt_ptx.cuh", "frt_epi.cuh", "frt_f4.cuh"],
                  "gemm_down": ["k_gemm_tc.cuh", "k_gemm_fp8.cu", "frt_ptx.cuh", "frt_epi.cuh", "frt_f4.cuh"],
                  "ffn_stack": ["k_stack_fp8.cu", "frt_ptx.cuh", "frt_epi.cuh"],
                  "nvfp4_norm_quant": ["k_nvfp4.cu", "frt_ptx.cuh", "frt_f4.cuh"],
                  "nvfp4_gemm": ["k_gemm_tc.cuh", "k_gemm_f4.cu", "frt_ptx.cuh", "frt_epi.cuh", "frt_f4.cuh"]}
FP4_STEP_NAMES = ["nvfp4_norm_quant", "nvfp4_gemm_gate_up", "nvfp4_gemm_down"]


# ----------------------------------------------------------------- helpers --

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            js = json.load(f)
        return {"hbm_gbs": js["hbm_gbs"], "bf16_tflops": js["bf16_tflops"],
                "bf16_tflops_sustained": js.get("bf16_tflops_sustained", js["bf16_tflops"]), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


def kernel_bytes_flops(wl, M, step):
    """Algorithmic bytes (minimum reads + writes) and FLOPs of one launch of
    one step of one layer, for M tokens."""
    d, ff = wl.d, wl.ff
    if step == 0:   # residual (+ hidden at layer 0 is not timed here) in, norm weight in, q_x out
        return 2 * M * d + 2 * d + M * d, 0
    if step == 1:   # W_gu + q_x in, q_h out (gated activation in the epilogue)
        return 2 * ff * d + M * d + M * ff, 2 * M * 2 * ff * d
    return d * ff + M * ff + 2 * M * d + 2 * M * d, 2 * M * d * ff   # W_down + q_h + residual in, out


def stack_bytes_flops(wl, M):
    """The persistent stack kernel (one launch for all L layers): every
    layer's FP8 weights, the residual and hidden inputs and the output; the
    L layers' GEMM FLOPs."""
    return wl.L * 3 * wl.d * wl.ff + 3 * 2 * M * wl.d, wl.L * 6.0 * M * wl.d * wl.ff


def layer_algorithmic_bytes(wl, M):
    """FP8 weights + BF16 residual in/out of one layer (intermediates excluded)."""
    return 3 * wl.d * wl.ff + 2 * 2 * M * wl.d


def l2_note():
    if WARM_L2:
        return "warm: not flushed between timed steps (diagnostic)"
    return "flushed between timed steps (%d MiB write)" % (L2_FLUSH_BYTES >> 20)


def fp4_layer_bytes_flops(wl, M):
    """NVFP4 layer: E2M1 weight codes (half a byte each) + their E4M3 block
    scales (one byte per 16) + BF16 residual in/out; 3 GEMMs of 2 M d ff FLOPs."""
    return 3 * wl.d * wl.ff // 2 + 3 * wl.d * wl.ff // 16 + 4 * M * wl.d, 6.0 * M * wl.d * wl.ff


def fp4_kernel_bytes_flops(wl, M, step):
    """Algorithmic bytes and FLOPs of one launch of one NVFP4 step, for M
    tokens (codes half a byte an element, E4M3 block scales one byte per 16)."""
    d, ff = wl.d, wl.ff
    if step == 0:   # residual + norm weight in, X codes and scales out
        return 2 * M * d + 2 * d + M * d // 2 + M * d // 16, 0
    if step == 1:   # [W_g; W_u] codes + scales and X in, A codes and scales out
        return (2 * ff * d // 2 + 2 * ff * d // 16 + M * d // 2 + M * d // 16 + M * ff // 2 + M * ff // 16,
                4.0 * M * d * ff)
    # W_d codes + scales and A in, residual in, out
    return d * ff // 2 + d * ff // 16 + M * ff // 2 + M * ff // 16 + 4 * M * d, 2.0 * M * d * ff


def source_code_only(text):
    """The code of a CUDA/C++ source without its comments and blank lines
    (string literals in these sources hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines()]
    return "\n".join(ln for ln in lines if ln.strip())


def source_hash(names):
    """Hash of the kernels' code (comments excluded), recorded with each ncu
    summary so that `traffic` is reported only for the code it was measured on."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "realtime_transformer_gb300", "csrc", n)) as f:
            h.update(source_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload, index=0):
    """dram read+write bytes per launch recorded from an ncu capture in
    profiles/ (the index-th kernel of the summary), if the kernel source has
    not changed since."""
    path = os.path.join(ROOT, "profiles", "ncu_%s_%s.md" % (kernel, workload))
    if not os.path.exists(path):
        return None
    rec, traffic = {}, []
    with open(path) as f:
        for line in f:
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                rec[k.strip()] = v.strip().strip("`")
                if k.strip() == "traffic_bytes_per_launch":
                    traffic.append(v.strip())
    if rec.get("source_sha256_16") != source_hash(KERNEL_SOURCES[kernel]):
        return None
    try:
        return int(float(traffic[index]))
    except (IndexError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    def __init__(self, device_index: int):
        self.proc = None
        ident = None
        try:
            props = torch.cuda.get_device_properties(device_index)
            uuid = getattr(props, "uuid", None)
            if uuid is not None:
                ident = "GPU-" + str(uuid) if not str(uuid).startswith("GPU-") else str(uuid)
        except Exception:
            ident = None
        self.ident = ident
        self.device_index = device_index

    def start(self):
        sel = ["-i", self.ident] if self.ident else []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", *sel, "--query-gpu=" + ",".join(CLOCK_FIELDS),
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= len(CLOCK_FIELDS) - 1]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def reduce_max(value: float, world: int, device) -> float:
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# -------------------------------------------------------------- CPU oracle --

def oracle_layers(wl, layers):
    """Oracle-quantised weights of the given layers (seeded like the GPU's)."""
    import oracle
    bits = synthetic.bf16_bits
    gen = "cuda" if torch.cuda.is_available() else "cpu"
    q = []
    for l in layers:
        w = synthetic.layer_weights(wl, l, device=gen)
        q.append(oracle.quantize_stack([{k: bits(v) for k, v in w.items()}])[0])
        del w
    return q


def oracle_sample(wl, q, s_x, s_h, r, h, budget_s):
    """Time the oracle, as it stands, on a bounded sample of the workload:
    `rows` tokens through the len(q) layers held in q (the stack's first
    ones), sized to about budget_s seconds.  Returns (tokens/s of the whole
    stack, scaled by L / len(q); the sample's seconds; rows)."""
    import oracle
    bits = synthetic.bf16_bits
    rb, hb = bits(r.cpu()), bits(h.cpu())
    t0 = time.perf_counter()
    oracle.stack_forward(q[:1], rb[:1], hb[:1], s_x, s_h, wl.act_id)
    t1 = max(time.perf_counter() - t0, 1e-6)
    rows = max(1, min(wl.M, int(budget_s / (t1 * len(q)))))
    t0 = time.perf_counter()
    oracle.stack_forward(q, rb[:rows], hb[:rows], s_x, s_h, wl.act_id)
    dt = time.perf_counter() - t0
    return rows / (dt * wl.L / len(q)), dt, rows


def sample_layers(wl):
    """How many of the stack's first layers the oracle sample runs."""
    per_layer = 3 * wl.d * wl.ff
    return max(1, min(wl.L, int(2.0e8 // per_layer)))


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------------- arms --

def gen_workload(wl, device):
    weights = [synthetic.layer_weights(wl, l, device=device) for l in range(wl.L)]
    r, h = synthetic.inputs(wl, device=device)
    calib = synthetic.calibration_batches(wl, device=device)
    return weights, r, h, calib


def run_reference(args, wl, world, rank):
    """The CPU oracle, as it stands, on this host's cores: each step a bounded
    sample of the workload (tokens through the stack's first layers, scaled
    to the whole stack); scales from the oracle's own calibration of those
    layers on a few rows."""
    if rank != 0:
        return None
    import oracle
    bits = synthetic.bf16_bits
    n_s = sample_layers(wl)
    q = oracle_layers(wl, range(n_s))
    r, h = synthetic.inputs(wl)
    calib = synthetic.calibration_batches(wl, M=min(wl.M, 8))
    s_x, s_h = oracle.calibrate_stack(q, [bits(a) for a, _ in calib], [bits(b) for _, b in calib], wl.act_id)
    budget = float(os.environ.get("FRT_REFERENCE_SECONDS", "60")) / max(1, args.steps + args.warmup)
    _, _, rows = oracle_sample(wl, q, s_x, s_h, r, h, budget)
    rb, hb = bits(r[:rows]), bits(h[:rows])
    for _ in range(args.warmup):
        oracle.stack_forward(q, rb, hb, s_x, s_h, wl.act_id)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.stack_forward(q, rb, hb, s_x, s_h, wl.act_id)
    dt = (time.perf_counter() - t0) * wl.L / n_s      # the whole stack, scaled from the sampled layers
    value = rows * args.steps / dt
    sample = "%d of %d tokens through %d of the %d layers per step, scaled to the stack" % (rows, wl.M, n_s, wl.L)
    line = {
        "impl": "reference", "metric": HEADLINE_METRIC if args.config is None else metric_of(wl), "value": value,
        "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp32 (E4M3/BF16 emulated)", "data": "synthetic",
        "config": config_of(wl),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


def metric_of(wl, variant="plain"):
    name = wl.name if variant == "plain" else "%s, %s" % (wl.name, VARIANTS[variant])
    return "FP8 FFN stack tokens/s (graph-replayed, %s)" % name


def config_of(wl):
    return {"workload": wl.name, "M": wl.M, "d": wl.d, "ff": wl.ff, "act": wl.act, "layers": wl.L,
            "weights": "E4M3 per-tensor", "residual": "BF16", "graph": "one CUDA graph per stack",
            "l2": l2_note(), "parallelism": "replicas"}


def timed_steps(stream, flush, fn, n, warm):
    """n steps of fn timed with CUDA events on `stream` (after `warm` untimed
    ones), L2 flushed before each unless --warm-l2; per-step milliseconds."""
    for _ in range(warm):
        with torch.cuda.stream(stream):
            if not WARM_L2:
                flush.zero_()
            fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for e0, e1 in evs:
            if not WARM_L2:
                flush.zero_()
            e0.record(stream)
            fn()
            e1.record(stream)
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in evs]


L2_BYTES = 129 * 1024 * 1024


def pipelined_e2e(stream, dev, replay, io, out, h_io, h_o, steps, warmup):
    """End to end as a serving loop runs it, for steps whose inputs exceed L2
    (so no flush is needed between them): step i+1's inputs are copied from
    pinned host memory into one of two device staging buffers on a copy stream
    while step i computes, and step i's output goes back to pinned host memory
    while step i+1 computes; a step copies its staged inputs into the graph's
    input buffer and its output into a staging buffer (device to device).  One
    pair of events brackets all `steps` steps, every host-to-device and
    device-to-host copy included.  Returns seconds for the steps."""
    cs = torch.cuda.Stream(device=dev)
    st_in = [torch.empty_like(io) for _ in range(2)]
    st_out = [torch.empty_like(out) for _ in range(2)]

    def run(n):
        in_ready, in_free = [torch.cuda.Event() for _ in range(2)], [torch.cuda.Event() for _ in range(2)]
        out_ready, out_free = [torch.cuda.Event() for _ in range(2)], [torch.cuda.Event() for _ in range(2)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        for b in range(2):
            in_free[b].record(stream)
            out_free[b].record(cs)
        e0.record(cs)

        def h2d(i):
            b = i % 2
            cs.wait_event(in_free[b])
            with torch.cuda.stream(cs):
                st_in[b].copy_(h_io, non_blocking=True)
            in_ready[b].record(cs)

        h2d(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                h2d(i + 1)
            stream.wait_event(in_ready[b])
            with torch.cuda.stream(stream):
                io.copy_(st_in[b])
                in_free[b].record(stream)
                replay()
                stream.wait_event(out_free[b])
                st_out[b].copy_(out)
                out_ready[b].record(stream)
            cs.wait_event(out_ready[b])
            with torch.cuda.stream(cs):
                h_o.copy_(st_out[b], non_blocking=True)
            out_free[b].record(cs)
        e1.record(cs)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1000.0

    run(warmup)
    return run(steps)


def run_ours(args, wl, world, rank, local):
    """One workload: the stack graph-replayed K times (CUDA events, L2 flushed
    between steps), end to end through the C ABI with pinned host buffers,
    the in-stack share of each kernel (graph_profile) for the dominant
    kernel's roofline, and the oracle on a bounded sample."""
    from realtime_transformer_gb300.ffn import FFNPlan
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    P = peaks()
    r, h = synthetic.inputs(wl, device=dev)
    calib = synthetic.calibration_batches(wl, device=dev)
    # residual and hidden side by side in one buffer: one host-to-device copy per step
    io = torch.stack([r, h]).contiguous()
    r, h = io[0], io[1]
    plan = FFNPlan(wl.d, wl.ff, wl.act, wl.M, wl.L)
    for l in range(wl.L):   # generated and loaded one layer at a time
        w = synthetic.layer_weights(wl, l, device=dev)
        plan.load_weights(l, w["w_norm"], w["w_gate"], w["w_up"], w["w_down"], fold_norm=args.variant == "fold",
                          digest=False)
        del w
    if args.variant == "ada":
        # one modulation row per token (the heavier AdaRMSNorm case); kept alive for the graph
        mods = [synthetic.modulation(wl, l, wl.M, dev) for l in range(wl.L)]
        plan.set_modulation(mods)
    plan.calibrate([a for a, _ in calib], [b for _, b in calib])
    out = torch.empty_like(r)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        plan.graph_capture(r, h, out, stream)
    torch.cuda.synchronize()
    replay = lambda: plan.graph_replay(wl.M, stream)

    if args.launch_list:
        # profiling aid: warm replays, then the given number inside an NVTX
        # range "replay" that ncu can select (--nvtx --nvtx-include "replay/")
        timed_steps(stream, flush, replay, 0, args.warmup)
        torch.cuda.nvtx.range_push("replay")
        with torch.cuda.stream(stream):
            for _ in range(args.launch_list):
                replay()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        plan.device_status(stream)
        plan.close()
        return {"launch_list": wl.name, "replays": args.launch_list, "launches_per_replay": 3 * wl.L}

    # warm-up, then exactly K timed steps between barriers
    timed_steps(stream, flush, replay, 0, args.warmup)
    barrier(world)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    t_wall0 = time.perf_counter()
    step_ms = timed_steps(stream, flush, replay, args.steps, 0)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    clocks = sampler.stop()
    barrier(world)
    plan.device_status(stream)
    total_s = sum(step_ms) / 1000.0
    total_s = reduce_max(total_s, world, dev)
    value = world * wl.M * args.steps / total_s
    ms_step = 1000.0 * total_s / args.steps

    # end to end through the public API: pinned host in, graph, host out
    h_io = io.cpu().pin_memory()
    h_o = torch.empty_like(out, device="cpu").pin_memory()

    def e2e_step():
        io.copy_(h_io, non_blocking=True)
        plan.graph_replay(wl.M, stream)
        h_o.copy_(out, non_blocking=True)

    # steps whose inputs exceed L2: the serving loop's overlap of the copies
    # with the previous and next steps' compute; else one step at a time, L2
    # flushed before each
    e2e_pipelined = io.numel() * io.element_size() > L2_BYTES and not WARM_L2
    if e2e_pipelined:
        e2e_s = reduce_max(pipelined_e2e(stream, dev, replay, io, out, h_io, h_o, args.steps, args.warmup), world,
                           dev)
    else:
        e2e_ms = timed_steps(stream, flush, e2e_step, args.steps, args.warmup)
        e2e_s = reduce_max(sum(e2e_ms) / 1000.0, world, dev)
    h2d = h_io.numel() * 2
    d2h = h_o.numel() * 2

    # in-stack share of every launch (stamped profiling replays of the same
    # graph, L2 flushed before each like the timed steps); the dominant kernel
    # is the step whose launches take the most of the stack
    n_prof = max(10, min(50, args.steps))
    shares = []
    for _ in range(n_prof):
        if not WARM_L2:
            with torch.cuda.stream(stream):
                flush.zero_()
        shares.append(plan.graph_profile(wl.M, n_replays=1, stream=stream))
    n_k = len(shares[0])
    med = [statistics.median(sh[k] for sh in shares) for k in range(n_k)]
    if n_k == 1:
        # the whole stack is one persistent launch
        kern_total = {"ffn_stack": med[0]}
        dom, launches = "ffn_stack", 1
        nbytes, flops = stack_bytes_flops(wl, wl.M)
    else:
        per_step = {STEP_NAMES[s]: [med[3 * l + s] for l in range(wl.L)] for s in range(3)}
        kern_total = {k: sum(v) for k, v in per_step.items()}
        dom, launches = max(kern_total, key=kern_total.get), wl.L
        nbytes, flops = kernel_bytes_flops(wl, wl.M, STEP_NAMES.index(dom))
    t_dom = kern_total[dom] / launches * 1e-6      # average in-stack duration of one launch
    long_step = ms_step >= 1.0
    fp8_peak = 2.0 * (P["bf16_tflops_sustained"] if long_step else P["bf16_tflops"])
    ridge = fp8_peak * 1e12 / (P["hbm_gbs"] * 1e9)
    tensor_bound = flops > 0 and flops / nbytes > ridge
    if tensor_bound:
        achieved = flops / t_dom / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": achieved / fp8_peak,
                "peak_note": "FP8 dense = 2 x %s bf16 (%s; nominal fp8/bf16 ratio 2)" % (
                    "sustained" if long_step else "burst", P["src"])}
    else:
        achieved = nbytes / t_dom / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": P["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / P["hbm_gbs"], "peak_note": "%s HBM copy bandwidth" % P["src"]}
    roof["kernel"] = dom
    roof["us_per_launch"] = kern_total[dom] / launches
    roof["timing"] = ("in-stack share of each launch (%%globaltimer stamps, median of %d profiled replays): "
                      "%d x us_per_launch = %.1f us of a %.1f us step" % (n_prof, launches, kern_total[dom],
                                                                          1000.0 * ms_step))
    roof["algorithmic_bytes"] = nbytes
    roof["flops"] = flops
    roof["traffic"] = profiled_traffic(dom, wl.name)

    layer_s = ms_step / 1000.0 / wl.L
    lb = layer_algorithmic_bytes(wl, wl.M)
    lf = 6.0 * wl.M * wl.d * wl.ff
    step_roof = {"bound": "hbm", "achieved": lb / layer_s / 1e9, "peak": P["hbm_gbs"], "unit": "GB/s",
                 "frac": lb / layer_s / 1e9 / P["hbm_gbs"], "tflops": lf / layer_s / 1e12}
    if lf / lb > ridge:
        step_roof = {"bound": "tensor", "achieved": lf / layer_s / 1e12, "peak": fp8_peak, "unit": "TFLOP/s",
                     "frac": lf / layer_s / 1e12 / fp8_peak, "hbm_gbs": lb / layer_s / 1e9}

    line = {
        "metric": metric_of(wl, args.variant),
        "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "us_per_layer": 1000.0 * ms_step / wl.L, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8_e4m3 (fp32 accumulate, bf16 residual)", "data": "synthetic",
        "config": config_of(wl) if args.variant == "plain" else dict(config_of(wl), variant=VARIANTS[args.variant]),
        "roofline": roof, "step_roofline": step_roof,
        "kernels_us_in_stack": {k: v / launches for k, v in kern_total.items()},
        "e2e": {"value": world * wl.M * args.steps / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": 1000.0 * e2e_s / args.steps,
                "timing": ("all steps between one pair of events; step i+1's inputs copied in (pinned host -> "
                           "device staging) and step i-1's output read back while step i computes, as a serving "
                           "loop overlaps them; inputs larger than L2, no flush") if e2e_pipelined else
                          ("per step, L2 flushed before each: host-to-device copy, graph replay, device-to-host "
                           "copy in order on one stream")},
        "gpu_launches": args.steps * n_k, "clocks": clocks, "wall_s_timed_region": t_wall,
    }
    sc = plan.scales()
    plan.close()
    del plan, flush
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.variant == "plain":
        n_s = sample_layers(wl)
        q = oracle_layers(wl, range(n_s))
        budget = float(os.environ.get("FRT_CPU_BASELINE_SECONDS", "6"))
        v, dt, rows = oracle_sample(wl, q, sc["s_x"][:n_s], sc["s_h"][:n_s], r, h, budget)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": "%d of %d tokens through %d of the %d layers (%.1f s), scaled to the "
                                          "stack" % (rows, wl.M, n_s, wl.L, dt)}
    return line


ALL_WORKLOADS = ["tiny", "vla_action_expert", "vla_prefix", "llm_decode", "long_prefill"]
HEADLINE = "long_prefill"   # the largest single-GPU workload: the line's top-level figures
HEADLINE_METRIC = "FP8 FFN stack tokens/s vs M (graph-replayed; headline: %s)" % HEADLINE


def run_all(args, world, rank, local):
    """The metric is quoted against M: every workload in one run, the
    headline's figures at the top level and each workload's under per_config."""
    per = {}
    for name in ALL_WORKLOADS:
        per[name] = run_ours(args, synthetic.WORKLOADS[name], world, rank, local)
    line = dict(per[HEADLINE])
    line["metric"] = HEADLINE_METRIC
    line["per_config"] = {
        name: {k: v for k, v in ln.items() if k in ("value", "ms_per_step", "us_per_layer", "roofline",
                                                   "step_roofline", "kernels_us_in_stack", "e2e", "cpu_baseline",
                                                   "clocks", "gpu_launches", "config")}
        for name, ln in per.items()}
    line["gpu_launches"] = sum(ln["gpu_launches"] for ln in per.values())
    line["gpu_launches_note"] = "all workloads' timed steps; the headline's own: %d" % per[HEADLINE]["gpu_launches"]
    return line


def qkv_config_of(wl):
    nq, nkv, hd, base = synthetic.ATTENTION[wl.name]
    return {"workload": wl.name + " attention input (QKV)", "M": wl.M, "d": wl.d, "n_q_heads": nq,
            "n_kv_heads": nkv, "head_dim": hd, "rope_base": base, "layers": wl.L, "weights": "E4M3 per-tensor",
            "graph": "the stack's L sublayer forwards in one CUDA graph (same input per layer)",
            "l2": l2_note(), "parallelism": "replicas"}


def run_qkv(args, wl, world, rank, local):
    """The attention-input sublayer (norm + FP8 fused-QKV GEMM + split/RoPE):
    one step = the L layers' sublayers, each on the workload's residual (the
    attention between them is not this library's), captured in one graph."""
    from realtime_transformer_gb300.qkv import QKVPlan
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    P = peaks()
    nq, nkv, hd, base = synthetic.ATTENTION[wl.name]
    N = (nq + 2 * nkv) * hd
    r, h = synthetic.inputs(wl, device=dev)
    calib = synthetic.calibration_batches(wl, device=dev)
    pos = torch.from_numpy(synthetic.positions(wl)).to(dev)
    plan = QKVPlan(wl.d, nq, nkv, hd, base, wl.M, wl.L)
    ws = [synthetic.qkv_weights(wl, l, device=dev) for l in range(wl.L)]
    for l, w in enumerate(ws):
        plan.load_weights(l, w["w_norm"], w["w_q"], w["w_k"], w["w_v"])
        plan.calibrate(l, [a for a, _ in calib], [b for _, b in calib] if l == 0 else None)
    outs = [plan._outs(wl.M, dev) for _ in range(wl.L)]
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def stack():
        for l in range(wl.L):
            plan.forward(l, r, h if l == 0 else None, pos, out=outs[l], stream=stream)

    with torch.cuda.stream(stream):
        stack()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            stack()
    torch.cuda.synchronize()

    def timed(fn, n, warm):
        for _ in range(warm):
            with torch.cuda.stream(stream):
                if not WARM_L2:
                    flush.zero_()
                fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        with torch.cuda.stream(stream):
            for e0, e1 in evs:
                if not WARM_L2:
                    flush.zero_()
                e0.record(stream)
                fn()
                e1.record(stream)
        torch.cuda.synchronize()
        return [e0.elapsed_time(e1) for e0, e1 in evs]

    timed(graph.replay, 0, args.warmup)
    barrier(world)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    t_wall0 = time.perf_counter()
    step_ms = timed(graph.replay, args.steps, 0)
    t_wall = time.perf_counter() - t_wall0
    clocks = sampler.stop()
    barrier(world)
    plan.device_status(stream)
    total_s = reduce_max(sum(step_ms) / 1000.0, world, dev)
    value = world * wl.M * args.steps / total_s
    ms_step = 1000.0 * total_s / args.steps

    # end to end: pinned host residual/hidden in, the graph, Q/K/V of every layer out
    h_r = r.cpu().pin_memory()
    h_h = h.cpu().pin_memory()
    h_out = [{k: torch.empty_like(o[k], device="cpu").pin_memory() for k in ("q", "k", "v")} for o in outs]

    def e2e_step():
        r.copy_(h_r, non_blocking=True)
        h.copy_(h_h, non_blocking=True)
        graph.replay()
        for ho, o in zip(h_out, outs):
            for k in ho:
                ho[k].copy_(o[k], non_blocking=True)

    e2e_ms = timed(e2e_step, args.steps, args.warmup)
    e2e_s = reduce_max(sum(e2e_ms) / 1000.0, world, dev)
    d2h = sum(t.numel() * 2 for ho in h_out for t in ho.values())

    # roofline of one sublayer (its three kernels together): weights + residual
    # in + Q/K/V out, against HBM or the FP8 tensor peak by intensity
    layer_s = ms_step / 1000.0 / wl.L
    nbytes = N * wl.d + 2 * wl.M * wl.d + 2 * wl.M * N
    flops = 2.0 * wl.M * wl.d * N
    fp8_peak = 2.0 * P["bf16_tflops"]
    if flops / nbytes > fp8_peak * 1e12 / (P["hbm_gbs"] * 1e9):
        ach = flops / layer_s / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": fp8_peak, "unit": "TFLOP/s", "frac": ach / fp8_peak,
                "peak_note": "FP8 dense = 2 x measured bf16 burst (%s)" % P["src"]}
    else:
        ach = nbytes / layer_s / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": P["hbm_gbs"], "unit": "GB/s", "frac": ach / P["hbm_gbs"],
                "peak_note": "%s HBM copy bandwidth" % P["src"]}
    roof.update({"kernel": "qkv sublayer (norm_quant + FP8 QKV GEMM + rope_split, graph-replayed)",
                 "us_per_launch": 1e6 * layer_s, "algorithmic_bytes": nbytes, "traffic": None})
    line = {
        "metric": "FP8 QKV sublayer tokens/s (graph-replayed, %s)" % wl.name, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "us_per_layer": 1e6 * layer_s, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8_e4m3 (fp32 accumulate, bf16 outputs)", "data": "synthetic", "config": qkv_config_of(wl),
        "roofline": roof,
        "e2e": {"value": world * wl.M * args.steps / e2e_s, "unit": "tokens/s",
                "h2d_bytes_per_step": h_r.numel() * 2 + h_h.numel() * 2, "d2h_bytes_per_step": d2h,
                "ms_per_step": 1000.0 * e2e_s / args.steps},
        "gpu_launches": args.steps * wl.L * 3, "clocks": clocks, "wall_s_timed_region": t_wall,
    }
    plan.close()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        bits = synthetic.bf16_bits
        w0 = {k: bits(v) for k, v in ws[0].items()}
        codes, s_qkv = oracle.quantize_qkv_weights(w0["w_q"], w0["w_k"], w0["w_v"])
        rows = min(wl.M, 16)
        s_x = oracle.calibrate_qkv_layer([bits(calib[0][0][:rows])], [bits(calib[0][1][:rows])], w0["w_norm"])
        f = oracle.rope_inv_freq(hd, base)
        p = synthetic.positions(wl)
        t0 = time.perf_counter()
        oracle.qkv_layer(bits(r[:rows]), bits(h[:rows]), w0["w_norm"], codes, s_x, s_qkv, nq, nkv, hd, p[:rows], f)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": rows / (dt * wl.L), "unit": "tokens/s", "cores": cpu_cores(),
                                "kind": "oracle", "sample": "%d of %d tokens through one of the %d layers, "
                                "scaled to the stack" % (rows, wl.M, wl.L)}
    return line


def run_fp4(args, wl, world, rank, local):
    """The NVFP4 variant of the FFN stack (norm + AWQ-free FP4 quantise; the
    gate/up NVFP4 GEMM forming G and U as NVFP4 and the FP4 -> FP4 gated
    activation in its epilogue; the NVFP4 down GEMM + residual): one step =
    the L layers on one batch, one CUDA graph."""
    from realtime_transformer_gb300.nvfp4 import FP4Plan
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    P = peaks()
    r, h = synthetic.inputs(wl, device=dev)
    calib = synthetic.calibration_batches(wl, device=dev)
    plan = FP4Plan(wl.d, wl.ff, wl.act, wl.M, wl.L)
    for l in range(wl.L):
        w = synthetic.layer_weights(wl, l, device=dev)
        plan.load_weights(l, w["w_norm"], w["w_gate"], w["w_up"], w["w_down"])
    plan.calibrate([a for a, _ in calib], [b for _, b in calib])
    out = torch.empty_like(r)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    with torch.cuda.stream(stream):
        plan.forward(r, h, out=out, stream=stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            plan.forward(r, h, out=out, stream=stream)
    torch.cuda.synchronize()

    if args.launch_list:
        # profiling aid: warm replays, then the given number inside an NVTX
        # range "replay" that ncu can select (--nvtx --nvtx-include "replay/")
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("replay")
        for _ in range(args.launch_list):
            graph.replay()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        plan.device_status(stream)
        plan.close()
        return {"launch_list": wl.name, "sublayer": "ffn_nvfp4", "replays": args.launch_list,
                "launches_per_replay": 3 * wl.L}

    def timed(fn, n, warm):
        for _ in range(warm):
            with torch.cuda.stream(stream):
                if not WARM_L2:
                    flush.zero_()
                fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        with torch.cuda.stream(stream):
            for e0, e1 in evs:
                if not WARM_L2:
                    flush.zero_()
                e0.record(stream)
                fn()
                e1.record(stream)
        torch.cuda.synchronize()
        return [e0.elapsed_time(e1) for e0, e1 in evs]

    timed(graph.replay, 0, args.warmup)
    barrier(world)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    t_wall0 = time.perf_counter()
    step_ms = timed(graph.replay, args.steps, 0)
    t_wall = time.perf_counter() - t_wall0
    clocks = sampler.stop()
    barrier(world)
    plan.device_status(stream)
    total_s = reduce_max(sum(step_ms) / 1000.0, world, dev)
    value = world * wl.M * args.steps / total_s
    ms_step = 1000.0 * total_s / args.steps

    # end to end: pinned host residual + hidden in, the graph, the output back
    h_io = torch.cat([r, h]).cpu().pin_memory()
    h_out = torch.empty_like(out, device="cpu").pin_memory()
    io = torch.empty_like(h_io, device=dev)

    def e2e_step():
        io.copy_(h_io, non_blocking=True)
        r.copy_(io[:wl.M])
        h.copy_(io[wl.M:])
        graph.replay()
        h_out.copy_(out, non_blocking=True)

    e2e_ms = timed(e2e_step, args.steps, args.warmup)
    e2e_s = reduce_max(sum(e2e_ms) / 1000.0, world, dev)

    # against HBM or the FP4 tensor peak by intensity (the sustained bf16
    # figure for steps of a millisecond and more, as the FP8 arm)
    long_step = ms_step >= 1.0
    fp4_peak = 6.0 * (P["bf16_tflops_sustained"] if long_step else P["bf16_tflops"])

    def roofline(nbytes, flops, secs):
        if flops / nbytes > fp4_peak * 1e12 / (P["hbm_gbs"] * 1e9):
            ach = flops / secs / 1e12
            return {"bound": "tensor", "achieved": ach, "peak": fp4_peak, "unit": "TFLOP/s", "frac": ach / fp4_peak,
                    "peak_note": "FP4 dense = 6 x measured bf16 %s (%s; nominal 13.5 / 2.25)" % (
                        "sustained" if long_step else "burst", P["src"])}
        ach = nbytes / secs / 1e9
        return {"bound": "hbm", "achieved": ach, "peak": P["hbm_gbs"], "unit": "GB/s", "frac": ach / P["hbm_gbs"],
                "peak_note": "%s HBM copy bandwidth" % P["src"]}

    # the dominant kernel: each launch's in-stack share of a replay (stamped
    # replays of the same forward, L2 flushed before each)
    n_prof = 20
    shares = []
    for _ in range(n_prof):
        if not WARM_L2:
            with torch.cuda.stream(stream):
                flush.zero_()
        shares.append(plan.forward_profile(r, h, out=out, n_replays=1, stream=stream))
    med = [statistics.median(sh[k] for sh in shares) for k in range(3 * wl.L)]
    kern_total = {FP4_STEP_NAMES[st]: sum(med[3 * l + st] for l in range(wl.L)) for st in range(3)}
    dom = max(kern_total, key=kern_total.get)
    nbytes, flops = fp4_kernel_bytes_flops(wl, wl.M, FP4_STEP_NAMES.index(dom))
    roof = roofline(nbytes, flops, kern_total[dom] / wl.L * 1e-6)
    roof.update({"kernel": dom, "us_per_launch": kern_total[dom] / wl.L,
                 "timing": "in-stack share of each launch (%%globaltimer stamps, median of %d profiled replays): "
                           "%d x us_per_launch = %.1f us of a %.1f us step" % (
                               n_prof, wl.L, kern_total[dom], 1000.0 * ms_step),
                 "algorithmic_bytes": nbytes, "flops": flops,
                 "traffic": (profiled_traffic("nvfp4_gemm", wl.name, index=FP4_STEP_NAMES.index(dom) - 1)
                             if dom != "nvfp4_norm_quant" else None)})
    # the layer (its three kernels together): FP4 weights and their scales +
    # the residual stream in and out
    layer_s = ms_step / 1000.0 / wl.L
    step_roof = roofline(*fp4_layer_bytes_flops(wl, wl.M), layer_s)
    line = {
        "metric": "NVFP4 FFN stack tokens/s (graph-replayed, %s)" % wl.name, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "us_per_layer": 1e6 * layer_s, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "nvfp4 (e2m1 + e4m3 block scales, fp32 accumulate, bf16 residual)", "data": "synthetic",
        "config": dict(config_of(wl), weights="NVFP4 (E2M1, E4M3 scale per 16, fp32 per tensor)",
                       activations="NVFP4, calibrated per-tensor scales", graph="one CUDA graph per stack"),
        "roofline": roof, "step_roofline": step_roof,
        "kernels_us_in_stack": {k: v / wl.L for k, v in kern_total.items()},
        "e2e": {"value": world * wl.M * args.steps / e2e_s, "unit": "tokens/s",
                "h2d_bytes_per_step": h_io.numel() * 2, "d2h_bytes_per_step": h_out.numel() * 2,
                "ms_per_step": 1000.0 * e2e_s / args.steps},
        "gpu_launches": args.steps * wl.L * 3, "clocks": clocks, "wall_s_timed_region": t_wall,
    }
    plan.close()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        bits = synthetic.bf16_bits
        w0 = {k: bits(v) for k, v in synthetic.layer_weights(wl, 0).items()}
        L0 = oracle.quantize_layer_nvfp4(w0["w_norm"], w0["w_gate"], w0["w_up"], w0["w_down"])
        rows = min(wl.M, 16)
        rc, hc = calib[0][0][:rows].cpu(), calib[0][1][:rows].cpu()
        sc, _ = oracle.calibrate_layer_nvfp4([bits(rc)], [bits(hc)], L0, wl.act_id)
        rr, hh = bits(r[:rows].cpu()), bits(h[:rows].cpu())
        t0 = time.perf_counter()
        oracle.ffn_layer_nvfp4(rr, hh, L0, sc, wl.act_id)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": rows / (dt * wl.L), "unit": "tokens/s", "cores": cpu_cores(),
                                "kind": "oracle", "sample": "%d of %d tokens through one of the %d layers, "
                                "scaled to the stack" % (rows, wl.M, wl.L)}
    return line


def run_fp8_gemm_peak(args, local):
    """Diagnostic: this library's FP8 GEMM (tcgen05, tiled role, CTA pairs)
    on 8192 x 8192 x 8192 E4M3 operands, timed with CUDA events -- the FP8
    dense throughput a long contraction reaches here, beside the nominal
    2 x bf16 proxy."""
    from realtime_transformer_gb300.ffn import FFNPlan
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    n = 8192
    plan = FFNPlan(256, 1024, "geglu_tanh", 64, 1)
    g = torch.Generator(device=dev).manual_seed(7)
    A = torch.randint(0, 0x7E, (n, n), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
    B = torch.randint(0, 0x7E, (n, n), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            plan.gemm(A, B, path=2, stream=stream)
        torch.cuda.synchronize()
        sampler = ClockSampler(local)
        sampler.start()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            plan.gemm(A, B, path=2, stream=stream)
        e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    plan.device_status()
    plan.close()
    ms = e0.elapsed_time(e1) / args.steps
    P = peaks()
    tf = 2.0 * n ** 3 / (ms * 1e-3) / 1e12
    return {"fp8_gemm_8192": {"tflops": tf, "ms": ms, "steps": args.steps,
                              "vs_2x_bf16_burst": tf / (2.0 * P["bf16_tflops"]),
                              "vs_2x_bf16_sustained": tf / (2.0 * P["bf16_tflops_sustained"]), "clocks": clocks}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=None, choices=sorted(synthetic.WORKLOADS),
                    help="one workload (default: the FFN stack times all five, the headline on %s; the other "
                         "sublayers default to %s)" % (HEADLINE, DEFAULT_CONFIG))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sublayer", choices=["ffn", "qkv", "ffn_nvfp4"], default="ffn",
                    help="ffn: the FFN stack (the default bench line); qkv: the attention-input projections; "
                         "ffn_nvfp4: the NVFP4 variant of the FFN stack")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling aid: run a plan of this many layers of the workload's shape "
                         "(the line is then not the workload's bench line)")
    ap.add_argument("--launch-list", type=int, default=0,
                    help="profiling aid: after the warm-up, run this many graph replays of one workload inside an "
                         "NVTX range \"replay\" and print no bench line")
    ap.add_argument("--fp8-gemm-peak", action="store_true",
                    help="diagnostic: time this library's FP8 GEMM on 8192^3 and print its TFLOP/s (no bench line)")
    ap.add_argument("--variant", choices=sorted(VARIANTS), default="plain",
                    help="FFN stack only: plain (the bench line), fold (norm weight folded into the gate/up "
                         "weights) or ada (AdaRMSNorm modulation)")
    ap.add_argument("--warm-l2", action="store_true",
                    help="diagnostic: do not flush L2 between timed steps (the line says so in config.l2)")
    args = ap.parse_args()
    global WARM_L2
    WARM_L2 = args.warm_l2
    if args.warmup < 3:
        args.warmup = 3
    all_ffn = (args.config is None and args.sublayer == "ffn" and args.layers == 0 and args.variant == "plain"
               and not args.launch_list)
    wl = synthetic.WORKLOADS[args.config or (HEADLINE if args.sublayer == "ffn" else DEFAULT_CONFIG)]
    if args.layers > 0:
        wl = wl.with_(L=args.layers, name=wl.name + "_%dlayers" % args.layers)
    if args.variant != "plain" and (args.sublayer != "ffn" or args.impl != "ours"):
        ap.error("--variant applies to the FFN stack of this implementation only")
    world, rank, local = dist_setup(args.gpus)
    if args.fp8_gemm_peak:
        line = run_fp8_gemm_peak(args, local)
    elif args.impl == "reference":
        line = run_reference(args, wl, world, rank)
    elif args.sublayer == "qkv":
        line = run_qkv(args, wl, world, rank, local)
    elif args.sublayer == "ffn_nvfp4":
        line = run_fp4(args, wl, world, rank, local)
    elif all_ffn:
        line = run_all(args, world, rank, local)
    else:
        line = run_ours(args, wl, world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
