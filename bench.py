#!/usr/bin/env python
"""Benchmark: dequant-fused 4-bit GEMV decode stack on one GB300.

Workload: one decode token (batch 1) through a stack of 32
Llama-3.1-8B-shaped layers, each the fused matvec chain
    RMSNorm->QKV 4096->6144 -> value-head copy (decode over one position)
    -> o_proj 4096->4096 (+ residual)
    -> gate.up 4096->2x14336 SwiGLU (post-attention RMSNorm fused)
    -> down 14336->4096 (+ residual)
with 4-bit group-64 planar weights.  A step is one token through all 32
layers: ONE qgemv_decode_stack call (4 streaming-kernel launches per layer,
chained with programmatic dependent launch, replayed from the call's CUDA
graph cache) reading 3.93 GB of distinct device weights, so no step's inputs
fit in the 129 MB L2.  The 32 layers are device copies of one seeded
synthetic layer.

Metric: algorithmic HBM GB/s (codes + scales + biases + activations read and
written, per the byte accounting of bit_group_quantized_qgemv_gb300.accounting)
divided by the device time of the step, plus us per decode matvec stack.

Timing: W warm-up and K timed steps on one stream, CUDA events around the K,
a barrier and torch.cuda.synchronize() on both sides, max over ranks.  The
same chain as a CUDA graph of single-op C-ABI launches (5 per layer) is
timed beside it ("unfused").  The roofline object is the dominant kernel,
gate.up SwiGLU: its average duration is timed by CUDA events around replays
of a graph of the token's 32 gate.up launches back to back.  `--op NAME`
times one fused op alone through CUDA-graph replays.  `--impl reference`
times the fp64 CPU oracle on a bounded row sample of the same layer instead.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "dequant-GEMV achieved HBM GB/s (% of GB300 peak); us per decode matvec stack"
LAYERS = 32
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["own", "reference"], default="own")
    p.add_argument("--layers", type=int, default=LAYERS)
    p.add_argument("--no-cpu-baseline", action="store_true",
                   help="skip the oracle CPU-baseline leg")
    p.add_argument("--no-unfused", action="store_true",
                   help="skip the single-op CUDA-graph comparison")
    p.add_argument("--op", default="stack",
                   help="time one op or configuration unit alone instead of the stack: "
                        "qkv, o_proj, swiglu, down, moe, moe_routed, lm_head, lm_head_argmax, "
                        "lm_head_sample, gemv1024, lut_layer, lut_lm_head, "
                        "qwen_stack, w2_layer, w8_layer, m2, m4, m8, m2_w2, m4_w2, m8_w2, "
                        "residual_rmsnorm, "
                        "or all")
    p.add_argument("--copies", type=int, default=0,
                   help="--op: device copies of the weights to rotate through (default: "
                        "enough to exceed 3x L2; 1 keeps them resident in L2, the "
                        "compute-only variant)")
    return p.parse_args()


def max_over_ranks(torch, values, device, world):
    """Each rank's timings -> their maximum over all ranks (the job's time,
    since every rank must finish); identity on one rank."""
    if world <= 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# The files the streaming kernels (and their launch plans) are built from:
# the ncu counters in profiles/traffic.json hold while these are unchanged.
STREAM_KERNEL_SOURCES = ("qgemv_args.h", "qgemv_device.cuh", "qgemv_stream.cuh",
                         "stream_norm_swiglu.cu", "stream_plain.cu")


def kernel_sources_digest():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_group_quantized_qgemv_gb300", "csrc")
    for name in STREAM_KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def recorded_traffic(kernel_key):
    """Per-launch DRAM bytes of the kernel from the committed ncu summary, if
    the kernel sources have not changed since it was taken; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel_key]
    except (OSError, KeyError, ValueError):
        return None
    if rec.get("sources_sha256") != kernel_sources_digest():
        return None
    return rec.get("dram_bytes_per_launch")


# --------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ own arm
def build_stack(torch, n_layers, device):
    import numpy as np

    import synth
    c = synth.LLAMA8B
    H, I = c["hidden"], c["inter"]
    layer = synth.llama_layer(1, 0, 4)

    def up(w):
        codes = torch.from_numpy(np.ascontiguousarray(w.codes).view(np.int32)).to(device)
        return (codes, torch.from_numpy(w.scales).to(device), torch.from_numpy(w.biases).to(device))

    base = {k: up(layer[k]) for k in ("qkv", "o", "gate", "up", "down")}
    g1 = torch.from_numpy(layer["gamma1"]).to(device)
    g2 = torch.from_numpy(layer["gamma2"]).to(device)
    layers = []
    for _ in range(n_layers):
        layers.append({k: tuple(t.clone() for t in v) for k, v in base.items()} |
                      {"attn_norm": g1.clone(), "mlp_norm": g2.clone()})
    x0 = torch.from_numpy(layer["x"]).to(device)
    bufs = {
        "x": torch.empty(H, dtype=torch.float16, device=device),
        "qkv": torch.empty((c["n_q"] + 2 * c["n_kv"]) * c["head_dim"], dtype=torch.float16,
                           device=device),
        "attn": torch.empty(c["n_q"] * c["head_dim"], dtype=torch.float16, device=device),
        "h": torch.empty(H, dtype=torch.float16, device=device),
        "act": torch.empty(I, dtype=torch.float16, device=device),
    }
    return layers, x0, bufs


def unfused_calls(q, layers, bufs, eps, events=None):
    """The same token as single-op C-ABI calls (5 per layer) on the current
    stream, for the comparison graph; `events[l]` = (start, end) recorded
    around layer l's gate.up SwiGLU launch."""
    import synth
    c = synth.LLAMA8B
    x, qkv, attn, h, act = bufs["x"], bufs["qkv"], bufs["attn"], bufs["h"], bufs["act"]
    for li, L in enumerate(layers):
        q.rmsnorm_qgemv(L["qkv"], x, L["attn_norm"], eps, y=qkv)
        q.decode_attention_seq1(qkv, c["n_q"], c["n_kv"], c["head_dim"], out=attn)
        q.qgemv_w4g64(L["o"], attn, y=h, residual=x)
        if events is not None:
            events[li][0].record()
        q.swiglu_qgemv(L["gate"], L["up"], h, L["mlp_norm"], eps, h=act)
        if events is not None:
            events[li][1].record()
        q.qgemv_w4g64(L["down"], act, y=x, residual=h)


def run_own(args):
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import bit_group_quantized_qgemv_gb300 as q
    from bit_group_quantized_qgemv_gb300 import accounting as acc
    import synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    c = synth.LLAMA8B
    n_layers = args.layers
    eps = 1e-5
    layers, x0, bufs = build_stack(torch, n_layers, device)
    ops = acc.llama8b_layer_ops(4)
    layer_bytes = acc.llama8b_layer_bytes(4)
    step_bytes = n_layers * layer_bytes
    shape = q.stack_shape(c["hidden"], c["n_q"], c["n_kv"], c["head_dim"], c["inter"], n_layers,
                          eps)
    descs = q.stack_layers(layers)
    work = torch.empty(q.decode_stack_workspace_bytes(shape), dtype=torch.uint8, device=device)
    x_in = x0.clone()
    y_out = torch.empty_like(x0)

    stream = torch.cuda.Stream(device)

    def step():
        q.decode_stack(descs, shape, x_in, y=y_out, workspace=work, stream=stream)

    torch.cuda.synchronize()
    step()                                        # sets the kernel's attributes
    torch.cuda.synchronize()
    if q.device_status() != 0:
        raise RuntimeError("device-side wait timed out during warm-up")

    K, W = args.steps, args.warmup
    gpu_id = str(local)
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        pass

    # ---- timed region: K steps of the device-resident stack, one launch each
    for _ in range(W):
        step()
    barrier()
    clocks = ClockSampler(gpu_id)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(K):
        step()
    t_end.record(stream)
    barrier()
    clk = clocks.stop()
    ms = t_start.elapsed_time(t_end)

    # ---- timed region: end to end through the public API with host buffers
    x_host = x0.cpu().pin_memory()
    y_host = torch.empty_like(x_host).pin_memory()

    def step_e2e():
        with torch.cuda.stream(stream):
            x_in.copy_(x_host, non_blocking=True)
            step()
            y_host.copy_(y_out, non_blocking=True)

    Ke = max(1, min(K, 1000))
    for _ in range(min(W, 20)):
        step_e2e()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(Ke):
        step_e2e()
    e1.record(stream)
    barrier()
    ms_e2e = e0.elapsed_time(e1)
    out_ok = bool(torch.isfinite(y_host.float()).all())
    # Per-token latency with the host waiting for each token's result before
    # issuing the next (wall clock, host sync after every token).
    lat = []
    for _ in range(min(Ke, 50)):
        t0 = time.perf_counter()
        step_e2e()
        stream.synchronize()
        lat.append((time.perf_counter() - t0) * 1e6)
    lat_us = statistics.median(lat)

    # ---- the same token as a CUDA graph of single-op launches
    # ---- the same token as a CUDA graph of single-op launches (+ the
    # attention copy), and the dominant kernel timed live inside it: CUDA
    # events (graph nodes) around every gate.up SwiGLU launch
    def timing_event():
        try:
            return torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            return torch.cuda.Event(enable_timing=True)

    with torch.cuda.stream(stream):
        bufs["x"].copy_(x0)
        unfused_calls(q, layers, bufs, eps)
    torch.cuda.synchronize()
    unfused = None
    if not args.no_unfused:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            unfused_calls(q, layers, bufs, eps)
        Ku = max(1, min(K, 1000))
        with torch.cuda.stream(stream):
            for _ in range(min(W, 20)):
                g.replay()
        barrier()
        u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        u0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(Ku):
                g.replay()
        u1.record(stream)
        barrier()
        ms_u = u0.elapsed_time(u1) / Ku
        unfused = {"us_per_step": round(ms_u * 1e3, 2),
                   "value": round(step_bytes / (ms_u * 1e-3) / 1e9, 1), "unit": "GB/s",
                   "launches_per_step": 5 * n_layers,
                   "how": "CUDA graph of 5 single-op C-ABI launches per layer (value-head "
                          "copy kernel included)"}
    ev = [(timing_event(), timing_event()) for _ in range(n_layers)]
    ge = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ge, stream=stream):
        unfused_calls(q, layers, bufs, eps, ev)
    sw_ms = []
    with torch.cuda.stream(stream):
        for _ in range(3):
            ge.replay()
    barrier()
    for _ in range(max(1, min(K // 100, 30))):
        with torch.cuda.stream(stream):
            ge.replay()
        barrier()
        sw_ms += [s_.elapsed_time(e_) for s_, e_ in ev]
    # The roofline kernel as it runs in a chain: a graph of this token's
    # n_layers gate.up launches back to back (each layer's own weights, more
    # bytes than L2), events around the replays.  Events around every single
    # launch (above) also time the launch gaps they force.
    gs = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gs, stream=stream):
        for L in layers:
            q.swiglu_qgemv(L["gate"], L["up"], bufs["h"], L["mlp_norm"], eps, h=bufs["act"])
    with torch.cuda.stream(stream):
        for _ in range(3):
            gs.replay()
    barrier()
    Rs = max(1, min(K // 10, 300))
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(Rs):
            gs.replay()
    s1.record(stream)
    barrier()
    sw_chain_ms = s0.elapsed_time(s1) / (Rs * n_layers)
    swiglu_bytes = dict(ops)["gate_up_swiglu"]
    status = q.device_status()

    ms, ms_e2e = max_over_ranks(torch, [ms, ms_e2e], device, world)

    peak, peak_kind = measured_peak()
    value = world * step_bytes * K / (ms * 1e-3) / 1e9
    e2e_value = world * step_bytes * Ke / (ms_e2e * 1e-3) / 1e9
    sw_avg = statistics.mean(sw_ms)
    achieved = swiglu_bytes / (sw_chain_ms * 1e-3) / 1e9
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline()
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(ms / K, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp16 activations, 4-bit g64 weights, fp32 accumulate",
        "data": "synthetic (seeded; %d device copies of one Llama-3.1-8B-shaped layer)" % n_layers,
        "config": {
            "workload": "Llama-3.1-8B-shaped decode layer x%d, w4g64, batch 1" % n_layers,
            "layers_per_step": n_layers,
            "bytes_per_step": step_bytes,
            "l2": "inputs larger than L2: %.2f GB of distinct weights per step" % (step_bytes / 1e9),
            "timing": "one qgemv_decode_stack call per step (4 streaming-kernel launches "
                      "per layer, programmatic dependent launch); CUDA events on the "
                      "launching stream",
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "us_per_step": round(ms / K * 1e3, 2),
        "us_per_layer": round(ms / K * 1e3 / n_layers, 3),
        "pct_of_peak": round(100.0 * value / world / peak, 1),
        "peak_hbm_gbs": peak,
        "peak_kind": peak_kind,
        "tok_s": round(1e3 * K / ms, 1),
        "roofline": {
            "kernel": "stream_kernel<4, kSwiglu> (swiglu_qgemv, gate.up 4096 -> 2 x 14336, "
                      "RMSNorm fused): the step's dominant kernel",
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": recorded_traffic("swiglu_qgemv_llama8b"),
            "algorithmic_bytes_per_launch": swiglu_bytes,
            "avg_launch_us": round(sw_chain_ms * 1e3, 3),
            "launches_timed": Rs * n_layers,
            "avg_launch_us_isolated": round(sw_avg * 1e3, 3),
            "peak_note": "of %s (MEASURED_PEAKS.json hbm_gbs); avg_launch_us: CUDA events "
                         "around replays of a graph of the token's %d gate.up launches back "
                         "to back (programmatic dependent launch between them, as in the "
                         "stack); avg_launch_us_isolated: events around each launch inside "
                         "the single-op graph of the token, which also times the launch "
                         "gaps the events force" % (peak_kind, n_layers),
        },
        "cpu_baseline": cpu,
        "e2e": {
            "value": round(e2e_value, 1),
            "unit": "GB/s",
            "h2d_bytes_per_step": int(x_host.numel() * 2),
            "d2h_bytes_per_step": int(y_host.numel() * 2),
            "steps": Ke,
            "how": "per token: pinned-host H2D of x, qgemv_decode_stack, D2H of y; "
                   "the tokens are queued back to back with no host sync between them, "
                   "so this is pipelined throughput, not per-token latency",
            "synced_us_per_token": round(lat_us, 1),
            "synced_how": "median wall-clock time of one token (H2D, stack, D2H) with the "
                          "host waiting for its result before the next, over %d tokens"
                          % min(Ke, 50),
        },
        "unfused": unfused,
        "gpu_launches": K * 4 * n_layers,
        "clocks": clk,
        "device_status": status,
        "output_finite": out_ok,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


OPS = ["qkv", "o_proj", "swiglu", "down", "moe", "moe_routed", "lm_head", "lm_head_argmax",
       "lm_head_sample", "gemv1024", "lut_layer", "lut_lm_head",
       "qwen_stack", "w2_layer", "w8_layer", "m2", "m4", "m8", "m2_w2", "m4_w2", "m8_w2",
       "residual_rmsnorm"]


def run_op(args):
    """One op (or one workload configuration's unit of work) timed alone:
    a CUDA graph of at least 32 calls on rotating device copies of the
    weights (more bytes than L2 unless `--copies` says otherwise), replayed;
    one JSON line per op: the mean over all replays (`us_per_call`) and
    p10 / p50 / p90 of 100-200 replays timed one by one (`us_per_call_pct`,
    per call).  `--op all` runs every entry of OPS."""
    names = OPS if args.op == "all" else [args.op]
    for name in names:
        run_one_op(args, name)
    return 0


def run_one_op(args, name):
    import numpy as np
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import bit_group_quantized_qgemv_gb300 as q
    from bit_group_quantized_qgemv_gb300 import accounting as acc
    import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    eps = 1e-5

    def up(w):
        return (torch.from_numpy(np.ascontiguousarray(w.codes).view(np.int32)).to(dev),
                torch.from_numpy(w.scales).to(dev), torch.from_numpy(w.biases).to(dev))

    c8, cq = synth.LLAMA8B, synth.QWEN06B
    H, I = c8["hidden"], c8["inter"]
    qkv_n = (c8["n_q"] + 2 * c8["n_kv"]) * c8["head_dim"]
    graph = True
    config = "config 1: Llama-3.1-8B-shaped layer op"
    if name in ("qkv", "o_proj", "swiglu", "down"):
        layer = synth.llama_layer(1, 0, 4)
        x = torch.from_numpy(layer["x"]).to(dev)
        ops = dict(acc.llama8b_layer_ops(4))
        xi = torch.randn(I, device=dev).half()
        g = torch.from_numpy(layer["gamma1" if name == "qkv" else "gamma2"]).to(dev)
        y = torch.empty(max(I, qkv_n), device=dev).half()
        if name == "swiglu":
            base = (up(layer["gate"]), up(layer["up"]))
            nbytes = ops["gate_up_swiglu"]
        else:
            key = {"qkv": "qkv", "o_proj": "o", "down": "down"}[name]
            base = (up(layer[key]),)
            nbytes = ops[{"qkv": "rmsnorm_qkv", "o_proj": "o_proj_residual",
                          "down": "down_residual"}[name]]

        def call(w):
            if name == "qkv":
                q.rmsnorm_qgemv(w[0], x, g, eps, y=y[:qkv_n])
            elif name == "o_proj":
                q.qgemv_w4g64(w[0], x, y=y[:H], residual=x)
            elif name == "swiglu":
                q.swiglu_qgemv(w[0], w[1], x, g, eps, h=y[:I])
            else:
                q.qgemv_w4g64(w[0], xi, y=y[:H], residual=x)
        launches = 1
    elif name in ("moe", "moe_routed"):
        config = "config 3: MoE token, 4 of 512 experts, combine + residual"
        gu, dn = synth.moe_experts(3, 0, 8)
        base = (up(gu), up(dn))
        nbytes = acc.moe_token_bytes()
        x = torch.from_numpy(synth.activation(synth.rng(3, 0, synth.TID["x"]), H)).to(dev)
        idx = torch.tensor([0, 3, 5, 6], dtype=torch.int32, device=dev)
        wt = torch.tensor([0.4, 0.3, 0.2, 0.1], dtype=torch.float32, device=dev)
        work = torch.empty(4 * 1024, dtype=torch.float32, device=dev)
        y = torch.empty(H, device=dev).half()
        launches = 2
        if name == "moe_routed":
            # the router on the GPU too: an 8 x 4096 router (the 8 resident
            # experts of the rotated copies), shared expert 0 + 3 routed
            config = ("config 3: MoE token with its routing on the GPU (router GEMV, top-K "
                      "selection, softmax) + 4 experts + combine + residual")
            wr = synth.quant_weight(synth.rng(3, 0, synth.TID["router"]), 8, H, 4)
            base = (up(gu), up(dn), up(wr))
            nbytes += acc.matvec_bytes(8, H, 4) + 4 * (4 + 4)
            rlog = torch.empty(8, device=dev).half()
            launches = 4

        def call(w):
            if name == "moe_routed":
                q.moe_router(w[2], x, top_k=4, shared=0, logits=rlog, idx=idx, wt=wt)
            q.moe_qgemv_combine(w[0], w[1], idx, wt, x, x, y=y, workspace=work)
    elif name in ("lm_head", "lm_head_argmax", "lm_head_sample", "gemv1024"):
        if name == "lm_head":
            config = "config 2: Qwen3-0.6B-shaped lm_head 1024->151936"
            N, K, wl = cq["vocab"], cq["hidden"], 2
        elif name == "lm_head_argmax":
            config = ("config 2: Qwen3-0.6B-shaped lm_head 1024->151936 with the greedy token "
                      "chosen on the GPU")
            N, K, wl = cq["vocab"], cq["hidden"], 2
        elif name == "lm_head_sample":
            config = ("config 2: Qwen3-0.6B-shaped lm_head 1024->151936 with top-k sampling "
                      "(k = 50, temperature 0.8) on the GPU")
            N, K, wl = cq["vocab"], cq["hidden"], 2
        else:
            config = "config 0: single 4-bit g64 GEMV 1024x1024"
            N, K, wl = 1024, 1024, 0
        w0 = synth.quant_weight(synth.rng(wl, 0, synth.TID["lm_head" if wl == 2 else "qkv"]), N, K)
        base = (up(w0),)
        nbytes = acc.matvec_bytes(N, K, 4)
        x = torch.from_numpy(synth.activation(synth.rng(wl, 0, synth.TID["x"]), K)).to(dev)
        y = torch.empty(N, device=dev).half()
        am_scratch = torch.zeros(q.argmax_scratch_bytes(), dtype=torch.uint8, device=dev)
        am_token = torch.empty(1, dtype=torch.int32, device=dev)
        u = torch.from_numpy(synth.uniforms(synth.rng(6, 0, synth.TID["u"]), 1)).to(dev)

        def call(w):
            if name == "lm_head_argmax":
                q.lm_head_argmax(w[0], x, logits=y, scratch=am_scratch, token=am_token)
            elif name == "lm_head_sample":
                q.lm_head_sample(w[0], x, 50, 0.8, u, logits=y, token=am_token)
            else:
                q.qgemv_w4g64(w[0], x, y=y)
        launches = 1 if name in ("lm_head", "gemv1024") else 2
    elif name in ("w2_layer", "w8_layer"):
        wb = 2 if name == "w2_layer" else 8
        config = ("config 4: the five matvecs of one 8B-shaped layer at 2-bit" if wb == 2 else
                  "Q8 group 64: the five matvecs of one 8B-shaped layer at 8-bit")
        layer = synth.llama_layer(4 if wb == 2 else 5, 0, wb)
        shapes = [("qkv", qkv_n, H), ("o", H, H), ("gate", I, H), ("up", I, H), ("down", H, I)]
        base = tuple(up(layer[k]) for k, _, _ in shapes)
        nbytes = sum(acc.matvec_bytes(n, k, wb) for _, n, k in shapes)
        xs = {H: torch.randn(H, device=dev).half(), I: torch.randn(I, device=dev).half()}
        y = torch.empty(max(I, qkv_n), device=dev).half()
        fn = q.qgemv_w2g64 if wb == 2 else q.qgemv_w8g64

        def call(w):
            for (key, n, k), wi in zip(shapes, w):
                fn(wi, xs[k], y=y[:n])
        launches = len(shapes)
    elif name in ("lut_layer", "lut_lm_head"):
        if name == "lut_layer":
            config = ("LUT / palettised 4-bit (16-entry fp16 table per row): the five matvecs "
                      "of one 8B-shaped layer")
            shapes = [("qkv", qkv_n, H), ("o", H, H), ("gate", I, H), ("up", I, H), ("down", H, I)]
        else:
            config = ("LUT / palettised 4-bit, one table for the tensor: Qwen3-0.6B-shaped "
                      "lm_head 1024->151936")
            shapes = [("lm_head", cq["vocab"], cq["hidden"])]
        lw = [synth.lut_weight(synth.rng(7, i, synth.TID["lut"]), n, k,
                               1 if name == "lut_layer" else n)
              for i, (_, n, k) in enumerate(shapes)]
        base = tuple((torch.from_numpy(w.codes.view(np.int32)).to(dev),
                      torch.from_numpy(w.lut).to(dev)) for w in lw)
        rpl = [w.rows_per_lut for w in lw]
        nbytes = sum(w.nbytes + 2 * w.K + 2 * w.N for w in lw)
        xs = {k: torch.randn(k, device=dev).half() for _, _, k in shapes}
        y = torch.empty(max(n for _, n, _ in shapes), device=dev).half()

        def call(w):
            for (key, n, k), wi, rows in zip(shapes, w, rpl):
                q.qgemv_lut4(wi[0], wi[1], xs[k], rows_per_lut=rows, y=y[:n])
        launches = len(shapes)
    elif name in ("m2", "m4", "m8", "m2_w2", "m4_w2", "m8_w2"):
        M = int(name[1])
        bits = 2 if name.endswith("w2") else 4
        config = "config 4: M=%d small batch, %d-bit, o_proj- and down-shaped" % (M, bits)
        shapes = [(H, H), (H, I)]
        base = tuple(up(synth.quant_weight(synth.rng(4, n + k, synth.TID["qkv"]), n, k, bits))
                     for n, k in shapes)
        nbytes = sum(acc.matvec_bytes(n, k, bits, M=M) for n, k in shapes)
        xs = [torch.randn(M, k, device=dev).half() for _, k in shapes]
        ys = [torch.empty(M, n, device=dev).half() for n, _ in shapes]
        fn = q.qgemv_w2g64 if bits == 2 else q.qgemv_w4g64

        def call(w):
            for wi, xi_, yi in zip(w, xs, ys):
                fn(wi, xi_, y=yi)
        # one launch per matrix (at M = 8 the down projection splits K over
        # clusters of two CTAs inside its one launch)
        launches = 2
    elif name == "residual_rmsnorm":
        config = "residual add + RMSNorm epilogue, hidden 4096 (qgemv_residual_rmsnorm)"
        K = H
        base = ((torch.from_numpy(synth.activation(synth.rng(1, 0, synth.TID["x"]), K)).to(dev),
                 torch.from_numpy(synth.activation(synth.rng(1, 0, synth.TID["residual"]), K)).to(dev),
                 torch.from_numpy(synth.norm_gamma(synth.rng(1, 0, synth.TID["gamma1"]), K)).to(dev)),)
        nbytes = 3 * 2 * K + 2 * 2 * K  # x, r, gamma read; h, xn written
        hbuf = torch.empty(K, device=dev).half()
        xnbuf = torch.empty(K, device=dev).half()

        def call(w):
            q.residual_rmsnorm(w[0][0], w[0][2], w[0][1], eps, h=hbuf, xn=xnbuf)
        launches = 1
    elif name == "qwen_stack":
        config = "config 2: Qwen3-0.6B-shaped decode stack, 28 layers + lm_head"
        graph = False  # one qgemv_decode_stack call (+ lm_head) per token
        nl = cq["layers"]
        r = lambda t: synth.rng(2, 0, synth.TID[t])  # noqa: E731
        Hq, Iq = cq["hidden"], cq["inter"]
        Dq = cq["n_q"] * cq["head_dim"]
        qn = (cq["n_q"] + 2 * cq["n_kv"]) * cq["head_dim"]
        one = {"qkv": up(synth.quant_weight(r("qkv"), qn, Hq)),
               "o": up(synth.quant_weight(r("o"), Hq, Dq)),
               "gate": up(synth.quant_weight(r("gate"), Iq, Hq)),
               "up": up(synth.quant_weight(r("up"), Iq, Hq)),
               "down": up(synth.quant_weight(r("down"), Hq, Iq)),
               "attn_norm": torch.from_numpy(synth.norm_gamma(r("gamma1"), Hq)).to(dev),
               "mlp_norm": torch.from_numpy(synth.norm_gamma(r("gamma2"), Hq)).to(dev)}
        layers = [{k: (tuple(t.clone() for t in v) if isinstance(v, tuple) else v.clone())
                   for k, v in one.items()} for _ in range(nl)]
        lm = up(synth.quant_weight(r("lm_head"), cq["vocab"], Hq))
        shape = q.stack_shape(Hq, cq["n_q"], cq["n_kv"], cq["head_dim"], Iq, nl, eps)
        descs = q.stack_layers(layers)
        work = torch.empty(q.decode_stack_workspace_bytes(shape), dtype=torch.uint8, device=dev)
        x = torch.from_numpy(synth.activation(r("x"), Hq)).to(dev)
        hidden = torch.empty(Hq, device=dev).half()
        logits = torch.empty(cq["vocab"], device=dev).half()
        layer_bytes = (acc.matvec_bytes(qn, Hq, 4, gamma=True) +
                       acc.matvec_bytes(Hq, Dq, 4, residual=True) +
                       acc.weight_bytes(2 * Iq, Hq, 4) + 2 * Hq + 2 * Hq + 2 * Iq +
                       acc.matvec_bytes(Hq, Iq, 4, residual=True))
        nbytes = nl * layer_bytes + acc.matvec_bytes(cq["vocab"], Hq, 4)
        base = (lm,)

        def call(w):
            q.decode_stack(descs, shape, x, y=hidden, workspace=work)
            q.qgemv_w4g64(w[0], hidden, y=logits)
        launches = 4 * nl + 1
    else:
        raise SystemExit("unknown op " + name)

    weight_bytes = sum(t.numel() * t.element_size() for wt in base for t in wt)
    copies = 1 if name == "qwen_stack" else max(2, int(3 * 129e6 // max(weight_bytes, 1)) + 1)
    if name == "gemv1024":
        copies = max(copies, 512)
    if name == "residual_rmsnorm":  # 24 KB of inputs: an L2-resident epilogue by nature
        copies = 4
    if args.copies > 0 and name != "qwen_stack":
        copies = args.copies
    ws = [base] + [tuple(tuple(t.clone() for t in wt) for wt in base) for _ in range(copies - 1)]
    n_graph = max(copies, 32)  # calls per captured graph, cycling over the copies

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in range(copies):
            call(ws[i])
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if graph:
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg):
            for i in range(n_graph):
                call(ws[i % copies])
        reps = max(1, args.steps // n_graph)
        for _ in range(max(3, args.warmup // n_graph)):
            cg.replay()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            cg.replay()
        e1.record()
        n_calls = reps * n_graph
        # Distribution: events around each of up to 200 further replays.
        pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(min(200, max(100, reps)))]
        for a_, b_ in pev:
            a_.record()
            cg.replay()
            b_.record()
    else:
        reps = max(1, min(args.steps, 300))
        for i in range(max(3, min(args.warmup, 20))):
            call(ws[0])
        torch.cuda.synchronize()
        e0.record()
        for i in range(reps):
            call(ws[0])
        e1.record()
        n_calls = reps
        pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(100)]
        for a_, b_ in pev:
            a_.record()
            call(ws[0])
            b_.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n_calls
    per = sorted(a_.elapsed_time(b_) / (n_graph if graph else 1) for a_, b_ in pev)
    pct = {"p10": round(per[len(per) // 10] * 1e3, 3), "p50": round(per[len(per) // 2] * 1e3, 3),
           "p90": round(per[(9 * len(per)) // 10] * 1e3, 3), "replays": len(per)}
    peak, peak_kind = measured_peak()
    gbs = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({"op": name, "config": config,
                      "metric": "achieved HBM GB/s of one unit (CUDA-graph replays)" if graph
                      else "achieved HBM GB/s of one unit (stream launches)",
                      "value": round(gbs, 1), "unit": "GB/s", "us_per_call": round(ms * 1e3, 3),
                      "us_per_call_pct": pct,
                      "bytes_per_call": nbytes, "launches_per_call": launches,
                      "weight_copies": copies,
                      "l2_resident": bool(copies * max(weight_bytes, nbytes) < 129e6),
                      "calls_timed": n_calls, "peak": peak,
                      "peak_kind": peak_kind, "frac": round(gbs / peak, 4),
                      "device_status": q.device_status()}), flush=True)


# ------------------------------------------------------- CPU baseline
def oracle_layer_sample(rows_frac: int):
    """Inputs of one Llama-8B-shaped layer with every matrix cut to its first
    N // rows_frac rows (rows_frac = 1 for the whole layer)."""
    import numpy as np

    import synth
    layer = synth.llama_layer(1, 0, 4)
    c = synth.LLAMA8B
    H, I = c["hidden"], c["inter"]

    def cut(w):
        n = max(1, w.N // rows_frac)
        return synth.QuantWeight(w.codes[:n], w.scales[:n], w.biases[:n], 4)

    sample = {k: cut(layer[k]) for k in ("qkv", "o", "gate", "up", "down")}
    g = synth.rng(1, 0, synth.TID["spare"])
    return sample, layer["gamma1"], layer["gamma2"], layer["x"], \
        synth.activation(g, c["n_q"] * c["head_dim"]), synth.activation(g, I), H


def oracle_step(sample, g1, g2, x, a, act):
    import oracle
    s = sample
    oracle.rmsnorm_qgemv(s["qkv"].codes, s["qkv"].scales, s["qkv"].biases, x, g1, 1e-5)
    oracle.qgemv(4, s["o"].codes, s["o"].scales, s["o"].biases, a, x[:s["o"].N])
    oracle.swiglu_qgemv((s["gate"].codes, s["gate"].scales, s["gate"].biases),
                        (s["up"].codes, s["up"].scales, s["up"].biases), x, g2, 1e-5)
    oracle.qgemv(4, s["down"].codes, s["down"].scales, s["down"].biases, act, x[:s["down"].N])


def accounting_module():
    """The byte-accounting module, loaded by file path: importing it through
    the package would run the package's __init__, which loads libqgemv.so,
    and the oracle arm must not map the product library."""
    import importlib.util
    name = "qgemv_accounting"
    if name in sys.modules:
        return sys.modules[name]
    path = os.path.join(ROOT, "bit_group_quantized_qgemv_gb300", "accounting.py")
    spec = importlib.util.spec_from_file_location(name, path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    sys.modules[name] = mod
    return mod


def sample_bytes(sample, H):
    acc = accounting_module()
    b = 0
    for k in ("qkv", "o", "gate", "up", "down"):
        w = sample[k]
        b += acc.weight_bytes(w.N, w.K, 4) + 2 * w.K + 2 * w.N
    return b + 2 * H * 2


def cpu_baseline():
    """The fp64 oracle as it stands, on this host's cores: one whole
    Llama-8B-shaped layer (all four matvecs), repeated to ~10+ s of CPU work."""
    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    sample, g1, g2, x, a, act, H = oracle_layer_sample(1)
    nbytes = sample_bytes(sample, H)
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle_step(sample, g1, g2, x, a, act)
        reps += 1
        el = time.perf_counter() - t0
        if el * cores >= 12.0 or reps >= 8:
            break
    return {"value": round(nbytes * reps / el / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": "%d pass(es) of one whole Llama-8B-shaped layer (QKV+norm, o_proj, "
                      "gate.up SwiGLU+norm, down), fp64 C oracle, %.1f s wall" % (reps, el)}


# ------------------------------------------------------ reference arm
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    rows_frac = 64
    sample, g1, g2, x, a, act, H = oracle_layer_sample(rows_frac)
    nbytes = sample_bytes(sample, H)
    for _ in range(args.warmup):
        oracle_step(sample, g1, g2, x, a, act)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(sample, g1, g2, x, a, act)
    el = time.perf_counter() - t0
    value = nbytes * args.steps / el / 1e9
    desc = ("1/%d of the rows of every matvec of one Llama-8B-shaped layer per step, "
            "fp64 C oracle" % rows_frac)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(el / max(1, args.steps) * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": "Llama-3.1-8B-shaped decode layer, w4g64, batch 1 (row sample)",
                   "rows_fraction": 1.0 / rows_frac, "bytes_per_step": nbytes},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.op != "stack":
        return run_op(args)
    return run_own(args)


if __name__ == "__main__":
    sys.exit(main())
