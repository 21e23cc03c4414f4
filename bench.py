#!/usr/bin/env python
"""Benchmark: dequant-fused 4-bit GEMV decode stack on one GB300.

Workload: one decode token (batch 1) through a stack of 32
Llama-3.1-8B-shaped layers, each the fused matvec chain
    rmsnorm_qgemv(QKV 4096->6144) -> decode_attention_seq1 (value-head copy)
    -> qgemv_w4g64(o_proj 4096->4096, + residual)
    -> swiglu_qgemv(gate.up 4096->2x14336, post-attention RMSNorm fused)
    -> qgemv_w4g64(down 14336->4096, + residual)
with 4-bit group-64 planar weights.  A step is one token through all 32
layers (3.93 GB of distinct device weights, so no step's inputs fit in the
129 MB L2).  The 32 layers are device copies of one seeded synthetic layer.

Metric: algorithmic HBM GB/s (codes + scales + biases + activations read and
written, per the byte accounting of bit_group_quantized_qgemv_gb300.accounting)
divided by the device time of the step, plus us per decode matvec stack.

Timing: the step is captured once as a CUDA graph of C-ABI calls; W warm-up
and K timed replays on one stream, CUDA events around the K, a barrier and
torch.cuda.synchronize() on both sides, max over ranks.  Events captured
around every gate.up SwiGLU launch give the dominant kernel's live duration.
`--impl reference` times the fp64 CPU oracle on a bounded row sample of the
same layer instead.
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
    return p.parse_args()


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


def kernel_sources_digest():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_group_quantized_qgemv_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
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
def build_stack(q, torch, n_layers, device):
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
                      {"gamma1": g1.clone(), "gamma2": g2.clone()})
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


def step_calls(q, layers, bufs, eps, events=None):
    """Enqueue one token through the stack (C-ABI calls on the current stream)."""
    import synth
    c = synth.LLAMA8B
    x, qkv, attn, h, act = bufs["x"], bufs["qkv"], bufs["attn"], bufs["h"], bufs["act"]
    for li, L in enumerate(layers):
        q.rmsnorm_qgemv(L["qkv"], x, L["gamma1"], eps, y=qkv)
        q.decode_attention_seq1(qkv, c["n_q"], c["n_kv"], c["head_dim"], out=attn)
        q.qgemv_w4g64(L["o"], attn, y=h, residual=x)
        if events is not None:
            events[li][0].record()
        q.swiglu_qgemv(L["gate"], L["up"], h, L["gamma2"], eps, h=act)
        if events is not None:
            events[li][1].record()
        q.qgemv_w4g64(L["down"], act, y=x, residual=h)


def run_own(args):
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import bit_group_quantized_qgemv_gb300 as q
    from bit_group_quantized_qgemv_gb300 import accounting as acc

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

    n_layers = args.layers
    eps = 1e-5
    layers, x0, bufs = build_stack(q, torch, n_layers, device)
    ops = acc.llama8b_layer_ops(4)
    layer_bytes = sum(b for _, b in ops) + 2 * 2 * 128 * 32  # + the value-head copy
    step_bytes = n_layers * layer_bytes
    swiglu_bytes = dict(ops)["gate_up_swiglu"]

    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        bufs["x"].copy_(x0)
        step_calls(q, layers, bufs, eps)          # eager warm-up (sets kernel attributes)
    torch.cuda.synchronize()
    if q.device_status() != 0:
        raise RuntimeError("device-side wait timed out during warm-up")

    def timing_event():
        # external=True makes a record inside graph capture a real event node
        try:
            return torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            return torch.cuda.Event(enable_timing=True)

    # One graph per ring slot, each with its own events around gate.up SwiGLU.
    ring = 4
    graphs, evsets = [], []
    for _ in range(ring):
        ev = [(timing_event(), timing_event()) for _ in range(n_layers)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step_calls(q, layers, bufs, eps, ev)
        graphs.append(g)
        evsets.append(ev)
    # End-to-end graph: H2D of the token's input from pinned host memory,
    # the stack, D2H of its output.
    x_host = x0.cpu().pin_memory()
    y_host = torch.empty_like(x_host).pin_memory()
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e, stream=stream):
        bufs["x"].copy_(x_host, non_blocking=True)
        step_calls(q, layers, bufs, eps)
        y_host.copy_(bufs["x"], non_blocking=True)
    torch.cuda.synchronize()

    K, W = args.steps, args.warmup
    gpu_id = "0"
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        gpu_id = str(local)

    # ---- timed region: K steps of the device-resident stack
    with torch.cuda.stream(stream):
        for i in range(W):
            graphs[i % ring].replay()
    barrier()
    clocks = ClockSampler(gpu_id)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record()
        for i in range(K):
            graphs[i % ring].replay()
        t_end.record()
    barrier()
    clk = clocks.stop()
    ms = t_start.elapsed_time(t_end)
    swiglu_ms = [a.elapsed_time(b) for ev in evsets for a, b in ev]
    # ---- timed region: end to end with host buffers
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    Ke = max(1, min(K, 1000))
    with torch.cuda.stream(stream):
        for _ in range(min(W, 20)):
            g_e2e.replay()
    barrier()
    with torch.cuda.stream(stream):
        e0.record()
        for _ in range(Ke):
            g_e2e.replay()
        e1.record()
    barrier()
    ms_e2e = e0.elapsed_time(e1)
    out_ok = bool(torch.isfinite(y_host.float()).all())
    status = q.device_status()

    if world > 1:
        t = torch.tensor([ms, ms_e2e], device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms, ms_e2e = float(t[0]), float(t[1])

    peak, peak_kind = measured_peak()
    value = world * step_bytes * K / (ms * 1e-3) / 1e9
    e2e_value = world * step_bytes * Ke / (ms_e2e * 1e-3) / 1e9
    sw_ms = statistics.mean(swiglu_ms)
    achieved = swiglu_bytes / (sw_ms * 1e-3) / 1e9
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
        "data": "synthetic (seeded; 32 device copies of one Llama-3.1-8B-shaped layer)",
        "config": {
            "workload": "Llama-3.1-8B-shaped decode layer x%d, w4g64, batch 1" % n_layers,
            "layers_per_step": n_layers,
            "bytes_per_step": step_bytes,
            "l2": "inputs larger than L2: %.2f GB of distinct weights per step" % (step_bytes / 1e9),
            "timing": "CUDA graph of C-ABI calls per step, CUDA events on the launching stream",
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "us_per_step": round(ms / K * 1e3, 2),
        "us_per_layer": round(ms / K * 1e3 / n_layers, 3),
        "pct_of_peak": round(100.0 * value / world / peak, 1),
        "peak_hbm_gbs": peak,
        "peak_kind": peak_kind,
        "tok_s": round(1e3 * K / ms, 1),
        "roofline": {
            "kernel": "swiglu_qgemv (gate.up 4096 -> 2 x 14336, RMSNorm fused)",
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": recorded_traffic("swiglu_qgemv_llama8b"),
            "algorithmic_bytes_per_launch": swiglu_bytes,
            "avg_launch_us": round(sw_ms * 1e3, 3),
            "launches_timed": len(swiglu_ms),
            "peak_note": "of %s (MEASURED_PEAKS.json hbm_gbs)" % peak_kind,
        },
        "cpu_baseline": cpu,
        "e2e": {
            "value": round(e2e_value, 1),
            "unit": "GB/s",
            "h2d_bytes_per_step": int(x_host.numel() * 2),
            "d2h_bytes_per_step": int(y_host.numel() * 2),
            "steps": Ke,
            "how": "CUDA graph per token: pinned-host H2D of x, the stack via C-ABI calls, D2H of y",
        },
        "gpu_launches": K * n_layers * 5,
        "clocks": clk,
        "device_status": status,
        "output_finite": out_ok,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


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


def sample_bytes(sample, H):
    from bit_group_quantized_qgemv_gb300 import accounting as acc
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
    return run_own(args)


if __name__ == "__main__":
    sys.exit(main())
