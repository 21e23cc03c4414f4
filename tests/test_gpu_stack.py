"""qgemv_decode_stack against the chain of single-op C-ABI calls.

The stack kernel performs, per layer, the same arithmetic and the same fp16
roundings as rmsnorm_qgemv -> decode_attention_seq1 -> qgemv_w4g64 (+x) ->
swiglu_qgemv (+norm) -> qgemv_w4g64 (+h), each of which is parity-tested
against the oracle.  The only difference is the order of the RMS sum, so
the outputs agree to far within the down projection's tolerance
2e-3 * sum|w||act| + |h| (evaluated by the oracle on the chain's inputs).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from qhelpers import check, dev16, dev_weight, plain_tol

pytestmark = pytest.mark.gpu

q = pytest.importorskip("bit_group_quantized_qgemv_gb300")


def make_layers(wl, n_layers, H, nq, nkv, hd, I):
    layers, host = [], []
    for l in range(n_layers):
        r = lambda t: synth.rng(wl, l, synth.TID[t])  # noqa: E731
        W = {"qkv": synth.quant_weight(r("qkv"), (nq + 2 * nkv) * hd, H),
             "o": synth.quant_weight(r("o"), H, nq * hd),
             "gate": synth.quant_weight(r("gate"), I, H), "up": synth.quant_weight(r("up"), I, H),
             "down": synth.quant_weight(r("down"), H, I)}
        g1, g2 = synth.norm_gamma(r("gamma1"), H), synth.norm_gamma(r("gamma2"), H)
        d = {k: dev_weight(v) for k, v in W.items()}
        d["attn_norm"], d["mlp_norm"] = dev16(g1), dev16(g2)
        layers.append(d)
        host.append(W)
    return layers, host


def chain(layers, x, nq, nkv, hd, eps):
    """Layer-by-layer chain of the single-op entry points; returns the final
    output and the last layer's (act, h) for the tolerance."""
    for L in layers:
        qkv = q.rmsnorm_qgemv(L["qkv"], x, L["attn_norm"], eps)
        attn = q.decode_attention_seq1(qkv, nq, nkv, hd)
        h = q.qgemv_w4g64(L["o"], attn, residual=x)
        act = q.swiglu_qgemv(L["gate"], L["up"], h, L["mlp_norm"], eps)
        x = q.qgemv_w4g64(L["down"], act, residual=h)
    return x, act, h


@pytest.mark.parametrize("shape", [
    dict(H=1024, nq=8, nkv=2, hd=128, I=2048, L=1),
    dict(H=1024, nq=8, nkv=2, hd=128, I=2048, L=3),
    dict(H=1024, nq=16, nkv=8, hd=128, I=3072, L=2),       # Qwen3-0.6B-shaped layers
    # Llama-3.1-8B-shaped: one layer.  With the synthetic recipe every weight
    # has mean -0.5 * scale (bias -8 * scale, codes uniform in 0..15), so a
    # common-mode component grows from layer to layer and the second 8B-sized
    # layer overflows fp16 in the op chain and the stack alike.
    dict(H=4096, nq=32, nkv=8, hd=128, I=14336, L=1),
])
def test_stack_matches_op_chain(shape):
    H, nq, nkv, hd, I, NL = (shape[k] for k in ("H", "nq", "nkv", "hd", "I", "L"))
    eps = 1e-5
    layers, host = make_layers(400 + H, NL, H, nq, nkv, hd, I)
    x = dev16(synth.activation(synth.rng(400, H, synth.TID["x"]), H))
    y_chain, act, h = chain(layers, x, nq, nkv, hd, eps)
    sh = q.stack_shape(H, nq, nkv, hd, I, NL, eps)
    y = q.decode_stack(layers, sh, x)
    torch.cuda.synchronize()
    down = host[-1]["down"]
    _, _, bound = oracle.qgemv(4, down.codes, down.scales, down.biases, act.cpu().numpy(),
                               h.cpu().numpy())
    check(y, y_chain.double().cpu().numpy(), plain_tol(bound), f"stack {shape}")
    # twice in a row on the same workspace gives the same result
    ws = torch.empty(q.decode_stack_workspace_bytes(sh), dtype=torch.uint8, device="cuda")
    y1 = q.decode_stack(layers, sh, x, workspace=ws)
    y2 = q.decode_stack(layers, sh, x, workspace=ws)
    assert torch.equal(y1, y2) and torch.equal(y1, y)
    assert q.device_status() == 0


def test_stack_rejects_bad_shapes():
    x = torch.zeros(1024, dtype=torch.float16, device="cuda")
    layers, _ = make_layers(401, 1, 1024, 8, 2, 128, 2048)
    for bad in (q.stack_shape(1000, 8, 2, 128, 2048, 1), q.stack_shape(1024, 8, 3, 128, 2048, 1),
                q.stack_shape(1024, 8, 2, 128, 2048, 0), q.stack_shape(1024, 8, 2, 128, 2048, 1, 0.0)):
        with pytest.raises(q.QgemvError):
            q.decode_stack(layers, bad, x, workspace=torch.empty(1 << 20, dtype=torch.uint8,
                                                                  device="cuda"))


def test_stack_graph_cache_and_caller_capture():
    """Repeated calls replay a cached graph; more distinct argument sets than
    the cache holds, and a call inside the caller's own stream capture, give
    the same bits as the first (captured) call."""
    H, nq, nkv, hd, I, NL = 1024, 8, 2, 128, 2048, 2
    layers, _ = make_layers(402, NL, H, nq, nkv, hd, I)
    sh = q.stack_shape(H, nq, nkv, hd, I, NL, 1e-5)
    arr = q.stack_layers(layers)
    x = dev16(synth.activation(synth.rng(402, H, synth.TID["x"]), H))
    ws = torch.empty(q.decode_stack_workspace_bytes(sh), dtype=torch.uint8, device="cuda")
    ref = q.decode_stack(arr, sh, x, workspace=ws).clone()
    ys = [torch.empty(H, dtype=torch.float16, device="cuda") for _ in range(6)]
    for rep in range(2):                       # 6 keys > 4 cached: evictions, then re-captures
        for y in ys:
            q.decode_stack(arr, sh, x, y=y, workspace=ws)
            torch.cuda.synchronize()
            assert torch.equal(y, ref), rep
    y = torch.empty(H, dtype=torch.float16, device="cuda")
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            q.decode_stack(arr, sh, x, y=y, workspace=ws)
    torch.cuda.synchronize()
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, ref)
    assert q.device_status() == 0


def test_bench_configuration_32_layers():
    """The configuration bench.py times: 32 device copies of one
    Llama-3.1-8B-shaped layer and the benchmark's input, one
    qgemv_decode_stack call.  The chain of single-op calls' last down
    projection is checked against the oracle on its own fp16 inputs
    (stage-isolated), and the stack's output against the chain within that
    projection's tolerance."""
    import bench
    c = synth.LLAMA8B
    layers, x0, _ = bench.build_stack(torch, 32, torch.device("cuda", 0))
    sh = q.stack_shape(c["hidden"], c["n_q"], c["n_kv"], c["head_dim"], c["inter"], 32, c["eps"])
    y = q.decode_stack(layers, sh, x0)
    y_chain, act, h = chain(layers, x0, c["n_q"], c["n_kv"], c["head_dim"], c["eps"])
    torch.cuda.synchronize()
    assert bool(torch.isfinite(y.float()).all())
    down = synth.llama_layer(1, 0, 4)["down"]
    y64, _, bound = oracle.qgemv(4, down.codes, down.scales, down.biases, act.cpu().numpy(),
                                 h.cpu().numpy())
    check(y_chain, y64, plain_tol(bound), "bench configuration: chain's last down vs oracle")
    check(y, y_chain.double().cpu().numpy(), plain_tol(bound),
          "bench configuration: stack vs single-op chain")
    assert q.device_status() == 0
