"""qgemv_decode_stack against the oracle, stage by stage.

The stack keeps its intermediates in the caller's workspace (qkv, h, act and
the x ping-pong, at the offsets qgemv_decode_stack_workspace_bytes sums), so
after a call they hold the last layer's stage inputs and outputs.  Each
stage is checked element by element against the oracle fed the stack's OWN
fp16 input to that stage (stage-isolated, so the bounds do not compound):

  qkv  = rmsnorm_qgemv(W_qkv, x_l, attn_norm)       oracle.rmsnorm_qgemv
  h    = W_o . value_heads(qkv) + x_l               oracle.qgemv (+ residual)
  act  = swiglu(W_gate, W_up, h, mlp_norm)          oracle.swiglu_qgemv
  y    = W_down . act + h                           oracle.qgemv (+ residual)

where x_l, the last layer's input, is the call's x for one layer and the
previous layer's output (in the ping-pong buffer) otherwise.  Running every
prefix of a stack (n_layers = 1, 2, 3, ...) as its own call checks every
layer.  The layer block is the pre-norm reading of INFERENCE_RESEARCH.md
section 1 (one command buffer for the whole stack, fused RMSNorm->QKV and
gate.up SwiGLU) with the seq-len-1 attention stand-in.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from qhelpers import check, dev16, dev_weight, plain_tol

pytestmark = pytest.mark.gpu

q = pytest.importorskip("bit_group_quantized_qgemv_gb300")


def _up256(b):
    return (b + 255) // 256 * 256


def workspace_views(ws, H, nq, nkv, hd, I):
    """fp16 views of the stack's workspace: qkv, h, act, x ping-pong."""
    nqkv = (nq + 2 * nkv) * hd
    sizes = [nqkv, H, I, H, H]
    views, off = [], 0
    for n in sizes:
        views.append(ws[off:off + 2 * n].view(torch.float16))
        off += _up256(2 * n)
    assert off <= ws.numel()
    return views


def value_heads(qkv, nq, nkv, hd):
    """Decode over one cached position: query head h reads value head
    h / (nq / nkv) (softmax of one score is 1)."""
    g = nq // nkv
    v0 = (nq + nkv) * hd
    return np.concatenate([qkv[v0 + (h // g) * hd: v0 + (h // g + 1) * hd] for h in range(nq)])


def check_last_layer(W, g1, g2, ws, x_call, y, NL, H, nq, nkv, hd, I, eps, what):
    qkv_d, h_d, act_d, xb0, xb1 = workspace_views(ws, H, nq, nkv, hd, I)
    x_l = x_call if NL == 1 else (xb0 if ((NL - 1) & 1) == 0 else xb1)
    x_l = x_l.cpu().numpy()
    qkv = qkv_d.cpu().numpy()
    h = h_d.cpu().numpy()
    act = act_d.cpu().numpy()
    g1 = g1.cpu().numpy() if torch.is_tensor(g1) else g1
    g2 = g2.cpu().numpy() if torch.is_tensor(g2) else g2
    w = W["qkv"]
    y64, _, bound = oracle.rmsnorm_qgemv(w.codes, w.scales, w.biases, x_l, g1, eps)
    check(qkv_d, y64, plain_tol(bound), f"{what}: qkv")
    w = W["o"]
    y64, _, bound = oracle.qgemv(4, w.codes, w.scales, w.biases,
                                 value_heads(qkv, nq, nkv, hd), x_l)
    check(h_d, y64, plain_tol(bound), f"{what}: o_proj + residual")
    gt, ut = W["gate"], W["up"]
    h64, _, tol = oracle.swiglu_qgemv((gt.codes, gt.scales, gt.biases),
                                      (ut.codes, ut.scales, ut.biases), h, g2, eps)
    check(act_d, h64, tol, f"{what}: gate.up SwiGLU")
    w = W["down"]
    y64, _, bound = oracle.qgemv(4, w.codes, w.scales, w.biases, act, h)
    check(y, y64, plain_tol(bound), f"{what}: down + residual")


def make_layers(wl, n_layers, H, nq, nkv, hd, I):
    layers, host = [], []
    for l in range(n_layers):
        r = lambda t: synth.rng(wl, l, synth.TID[t])  # noqa: E731
        W = {"qkv": synth.quant_weight(r("qkv"), (nq + 2 * nkv) * hd, H),
             "o": synth.quant_weight(r("o"), H, nq * hd),
             "gate": synth.quant_weight(r("gate"), I, H), "up": synth.quant_weight(r("up"), I, H),
             "down": synth.quant_weight(r("down"), H, I),
             "g1": synth.norm_gamma(r("gamma1"), H), "g2": synth.norm_gamma(r("gamma2"), H)}
        d = {k: dev_weight(W[k]) for k in ("qkv", "o", "gate", "up", "down")}
        d["attn_norm"], d["mlp_norm"] = dev16(W["g1"]), dev16(W["g2"])
        layers.append(d)
        host.append(W)
    return layers, host


@pytest.mark.parametrize("shape", [
    dict(H=1024, nq=16, nkv=8, hd=128, I=3072, L=3, wl=410),    # Qwen3-0.6B-shaped layers
    dict(H=1024, nq=8, nkv=2, hd=128, I=2048, L=3, wl=411),
    dict(H=2048, nq=16, nkv=4, hd=128, I=5120, L=2, wl=412),
    # Llama-3.1-8B-shaped: one layer (a second distinct layer overflows fp16
    # with the synthetic weights' common-mode component)
    dict(H=4096, nq=32, nkv=8, hd=128, I=14336, L=1, wl=413),
])
def test_stack_stages_against_oracle_every_prefix(shape):
    H, nq, nkv, hd, I, NL, wl = (shape[k] for k in ("H", "nq", "nkv", "hd", "I", "L", "wl"))
    eps = 1e-5
    layers, host = make_layers(wl, NL, H, nq, nkv, hd, I)
    x = dev16(synth.activation(synth.rng(wl, 99, synth.TID["x"]), H))
    for nl in range(1, NL + 1):
        sh = q.stack_shape(H, nq, nkv, hd, I, nl, eps)
        ws = torch.empty(q.decode_stack_workspace_bytes(sh), dtype=torch.uint8, device="cuda")
        y = q.decode_stack(layers[:nl], sh, x, workspace=ws)
        torch.cuda.synchronize()
        W = host[nl - 1]
        check_last_layer(W, W["g1"], W["g2"], ws, x, y, nl, H, nq, nkv, hd, I, eps,
                         f"{shape} layer {nl - 1}")
    assert q.device_status() == 0


def test_bench_configuration_last_layer_against_oracle():
    """The configuration bench.py times (32 device copies of one seeded
    Llama-3.1-8B-shaped layer, the benchmark's input, one qgemv_decode_stack
    call): the last layer's four stages against the oracle on the stack's
    own inputs, and layers 1..3 through the prefixes of the same stack."""
    import bench
    c = synth.LLAMA8B
    H, nq, nkv, hd, I = c["hidden"], c["n_q"], c["n_kv"], c["head_dim"], c["inter"]
    layers, x0, _ = bench.build_stack(torch, 32, torch.device("cuda", 0))
    src = synth.llama_layer(1, 0, 4)
    for nl in (1, 2, 3, 32):
        sh = q.stack_shape(H, nq, nkv, hd, I, nl, c["eps"])
        ws = torch.empty(q.decode_stack_workspace_bytes(sh), dtype=torch.uint8, device="cuda")
        y = q.decode_stack(layers[:nl], sh, x0, workspace=ws)
        torch.cuda.synchronize()
        assert bool(torch.isfinite(y.float()).all())
        check_last_layer(src, src["gamma1"], src["gamma2"], ws, x0, y, nl, H, nq, nkv, hd, I,
                         c["eps"], f"bench configuration, {nl} layers")
    assert q.device_status() == 0
