"""Full-size parity: every workload configuration at its stated sizes, in the
launch configuration the benchmark uses, checked element by element against
the fp64 oracle (stage-isolated: each kernel gets its own fp16 input, so
tolerance bounds do not compound along a layer).

  config 0  single 4-bit GEMV 1024 x 1024, seed 0
  config 1  Llama-3.1-8B-shaped layer: RMSNorm->QKV 4096->6144, o_proj
            4096->4096 + residual, gate.up 4096->2x14336 SwiGLU (+ norm),
            down 14336->4096 + residual
  config 2  Qwen3-0.6B-shaped layer ops and the lm_head 1024->151936
  config 3  MoE layer: 512 experts resident (3.6 GB), 16 tokens, K = 4
            (shared expert 0 + 3 routed), weighted combine + residual
  config 4  2-bit at the config-1 shapes, and M in {1, 2, 4, 8} for 4-bit
            and 2-bit
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from qhelpers import check, dev16, dev_weight, plain_tol

pytestmark = pytest.mark.gpu

q = pytest.importorskip("bit_group_quantized_qgemv_gb300")


@pytest.fixture(scope="module")
def llama():
    return synth.llama_layer(1, 0, 4)


def test_config0_single_gemv():
    w = synth.quant_weight(synth.rng(0, 0, synth.TID["qkv"]), 1024, 1024, 4)
    x = synth.activation(synth.rng(0, 0, synth.TID["x"]), 1024)
    y = q.qgemv_w4g64(dev_weight(w), dev16(x))
    y64, _, bound = oracle.qgemv(4, w.codes, w.scales, w.biases, x)
    check(y, y64, plain_tol(bound), "config 0")


def test_config1_layer_stage_isolated(llama):
    L = llama
    c = synth.LLAMA8B
    eps = c["eps"]
    x = L["x"]
    # RMSNorm -> QKV
    qkv = q.rmsnorm_qgemv(dev_weight(L["qkv"]), dev16(x), dev16(L["gamma1"]), eps)
    y64, _, bound = oracle.rmsnorm_qgemv(L["qkv"].codes, L["qkv"].scales, L["qkv"].biases, x,
                                         L["gamma1"], eps)
    check(qkv, y64, plain_tol(bound), "config 1 rmsnorm_qkv")
    # value-head copy (bit-exact)
    attn = q.decode_attention_seq1(qkv, c["n_q"], c["n_kv"], c["head_dim"])
    v = qkv.cpu().numpy()[(c["n_q"] + c["n_kv"]) * c["head_dim"]:].reshape(c["n_kv"], -1)
    assert np.array_equal(attn.cpu().numpy(), np.repeat(v, c["n_q"] // c["n_kv"], axis=0).reshape(-1))
    # o_proj + residual, fed the GPU's own attention output
    a16 = attn.cpu().numpy()
    h = q.qgemv_w4g64(dev_weight(L["o"]), attn, residual=dev16(x))
    y64, _, bound = oracle.qgemv(4, L["o"].codes, L["o"].scales, L["o"].biases, a16, x)
    check(h, y64, plain_tol(bound), "config 1 o_proj")
    # gate.up SwiGLU with the post-attention norm
    h16 = h.cpu().numpy()
    act = q.swiglu_qgemv(dev_weight(L["gate"]), dev_weight(L["up"]), h, dev16(L["gamma2"]), eps)
    g = L["gate"]
    u = L["up"]
    h64, _, tol = oracle.swiglu_qgemv((g.codes, g.scales, g.biases), (u.codes, u.scales, u.biases),
                                      h16, L["gamma2"], eps)
    check(act, h64, tol, "config 1 swiglu")
    # down + residual
    act16 = act.cpu().numpy()
    out = q.qgemv_w4g64(dev_weight(L["down"]), act, residual=h)
    y64, _, bound = oracle.qgemv(4, L["down"].codes, L["down"].scales, L["down"].biases, act16, h16)
    check(out, y64, plain_tol(bound), "config 1 down")
    assert q.device_status() == 0


def test_config2_qwen_ops_and_lm_head():
    c = synth.QWEN06B
    H, I, eps = c["hidden"], c["inter"], c["eps"]
    qkv_n = (c["n_q"] + 2 * c["n_kv"]) * c["head_dim"]
    Dq = c["n_q"] * c["head_dim"]
    r = lambda t: synth.rng(2, 0, synth.TID[t])  # noqa: E731
    W = {"qkv": synth.quant_weight(r("qkv"), qkv_n, H), "o": synth.quant_weight(r("o"), H, Dq),
         "gate": synth.quant_weight(r("gate"), I, H), "up": synth.quant_weight(r("up"), I, H),
         "down": synth.quant_weight(r("down"), H, I),
         "lm_head": synth.quant_weight(r("lm_head"), c["vocab"], H)}
    g1, g2 = synth.norm_gamma(r("gamma1"), H), synth.norm_gamma(r("gamma2"), H)
    x = synth.activation(r("x"), H)
    xa = synth.activation(synth.rng(2, 1, synth.TID["x"]), Dq)
    xi = synth.activation(synth.rng(2, 2, synth.TID["x"]), I)
    y = q.rmsnorm_qgemv(dev_weight(W["qkv"]), dev16(x), dev16(g1), eps)
    y64, _, b = oracle.rmsnorm_qgemv(W["qkv"].codes, W["qkv"].scales, W["qkv"].biases, x, g1, eps)
    check(y, y64, plain_tol(b), "qwen qkv")
    y = q.qgemv_w4g64(dev_weight(W["o"]), dev16(xa), residual=dev16(x))
    y64, _, b = oracle.qgemv(4, W["o"].codes, W["o"].scales, W["o"].biases, xa, x)
    check(y, y64, plain_tol(b), "qwen o_proj")
    y = q.swiglu_qgemv(dev_weight(W["gate"]), dev_weight(W["up"]), dev16(x), dev16(g2), eps)
    gw, uw = W["gate"], W["up"]
    h64, _, tol = oracle.swiglu_qgemv((gw.codes, gw.scales, gw.biases),
                                      (uw.codes, uw.scales, uw.biases), x, g2, eps)
    check(y, h64, tol, "qwen swiglu")
    y = q.qgemv_w4g64(dev_weight(W["down"]), dev16(xi), residual=dev16(x))
    y64, _, b = oracle.qgemv(4, W["down"].codes, W["down"].scales, W["down"].biases, xi, x)
    check(y, y64, plain_tol(b), "qwen down")
    y = q.qgemv_w4g64(dev_weight(W["lm_head"]), dev16(x))
    y64, _, b = oracle.qgemv(4, W["lm_head"].codes, W["lm_head"].scales, W["lm_head"].biases, x)
    check(y, y64, plain_tol(b), "qwen lm_head")


def test_config3_moe_512_experts_16_tokens():
    m = synth.MOE
    E, H, I, K = m["n_experts"], m["hidden"], m["inter"], m["top_k"]
    tokens = []
    for t in range(m["tokens"]):
        idx, wt = synth.routing(synth.rng(3, t, synth.TID["routing"]), E, K)
        x = synth.activation(synth.rng(3, t, synth.TID["x"]), H)
        tokens.append((idx, wt, x))
    used = sorted({int(e) for idx, _, _ in tokens for e in idx})
    experts = {e: synth.moe_expert(3, 0, e) for e in used}
    # Full resident layout: 512 expert slots; only the used experts are filled
    # (the kernels read no other slot).
    gw, dw = H // 8, I // 8
    gu_c = torch.empty((E, 2 * I, gw), dtype=torch.int32, device="cuda")
    gu_s = torch.empty((E, 2 * I, H // 64), dtype=torch.float16, device="cuda")
    gu_b = torch.empty_like(gu_s)
    dn_c = torch.empty((E, H, dw), dtype=torch.int32, device="cuda")
    dn_s = torch.empty((E, H, I // 64), dtype=torch.float16, device="cuda")
    dn_b = torch.empty_like(dn_s)
    for e, (gu, dn) in experts.items():
        gu_c[e].copy_(torch.from_numpy(gu.codes.view(np.int32)))
        gu_s[e].copy_(torch.from_numpy(gu.scales))
        gu_b[e].copy_(torch.from_numpy(gu.biases))
        dn_c[e].copy_(torch.from_numpy(dn.codes.view(np.int32)))
        dn_s[e].copy_(torch.from_numpy(dn.scales))
        dn_b[e].copy_(torch.from_numpy(dn.biases))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for t, (idx, wt, x) in enumerate(tokens):
        y = q.moe_qgemv_combine((gu_c, gu_s, gu_b), (dn_c, dn_s, dn_b),
                                torch.from_numpy(idx).cuda(), torch.from_numpy(wt).cuda(),
                                dev16(x), dev16(x), err_flag=err)
        # oracle over the same experts, renumbered 0..3
        sub_gu = synth.QuantWeight(np.stack([experts[int(e)][0].codes for e in idx]),
                                   np.stack([experts[int(e)][0].scales for e in idx]),
                                   np.stack([experts[int(e)][0].biases for e in idx]), 4)
        sub_dn = synth.QuantWeight(np.stack([experts[int(e)][1].codes for e in idx]),
                                   np.stack([experts[int(e)][1].scales for e in idx]),
                                   np.stack([experts[int(e)][1].biases for e in idx]), 4)
        y64, _, tol, e_flag = oracle.moe_qgemv_combine(
            (sub_gu.codes, sub_gu.scales, sub_gu.biases), (sub_dn.codes, sub_dn.scales,
                                                           sub_dn.biases),
            np.arange(K, dtype=np.int32), wt, x, x)
        assert e_flag == 0
        check(y, y64, tol, f"config 3 token {t}")
    assert int(err.item()) == 0
    assert q.device_status() == 0


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_config4_bits_and_small_batch(bits, M):
    # the config-1 shapes: o_proj-like 4096x4096 and down-like 4096x14336
    for (N, K) in [(4096, 4096), (4096, 14336)]:
        w = synth.quant_weight(synth.rng(4, N + K, synth.TID["qkv"]), N, K, bits)
        x = synth.activation(synth.rng(4, K, synth.TID["x"]), K, M)
        fn = q.qgemv_w4g64 if bits == 4 else q.qgemv_w2g64
        y = fn(dev_weight(w), dev16(x))
        y64, _, bound = oracle.qgemv(bits, w.codes, w.scales, w.biases, x)
        check(y, y64, plain_tol(bound), f"config 4 w{bits} M={M} {N}x{K}")


def test_config4_two_bit_layer_shapes():
    for name, (N, K) in {"qkv": (6144, 4096), "gate": (14336, 4096)}.items():
        w = synth.quant_weight(synth.rng(4, 1, synth.TID[name]), N, K, 2)
        x = synth.activation(synth.rng(4, 2, synth.TID["x"]), K)
        y = q.qgemv_w2g64(dev_weight(w), dev16(x))
        y64, _, bound = oracle.qgemv(2, w.codes, w.scales, w.biases, x)
        check(y, y64, plain_tol(bound), f"config 4 w2 {name}")


def test_q8_layer_shapes():
    """8-bit (Q8 group 64) at the Llama-3.1-8B layer's matvec shapes, in the
    streaming launch the benchmark's w8_layer unit times."""
    shapes = {"qkv": (6144, 4096), "o": (4096, 4096), "gate": (14336, 4096),
              "down": (4096, 14336)}
    for name, (N, K) in shapes.items():
        w = synth.quant_weight(synth.rng(5, 0, synth.TID[name]), N, K, 8)
        x = synth.activation(synth.rng(5, 1, synth.TID["x"], K), K)
        y = q.qgemv_w8g64(dev_weight(w), dev16(x))
        y64, _, bound = oracle.qgemv(8, w.codes, w.scales, w.biases, x)
        check(y, y64, plain_tol(bound), f"q8 {name}")
