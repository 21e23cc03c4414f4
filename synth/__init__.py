"""Seeded synthetic inputs for the quantized GEMV workloads.

This module only draws random numbers in the shapes, ranges and structure of
the workloads; it holds none of the method's arithmetic (no unpacking, no
dequantisation, no products).  Both the CUDA path's tests/benchmark and the
fp64 oracle consume what it returns.

Generator: numpy PCG64 seeded by ``SeedSequence([workload, layer, tensor_id,
expert])``.  Uniform codes are drawn as uniform random uint32 words, which is
exactly 8 i.i.d. uniform 4-bit codes (or 16 uniform 2-bit codes) per word.

Tensor ids (the third seed word):
    1 QKV / generic weight    2 o_proj           3 gate         4 up
    5 down                    6 lm_head          7 MoE gate.up  8 MoE down
    10 x (activation)         11 residual        12 norm gamma (first norm)
    13 norm gamma (second)    14 MoE routing     15 spare weight
    16 MoE router weight      17 logits          18 sampling uniforms
    19 LUT (palettised) weight

Workloads (the first seed word): 0 the 1024 x 1024 GEMV, 1 the
Llama-3.1-8B-shaped layer, 2 the Qwen3-0.6B-shaped stack, 3 the MoE, 4 the
2-bit layer and small batches, 5 the 8-bit (Q8) layer, 6 top-k sampling,
7 the LUT / palettised layer.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

TID = {
    "qkv": 1, "o": 2, "gate": 3, "up": 4, "down": 5, "lm_head": 6,
    "moe_gu": 7, "moe_down": 8, "x": 10, "residual": 11, "gamma1": 12,
    "gamma2": 13, "routing": 14, "spare": 15, "router": 16, "logits": 17,
    "u": 18, "lut": 19,
}


def rng(workload: int, layer: int, tensor: int, expert: int = 0) -> np.random.Generator:
    """Independent PCG64 stream for one tensor of one workload."""
    return np.random.Generator(np.random.PCG64(
        np.random.SeedSequence([int(workload), int(layer), int(tensor), int(expert)])))


@dataclass
class QuantWeight:
    """Planar quantized weight: codes uint32 [N][K*bits/32], scales and
    biases fp16 [N][K/64]."""
    codes: np.ndarray
    scales: np.ndarray
    biases: np.ndarray
    bits: int

    @property
    def N(self) -> int:
        return self.codes.shape[-2]

    @property
    def K(self) -> int:
        return self.codes.shape[-1] * 32 // self.bits

    def nbytes(self) -> int:
        return self.codes.nbytes + self.scales.nbytes + self.biases.nbytes


def quant_weight(g: np.random.Generator, N: int, K: int, bits: int = 4,
                 lead: tuple = ()) -> QuantWeight:
    """Draw a weight in the workloads' recipe.

    4-bit: codes uniform 0..15; scale ~ U(0.005, 0.02) rounded to fp16;
    bias = fp16(-8 * scale + N(0, 0.001)) per (row, group).
    2-bit: codes uniform 0..3; scale ~ U(0.02, 0.08) rounded to fp16;
    bias = fp16(-1.5 * scale), no noise.
    8-bit: codes uniform 0..255; scale ~ U(0.0003125, 0.00125) (the 4-bit
    range / 16, so weights span the same range) rounded to fp16;
    bias = fp16(-128 * scale + N(0, 0.001)).
    ``lead`` prepends leading dimensions (e.g. (E,) for expert stacks).
    """
    assert bits in (2, 4, 8) and K % 64 == 0
    words = K * bits // 32
    G = K // 64
    codes = g.integers(0, 0xFFFFFFFF, size=lead + (N, words), dtype=np.uint32,
                       endpoint=True)
    if bits == 4:
        s = g.uniform(0.005, 0.02, size=lead + (N, G)).astype(np.float16)
        noise = g.normal(0.0, 0.001, size=lead + (N, G))
        b = (-8.0 * s.astype(np.float64) + noise).astype(np.float16)
    elif bits == 8:
        s = g.uniform(0.0003125, 0.00125, size=lead + (N, G)).astype(np.float16)
        noise = g.normal(0.0, 0.001, size=lead + (N, G))
        b = (-128.0 * s.astype(np.float64) + noise).astype(np.float16)
    else:
        s = g.uniform(0.02, 0.08, size=lead + (N, G)).astype(np.float16)
        b = (-1.5 * s.astype(np.float64)).astype(np.float16)
    return QuantWeight(codes, s, b, bits)


def activation(g: np.random.Generator, K: int, M: int | None = None) -> np.ndarray:
    """fp16 activations ~ N(0, 1); shape [K] or [M][K]."""
    shape = (K,) if M is None else (M, K)
    return g.normal(0.0, 1.0, size=shape).astype(np.float16)


def norm_gamma(g: np.random.Generator, K: int) -> np.ndarray:
    """RMSNorm weight ~ N(1, 0.05) in fp16."""
    return g.normal(1.0, 0.05, size=K).astype(np.float16)


def routing(g: np.random.Generator, n_experts: int, top_k: int = 4,
            shared: int = 0):
    """One token's routing: the shared expert plus top_k-1 experts drawn
    uniformly without replacement from the others; weights are the softmax
    of top_k N(0,1) logits (computed in fp64, stored fp32)."""
    others = np.array([e for e in range(n_experts) if e != shared], np.int64)
    routed = g.choice(others, size=top_k - 1, replace=False)
    idx = np.concatenate([[shared], routed]).astype(np.int32)
    logits = g.normal(0.0, 1.0, size=top_k)
    ex = np.exp(logits - logits.max())
    wt = (ex / ex.sum()).astype(np.float32)
    return idx, wt


@dataclass
class LutWeight:
    """A LUT / palettised 4-bit weight: uint32 codes [N][K/8] (8 indices per
    word, low nibble first) and fp16 tables [n_luts][16], table t serving
    rows t*rows_per_lut .. +rows_per_lut-1."""
    codes: np.ndarray
    lut: np.ndarray
    rows_per_lut: int

    @property
    def N(self) -> int:
        return self.codes.shape[0]

    @property
    def K(self) -> int:
        return self.codes.shape[1] * 8

    @property
    def nbytes(self) -> int:
        return self.codes.nbytes + self.lut.nbytes


def lut_weight(g: np.random.Generator, N: int, K: int, rows_per_lut: int = 1,
               spread: float = 0.02) -> LutWeight:
    """Uniform random indices (uniform uint32 words) and, per table, 16
    sorted N(0, spread) values in fp16 (the shape of a k-means palette)."""
    codes = g.integers(0, 2**32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32)
    n_luts = -(-N // rows_per_lut)
    lut = np.sort(g.normal(0.0, spread, size=(n_luts, 16)), axis=1).astype(np.float16)
    return LutWeight(codes, lut, rows_per_lut)


def logits(g: np.random.Generator, N: int, spread: float = 2.5, peaks: int = 8,
           step: float | None = None) -> np.ndarray:
    """fp16 next-token logits [N]: N(0, spread) with ``peaks`` entries raised
    by U(6, 12) (a few likely tokens); with ``step``, every value is rounded
    to a multiple of it (many exact ties)."""
    v = g.normal(0.0, spread, size=N)
    if peaks:
        at = g.choice(N, size=min(peaks, N), replace=False)
        v[at] += g.uniform(6.0, 12.0, size=at.size)
    if step is not None:
        v = np.round(v / step) * step
    return v.astype(np.float16)


def uniforms(g: np.random.Generator, n: int) -> np.ndarray:
    """fp32 uniforms in [0, 1) (the random numbers a sampler is given)."""
    return g.random(n, dtype=np.float32)


# ------------------------------------------------------------------ shapes

#: Llama-3.1-8B-shaped decode layer (hidden 4096, 32 q + 8 kv heads x 128).
LLAMA8B = dict(hidden=4096, n_q=32, n_kv=8, head_dim=128, inter=14336, eps=1e-5)
#: Qwen3-0.6B-shaped decode stack (28 layers, hidden 1024, 16 q + 8 kv x 128).
QWEN06B = dict(hidden=1024, n_q=16, n_kv=8, head_dim=128, inter=3072, layers=28,
               vocab=151936, eps=1e-5)
#: MoE expert layer: 512 experts, hidden 4096, expert intermediate 1024, K=4.
MOE = dict(hidden=4096, inter=1024, n_experts=512, top_k=4, tokens=16)


def llama_layer(workload: int, layer: int, bits: int = 4) -> dict:
    """Weights and inputs of one Llama-8B-shaped layer (bits 4, 2 or 8)."""
    c = LLAMA8B
    H, I = c["hidden"], c["inter"]
    qkv_n = (c["n_q"] + 2 * c["n_kv"]) * c["head_dim"]
    return dict(
        qkv=quant_weight(rng(workload, layer, TID["qkv"]), qkv_n, H, bits),
        o=quant_weight(rng(workload, layer, TID["o"]), H, c["n_q"] * c["head_dim"], bits),
        gate=quant_weight(rng(workload, layer, TID["gate"]), I, H, bits),
        up=quant_weight(rng(workload, layer, TID["up"]), I, H, bits),
        down=quant_weight(rng(workload, layer, TID["down"]), H, I, bits),
        gamma1=norm_gamma(rng(workload, layer, TID["gamma1"]), H),
        gamma2=norm_gamma(rng(workload, layer, TID["gamma2"]), H),
        x=activation(rng(workload, layer, TID["x"]), H),
    )


def moe_expert(workload: int, layer: int, e: int, hidden: int | None = None,
               inter: int | None = None):
    """Expert e of an MoE layer: gate.up [2I][H/8] (gate rows 0..I-1, then up
    rows) and down [H][I/8], each from its own seeded stream."""
    H = MOE["hidden"] if hidden is None else hidden
    I = MOE["inter"] if inter is None else inter
    gu = quant_weight(rng(workload, layer, TID["moe_gu"], e), 2 * I, H, 4)
    dn = quant_weight(rng(workload, layer, TID["moe_down"], e), H, I, 4)
    return gu, dn


def moe_experts(workload: int, layer: int, n_experts: int, hidden: int | None = None,
                inter: int | None = None):
    """Stacked experts: gate.up [E][2I][H/8] and down [E][H][I/8] (host arrays).

    Expert e is identical to ``moe_expert(workload, layer, e)``.
    """
    parts = [moe_expert(workload, layer, e, hidden, inter) for e in range(n_experts)]
    gu = QuantWeight(np.stack([p[0].codes for p in parts]),
                     np.stack([p[0].scales for p in parts]),
                     np.stack([p[0].biases for p in parts]), 4)
    dn = QuantWeight(np.stack([p[1].codes for p in parts]),
                     np.stack([p[1].scales for p in parts]),
                     np.stack([p[1].biases for p in parts]), 4)
    return gu, dn
