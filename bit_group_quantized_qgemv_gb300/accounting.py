"""Algorithmic byte accounting of the quantized GEMV workloads.

Bytes per weight: 4-bit g64 = 0.5 (code) + 2 * 2 / 64 (fp16 scale and bias
per 64 weights) = 0.5625; 2-bit = 0.25 + 0.0625 = 0.3125.  A matvec moves
its packed codes, scales and biases once, plus its activations and output:
    bytes = N*K*B/w + M*K*2 (x) + M*N*2 (y) [+ K*2 (gamma)] [+ M*N*2 (residual)].
Decode latency is bandwidth-bound, time ~= bytes / bandwidth ("Boosting
inference speed on Apple Silicon", INFERENCE_RESEARCH.md, TL;DR).  The MoE
expert of the hada.io page (topic 27758, "SSD Expert Streaming", about
6.75 MB per expert) is gate.up 4096 -> 2 x 1024 plus down 1024 -> 4096.
"""
from __future__ import annotations


def weight_bytes(N: int, K: int, bits: int) -> int:
    """Packed codes + fp16 scales + fp16 biases of an N x K weight."""
    assert K % 64 == 0
    return N * K * bits // 8 + 2 * 2 * N * (K // 64)


def matvec_bytes(N: int, K: int, bits: int = 4, M: int = 1, gamma: bool = False,
                 residual: bool = False) -> int:
    b = weight_bytes(N, K, bits) + 2 * M * K + 2 * M * N
    if gamma:
        b += 2 * K
    if residual:
        b += 2 * M * N
    return b


def expert_bytes(hidden: int = 4096, inter: int = 1024, bits: int = 4) -> int:
    """One MoE expert: gate.up (2*inter x hidden) + down (hidden x inter)."""
    return weight_bytes(2 * inter, hidden, bits) + weight_bytes(hidden, inter, bits)


def llama8b_layer_ops(bits: int = 4):
    """(name, algorithmic bytes) of each matvec of the Llama-8B-shaped layer."""
    H, I, qkv = 4096, 14336, (32 + 16) * 128
    return [
        ("rmsnorm_qkv", matvec_bytes(qkv, H, bits, gamma=True)),
        ("o_proj_residual", matvec_bytes(H, 32 * 128, bits, residual=True)),
        ("gate_up_swiglu", 2 * weight_bytes(I, H, bits) + 2 * H + 2 * H + 2 * I),
        ("down_residual", matvec_bytes(H, I, bits, residual=True)),
    ]


def llama8b_layer_bytes(bits: int = 4) -> int:
    return sum(b for _, b in llama8b_layer_ops(bits))


def moe_token_bytes(top_k: int = 4, hidden: int = 4096, inter: int = 1024) -> int:
    """Per token: top_k experts + x + residual + y + (idx, weight) per expert."""
    return top_k * expert_bytes(hidden, inter) + 3 * 2 * hidden + top_k * 8
