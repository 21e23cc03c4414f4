"""qgemv_lm_head_argmax: greedy lm_head on the GPU.

The logits must match the fp64 oracle within the matvec tolerance; the
token is an integer decided by floating point, so it is compared where it is
unique: bit-exactly with the lowest index of the largest returned logit, and
as a valid pick against the oracle (its oracle logit within the tolerance of
the oracle's maximum).  Shapes: the full Qwen3-0.6B-shaped lm_head
(151936 x 1024, the fused streaming launch), a ragged one, one the generic
fallback takes; ties, all-negative logits, and a scratch reused across calls.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from qhelpers import check, dev16, dev_weight, plain_tol

pytestmark = pytest.mark.gpu

q = pytest.importorskip("bit_group_quantized_qgemv_gb300")


def W(seed, N, K):
    return synth.quant_weight(synth.rng(500, seed, 1), N, K, 4)


def X(seed, K):
    return synth.activation(synth.rng(500, seed, 10), K)


def check_argmax(w, x, what, scratch=None):
    tok, logits = q.lm_head_argmax(dev_weight(w), dev16(x), scratch=scratch)
    y64, _, bound = oracle.qgemv(4, w.codes, w.scales, w.biases, x)
    tol = plain_tol(bound)
    check(logits, y64, tol, what + " logits")
    t = int(tok.item())
    got = logits.cpu().numpy()
    assert t == int(np.argmax(got)), f"{what}: token {t} is not the first maximum of the logits"
    best = int(np.argmax(y64))
    assert y64[t] >= y64[best] - (tol[t] + tol[best]), f"{what}: token {t} is not a valid pick"
    return t, got


@pytest.mark.parametrize("N,K", [(151936, 1024), (1000, 2048), (333, 960), (7, 4096)])
def test_lm_head_argmax_parity(N, K):
    check_argmax(W(N + K, N, K), X(N, K), f"argmax N={N} K={K}")


@pytest.mark.parametrize("K", [1024, 960])
def test_ties_pick_the_lowest_index(K):
    N = 300
    w = W(K, N, K)
    w.codes[:] = 0
    w.scales[:] = 1.0
    w.biases[:] = 0.0
    w.biases[[5, 7, 250], 0] = 1.0          # rows 5, 7, 250 get the same largest logit
    x = np.zeros(K, np.float16)
    x[:64] = 1.0
    t, got = check_argmax(w, x, f"ties K={K}")
    assert t == 5 and got[5] == got[7] == got[250] == 64.0


def test_all_negative_logits():
    N, K = 4096, 1024
    w = W(3, N, K)
    g = np.random.default_rng(3)            # every logit negative, all distinct rows
    w.biases[:] = (-(0.01 + 0.04 * g.random(w.biases.shape))).astype(np.float16)
    w.codes[:] = 0
    x = np.abs(X(3, K)).astype(np.float16)
    x[x == 0] = np.float16(0.5)
    t, got = check_argmax(w, x, "all negative")
    assert got.max() < 0


def test_scratch_is_left_zero_and_reused():
    N, K = 20000, 1024
    scratch = torch.zeros(q.argmax_scratch_bytes(), dtype=torch.uint8, device="cuda")
    for seed in range(4):
        check_argmax(W(40 + seed, N, K), X(40 + seed, K), f"reuse {seed}", scratch=scratch)
        torch.cuda.synchronize()
        assert int(scratch.sum().item()) == 0
    assert q.device_status() == 0
