"""Seeded random cases for top-k sampling and the LUT GEMV against the oracle.

Each case draws its shape and parameters from a fixed seed: for sampling N,
top_k, the temperature, how coarse a grid the logits are rounded to (from
none to a few values, i.e. from no ties to thousands) and whether the
logits start 16-byte aligned; for the LUT GEMV N, K, rows_per_lut and a
residual.  The checks are those of tests/test_gpu_sample.py and
tests/test_gpu_lut.py: candidates bit-exact, weights and token within the
derived bounds; outputs within the matvec tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from qhelpers import check, dev16, plain_tol
from test_gpu_sample import assert_token

pytestmark = pytest.mark.gpu

q = pytest.importorskip("bit_group_quantized_qgemv_gb300")


@pytest.mark.parametrize("case", range(24))
def test_sample_fuzz(case):
    g = np.random.default_rng(9000 + case)
    N = int(g.choice([int(g.integers(1, 64)), int(g.integers(64, 5000)),
                      int(g.integers(5000, 200000))]))
    k = int(min(N, g.choice([1, int(g.integers(1, 33)), int(g.integers(33, 257)),
                             int(g.integers(257, 1025))])))
    T = float(g.choice([0.05, 0.5, 0.8, 1.0, 2.0]))
    step = [None, None, 0.25, 1.0, 8.0, 1000.0][int(g.integers(0, 6))]
    lv = synth.logits(synth.rng(6, 5000 + case, synth.TID["logits"]), N, step=step)
    offset = int(g.integers(0, 2))  # 1: the logits start 2 bytes past a 16-byte boundary
    buf = dev16(np.concatenate([np.zeros(offset, np.float16), lv]))
    ld = buf[offset:]
    u = float(synth.uniforms(synth.rng(6, 5000 + case, synth.TID["u"]), 1)[0])
    ud = torch.tensor([u], dtype=torch.float32, device="cuda")
    tok, idx, prob = q.sample_topk(ld, k, T, ud, want_topk=True)
    _, cand, cum = oracle.lm_head_sample(lv, k, T, u)
    what = f"case {case}: N={N} k={k} T={T} step={step} offset={offset}"
    assert np.array_equal(idx.cpu().numpy(), cand), what
    p64 = np.diff(np.concatenate([[0.0], cum]))
    assert np.allclose(prob.cpu().numpy(), p64, rtol=1e-4, atol=1e-6), what
    assert_token(int(tok.item()), lv, k, T, u, what)


@pytest.mark.parametrize("case", range(16))
def test_lut_fuzz(case):
    g = np.random.default_rng(9100 + case)
    N = int(g.choice([int(g.integers(1, 40)), int(g.integers(40, 3000)),
                      int(g.integers(3000, 20000))]))
    K = 64 * int(g.integers(1, 257))  # 64 .. 16384
    R = int(g.choice([1, int(g.integers(1, 9)), int(g.integers(9, 200)), N]))
    w = synth.lut_weight(synth.rng(7, 5000 + case, synth.TID["lut"]), N, K, R)
    x = synth.activation(synth.rng(7, 5000 + case, synth.TID["x"]), K)
    r = synth.activation(synth.rng(7, 5000 + case, synth.TID["residual"]), N) if case % 2 else None
    y = q.qgemv_lut4(torch.from_numpy(w.codes.view(np.int32)).cuda(),
                     torch.from_numpy(w.lut).cuda(), dev16(x), rows_per_lut=R,
                     residual=None if r is None else dev16(r))
    y64, _, bound = oracle.lut_qgemv(w.codes, w.lut, R, x, r)
    check(y, y64, plain_tol(bound), f"lut case {case}: N={N} K={K} R={R}")
