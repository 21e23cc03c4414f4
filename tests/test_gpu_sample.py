"""qgemv_sample_topk / qgemv_lm_head_sample: top-k sampling on the GPU.

The candidates (which top_k logits, in which order) are integer work on the
fp16 bits and must equal the oracle's exactly.  The weights are fp32 on the
GPU and fp64 in the oracle: the normalised weights must agree within
1e-6 + 1e-4 relative, and the token, an index decided by
floating point, is compared where it is unique: it must be the oracle's
token whenever u lies more than CDF_TOL from every boundary of the oracle's
running sum, and otherwise one of the two candidates beside that boundary.

CDF_TOL: the weight exp(a), a = (l_j - l_0) / T <= 0, carries a relative
error of at most |a| 2^-23 (the subtraction and division, each rounded once)
plus 2 ulp (expf), so an absolute error of at most e^-1 2^-23 + 2^-22 p_j;
summed over k <= 1024 candidates and divided by the total (>= 1, since
p_0 = 1) that is below 5e-5, plus the scan's own rounding (about 2^-20).
1e-4 covers it.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from qhelpers import check, dev16, dev_weight, plain_tol

pytestmark = pytest.mark.gpu

q = pytest.importorskip("bit_group_quantized_qgemv_gb300")

CDF_TOL = 1e-4


def L(seed, N, **kw):
    return synth.logits(synth.rng(6, seed, synth.TID["logits"]), N, **kw)


def U(seed, n):
    return synth.uniforms(synth.rng(6, seed, synth.TID["u"]), n)


def run(logits_dev, k, T, u):
    ud = torch.tensor([u], dtype=torch.float32, device="cuda")
    tok, idx, prob = q.sample_topk(logits_dev, k, T, ud, want_topk=True)
    return int(tok.item()), idx.cpu().numpy(), prob.cpu().numpy()


def check_sample(lv, k, T, us, what, logits_dev=None):
    """lv: the fp16 logits (numpy) the GPU samples from."""
    if logits_dev is None:
        logits_dev = dev16(lv)
    _, cand, cum = oracle.lm_head_sample(lv, k, T, 0.0)
    p64 = np.diff(np.concatenate([[0.0], cum]))
    for u in us:
        tok, idx, prob = run(logits_dev, k, T, float(u))
        assert np.array_equal(idx, cand), (
            f"{what}: candidates differ at {np.flatnonzero(idx != cand)[:8]}")
        assert np.allclose(prob, p64, rtol=1e-4, atol=1e-6), (
            f"{what}: weights off by {np.max(np.abs(prob - p64)):.3g}")
        assert_token(tok, lv, k, T, float(u), what)


def assert_token(tok, lv, k, T, u, what):
    """The oracle's token, or its neighbour across a running-sum boundary
    within CDF_TOL of u."""
    want, cand, cum = oracle.lm_head_sample(lv, k, T, u)
    if tok == want:
        return
    pos = np.flatnonzero(cand == tok)
    assert pos.size == 1, f"{what}: token {tok} is not a candidate"
    j, jw = int(pos[0]), int(np.flatnonzero(cand == want)[0])
    boundary = cum[min(j, jw)]               # the running-sum boundary between them
    assert abs(j - jw) == 1 and abs(u - boundary) <= CDF_TOL, (
        f"{what}: u={u} gives {tok} (position {j}), oracle {want} (position {jw})")


def midpoints(lv, k, T):
    """u at the middle of every bracket of the oracle's running sum wider than
    2 CDF_TOL: there the token is unique."""
    _, _, cum = oracle.lm_head_sample(lv, k, T, 0.0)
    lo = np.concatenate([[0.0], cum[:-1]])
    keep = (cum - lo) > 2 * CDF_TOL
    return ((lo + cum) / 2)[keep][:64]


@pytest.mark.parametrize("N,k,T", [(151936, 1, 1.0), (151936, 2, 0.7), (151936, 50, 0.8),
                                   (151936, 1024, 1.5), (128256, 40, 1.0),
                                   (1001, 7, 1.0), (9, 3, 2.0), (1, 1, 1.0), (5, 5, 0.5)])
def test_sample_topk_parity(N, k, T):
    lv = L(N + k, N)
    us = np.concatenate([U(N + k, 12), [0.0, 0.5, 0.99999994]]).astype(np.float32)
    check_sample(lv, k, T, us, f"sample N={N} k={k} T={T}")


@pytest.mark.parametrize("N,k,T", [(151936, 50, 0.8), (151936, 1024, 1.0), (2000, 300, 3.0)])
def test_sample_topk_bracket_midpoints_are_exact(N, k, T):
    lv = L(N + 3, N)
    for u in midpoints(lv, k, T):
        tok, _, _ = run(dev16(lv), k, T, float(u))
        assert tok == oracle.lm_head_sample(lv, k, T, float(u))[0], f"u={u}"


@pytest.mark.parametrize("N,k,step", [(151936, 50, 0.5), (151936, 1000, 1.0), (4096, 64, 4.0),
                                      (50000, 17, 100.0)])
def test_sample_topk_ties_take_the_lowest_indices(N, k, step):
    # values rounded to a coarse grid: thousands of logits equal to the k-th
    lv = L(N + 11, N, step=step)
    check_sample(lv, k, 1.0, U(N + 11, 6), f"ties N={N} k={k} step={step}")


def test_sample_topk_all_equal_and_signed_zeros():
    lv = np.zeros(1000, np.float16)
    lv[1::3] = -0.0                          # -0 and +0 are the same value
    _, idx, prob = run(dev16(lv), 40, 1.0, 0.3)
    assert idx.tolist() == list(range(40))
    assert np.allclose(prob, 1.0 / 40, rtol=1e-6)
    check_sample(lv, 40, 1.0, U(5, 8), "all equal")


def test_sample_topk_extreme_values():
    lv = L(21, 5000)
    lv[[10, 20]] = np.float16(65504.0)      # the largest finite fp16, twice
    lv[30] = np.float16(-65504.0)
    lv[40:50] = np.float16(6e-8)            # subnormals
    lv[50:60] = np.float16(-6e-8)
    check_sample(lv, 20, 1.0, U(21, 6), "extreme values")
    lv = -np.abs(L(22, 5000)) - np.float16(1000.0)   # all negative and far apart from 0
    check_sample(lv.astype(np.float16), 100, 0.05, U(22, 6), "all negative")


def test_sample_topk_unaligned_logits_and_the_largest_n():
    lv = L(31, 50001)
    buf = dev16(np.concatenate([[0.0], lv]).astype(np.float16))
    check_sample(lv, 33, 1.0, U(31, 4), "unaligned", logits_dev=buf[1:])   # 2-byte aligned only
    N = 786432                               # QGEMV_SAMPLE_MAX_N
    lv = L(32, N)
    check_sample(lv, 1024, 1.0, U(32, 3), "largest N")


def test_sample_topk_temperature_limits():
    lv = L(41, 151936)
    best = int(np.argmax(lv))                # first maximum
    for u in (0.0, 0.5, 0.99):
        tok, _, _ = run(dev16(lv), 50, 1e-3, u)
        assert tok == best
    tok, _, _ = run(dev16(lv), 1, 5.0, 0.99)
    assert tok == best


def test_sample_frequencies_follow_the_weights():
    # one graph, replayed with a fresh u each time: the token frequencies over
    # a grid of u follow the normalised weights
    lv = np.array([0.0, 1.0, 0.5, -1.0, 2.0, 1.0, -3.0, 0.25], np.float16)
    ld = dev16(lv)
    ud = torch.zeros(1, dtype=torch.float32, device="cuda")
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    q.sample_topk(ld, 4, 0.8, ud, token=tok)         # warm-up outside capture
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        q.sample_topk(ld, 4, 0.8, ud, token=tok, stream=s)
    n = 2000
    us = (np.arange(n) + 0.5) / n
    counts = {}
    for u in us:
        ud.fill_(float(u))
        g.replay()
        t = int(tok.item())
        counts[t] = counts.get(t, 0) + 1
    _, cand, cum = oracle.lm_head_sample(lv, 4, 0.8, 0.0)
    p = np.diff(np.concatenate([[0.0], cum]))
    assert set(counts) == set(cand.tolist())
    freq = np.array([counts[int(c)] for c in cand]) / n
    assert np.allclose(freq, p, atol=2.0 / n)


@pytest.mark.parametrize("N,K,k", [(151936, 1024, 50), (1000, 2048, 20), (333, 960, 5)])
def test_lm_head_sample_parity(N, K, k):
    w = synth.quant_weight(synth.rng(6, N + K, synth.TID["lm_head"]), N, K, 4)
    x = synth.activation(synth.rng(6, N, synth.TID["x"]), K)
    u = float(U(N + K, 1)[0])
    ud = torch.tensor([u], dtype=torch.float32, device="cuda")
    tok, logits, idx, prob = q.lm_head_sample(dev_weight(w), dev16(x), k, 0.8, ud, want_topk=True)
    y64, _, bound = oracle.qgemv(4, w.codes, w.scales, w.biases, x)
    check(logits, y64, plain_tol(bound), f"lm_head_sample N={N} K={K} logits")
    # the sampling is checked on the logits the GPU produced
    lv = logits.cpu().numpy()
    _, cand, _ = oracle.lm_head_sample(lv, k, 0.8, u)
    assert np.array_equal(idx.cpu().numpy(), cand)
    assert_token(int(tok.item()), lv, k, 0.8, u, f"lm_head_sample N={N} K={K} token")
    check_sample(lv, k, 0.8, [u], f"lm_head_sample N={N} K={K}", logits_dev=logits)


def test_lm_head_sample_in_a_captured_graph():
    # the GEMV and the sampler as graph nodes joined by a programmatic
    # dependency: every replay (with a fresh u) equals the eager call
    N, K, k = 151936, 1024, 50
    w = synth.quant_weight(synth.rng(6, 77, synth.TID["lm_head"]), N, K, 4)
    x = dev16(synth.activation(synth.rng(6, 78, synth.TID["x"]), K))
    wd = dev_weight(w)
    ud = torch.zeros(1, dtype=torch.float32, device="cuda")
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.empty(N, dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    q.lm_head_sample(wd, x, k, 0.8, ud, logits=logits, token=tok)  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        q.lm_head_sample(wd, x, k, 0.8, ud, logits=logits, token=tok, stream=s)
    for u in U(79, 16):
        ud.fill_(float(u))
        g.replay()
        got = int(tok.item())
        want, _, _, _ = q.lm_head_sample(wd, x, k, 0.8, torch.tensor([float(u)], device="cuda"))
        assert got == int(want.item()), f"u={u}"
