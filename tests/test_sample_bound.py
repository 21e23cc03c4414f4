"""The 1e-4 running-sum bound the sampling parity tests use (CPU only).

The GPU computes the weights p_j = exp((l_j - l_0) / T) in fp32 and their
running sum in a fixed order: lane l of one warp sums candidates
[l E, l E + E) in turn (E = ceil(k / 32)), a 32-lane inclusive scan adds the
lanes' totals, and each lane then walks its own candidates again.  Here that
order is replayed in numpy float32, with every weight pushed off its fp64
value by the whole relative error the derivation allows it, |a| 2^-23 (the
rounded subtraction and division of its argument a) plus 2^-22 (2 ulp of an
fp32 exp), in a sign pattern that does not cancel, and the normalised
running sums are compared with the oracle's fp64 ones: the largest
difference must stay below the bound, for k up to 1024.
"""
import numpy as np
import pytest

import oracle
import synth

CDF_TOL = 1e-4


def gpu_order_running_sums(p32, k):
    E = (k + 31) // 32
    parts = np.zeros(32, np.float32)
    for lane in range(32):
        acc = np.float32(0.0)
        for i in range(lane * E, min(lane * E + E, k)):
            acc = np.float32(acc + p32[i])
        parts[lane] = acc
    inc = parts.copy()
    o = 1
    while o < 32:  # Hillis-Steele inclusive scan, as the shuffles do it
        prev = inc.copy()
        for lane in range(o, 32):
            inc[lane] = np.float32(prev[lane] + prev[lane - o])
        o *= 2
    total = inc[31]
    cum = np.zeros(k, np.float32)
    for lane in range(32):
        run = np.float32(inc[lane] - parts[lane])
        for i in range(lane * E, min(lane * E + E, k)):
            run = np.float32(run + p32[i])
            cum[i] = run
    return cum, total


@pytest.mark.parametrize("k,T,step,seed", [(1024, 1.0, None, 1), (1024, 5.0, None, 2),
                                           (1024, 0.05, None, 3), (1024, 1.0, 1000.0, 4),
                                           (512, 0.8, 0.25, 5), (50, 0.8, None, 6),
                                           (1000, 2.0, None, 7)])
def test_running_sum_bound(k, T, step, seed):
    lv = synth.logits(synth.rng(6, 7000 + seed, synth.TID["logits"]), 200000, step=step)
    _, cand, cum64 = oracle.lm_head_sample(lv, k, T, 0.0)
    l = lv.astype(np.float64)[cand]
    a = (l - l[0]) / T
    p64 = np.exp(a)
    rel = np.abs(a) * 2.0**-23 + 2.0**-22
    sign = np.where(np.arange(k) % 3 == 0, -1.0, 1.0)  # errors that do not cancel out
    p32 = (p64 * (1.0 + sign * rel)).astype(np.float32)
    cum32, total32 = gpu_order_running_sums(p32, k)
    err = np.max(np.abs(cum32.astype(np.float64) / np.float64(total32) - cum64))
    assert err < CDF_TOL, err
