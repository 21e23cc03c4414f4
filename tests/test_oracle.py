"""Pins for the fp64 oracle, against things other than the oracle itself.

Each check ties the oracle to mathematics or to an independent computation:
hand-worked examples (tests/golden), closed forms, invariants, library
routines (numpy's binary16 conversion, scipy's logistic function) and a
numpy brute force that unpacks codes through a byte view instead of the
oracle's word shifts.  CPU only.
"""
import sys

import numpy as np
import pytest
from scipy.special import expit

import oracle
import synth
from conftest import load_golden

assert sys.byteorder == "little"


# ------------------------------------------------------------ independent
def np_unpack(codes, bits):
    """Unpack packed rows through a little-endian byte view (independent of
    the oracle's word/shift arithmetic).  Returns int64 [..., K]."""
    b = np.ascontiguousarray(codes).view(np.uint8)
    if bits == 8:
        parts = [b]
    elif bits == 4:
        parts = [b & 0xF, b >> 4]
    else:
        parts = [(b >> s) & 0x3 for s in (0, 2, 4, 6)]
    q = np.stack(parts, axis=-1)
    return q.reshape(*codes.shape[:-1], -1).astype(np.int64)


def np_dense(w):
    q = np_unpack(w.codes, w.bits)
    s = np.repeat(w.scales.astype(np.float64), 64, axis=-1)
    b = np.repeat(w.biases.astype(np.float64), 64, axis=-1)
    return q * s + b


def small_weight(seed, N, K, bits=4):
    return synth.quant_weight(synth.rng(100, seed, 15), N, K, bits)


# ------------------------------------------------------------------- fp16
def test_half_to_double_all_patterns():
    lib = oracle.lib()
    pats = np.arange(65536, dtype=np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([lib.oracle_half_to_double(int(p)) for p in pats])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_double_to_half_matches_numpy_rne():
    g = np.random.default_rng(7)
    vals = np.concatenate([
        g.normal(0, 1, 4000), g.normal(0, 1e-5, 2000), g.normal(0, 3e4, 2000),
        g.uniform(-70000, 70000, 1000),
        # exact ties between neighbouring fp16 values (normal and subnormal)
        (np.arange(-600, 600, dtype=np.float64) + 0.5) * 2.0**-24,
        (np.arange(1024, 2048, dtype=np.float64) + 0.5) * 2.0**-10,
        [0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 2.0**-24, 2.0**-25,
         3 * 2.0**-26, 2.0**-14, np.inf, -np.inf],
    ])
    lib = oracle.lib()
    got = np.array([lib.oracle_double_to_half(float(v)) for v in vals], np.uint16)
    ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


# ----------------------------------------------------------------- unpack
@pytest.mark.parametrize("bits", [2, 4, 8])
def test_unpack_against_byte_view(bits):
    g = np.random.default_rng(bits)
    row = g.integers(0, 2**32, size=8, dtype=np.uint64).astype(np.uint32)
    K = 8 * 32 // bits
    ref = np_unpack(row[None, :], bits)[0]
    got = [oracle.code(row, bits, k) for k in range(K)]
    assert np.array_equal(np.array(got), ref)


# ---------------------------------------------------------- hand examples
def test_hand_example_a():
    d = load_golden("hand_example_a.txt")
    words = np.array([int(w, 16) for w in d["words"].split()], np.uint32)[None, :]
    s = np.array([[float(d["scales"])]], np.float16)
    b = np.array([[float(d["biases"])]], np.float16)
    x = np.array([float(v) for v in d["x"].split()], np.float16)
    y64, y16, _ = oracle.qgemv(4, words, s, b, x)
    assert y64[0] == float(d["y"])
    assert float(y16[0]) == float(d["y"])
    # the fixture's misread value really is what the other order gives
    assert float(d["y_high_nibble_first"]) != float(d["y"])
    q_hi = np.array([7 - k for k in range(8)] + [0] * 56)
    xv = x.astype(np.float64)
    assert np.sum((0.5 * q_hi - 4) * xv * (np.arange(64) < 8)) == float(d["y_high_nibble_first"])


def test_hand_example_c_8bit():
    d = load_golden("hand_example_c.txt")
    words = np.array([int(w, 16) for w in d["words"].split()], np.uint32)[None, :]
    s = np.array([[float(d["scales"])]], np.float16)
    b = np.array([[float(d["biases"])]], np.float16)
    x = np.array([float(v) for v in d["x"].split()], np.float16)
    y64, y16, _ = oracle.qgemv(8, words, s, b, x)
    assert y64[0] == float(d["y"])
    assert float(y16[0]) == float(d["y"])
    # the fixture's misread value really is what the other byte order gives
    assert float(d["y_high_byte_first"]) != float(d["y"])
    q_hi = np.array([3, 2, 1, 0, 7, 6, 5, 4] + [0] * 56)
    xv = x.astype(np.float64)
    assert np.sum((0.5 * q_hi - 16) * xv * (np.arange(64) < 8)) == float(d["y_high_byte_first"])


def test_hand_example_b():
    d = load_golden("hand_example_b.txt")
    r0 = [int(w, 16) for w in d["row0_words"].split()] * 8
    r1 = [int(w, 16) for w in d["row1_words"].split()] * 8
    codes = np.array([r0, r1], np.uint32)
    s = np.array([float(v) for v in d["scales"].split()], np.float16).reshape(2, 2)
    b = np.array([float(v) for v in d["biases"].split()], np.float16).reshape(2, 2)
    x = np.array([float(d["x_even"]) if k % 2 == 0 else float(d["x_odd"])
                  for k in range(128)], np.float16)
    want = [float(v) for v in d["y"].split()]
    y64, y16, _ = oracle.qgemv(4, codes, s, b, x)
    assert list(y64) == want
    assert [float(v) for v in y16] == want
    # codes really are q = (3k + n) mod 16
    q = np_unpack(codes, 4)
    assert np.array_equal(q, [[(3 * k + n) % 16 for k in range(128)] for n in range(2)])
    # feeding the transposed scale/bias layout gives the fixture's misread
    sT = np.ascontiguousarray(s.reshape(-1).reshape(2, 2).T)
    bT = np.ascontiguousarray(b.reshape(-1).reshape(2, 2).T)
    y_mis, _, _ = oracle.qgemv(4, codes, sT, bT, x)
    assert list(y_mis) == [float(v) for v in d["y_transposed_scales"].split()]


# ------------------------------------------------------------- invariants
def test_zero_codes_give_bias_path():
    w = small_weight(1, 7, 256)
    w.codes[:] = 0
    x = synth.activation(synth.rng(100, 1, 10), 256)
    y64, _, _ = oracle.qgemv(4, w.codes, w.scales, w.biases, x)
    xs = x.astype(np.float64).reshape(4, 64).sum(axis=1)
    ref = (w.biases.astype(np.float64) * xs[None, :]).sum(axis=1)
    assert np.allclose(y64, ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("bits,K", [(4, 64), (4, 128), (2, 128)])
def test_unit_scale_zero_bias_is_integer_dot(bits, K):
    g = np.random.default_rng(K + bits)
    w = small_weight(2, 5, K, bits)
    w.scales[:] = 1.0
    w.biases[:] = 0.0
    x = g.integers(-1, 2, size=K).astype(np.float16)
    y64, y16, _ = oracle.qgemv(bits, w.codes, w.scales, w.biases, x)
    q = np_unpack(w.codes, bits)
    ref = q @ x.astype(np.int64)
    assert np.array_equal(y64, ref.astype(np.float64))
    assert np.array_equal(y16.astype(np.float64), ref.astype(np.float64))


def test_unit_scale_zero_bias_is_integer_dot_8bit():
    # eight nonzero activations in {-1, 1}: |y| <= 8 * 255 = 2040, exact in fp16
    K = 128
    g = np.random.default_rng(8)
    w = small_weight(2, 5, K, 8)
    w.scales[:] = 1.0
    w.biases[:] = 0.0
    x = np.zeros(K, np.float16)
    x[g.choice(K, size=8, replace=False)] = g.choice([-1.0, 1.0], size=8)
    y64, y16, _ = oracle.qgemv(8, w.codes, w.scales, w.biases, x)
    q = np_unpack(w.codes, 8)
    ref = q @ x.astype(np.int64)
    assert np.array_equal(y64, ref.astype(np.float64))
    assert np.array_equal(y16.astype(np.float64), ref.astype(np.float64))


# -------------------------------------------------------- brute force
@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("N,K,M", [(1, 64, 1), (3, 192, 2), (17, 320, 3), (64, 512, 8)])
def test_brute_force_dense(bits, N, K, M):
    w = small_weight(N * 1000 + K, N, K, bits)
    x = synth.activation(synth.rng(100, N, 10, K), K, M)
    r = synth.activation(synth.rng(100, N, 11, K), N, M)
    W = np_dense(w)
    for res in (None, r):
        y64, y16, bound = oracle.qgemv(bits, w.codes, w.scales, w.biases, x, res)
        ref = x.astype(np.float64) @ W.T
        mag = np.abs(x.astype(np.float64)) @ np.abs(W).T
        if res is not None:
            ref = ref + res.astype(np.float64)
            mag = mag + np.abs(res.astype(np.float64))
        assert np.allclose(y64, ref, rtol=1e-12, atol=1e-12 * mag.max())
        assert np.allclose(bound, mag, rtol=1e-12)
        assert np.array_equal(y16, y64.astype(np.float16))


def test_four_bit_reencoded_as_eight_bit():
    K, N = 256, 7
    w4 = small_weight(5, N, K, 4)
    q = np_unpack(w4.codes, 4)                       # values 0..15
    # repack the same codes 4 per word, one per byte, low byte first
    q4 = q.reshape(N, K // 4, 4).astype(np.uint64)
    words8 = np.zeros((N, K // 4), np.uint64)
    for j in range(4):
        words8 |= q4[:, :, j] << np.uint64(8 * j)
    words8 = words8.astype(np.uint32)
    x = synth.activation(synth.rng(100, 5, 10), K)
    y4, _, _ = oracle.qgemv(4, w4.codes, w4.scales, w4.biases, x)
    y8, _, _ = oracle.qgemv(8, words8, w4.scales, w4.biases, x)
    assert np.array_equal(y4, y8)


def test_two_bit_reencoded_as_four_bit():
    K, N = 256, 9
    w2 = small_weight(3, N, K, 2)
    q = np_unpack(w2.codes, 2)                       # values 0..3
    # repack the same codes 8 per word, low nibble first
    q8 = q.reshape(N, K // 8, 8).astype(np.uint64)
    words4 = np.zeros((N, K // 8), np.uint64)
    for j in range(8):
        words4 |= q8[:, :, j] << np.uint64(4 * j)
    words4 = words4.astype(np.uint32)
    x = synth.activation(synth.rng(100, 3, 10), K)
    y2, _, _ = oracle.qgemv(2, w2.codes, w2.scales, w2.biases, x)
    y4, _, _ = oracle.qgemv(4, words4, w2.scales, w2.biases, x)
    assert np.array_equal(y2, y4)


# ------------------------------------------------------------- RMSNorm
def test_rmsnorm_closed_form_constant_input():
    K, eps = 512, 1e-5
    for c in (0.25, 1.0, -3.0, 100.0):
        x = np.full(K, c, np.float16)
        gamma = np.ones(K, np.float16)
        xn = oracle.rmsnorm(x, gamma, eps)
        cv = float(np.float16(c))
        assert np.allclose(xn, cv / np.sqrt(cv * cv + eps), rtol=1e-14)


def test_rmsnorm_against_numpy_and_scale_invariance():
    K, eps = 1024, 1e-5
    x = synth.activation(synth.rng(100, 4, 10), K)
    gamma = synth.norm_gamma(synth.rng(100, 4, 12), K)
    xn = oracle.rmsnorm(x, gamma, eps)
    xd = x.astype(np.float64)
    ref = xd / np.sqrt(np.mean(xd * xd) + eps) * gamma.astype(np.float64)
    assert np.allclose(xn, ref, rtol=1e-13)
    x4 = (x.astype(np.float64) * 4).astype(np.float16)   # exact scaling by 4
    xn4 = oracle.rmsnorm(x4, gamma, eps)
    assert np.allclose(xn4, xn, rtol=1e-5)                # equal up to eps


def test_rmsnorm_qgemv_composes():
    N, K, eps = 33, 256, 1e-5
    w = small_weight(5, N, K)
    x = synth.activation(synth.rng(100, 5, 10), K)
    gamma = synth.norm_gamma(synth.rng(100, 5, 12), K)
    y64, y16, bound = oracle.rmsnorm_qgemv(w.codes, w.scales, w.biases, x, gamma, eps)
    xd = x.astype(np.float64)
    xn = xd / np.sqrt(np.mean(xd * xd) + eps) * gamma.astype(np.float64)
    W = np_dense(w)
    assert np.allclose(y64, W @ xn, rtol=1e-12, atol=1e-12)
    assert np.allclose(bound, np.abs(W) @ np.abs(xn), rtol=1e-12)
    assert np.array_equal(y16, y64.astype(np.float16))


# -------------------------------------------------------------- SwiGLU
def test_silu_against_logistic():
    for z in np.linspace(-30, 30, 601):
        assert oracle.silu(z) == pytest.approx(z * expit(z), rel=1e-14, abs=1e-300)


def test_swiglu_zero_gate_gives_zero():
    I, K = 16, 128
    gate, up = small_weight(6, I, K), small_weight(7, I, K)
    gate.codes[:] = 0
    gate.biases[:] = 0
    x = synth.activation(synth.rng(100, 6, 10), K)
    h64, h16, _ = oracle.swiglu_qgemv((gate.codes, gate.scales, gate.biases),
                                      (up.codes, up.scales, up.biases), x)
    assert np.all(h64 == 0.0) and np.all(h16.astype(np.float64) == 0.0)


@pytest.mark.parametrize("with_norm", [False, True])
def test_swiglu_brute_force(with_norm):
    I, K, eps = 24, 320, 1e-5
    gate, up = small_weight(8, I, K), small_weight(9, I, K)
    x = synth.activation(synth.rng(100, 8, 10), K)
    gamma = synth.norm_gamma(synth.rng(100, 8, 12), K) if with_norm else None
    h64, h16, tol = oracle.swiglu_qgemv((gate.codes, gate.scales, gate.biases),
                                        (up.codes, up.scales, up.biases), x, gamma)
    xt = x.astype(np.float64)
    if with_norm:
        xt = xt / np.sqrt(np.mean(xt * xt) + eps) * gamma.astype(np.float64)
    Wg, Wu = np_dense(gate), np_dense(up)
    g, u = Wg @ xt, Wu @ xt
    h = g * expit(g) * u
    assert np.allclose(h64, h, rtol=1e-11, atol=1e-12)
    assert np.array_equal(h16, h64.astype(np.float16))
    dg = 2e-3 * (np.abs(Wg) @ np.abs(xt))
    du = 2e-3 * (np.abs(Wu) @ np.abs(xt))
    ref_tol = 1.1 * np.abs(u) * dg + np.abs(g * expit(g)) * du + np.abs(h) * 2.0**-11 + 1e-5
    assert np.allclose(tol, ref_tol, rtol=1e-10)


# ----------------------------------------------------------------- MoE
def _moe_small(E=6, H=128, I=64, seed=11):
    gu, dn = synth.moe_experts(100, seed, E, hidden=H, inter=I)
    x = synth.activation(synth.rng(100, seed, 10), H)
    r = synth.activation(synth.rng(100, seed, 11), H)
    return gu, dn, x, r


def _np_moe(gu, dn, idx, wt, x, r):
    I = gu.codes.shape[1] // 2
    xt = x.astype(np.float64)
    y = r.astype(np.float64).copy()
    for e, w in zip(idx, wt):
        if e < 0 or e >= gu.codes.shape[0]:
            continue
        Wgu = np_dense(synth.QuantWeight(gu.codes[e], gu.scales[e], gu.biases[e], 4))
        g, u = Wgu[:I] @ xt, Wgu[I:] @ xt
        h = g * expit(g) * u
        Wd = np_dense(synth.QuantWeight(dn.codes[e], dn.scales[e], dn.biases[e], 4))
        y += float(w) * (Wd @ h)
    return y


def _call_moe(gu, dn, idx, wt, x, r):
    return oracle.moe_qgemv_combine((gu.codes, gu.scales, gu.biases),
                                    (dn.codes, dn.scales, dn.biases), idx, wt, x, r)


def test_moe_brute_force_and_topk1_reduction():
    gu, dn, x, r = _moe_small()
    idx = np.array([0, 4, 2, 5], np.int32)
    wt = np.array([0.4, 0.3, 0.2, 0.1], np.float32)
    y64, y16, tol, err = _call_moe(gu, dn, idx, wt, x, r)
    assert err == 0
    assert np.allclose(y64, _np_moe(gu, dn, idx, wt, x, r), rtol=1e-11, atol=1e-11)
    assert np.array_equal(y16, y64.astype(np.float16))
    # top_k = 1, weight 1, zero residual: qgemv(down_e, swiglu(gate_e, up_e, x))
    e, I = 3, gu.codes.shape[1] // 2
    zero = np.zeros_like(r)
    y1, _, _, _ = _call_moe(gu, dn, np.array([e], np.int32), np.array([1.0], np.float32), x, zero)
    h, _, _ = oracle.swiglu_qgemv((gu.codes[e][:I], gu.scales[e][:I], gu.biases[e][:I]),
                                  (gu.codes[e][I:], gu.scales[e][I:], gu.biases[e][I:]), x)
    yd, _ = oracle.matvec_f64(4, dn.codes[e], dn.scales[e], dn.biases[e], h)
    assert np.allclose(y1, yd, rtol=1e-13, atol=1e-13)


def test_moe_permutation_and_weight_swap():
    gu, dn, x, r = _moe_small(seed=12)
    idx = np.array([0, 1, 2, 3], np.int32)
    wt = np.array([0.5, 0.25, 0.15, 0.1], np.float32)
    y, _, _, _ = _call_moe(gu, dn, idx, wt, x, r)
    perm = np.array([2, 0, 3, 1])
    yp, _, _, _ = _call_moe(gu, dn, idx[perm], wt[perm], x, r)
    assert np.allclose(y, yp, rtol=1e-12, atol=1e-12)
    ys, _, _, _ = _call_moe(gu, dn, idx, wt[[1, 0, 2, 3]], x, r)
    assert not np.allclose(y, ys, rtol=1e-6, atol=1e-6)


def test_moe_bad_index_sets_flag_and_drops_expert():
    gu, dn, x, r = _moe_small(seed=13)
    wt = np.array([0.4, 0.3, 0.2, 0.1], np.float32)
    for bad in (-1, 6, 1 << 30):
        idx = np.array([0, bad, 2, 5], np.int32)
        y, _, _, err = _call_moe(gu, dn, idx, wt, x, r)
        assert err == 1
        keep = np.array([0, 2, 5], np.int32)
        yk, _, _, errk = _call_moe(gu, dn, keep, wt[[0, 2, 3]], x, r)
        assert errk == 0
        assert np.array_equal(y, yk)


def _np_moe_tol(gu, dn, idx, wt, x, r):
    """The propagated MoE tolerance, computed from dense numpy matrices built
    through the byte-view unpack: per valid expert, the SwiGLU bound tol_h
    of its h, then 2e-3 * (sum_k |wt_k| sum_j |Wd_nj| (|h_kj| + tol_h_kj / 2e-3)
    + |r_n|) + 1e-5."""
    I = gu.codes.shape[1] // 2
    xt = x.astype(np.float64)
    mag = np.zeros(dn.codes.shape[1])
    for e, w in zip(idx, wt):
        if e < 0 or e >= gu.codes.shape[0]:
            continue
        Wgu = np_dense(synth.QuantWeight(gu.codes[e], gu.scales[e], gu.biases[e], 4))
        Wg, Wu = Wgu[:I], Wgu[I:]
        g, u = Wg @ xt, Wu @ xt
        sg = g * expit(g)
        h = sg * u
        dg = 2e-3 * (np.abs(Wg) @ np.abs(xt))
        du = 2e-3 * (np.abs(Wu) @ np.abs(xt))
        tol_h = 1.1 * np.abs(u) * dg + np.abs(sg) * du + np.abs(h) * 2.0**-11 + 1e-5
        Wd = np_dense(synth.QuantWeight(dn.codes[e], dn.scales[e], dn.biases[e], 4))
        mag += abs(float(w)) * (np.abs(Wd) @ (np.abs(h) + tol_h / 2e-3))
    return 2e-3 * (mag + np.abs(r.astype(np.float64))) + 1e-5


@pytest.mark.parametrize("idx,wt", [
    ([0, 4, 2, 5], [0.4, 0.3, 0.2, 0.1]),
    ([3, 1, 3, 0], [0.7, -0.45, 0.25, 0.5]),       # a negative weight and a repeated expert
    ([2, 9, -3, 5], [0.25, 0.25, 0.25, 0.25]),     # two indices out of range
])
def test_moe_tolerance_brute_force(idx, wt):
    gu, dn, x, r = _moe_small(seed=15)
    idx = np.array(idx, np.int32)
    wt = np.array(wt, np.float32)
    _, _, tol, _ = _call_moe(gu, dn, idx, wt, x, r)
    ref = _np_moe_tol(gu, dn, idx, wt, x, r)
    assert np.allclose(tol, ref, rtol=1e-10, atol=0)
    # without the residual the |r| term is gone: tol falls by exactly 2e-3 |r|
    _, _, tol0, _ = _call_moe(gu, dn, idx, wt, x, np.zeros_like(r))
    assert np.allclose(tol - tol0, 2e-3 * np.abs(r.astype(np.float64)), rtol=1e-9, atol=1e-15)


def test_moe_duplicate_index_counts_twice():
    gu, dn, x, r = _moe_small(seed=14)
    zero = np.zeros_like(r)
    y2, _, _, _ = _call_moe(gu, dn, np.array([1, 1], np.int32),
                            np.array([0.25, 0.25], np.float32), x, zero)
    y1, _, _, _ = _call_moe(gu, dn, np.array([1], np.int32),
                            np.array([0.5], np.float32), x, zero)
    assert np.allclose(y2, y1, rtol=1e-13, atol=1e-13)


# ----------------------------------------------------------- MoE routing
def test_moe_route_hand_example():
    # E = 6, shared expert 0, top_k = 4: routed = 3 (3.0), then 1 and 5 tie
    # at 2.0 and the lower index comes first
    logits = np.array([0.5, 2.0, 1.0, 3.0, -1.0, 2.0], np.float16)
    idx, wt = oracle.moe_route(logits, 4, 0)
    assert idx.tolist() == [0, 3, 1, 5]
    e = np.exp(np.array([0.5, 3.0, 2.0, 2.0]))
    assert np.allclose(wt, e / e.sum(), rtol=1e-15)


def test_moe_route_equal_logits_and_no_shared_expert():
    idx, wt = oracle.moe_route(np.zeros(10, np.float16), 4, 0)
    assert idx.tolist() == [0, 1, 2, 3] and np.allclose(wt, 0.25, rtol=1e-15)
    idx, wt = oracle.moe_route(np.zeros(10, np.float16), 3, -1)
    assert idx.tolist() == [0, 1, 2] and np.allclose(wt, 1 / 3, rtol=1e-15)


@pytest.mark.parametrize("E,top_k,shared", [(512, 4, 0), (64, 8, -1), (33, 1, 5), (16, 2, 15)])
def test_moe_route_against_stable_sort(E, top_k, shared):
    g = np.random.default_rng(E + top_k)
    logits = g.normal(0, 1, E).astype(np.float16)
    logits[g.choice(E, size=E // 4)] = logits[0]          # plenty of exact ties
    idx, wt = oracle.moe_route(logits, top_k, shared)
    # independent selection: a stable sort on the negated logits keeps the
    # lower index first among equal values
    order = [e for e in np.argsort(-logits.astype(np.float64), kind="stable") if e != shared]
    want = ([shared] if shared >= 0 else []) + order[:top_k - (1 if shared >= 0 else 0)]
    assert idx.tolist() == [int(v) for v in want]
    sel = logits.astype(np.float64)[want]
    assert abs(wt.sum() - 1.0) < 1e-15
    # the softmax of the chosen logits, ranked like them
    assert np.allclose(wt, np.exp(sel - sel.max()) / np.exp(sel - sel.max()).sum(), rtol=1e-14)
    assert np.all(np.diff(wt[1 if shared >= 0 else 0:]) <= 1e-15)


# ------------------------------------------------------ top-k sampling
def test_lm_head_sample_hand_example():
    # logits 1, 3, 2, 3: top 3 = indices 1 and 3 (tie at 3.0, lower first),
    # then 2; weights 1, 1, e^-1 at T = 1
    logits = np.array([1.0, 3.0, 2.0, 3.0], np.float16)
    tot = 2.0 + np.exp(-1.0)
    for u, want in ((0.2, 1), (0.5, 3), (0.9, 2), (0.0, 1)):
        tok, cand, cum = oracle.lm_head_sample(logits, 3, 1.0, u)
        assert tok == want and cand.tolist() == [1, 3, 2]
        assert np.allclose(cum, np.array([1.0, 2.0, tot]) / tot, rtol=1e-15)


def test_lm_head_sample_top1_is_greedy_and_temperature():
    g = np.random.default_rng(7)
    logits = g.normal(0, 2, 1000).astype(np.float16)
    best = int(np.argmax(logits))
    for u in (0.0, 0.5, 0.999):
        assert oracle.lm_head_sample(logits, 1, 0.7, u)[0] == best
    # a tiny temperature puts all the weight on the largest logit
    assert oracle.lm_head_sample(logits, 40, 1e-4, 0.999)[0] == best


def test_lm_head_sample_frequencies_follow_the_softmax():
    # a fine grid of u visits each candidate in proportion to its weight
    logits = np.array([0.0, 1.0, 0.5, -1.0, 2.0, 1.0], np.float16)
    k, T = 4, 0.8
    us = (np.arange(20000) + 0.5) / 20000
    toks = [oracle.lm_head_sample(logits, k, T, u)[0] for u in us]
    _, cand, _ = oracle.lm_head_sample(logits, k, T, 0.0)
    lv = logits.astype(np.float64)[cand]
    p = np.exp((lv - lv.max()) / T)
    p /= p.sum()
    freq = np.array([toks.count(int(c)) for c in cand]) / len(us)
    assert cand.tolist() == [4, 1, 5, 2]
    assert np.allclose(freq, p, atol=1e-4)


def test_lm_head_sample_boundaries():
    # two equal logits: running sums exactly 0.5 and 1.0, so u = 0.5 is not
    # exceeded by the first (the pick needs a strictly larger running sum)
    lv = np.array([2.0, 2.0, -1.0], np.float16)
    assert oracle.lm_head_sample(lv, 2, 1.0, 0.5)[0] == 1
    assert oracle.lm_head_sample(lv, 2, 1.0, 0.4999)[0] == 0
    # no running sum exceeds u >= 1: the last candidate
    assert oracle.lm_head_sample(lv, 3, 1.0, 1.0)[0] == 2
    # ties among the top values go to the lower index even when they are not first
    lv = np.array([0.0, 1.0, 3.0, 1.0, 1.0], np.float16)
    assert oracle.lm_head_sample(lv, 3, 1.0, 0.0)[1].tolist() == [2, 1, 3]


# ------------------------------------------------------ LUT / palettised
def _unpack4(codes):
    """Byte-view unpack of 4-bit codes, low nibble first (independent of the
    oracle's oracle_code)."""
    b = np.ascontiguousarray(codes).view(np.uint8)
    return np.stack([b & 15, b >> 4], axis=-1).reshape(codes.shape[0], -1).astype(np.int64)


def _lut_fixture():
    d = load_golden("hand_example_d_lut.txt")
    w0 = [int(w, 16) for w in d["words0"].split()]
    w1 = [int(w, 16) for w in d["words1"].split()]
    codes = np.array([w0, w1], np.uint32)
    lut = np.array([[float(v) for v in d["lut0"].split()],
                    [float(v) for v in d["lut1"].split()]], np.float16)
    K = int(d["K"])
    x = np.where(np.arange(K) % 2 == 0, float(d["x_even"]), float(d["x_odd"])).astype(np.float16)
    return d, codes, lut, x


def test_lut_hand_example_d():
    d, codes, lut, x = _lut_fixture()
    y64, y16, bound = oracle.lut_qgemv(codes, lut, 1, x)
    assert y64.tolist() == [float(v) for v in d["y"].split()]
    assert y16.astype(np.float64).tolist() == [float(v) for v in d["y"].split()]
    assert bound.tolist() == [float(v) for v in d["bound"].split()]
    # one table for both rows
    y64s, _, _ = oracle.lut_qgemv(codes, lut[:1], 2, x)
    assert y64s[1] == float(d["y1_shared_table"]) and y64s[0] == y64[0]
    # the fixture's misread value is what reading the nibbles high first gives
    q = _unpack4(codes)[1]
    q_hi = q.reshape(-1, 8)[:, ::-1].reshape(-1)
    lv = lut[1].astype(np.float64)
    assert np.dot(lv[q_hi], x.astype(np.float64)) == float(d["y1_high_nibble_first"])


@pytest.mark.parametrize("N,K,R,seed", [(7, 64, 1, 1), (33, 192, 4, 2), (16, 1024, 16, 3),
                                        (5, 128, 3, 4)])
def test_lut_brute_force(N, K, R, seed):
    g = np.random.default_rng(seed)
    codes = g.integers(0, 2**32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32)
    lut = g.normal(0, 0.05, size=(-(-N // R), 16)).astype(np.float16)
    x = g.normal(0, 1, size=K).astype(np.float16)
    r = g.normal(0, 1, size=N).astype(np.float16)
    w = lut.astype(np.float64)[np.arange(N)[:, None] // R, _unpack4(codes)]
    want = w @ x.astype(np.float64) + r.astype(np.float64)
    y64, y16, bound = oracle.lut_qgemv(codes, lut, R, x, r)
    assert np.allclose(y64, want, rtol=1e-12, atol=1e-12)
    assert np.allclose(bound, np.abs(w) @ np.abs(x.astype(np.float64)) + np.abs(r.astype(np.float64)),
                       rtol=1e-12)
    assert np.array_equal(y16, want.astype(np.float16))


def test_lut_affine_table_is_the_q4_format():
    # lut[v] = v * s + b (exact in fp16) is the 4-bit g64 format with that
    # scale and bias in every group of the row
    g = np.random.default_rng(11)
    N, K = 9, 256
    codes = g.integers(0, 2**32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32)
    s = (g.integers(1, 64, size=N) / 256).astype(np.float16)
    b = (-g.integers(0, 64, size=N) / 64).astype(np.float16)
    lut = (np.arange(16)[None, :] * s.astype(np.float64)[:, None]
           + b.astype(np.float64)[:, None]).astype(np.float16)
    assert np.array_equal(lut.astype(np.float64),
                          np.arange(16)[None, :] * s.astype(np.float64)[:, None]
                          + b.astype(np.float64)[:, None])
    x = g.normal(0, 1, size=K).astype(np.float16)
    y_lut, _, _ = oracle.lut_qgemv(codes, lut, 1, x)
    sc = np.repeat(s[:, None], K // 64, axis=1)
    bi = np.repeat(b[:, None], K // 64, axis=1)
    y_q4, _, _ = oracle.qgemv(4, codes, sc, bi, x)
    assert np.allclose(y_lut, y_q4, rtol=1e-13, atol=1e-13)


def test_lut_relabelling_and_shared_tables():
    g = np.random.default_rng(12)
    N, K = 12, 512
    codes = g.integers(0, 2**32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32)
    lut = g.normal(0, 0.1, size=(N, 16)).astype(np.float16)
    x = g.normal(0, 1, size=K).astype(np.float16)
    y, _, _ = oracle.lut_qgemv(codes, lut, 1, x)
    # relabel: entry v moves to perm[v] and every code follows it
    perm = g.permutation(16)
    q = _unpack4(codes)
    q2 = perm[q]
    nib = q2.reshape(N, K // 8, 8).astype(np.uint64) << (4 * np.arange(8, dtype=np.uint64))
    codes2 = nib.sum(axis=-1).astype(np.uint32)
    lut2 = np.empty_like(lut)
    lut2[:, perm] = lut
    y2, _, _ = oracle.lut_qgemv(codes2, lut2, 1, x)
    assert np.array_equal(y, y2)
    # one table per 4 rows equals per-row tables that repeat it
    shared = lut[::4]
    ya, _, _ = oracle.lut_qgemv(codes, shared, 4, x)
    yb, _, _ = oracle.lut_qgemv(codes, np.repeat(shared, 4, axis=0), 1, x)
    assert np.array_equal(ya, yb)
