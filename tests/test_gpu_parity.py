"""Parity of every C-ABI entry point against the fp64 oracle on the GPU.

Sizes span several tiles, ragged tails (N not a multiple of any row band),
both the streaming kernel (K a multiple of 1024, aligned pointers, M = 1) and
the generic kernel (other K, misaligned pointers, M > 1), and the degenerate
cases (one row, one group, zero weights, integer-exact inputs).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import load_golden
from qhelpers import check, dev16, dev_weight, plain_tol

pytestmark = pytest.mark.gpu

q = pytest.importorskip("bit_group_quantized_qgemv_gb300")


def W(seed, N, K, bits=4):
    return synth.quant_weight(synth.rng(200, seed, 1), N, K, bits)


def X(seed, K, M=None):
    return synth.activation(synth.rng(200, seed, 10), K, M)


def run_plain(bits, w, x, residual=None, y=None):
    fn = {4: q.qgemv_w4g64, 2: q.qgemv_w2g64, 8: q.qgemv_w8g64}[bits]
    return fn(dev_weight(w), x if torch.is_tensor(x) else dev16(x),
              y=y, residual=None if residual is None else
              (residual if torch.is_tensor(residual) else dev16(residual)))


# ------------------------------------------------------------ hand examples
def test_hand_example_a_exact():
    d = load_golden("hand_example_a.txt")
    words = np.array([int(v, 16) for v in d["words"].split()], np.uint32)
    x = np.array([float(v) for v in d["x"].split()], np.float16)
    for reps in (1, 16):          # K = 64 (generic kernel) and K = 1024 (streaming)
        w = synth.QuantWeight(np.tile(words, reps)[None, :],
                              np.full((1, reps), float(d["scales"]), np.float16),
                              np.full((1, reps), float(d["biases"]), np.float16), 4)
        xx = np.concatenate([x, np.zeros(64 * (reps - 1), np.float16)])
        y = run_plain(4, w, xx)
        assert float(y[0]) == float(d["y"])


def test_hand_example_c_8bit_exact():
    d = load_golden("hand_example_c.txt")
    words = np.array([int(v, 16) for v in d["words"].split()], np.uint32)
    x = np.array([float(v) for v in d["x"].split()], np.float16)
    for reps in (1, 16):          # K = 64 (generic kernel) and K = 1024 (streaming)
        w = synth.QuantWeight(np.tile(words, reps)[None, :],
                              np.full((1, reps), float(d["scales"]), np.float16),
                              np.full((1, reps), float(d["biases"]), np.float16), 8)
        xx = np.concatenate([x, np.zeros(64 * (reps - 1), np.float16)])
        y = run_plain(8, w, xx)
        assert float(y[0]) == float(d["y"])


def test_hand_example_b_exact():
    d = load_golden("hand_example_b.txt")
    r0 = [int(v, 16) for v in d["row0_words"].split()] * 8
    r1 = [int(v, 16) for v in d["row1_words"].split()] * 8
    codes = np.array([r0, r1], np.uint32)
    s = np.array([float(v) for v in d["scales"].split()], np.float16).reshape(2, 2)
    b = np.array([float(v) for v in d["biases"].split()], np.float16).reshape(2, 2)
    x = np.array([1.0 if k % 2 == 0 else -0.5 for k in range(128)], np.float16)
    y = run_plain(4, synth.QuantWeight(codes, s, b, 4), x)
    assert [float(v) for v in y.cpu()] == [float(v) for v in d["y"].split()]


# ------------------------------------------------------------- plain GEMV
FAST = [(4, 1024, 1024), (4, 7, 1024), (4, 1000, 2048), (4, 333, 3072), (4, 4099, 4096),
        (4, 601, 14336), (2, 513, 2048), (2, 300, 4096), (2, 97, 14336), (4, 1, 4096),
        (4, 152, 1024), (4, 153, 2048)]
GENERIC = [(4, 5, 64), (4, 17, 192), (4, 33, 960), (4, 3, 1088), (2, 9, 128), (2, 40, 1024),
           (2, 11, 3072)]
# 8-bit (Q8 group 64): streaming shapes (ragged bands, K up to 14336) and
# shapes the generic kernel takes
EIGHT = [(8, 1000, 2048), (8, 4099, 4096), (8, 601, 14336), (8, 7, 1024), (8, 153, 2048),
         (8, 5, 64), (8, 33, 960), (8, 3, 1088)]


@pytest.mark.parametrize("bits,N,K", FAST + GENERIC + EIGHT)
@pytest.mark.parametrize("with_res", [False, True])
def test_plain_parity(bits, N, K, with_res):
    w = W(N * 7 + K + bits, N, K, bits)
    x = X(N + K, K)
    r = X(N * 3 + K + 1, N) if with_res else None
    y = run_plain(bits, w, x, r)
    y64, _, bound = oracle.qgemv(bits, w.codes, w.scales, w.biases, x, r)
    check(y, y64, plain_tol(bound), f"w{bits} N={N} K={K} res={with_res}")


@pytest.mark.parametrize("bits", [4, 2, 8])
@pytest.mark.parametrize("M", [2, 3, 8])
def test_small_batch(bits, M):
    N, K = 203, 2048
    w = W(M * 11 + bits, N, K, bits)
    x = X(M * 13 + bits, K, M)
    r = X(M * 17 + bits, N, M)
    y = run_plain(bits, w, x, r)
    y64, _, bound = oracle.qgemv(bits, w.codes, w.scales, w.biases, x, r)
    check(y, y64, plain_tol(bound), f"w{bits} M={M}")
    # row m of the batched call agrees with the M = 1 call on x[m]
    for m in range(M):
        y1 = run_plain(bits, w, x[m], r[m])
        check(y[m], y1.double().cpu().numpy(), plain_tol(bound[m]), f"row {m}")


def test_misaligned_pointers_take_generic_path():
    N, K = 257, 4096
    w = W(5, N, K)
    x = X(6, K)
    xd = dev16(np.concatenate([[0], x]).astype(np.float16))[1:]      # 2-byte offset
    codes, s, b = dev_weight(w)
    s2 = dev16(np.concatenate([[0], w.scales.reshape(-1)]).astype(np.float16))[1:].view(N, -1)
    y = q.qgemv_w4g64((codes, s2, b), xd)
    y64, _, bound = oracle.qgemv(4, w.codes, w.scales, w.biases, x)
    check(y, y64, plain_tol(bound), "misaligned")


def test_inplace_residual():
    N, K = 777, 4096
    w = W(8, N, K)
    x = X(9, K)
    r = X(10, N)
    y = dev16(r)
    run_plain(4, w, x, residual=y, y=y)
    y64, _, bound = oracle.qgemv(4, w.codes, w.scales, w.biases, x, r)
    check(y, y64, plain_tol(bound), "in-place residual")


@pytest.mark.parametrize("bits,K", [(4, 1024), (4, 64), (2, 2048)])
def test_integer_dot_is_exact(bits, K):
    N = 64
    g = np.random.default_rng(K)
    w = W(11, N, K, bits)
    w.scales[:] = 1.0
    w.biases[:] = 0.0
    x = g.integers(-1, 2, size=K).astype(np.float16)
    y = run_plain(bits, w, x)
    y64, _, _ = oracle.qgemv(bits, w.codes, w.scales, w.biases, x)
    assert np.array_equal(y.double().cpu().numpy(), y64)


def test_zero_weights_give_exact_zero_and_residual():
    N, K = 300, 4096
    w = W(12, N, K)
    w.codes[:] = 0
    w.biases[:] = 0
    x = X(13, K)
    r = X(14, N)
    assert np.all(run_plain(4, w, x).cpu().numpy() == 0)
    assert np.array_equal(run_plain(4, w, x, r).cpu().numpy(), r)


def test_zero_codes_bias_path():
    N, K = 64, 2048
    w = W(15, N, K)
    w.codes[:] = 0
    x = X(16, K)
    y = run_plain(4, w, x)
    y64, _, bound = oracle.qgemv(4, w.codes, w.scales, w.biases, x)
    check(y, y64, plain_tol(bound), "zero codes")


# ------------------------------------------------------- RMSNorm -> GEMV
@pytest.mark.parametrize("N,K", [(1000, 1024), (4096, 4096), (37, 2048), (10, 192), (9, 1088)])
def test_rmsnorm_qgemv(N, K):
    w = W(N + K + 1, N, K)
    x = X(N + 2, K)
    gamma = synth.norm_gamma(synth.rng(200, N, 12), K)
    y = q.rmsnorm_qgemv(dev_weight(w), dev16(x), dev16(gamma), 1e-5)
    y64, _, bound = oracle.rmsnorm_qgemv(w.codes, w.scales, w.biases, x, gamma, 1e-5)
    check(y, y64, plain_tol(bound), f"rmsnorm N={N} K={K}")


# ---------------------------------------------------------------- SwiGLU
@pytest.mark.parametrize("I,K", [(700, 1024), (3072, 1024), (1433, 4096), (50, 320), (8, 64)])
@pytest.mark.parametrize("norm", [False, True])
def test_swiglu_qgemv(I, K, norm):
    gate, up = W(I + 1, I, K), W(I + 2, I, K)
    x = X(I + 3, K)
    gamma = synth.norm_gamma(synth.rng(200, I, 13), K) if norm else None
    h = q.swiglu_qgemv(dev_weight(gate), dev_weight(up), dev16(x),
                       None if gamma is None else dev16(gamma), 1e-5)
    h64, _, tol = oracle.swiglu_qgemv((gate.codes, gate.scales, gate.biases),
                                      (up.codes, up.scales, up.biases), x, gamma, 1e-5)
    check(h, h64, tol, f"swiglu I={I} K={K} norm={norm}")


# ------------------------------------------------------------------- MoE
def moe_case(E, H, I, seed):
    gu, dn = synth.moe_experts(201, seed, E, hidden=H, inter=I)
    x = X(seed + 30, H)
    r = X(seed + 31, H)
    return gu, dn, x, r


def run_moe(gu, dn, idx, wt, x, r, err=None):
    return q.moe_qgemv_combine(dev_weight(gu), dev_weight(dn),
                               torch.from_numpy(np.asarray(idx, np.int32)).cuda(),
                               torch.from_numpy(np.asarray(wt, np.float32)).cuda(),
                               dev16(x), None if r is None else dev16(r), err_flag=err)


@pytest.mark.parametrize("E,H,I,top_k", [(8, 1024, 1024, 4), (6, 2048, 1024, 4),
                                         (5, 1024, 2048, 3), (7, 256, 128, 4),
                                         (4, 1024, 1024, 1), (9, 1024, 1024, 8)])
def test_moe_parity(E, H, I, top_k):
    gu, dn, x, r = moe_case(E, H, I, E + H + I + top_k)
    g = np.random.default_rng(E * top_k)
    idx = g.choice(E, size=top_k, replace=False).astype(np.int32)
    wt = g.dirichlet(np.ones(top_k)).astype(np.float32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = run_moe(gu, dn, idx, wt, x, r, err)
    y64, _, tol, e = oracle.moe_qgemv_combine((gu.codes, gu.scales, gu.biases),
                                              (dn.codes, dn.scales, dn.biases), idx, wt, x, r)
    assert e == 0 and int(err.item()) == 0
    check(y, y64, tol, f"moe E={E} H={H} I={I} k={top_k}")


@pytest.mark.parametrize("H,I", [(1024, 1024), (256, 128)])
def test_moe_bad_and_repeated_indices(H, I):
    E = 6
    gu, dn, x, r = moe_case(E, H, I, 77 + H)
    wt = np.array([0.4, 0.3, 0.2, 0.1], np.float32)
    for idx in ([0, -1, 2, 5], [0, 6, 2, 1 << 30], [3, 3, 1, 1], [-5, 99, 7, 6]):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        y = run_moe(gu, dn, idx, wt, x, r, err)
        y64, _, tol, e = oracle.moe_qgemv_combine((gu.codes, gu.scales, gu.biases),
                                                  (dn.codes, dn.scales, dn.biases),
                                                  np.array(idx, np.int32), wt, x, r)
        assert int(err.item()) == e, idx
        check(y, y64, tol, f"moe idx={idx}")


def test_moe_null_residual_and_err_flag():
    gu, dn, x, _ = moe_case(4, 1024, 1024, 5)
    idx, wt = [1, 0, 3, 2], [0.25, 0.25, 0.25, 0.25]
    y = run_moe(gu, dn, idx, wt, x, None)
    y64, _, tol, _ = oracle.moe_qgemv_combine((gu.codes, gu.scales, gu.biases),
                                              (dn.codes, dn.scales, dn.biases),
                                              np.array(idx, np.int32), np.array(wt, np.float32),
                                              x, None)
    check(y, y64, tol, "moe no residual")


# ------------------------------------------------------- attention stand-in
@pytest.mark.parametrize("n_q,n_kv,d", [(32, 8, 128), (16, 8, 128), (4, 4, 64), (6, 1, 32)])
def test_attention_seq1_copies_value_heads(n_q, n_kv, d):
    qkv = X(n_q * 100 + n_kv, (n_q + 2 * n_kv) * d)
    out = q.decode_attention_seq1(dev16(qkv), n_q, n_kv, d).cpu().numpy()
    v = qkv[(n_q + n_kv) * d:].reshape(n_kv, d)
    ref = np.repeat(v, n_q // n_kv, axis=0).reshape(-1)
    assert np.array_equal(out.view(np.uint16), ref.view(np.uint16))


def test_no_device_side_timeouts():
    assert q.device_status() == 0


# ------------------------------------------------- residual + RMSNorm epilogue
@pytest.mark.parametrize("K,with_res", [(4096, True), (1024, True), (14336, True), (333, True),
                                        (4096, False), (1, True)])
def test_residual_rmsnorm(K, with_res):
    eps = 1e-5
    x = X(K + 1, K)
    r = X(K + 2, K) if with_res else None
    gamma = synth.norm_gamma(synth.rng(200, K, 13), K)
    h, xn = q.residual_rmsnorm(dev16(x), dev16(gamma), None if r is None else dev16(r), eps)
    # h: the exact sum rounded once to fp16, bit for bit
    h16 = (x.astype(np.float64) + r.astype(np.float64)).astype(np.float16) if with_res else x
    assert np.array_equal(h.cpu().numpy().view(np.uint16), h16.view(np.uint16))
    xn64 = oracle.rmsnorm(h16, gamma, eps)
    tol = (2.0 ** -11 + 1e-5) * np.abs(xn64) + 1e-7   # one fp16 rounding + fp32 sums
    check(xn, xn64, tol, f"residual_rmsnorm K={K} res={with_res}")
