"""The small-batch GEMV (M = 2..8) against the oracle.

M >= 3 runs on the tensor-core kernel, and so does M = 2 on short ops (K <=
4096, at most 128 KB of weights per SM; longer ones take the CUDA-core
small-batch kernel).  The tensor-core kernel stages the batch's activations
in shared memory (2 * M_pad * K bytes, M_pad = 4 or 8): one CTA per tile
when they are small, else K split over a thread-block cluster of 4 (or 2)
CTAs whose fp32 partials meet in rank 0 (M >= 5 from K = 8192, every M >=
3 from K = 14336), and passes of at most 4 rows only when even that cannot
hold them.  Shapes here cover every plan: whole rows of 512 to 4096 k in
one stage, chunked rows, ragged 16-row tiles, bands of a few rows, cluster
splits, residuals, 2-bit codes, exact integer dots (scale 1, bias 0, x in
{-1, 0, 1}), and activations whose pre-divided copies (x / 16, x / 64) are
fp16 subnormals.  Every output is checked against the fp64 oracle within
the matvec tolerance, and each batch row against the M = 1 call on that
row.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from qhelpers import check, dev16, dev_weight, plain_tol

pytestmark = pytest.mark.gpu

q = pytest.importorskip("bit_group_quantized_qgemv_gb300")


def W(seed, N, K, bits):
    return synth.quant_weight(synth.rng(500, seed, 1), N, K, bits)


def X(seed, K, M):
    return synth.activation(synth.rng(500, seed, 10), K, M)


def run(bits, w, x, r=None):
    fn = q.qgemv_w4g64 if bits == 4 else q.qgemv_w2g64
    return fn(dev_weight(w), dev16(x), residual=None if r is None else dev16(r))


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("M,N,K", [
    (2, 203, 512), (3, 77, 1024), (4, 1000, 3072), (5, 4096, 4096), (8, 4099, 4096), (3, 500, 512),
    (6, 1000, 14336), (7, 64, 14336),
    (8, 17, 8192), (7, 301, 8192), (2, 96, 14336), (4, 1001, 14336), (5, 333, 14336),
    (8, 4096, 14336), (6, 2, 2048), (8, 1, 1024), (2, 151936 // 8, 1024),
    (4, 300, 16384), (8, 333, 16384), (5, 97, 32768), (3, 40, 32768),
    (8, 1, 14336), (4, 1, 14336), (5, 4096 + 15, 8192),
    (8, 151936 // 4, 1024), (4, 1024, 3072), (6, 3072, 1024),
])
def test_batch_parity(bits, M, N, K):
    w = W(N + K + M + bits, N, K, bits)
    x = X(M + K, K, M)
    r = X(M + N, N, M) if (N + M) % 2 else None
    y = run(bits, w, x, r)
    y64, _, bound = oracle.qgemv(bits, w.codes, w.scales, w.biases, x, r)
    check(y, y64, plain_tol(bound), f"w{bits} M={M} N={N} K={K}")
    if N * K <= 4096 * 4096:
        for m in range(M):
            y1 = run(bits, w, x[m], None if r is None else r[m])
            check(y[m], y1.double().cpu().numpy(), plain_tol(bound[m]), f"row {m}")


@pytest.mark.parametrize("bits,K", [(4, 1024), (2, 2048)])
def test_batch_integer_dot_is_exact(bits, K):
    """scale 1, bias 0, x in {-1, 0, 1}: every product and partial sum is an
    integer far below 2^24, so the result is the integer dot product exactly
    (for 2-bit, x / 64 stays an exact fp16)."""
    N, M = 64, 8
    w = W(K + bits, N, K, bits)
    w.scales[:] = np.float16(1.0)
    w.biases[:] = np.float16(0.0)
    g = np.random.default_rng(K)
    x = g.integers(-1, 2, size=(M, K)).astype(np.float16)
    y = run(bits, w, x).cpu().numpy().astype(np.float64)
    y64, _, _ = oracle.qgemv(bits, w.codes, w.scales, w.biases, x)
    assert np.array_equal(y, y64)


def test_batch_tiny_activations():
    """Activations near the bottom of fp16 (their x / 16 and x / 64 copies
    are subnormal and rounded): still within the tolerance."""
    N, K, M = 300, 2048, 8
    for bits in (4, 2):
        w = W(7 + bits, N, K, bits)
        x = X(9, K, M)
        x[1] *= np.float16(2.0 ** -12)           # |x| ~ 2^-12: x / 64 subnormal
        x[3, ::3] = np.float16(6.1e-5)           # smallest normal fp16
        x[5, ::7] = np.float16(2.0 ** -24)       # smallest subnormal
        y = run(bits, w, x)
        y64, _, bound = oracle.qgemv(bits, w.codes, w.scales, w.biases, x)
        check(y, y64, plain_tol(bound), f"tiny activations w{bits}")


def test_batch_inplace_residual_and_guards():
    N, K, M = 1003, 4096, 6
    w = W(11, N, K, 4)
    x = X(12, K, M)
    r = X(13, N, M)
    G = 256
    buf = torch.full((M * N + 2 * G,), 0x7E5A, dtype=torch.int16, device="cuda")
    yv = buf[G:G + M * N].view(torch.float16).view(M, N)
    yv.copy_(dev16(r))
    q.qgemv_w4g64(dev_weight(w), dev16(x), y=yv, residual=yv)   # residual == y
    torch.cuda.synchronize()
    raw = buf.cpu().numpy()
    assert np.all(raw[:G] == 0x7E5A) and np.all(raw[G + M * N:] == 0x7E5A)
    y64, _, bound = oracle.qgemv(4, w.codes, w.scales, w.biases, x, r)
    check(yv, y64, plain_tol(bound), "in-place residual")
    assert q.device_status() == 0


@pytest.mark.parametrize("M,N,K", [(8, 1003, 14336), (5, 77, 32768)])
def test_batch_cluster_split_inplace_residual_and_guards(M, N, K):
    """The cluster-split path (rank 0 adds the other ranks' partials and
    writes y) with y aliasing the residual, inside guard bands."""
    w = W(13 + K, N, K, 4)
    x = X(14 + K, K, M)
    r = X(15 + N, N, M)
    G = 256
    buf = torch.full((M * N + 2 * G,), 0x7E5A, dtype=torch.int16, device="cuda")
    yv = buf[G:G + M * N].view(torch.float16).view(M, N)
    yv.copy_(dev16(r))
    q.qgemv_w4g64(dev_weight(w), dev16(x), y=yv, residual=yv)
    torch.cuda.synchronize()
    raw = buf.cpu().numpy()
    assert np.all(raw[:G] == 0x7E5A) and np.all(raw[G + M * N:] == 0x7E5A)
    y64, _, bound = oracle.qgemv(4, w.codes, w.scales, w.biases, x, r)
    check(yv, y64, plain_tol(bound), f"cluster split M={M} K={K}")
    assert q.device_status() == 0


@pytest.mark.parametrize("M", [2, 4, 8])
def test_batch_misaligned_activations_take_generic_path(M):
    """Activations 2 bytes off a 16-byte boundary: neither small-batch
    kernel applies (both read x with 16-byte loads), the generic kernel
    takes the call, same results."""
    N, K = 301, 4096
    w = W(21 + M, N, K, 4)
    x = X(22 + M, K, M)
    flat = np.concatenate([[0], x.reshape(-1)]).astype(np.float16)
    xd = dev16(flat)[1:].view(M, K)
    assert xd.data_ptr() % 16 == 2
    y = q.qgemv_w4g64(dev_weight(w), xd)
    y64, _, bound = oracle.qgemv(4, w.codes, w.scales, w.biases, x)
    check(y, y64, plain_tol(bound), f"misaligned M={M}")
