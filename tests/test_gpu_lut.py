"""qgemv_lut4: the LUT / palettised 4-bit GEMV against the fp64 oracle.

Every output within |y - y_ref| <= 2e-3 * sum|w||x| + 1e-5 (the products of
table entries and activations are exact on both sides; only the fp32
accumulation order differs).  Shapes: the Llama-3.1-8B-shaped matvecs
(each of the three kernel configurations: K <= 2048, K <= 4096, longer),
the Qwen3-0.6B-shaped lm_head with one table for the whole tensor, tables
shared by groups of rows that do not divide N, ragged and tiny shapes, the
longest K, residuals, and tables holding extreme fp16 values.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from qhelpers import check, dev16, plain_tol

pytestmark = pytest.mark.gpu

q = pytest.importorskip("bit_group_quantized_qgemv_gb300")


def W(seed, N, K, R):
    return synth.lut_weight(synth.rng(7, seed, synth.TID["lut"]), N, K, R)


def X(seed, K):
    return synth.activation(synth.rng(7, seed, synth.TID["x"]), K)


def run(w, x, residual=None):
    codes = torch.from_numpy(w.codes.view(np.int32)).cuda()
    lut = torch.from_numpy(w.lut).cuda()
    r = None if residual is None else dev16(residual)
    return q.qgemv_lut4(codes, lut, dev16(x), rows_per_lut=w.rows_per_lut, residual=r)


@pytest.mark.parametrize("N,K,R", [
    (6144, 4096, 1),      # QKV-shaped, K <= 4096 configuration
    (4096, 4096, 1),      # o_proj
    (14336, 4096, 1),     # gate / up
    (4096, 14336, 1),     # down: the long-row configuration
    (151936, 1024, 151936),  # lm_head, one table for the tensor (K <= 2048 configuration)
    (1001, 2048, 64),     # tables shared by 64 rows, 1001 not a multiple
    (333, 960, 7),
    (7, 64, 1),
    (1, 16384, 1),        # the longest K
    (5, 6144, 2),
])
def test_lut_parity(N, K, R):
    w = W(N + K + R, N, K, R)
    x = X(N + K, K)
    y = run(w, x)
    y64, _, bound = oracle.lut_qgemv(w.codes, w.lut, R, x)
    check(y, y64, plain_tol(bound), f"lut N={N} K={K} R={R}")


@pytest.mark.parametrize("N,K", [(4096, 4096), (300, 1024), (77, 14336)])
def test_lut_residual(N, K):
    w = W(N + 1, N, K, 1)
    x = X(N + 2, K)
    r = X(N + 3, N)
    y = run(w, x, r)
    y64, _, bound = oracle.lut_qgemv(w.codes, w.lut, 1, x, r)
    check(y, y64, plain_tol(bound), f"lut residual N={N} K={K}")


def test_lut_extreme_tables():
    # entries at the ends of fp16 (65504, the smallest subnormal, signed
    # zeros) with small activations: the products stay exact, the sums fp32
    N, K = 64, 2048
    w = W(5, N, K, 1)
    ext = np.array([65504.0, -65504.0, 6e-8, -6e-8, 0.0, -0.0, 1.0, -1.0,
                    2048.0, -2048.0, 0.5, 3e-5, -3e-5, 100.0, -100.0, 7.0], np.float16)
    w.lut[:] = ext
    w.lut[1::2] = ext[::-1]
    x = (X(6, K).astype(np.float32) * 1e-4).astype(np.float16)
    y = run(w, x)
    y64, _, bound = oracle.lut_qgemv(w.codes, w.lut, 1, x)
    check(y, y64, plain_tol(bound), "lut extreme tables")


def test_lut_single_code_rows_pick_one_entry():
    # every code of row n equals n % 16, x = 1: y[n] = K * lut[n][n % 16], exact
    N, K = 48, 256
    w = W(7, N, K, 1)
    nib = (np.arange(N) % 16).astype(np.uint32)
    w.codes[:] = (nib * 0x11111111)[:, None]
    w.lut[:] = (np.arange(16, dtype=np.float16)[None, :] * 0.125 - 1.0).astype(np.float16)
    x = np.ones(K, np.float16)
    y = run(w, x).cpu().numpy().astype(np.float64)
    want = K * (nib.astype(np.float64) * 0.125 - 1.0)
    assert np.array_equal(y, want.astype(np.float16).astype(np.float64))
