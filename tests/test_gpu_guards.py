"""Guard bands and the bounded-wait self-test.

Every entry point may write only its output (and its workspace): outputs and
workspaces are views into larger device buffers whose margins hold a
sentinel bit pattern, which must be bit-identical after the call, while the
output itself is checked against the oracle (stand-in for a memory checker,
which this GPU pool does not offer).  The self-test makes a device wait that
nothing satisfies run out: the kernel must give up, report it through
qgemv_device_status and leave the context usable.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import synth
from qhelpers import check, dev16, dev_weight, plain_tol

pytestmark = pytest.mark.gpu

q = pytest.importorskip("bit_group_quantized_qgemv_gb300")

G = 256  # guard elements on each side (keeps 16-byte and 256-byte alignment)
SENTINEL = {torch.float16: (torch.int16, 0x7E5A), torch.float32: (torch.int32, 0x7FA5A5A5),
            torch.uint8: (torch.uint8, 0xA5)}


def guarded(n, dtype=torch.float16):
    """(buffer, view of n elements between two guard bands)."""
    buf = torch.empty(n + 2 * G, dtype=dtype, device="cuda")
    itype, pat = SENTINEL[dtype]
    buf.view(itype).fill_(pat)
    return buf, buf[G:G + n]


def assert_guards(buf, n, what):
    itype, pat = SENTINEL[buf.dtype]
    raw = buf.view(itype).cpu().numpy()
    head, tail = raw[:G], raw[G + n:]
    want = np.array(pat, dtype=raw.dtype)
    assert np.all(head == want), f"{what}: {int(np.count_nonzero(head != want))} guard values before the output overwritten"
    assert np.all(tail == want), f"{what}: {int(np.count_nonzero(tail != want))} guard values after the output overwritten"


def W(seed, N, K, bits=4):
    return synth.quant_weight(synth.rng(300, seed, 1), N, K, bits)


def X(seed, K, M=None):
    return synth.activation(synth.rng(300, seed, 10), K, M)


@pytest.mark.parametrize("bits,N,K,M", [
    (4, 1000, 2048, 1),    # streaming kernel, ragged row bands
    (4, 4099, 4096, 1),
    (2, 97, 14336, 1),
    (4, 33, 960, 1),       # generic kernel
    (4, 601, 4096, 3),     # small-batch kernel
    (4, 100, 2048, 8),
    (2, 203, 14336, 8),    # small-batch, two passes of 4 rows
    (8, 1000, 2048, 1),    # 8-bit streaming
    (8, 203, 4096, 3),     # 8-bit, M > 1 (generic kernel)
])
def test_plain_writes_only_y(bits, N, K, M):
    w = W(N + K + M, N, K, bits)
    x = X(N + M, K, None if M == 1 else M)
    r = X(N + 7, N, None if M == 1 else M)
    buf, y = guarded(M * N)
    y = y.view(N) if M == 1 else y.view(M, N)
    fn = {4: q.qgemv_w4g64, 2: q.qgemv_w2g64, 8: q.qgemv_w8g64}[bits]
    fn(dev_weight(w), dev16(x), y=y, residual=dev16(r))
    torch.cuda.synchronize()
    assert_guards(buf, M * N, f"w{bits} N={N} K={K} M={M}")
    y64, _, bound = oracle.qgemv(bits, w.codes, w.scales, w.biases, x, r)
    check(y, y64, plain_tol(bound), f"guarded w{bits} N={N} K={K} M={M}")


@pytest.mark.parametrize("N,K", [(1000, 1024), (37, 2048), (9, 1088)])
def test_rmsnorm_writes_only_y(N, K):
    w = W(N + K, N, K)
    x = X(N + 1, K)
    gamma = synth.norm_gamma(synth.rng(300, N, 12), K)
    buf, y = guarded(N)
    q.rmsnorm_qgemv(dev_weight(w), dev16(x), dev16(gamma), 1e-5, y=y)
    torch.cuda.synchronize()
    assert_guards(buf, N, f"rmsnorm N={N} K={K}")
    y64, _, bound = oracle.rmsnorm_qgemv(w.codes, w.scales, w.biases, x, gamma, 1e-5)
    check(y, y64, plain_tol(bound), f"guarded rmsnorm N={N} K={K}")


@pytest.mark.parametrize("I,K", [(1433, 4096), (50, 320)])
def test_swiglu_writes_only_h(I, K):
    gate, up = W(I + 1, I, K), W(I + 2, I, K)
    x = X(I + 3, K)
    gamma = synth.norm_gamma(synth.rng(300, I, 13), K)
    buf, h = guarded(I)
    q.swiglu_qgemv(dev_weight(gate), dev_weight(up), dev16(x), dev16(gamma), 1e-5, h=h)
    torch.cuda.synchronize()
    assert_guards(buf, I, f"swiglu I={I} K={K}")
    h64, _, tol = oracle.swiglu_qgemv((gate.codes, gate.scales, gate.biases),
                                      (up.codes, up.scales, up.biases), x, gamma, 1e-5)
    check(h, h64, tol, f"guarded swiglu I={I} K={K}")


@pytest.mark.parametrize("E,H,I,top_k", [(6, 1024, 1024, 4), (5, 256, 128, 3)])
def test_moe_writes_only_y_and_workspace(E, H, I, top_k):
    gu, dn = synth.moe_experts(301, E + H, E, hidden=H, inter=I)
    x, r = X(E + 1, H), X(E + 2, H)
    g = np.random.default_rng(E + H)
    idx = g.choice(E, size=top_k, replace=False).astype(np.int32)
    wt = g.dirichlet(np.ones(top_k)).astype(np.float32)
    ybuf, y = guarded(H)
    nws = q.moe_workspace_bytes(top_k, I) // 4
    wbuf, ws = guarded(nws, torch.float32)
    q.moe_qgemv_combine(dev_weight(gu), dev_weight(dn), torch.from_numpy(idx).cuda(),
                        torch.from_numpy(wt).cuda(), dev16(x), dev16(r), y=y, workspace=ws)
    torch.cuda.synchronize()
    assert_guards(ybuf, H, "moe y")
    assert_guards(wbuf, nws, "moe workspace")
    y64, _, tol, _ = oracle.moe_qgemv_combine((gu.codes, gu.scales, gu.biases),
                                              (dn.codes, dn.scales, dn.biases), idx, wt, x, r)
    check(y, y64, tol, f"guarded moe E={E} H={H} I={I} k={top_k}")


@pytest.mark.parametrize("N,K,R", [(1000, 2048, 1), (301, 4096, 3), (77, 14336, 77)])
def test_lut_writes_only_y(N, K, R):
    w = synth.lut_weight(synth.rng(300, N + K, 19), N, K, R)
    x = X(N + 5, K)
    r = X(N + 6, N)
    buf, y = guarded(N)
    codes = torch.from_numpy(w.codes.view(np.int32)).cuda()
    q.qgemv_lut4(codes, torch.from_numpy(w.lut).cuda(), dev16(x), rows_per_lut=R, y=y,
                 residual=dev16(r))
    torch.cuda.synchronize()
    assert_guards(buf, N, f"lut N={N} K={K} R={R}")
    y64, _, bound = oracle.lut_qgemv(w.codes, w.lut, R, x, r)
    check(y, y64, plain_tol(bound), f"guarded lut N={N} K={K} R={R}")


def test_attention_seq1_writes_only_out():
    n_q, n_kv, d = 6, 2, 64
    qkv = X(5, (n_q + 2 * n_kv) * d)
    buf, out = guarded(n_q * d)
    q.decode_attention_seq1(dev16(qkv), n_q, n_kv, d, out=out)
    torch.cuda.synchronize()
    assert_guards(buf, n_q * d, "attention_seq1")
    v = qkv[(n_q + n_kv) * d:].reshape(n_kv, d)
    ref = np.repeat(v, n_q // n_kv, axis=0).reshape(-1)
    assert np.array_equal(out.cpu().numpy().view(np.uint16), ref.view(np.uint16))


def test_decode_stack_writes_only_y_and_workspace():
    H, nq, nkv, hd, I, NL = 1024, 8, 2, 128, 2048, 2
    layers = []
    for l in range(NL):
        r = lambda t: synth.rng(302, l, synth.TID[t])  # noqa: E731
        d = {"qkv": synth.quant_weight(r("qkv"), (nq + 2 * nkv) * hd, H),
             "o": synth.quant_weight(r("o"), H, nq * hd),
             "gate": synth.quant_weight(r("gate"), I, H), "up": synth.quant_weight(r("up"), I, H),
             "down": synth.quant_weight(r("down"), H, I)}
        d = {k: dev_weight(v) for k, v in d.items()}
        d["attn_norm"] = dev16(synth.norm_gamma(r("gamma1"), H))
        d["mlp_norm"] = dev16(synth.norm_gamma(r("gamma2"), H))
        layers.append(d)
    sh = q.stack_shape(H, nq, nkv, hd, I, NL, 1e-5)
    x = dev16(X(303, H))
    nws = q.decode_stack_workspace_bytes(sh)
    ybuf, y = guarded(H)
    wbuf, ws = guarded(nws, torch.uint8)
    q.decode_stack(layers, sh, x, y=y, workspace=ws)
    torch.cuda.synchronize()
    assert_guards(ybuf, H, "decode stack y")
    assert_guards(wbuf, nws, "decode stack workspace")
    y_ref = q.decode_stack(layers, sh, x)
    assert torch.equal(y, y_ref)
    assert bool(torch.isfinite(y.float()).all())


def test_bounded_wait_gives_up_and_context_survives():
    assert q.device_status() == 0          # (read and clear)
    t0 = time.perf_counter()
    q.selftest_wait_timeout(5000)          # 5 ms on a barrier nothing arrives on
    flags = q.device_status()              # synchronises
    elapsed = time.perf_counter() - t0
    assert flags & 1, "the bounded wait did not report its timeout"
    assert 0.004 <= elapsed < 5.0, elapsed
    assert q.device_status() == 0          # the word was cleared by the read
    # the context still works: a streaming-kernel parity case
    w = W(9, 1000, 4096)
    x = X(10, 4096)
    y = q.qgemv_w4g64(dev_weight(w), dev16(x))
    y64, _, bound = oracle.qgemv(4, w.codes, w.scales, w.biases, x)
    check(y, y64, plain_tol(bound), "after the self-test")
    assert q.device_status() == 0
