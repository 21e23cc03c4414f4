"""Guard bands around the outputs of the sampling, greedy lm_head, router
and residual+RMSNorm entry points.

Each output (token, candidate indices and weights, logits, expert indices and
weights, h, xn, the argmax scratch) is a view into a larger device buffer
whose margins hold a sentinel bit pattern that must be bit-identical after
the call: a write of even one element past an output's end is caught, which
the parity checks (that read exactly the output's elements) cannot see.  The
outputs themselves are checked as in the parity tests.  Sampling k covers
the rank-counting sort (k <= 256) and the bitonic network (k > 256).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from qhelpers import check, dev16, dev_weight, plain_tol

pytestmark = pytest.mark.gpu

q = pytest.importorskip("bit_group_quantized_qgemv_gb300")

G = 256  # guard elements on each side
SENTINEL = {torch.float16: (torch.int16, 0x7E5A), torch.float32: (torch.int32, 0x7FA5A5A5),
            torch.int32: (torch.int32, 0x5A5A5A5A), torch.uint8: (torch.uint8, 0xA5)}


def guarded(n, dtype):
    buf = torch.empty(n + 2 * G, dtype=dtype, device="cuda")
    itype, pat = SENTINEL[dtype]
    buf.view(itype).fill_(pat)
    return buf, buf[G:G + n]


def assert_guards(buf, n, what):
    itype, pat = SENTINEL[buf.dtype]
    raw = buf.view(itype).cpu().numpy()
    want = np.array(pat, dtype=raw.dtype)
    assert np.all(raw[:G] == want), f"{what}: guard before the output overwritten"
    assert np.all(raw[G + n:] == want), f"{what}: guard after the output overwritten"


def _logits(N, seed, step=None):
    return synth.logits(synth.rng(6, seed, synth.TID["spare"]), N, step=step)


@pytest.mark.parametrize("N,k", [(151936, 1), (151936, 50), (151936, 300), (128256, 1024),
                                 (1001, 257), (9, 9)])
def test_sample_topk_writes_only_its_outputs(N, k):
    lg = _logits(N, N + k, step=0.25 if k > 256 else None)
    u = np.float32(0.6180339)
    tbuf, tok = guarded(1, torch.int32)
    ibuf, cidx = guarded(k, torch.int32)
    pbuf, cprob = guarded(k, torch.float32)
    ud = torch.tensor([u], dtype=torch.float32, device="cuda")
    q.sample_topk(dev16(lg), k, 0.8, ud, token=tok, want_topk=True, topk_idx=cidx, topk_prob=cprob)
    torch.cuda.synchronize()
    assert_guards(tbuf, 1, f"sample token N={N} k={k}")
    assert_guards(ibuf, k, f"sample candidates N={N} k={k}")
    assert_guards(pbuf, k, f"sample weights N={N} k={k}")
    _, cand, _ = oracle.lm_head_sample(lg, k, 0.8, float(u))
    assert np.array_equal(cidx.cpu().numpy(), cand), f"candidates N={N} k={k}"
    assert int(tok.item()) in cand.tolist()


def test_lm_head_sample_writes_only_its_outputs():
    N, K, k = 4099, 1024, 64
    w = synth.quant_weight(synth.rng(6, 1, synth.TID["lm_head"]), N, K, 4)
    x = synth.activation(synth.rng(6, 1, synth.TID["x"]), K)
    lbuf, lg = guarded(N, torch.float16)
    tbuf, tok = guarded(1, torch.int32)
    ibuf, cidx = guarded(k, torch.int32)
    pbuf, cprob = guarded(k, torch.float32)
    ud = torch.tensor([0.25], dtype=torch.float32, device="cuda")
    q.lm_head_sample(dev_weight(w), dev16(x), k, 1.0, ud, logits=lg, token=tok, want_topk=True,
                     topk_idx=cidx, topk_prob=cprob)
    torch.cuda.synchronize()
    for buf, n, what in ((lbuf, N, "logits"), (tbuf, 1, "token"), (ibuf, k, "candidates"),
                         (pbuf, k, "weights")):
        assert_guards(buf, n, "lm_head_sample " + what)
    y64, _, bound = oracle.qgemv(4, w.codes, w.scales, w.biases, x)
    check(lg, y64, plain_tol(bound), "guarded lm_head_sample logits")
    _, cand, _ = oracle.lm_head_sample(lg.cpu().numpy(), k, 1.0, 0.25)
    assert np.array_equal(cidx.cpu().numpy(), cand)


@pytest.mark.parametrize("N,K", [(151936, 1024), (1001, 2048), (77, 960)])
def test_lm_head_argmax_writes_only_its_outputs(N, K):
    w = synth.quant_weight(synth.rng(6, N, synth.TID["lm_head"]), N, K, 4)
    x = synth.activation(synth.rng(6, N, synth.TID["x"]), K)
    lbuf, lg = guarded(N, torch.float16)
    tbuf, tok = guarded(1, torch.int32)
    nsc = q.argmax_scratch_bytes()
    sbuf, scratch = guarded(nsc, torch.uint8)
    scratch.zero_()
    for _ in range(2):   # the scratch is left zeroed for the next call
        q.lm_head_argmax(dev_weight(w), dev16(x), logits=lg, scratch=scratch, token=tok)
        torch.cuda.synchronize()
        assert_guards(lbuf, N, "argmax logits")
        assert_guards(tbuf, 1, "argmax token")
        assert_guards(sbuf, nsc, "argmax scratch")
        assert int(scratch.cpu().numpy().sum()) == 0
        lv = lg.cpu().numpy()
        assert int(tok.item()) == int(np.argmax(lv))
    y64, _, bound = oracle.qgemv(4, w.codes, w.scales, w.biases, x)
    check(lg, y64, plain_tol(bound), f"guarded argmax logits N={N}")


@pytest.mark.parametrize("E,H,top_k,shared", [(512, 4096, 4, 0), (33, 960, 3, -1)])
def test_moe_router_writes_only_its_outputs(E, H, top_k, shared):
    w = synth.quant_weight(synth.rng(3, E + 1, synth.TID["router"]), E, H, 4)
    x = synth.activation(synth.rng(3, E + 1, synth.TID["x"]), H)
    lbuf, lg = guarded(E, torch.float16)
    ibuf, idx = guarded(top_k, torch.int32)
    wbuf, wt = guarded(top_k, torch.float32)
    q.moe_router(dev_weight(w), dev16(x), top_k=top_k, shared=shared, logits=lg, idx=idx, wt=wt)
    torch.cuda.synchronize()
    assert_guards(lbuf, E, "router logits")
    assert_guards(ibuf, top_k, "router indices")
    assert_guards(wbuf, top_k, "router weights")
    want_idx, want_wt = oracle.moe_route(lg.cpu().numpy(), top_k, shared)
    assert idx.cpu().numpy().tolist() == want_idx.tolist()
    assert np.allclose(wt.cpu().numpy().astype(np.float64), want_wt, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("K,with_res", [(4096, True), (1000, True), (1024, False)])
def test_residual_rmsnorm_writes_only_its_outputs(K, with_res):
    eps = 1e-5
    x = synth.activation(synth.rng(300, K, 10), K)
    r = synth.activation(synth.rng(300, K, 11), K) if with_res else None
    gamma = synth.norm_gamma(synth.rng(300, K, 13), K)
    xbuf, xn = guarded(K, torch.float16)
    hbuf, h = guarded(K, torch.float16)
    q.residual_rmsnorm(dev16(x), dev16(gamma), None if r is None else dev16(r), eps,
                       h=h if with_res else None, xn=xn)
    torch.cuda.synchronize()
    assert_guards(xbuf, K, "residual_rmsnorm xn")
    assert_guards(hbuf, K, "residual_rmsnorm h")
    h16 = (x.astype(np.float64) + r.astype(np.float64)).astype(np.float16) if with_res else x
    if with_res:
        assert np.array_equal(h.cpu().numpy().view(np.uint16), h16.view(np.uint16))
    else:
        # without a residual h is x itself and the h buffer is not written
        assert np.all(h.view(torch.int16).cpu().numpy() == np.int16(0x7E5A))
    xn64 = oracle.rmsnorm(h16, gamma, eps)
    check(xn, xn64, (2.0 ** -11 + 1e-5) * np.abs(xn64) + 1e-7, f"residual_rmsnorm K={K}")
