"""qgemv_moe_router: MoE routing on the GPU.

The router logits must match the fp64 oracle within the matvec tolerance;
the chosen experts are decided by floating point on those fp16 logits, so
the oracle's routing (oracle.moe_route) is run on the GPU's own logits and
must choose the same experts, in the same order, bit-exactly; the weights
(fp32 softmax on the GPU) must match its fp64 softmax.  End to end, the
device indices and weights feed moe_qgemv_combine.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from qhelpers import check, dev16, dev_weight, plain_tol

pytestmark = pytest.mark.gpu

q = pytest.importorskip("bit_group_quantized_qgemv_gb300")


def route_and_check(w, x, top_k, shared, what):
    idx, wt, logits = q.moe_router(dev_weight(w), dev16(x), top_k=top_k, shared=shared)
    y64, _, bound = oracle.qgemv(4, w.codes, w.scales, w.biases, x)
    check(logits, y64, plain_tol(bound), what + " logits")
    want_idx, want_wt = oracle.moe_route(logits.cpu().numpy(), top_k, shared)
    assert idx.cpu().numpy().tolist() == want_idx.tolist(), what
    assert np.allclose(wt.cpu().numpy().astype(np.float64), want_wt, rtol=2e-6, atol=1e-7), what
    return idx, wt


@pytest.mark.parametrize("E,H,top_k,shared", [(512, 4096, 4, 0), (64, 1024, 8, -1),
                                              (33, 960, 1, 5), (512, 1024, 2, 511)])
def test_router_parity(E, H, top_k, shared):
    w = synth.quant_weight(synth.rng(3, E, synth.TID["router"]), E, H, 4)
    x = synth.activation(synth.rng(3, E, synth.TID["x"]), H)
    route_and_check(w, x, top_k, shared, f"router E={E} H={H} k={top_k} shared={shared}")


def test_router_ties_pick_lower_indices():
    E, H = 40, 1024
    w = synth.quant_weight(synth.rng(3, 1, synth.TID["router"]), E, H, 4)
    w.codes[:] = 0
    w.scales[:] = 1.0
    w.biases[:] = 0.0
    w.biases[[9, 17, 30], 0] = 0.5          # three routed experts tie above the rest
    x = np.zeros(H, np.float16)
    x[:64] = 1.0
    idx, wt = route_and_check(w, x, 4, 0, "router ties")
    assert idx.cpu().numpy().tolist() == [0, 9, 17, 30]


def test_router_feeds_moe_combine():
    E, H, I, top_k = 8, 1024, 1024, 4
    wr = synth.quant_weight(synth.rng(3, 2, synth.TID["router"]), E, H, 4)
    gu, dn = synth.moe_experts(3, 2, E, hidden=H, inter=I)
    x = synth.activation(synth.rng(3, 2, synth.TID["x"]), H)
    idx, wt = route_and_check(wr, x, top_k, 0, "router e2e")
    y = q.moe_qgemv_combine(dev_weight(gu), dev_weight(dn), idx, wt, dev16(x), dev16(x))
    y64, _, tol, err = oracle.moe_qgemv_combine((gu.codes, gu.scales, gu.biases),
                                                (dn.codes, dn.scales, dn.biases),
                                                idx.cpu().numpy(), wt.cpu().numpy(), x, x)
    assert err == 0
    check(y, y64, tol, "routed MoE token")
    assert q.device_status() == 0
