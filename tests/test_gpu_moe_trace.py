"""MoE index handling, bit-exactly: what each CTA of the two MoE kernels read
and used (moe_qgemv_combine_traced) against the routing it was given.

The routing decisions (hada.io topic 27758, "Architecture du modele": K = 4
of 512 experts, one shared) must be honoured exactly: every launched CTA of
both phases must have read the caller's expert_idx and expert_w bit for bit,
used exactly the in-range indices, and skipped (expert -1, weight bits 0)
the out-of-range ones; a repeated index is used twice.  The output is also
checked against the oracle within the MoE tolerance, so the traced call is
the same computation as the plain one.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from qhelpers import check, dev16, dev_weight

pytestmark = pytest.mark.gpu

q = pytest.importorskip("bit_group_quantized_qgemv_gb300")


def expected_records(idx, wt, E):
    idx = np.asarray(idx, np.int32)
    wbits = np.asarray(wt, np.float32).view(np.uint32).astype(np.int64)
    ok = (idx >= 0) & (idx < E)
    rec = np.stack([idx.astype(np.int64), wbits, np.where(ok, idx, -1).astype(np.int64),
                    np.where(ok, wbits, 0)], axis=1)
    return rec.astype(np.uint32)


def run_traced(gu, dn, idx, wt, x, r, trace_ctas=512):
    E = gu.codes.shape[0]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx_d = torch.as_tensor(np.asarray(idx, np.int32)).cuda() if not torch.is_tensor(idx) else idx
    wt_d = torch.as_tensor(np.asarray(wt, np.float32)).cuda() if not torch.is_tensor(wt) else wt
    y, trace, launched = q.moe_qgemv_combine_traced(dev_weight(gu), dev_weight(dn), idx_d, wt_d,
                                                    dev16(x), dev16(r), trace_ctas=trace_ctas,
                                                    err_flag=err)
    torch.cuda.synchronize()
    tr = trace.cpu().numpy().view(np.uint32)
    want = expected_records(idx_d.cpu().numpy(), wt_d.cpu().numpy(), E)
    for p in range(2):
        n = min(launched[p], trace_ctas)
        assert launched[p] >= 1
        got = tr[p, :n]
        assert np.array_equal(got, np.broadcast_to(want, got.shape)), \
            f"phase {p}: a CTA consumed other (idx, wt) bits than given"
        # records of CTAs that were never launched stay untouched
        assert np.all(tr[p, n:] == 0xFFFFFFFF)
    ok = np.all((idx_d.cpu().numpy() >= 0) & (idx_d.cpu().numpy() < E))
    assert int(err.item()) == (0 if ok else 1)
    y64, _, tol, err_o = oracle.moe_qgemv_combine((gu.codes, gu.scales, gu.biases),
                                                  (dn.codes, dn.scales, dn.biases),
                                                  idx_d.cpu().numpy(), wt_d.cpu().numpy(), x, r)
    check(y, y64, tol, "traced MoE output")
    assert err_o == int(err.item())
    return launched


@pytest.mark.parametrize("H,I,path", [(4096, 1024, "stream"), (1024, 1024, "stream"),
                                      (320, 192, "generic")])
@pytest.mark.parametrize("case", ["valid", "bad_and_repeated", "weight_bits"])
def test_moe_trace_records_the_given_routing(H, I, path, case):
    E = 12
    gu, dn = synth.moe_experts(310, H, E, hidden=H, inter=I)
    x = synth.activation(synth.rng(310, H, 10), H)
    r = synth.activation(synth.rng(310, H, 11), H)
    if case == "valid":
        idx, wt = [0, 7, 3, 11], [0.4, 0.3, 0.2, 0.1]
    elif case == "bad_and_repeated":
        idx, wt = [5, -1, 5, 12, 1 << 30, 2], [0.25, 0.5, 0.125, 0.75, 0.3, 0.1]
    else:   # signed zero, a subnormal and a negative weight: compared as bits
        idx, wt = [4, 9, 1], [-0.0, np.float32(1e-41), -0.75]
    trace_ctas = 4096 if path == "generic" else 512
    launched = run_traced(gu, dn, idx, wt, x, r, trace_ctas)
    if path == "stream":
        assert max(launched) <= 152 * 2
    else:
        assert launched[0] == (len(idx) * I + 7) // 8


def test_moe_trace_of_router_output():
    """Indices and weights produced on the device by qgemv_moe_router are
    consumed by both phases exactly as the router wrote them."""
    E, H, I = 16, 1024, 1024
    gu, dn = synth.moe_experts(311, 0, E, hidden=H, inter=I)
    wr = synth.quant_weight(synth.rng(311, 0, synth.TID["router"]), E, H, 4)
    x = synth.activation(synth.rng(311, 0, 10), H)
    idx, wt, _ = q.moe_router(dev_weight(wr), dev16(x), top_k=4, shared=0)
    run_traced(gu, dn, idx, wt, x, x)
    assert q.device_status() == 0
