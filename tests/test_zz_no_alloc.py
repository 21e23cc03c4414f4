"""The allocation-free MoE entry point against the regular one.

moe_qgemv_combine_noalloc serves callers that cannot allocate device memory
(a plugin whose host application owns every allocation, or a loop that may
not allocate once running): it replaces the caller's workspace with the
library's fixed device scratch array.  These tests call it through the C ABI
and check that, on two calls in a row, its output matches moe_qgemv_combine
with a caller workspace, within the tolerance the MoE parity tests use.
The file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from qhelpers import check, dev16, dev_weight

pytestmark = pytest.mark.gpu

q = pytest.importorskip("bit_group_quantized_qgemv_gb300")


@pytest.mark.parametrize("E,H,I", [(8, 1024, 1024), (6, 256, 128)])
def test_noalloc_matches_workspace_entry_point_twice(E, H, I):
    gu, dn = synth.moe_experts(301, E, E, hidden=H, inter=I)
    gud, dnd = dev_weight(gu), dev_weight(dn)
    g = np.random.default_rng(E + H)
    for call in range(2):
        idx = g.choice(E, size=4, replace=False).astype(np.int32)
        wt = g.dirichlet(np.ones(4)).astype(np.float32)
        x = synth.activation(synth.rng(301, call, 10, H), H)
        r = synth.activation(synth.rng(301, call, 11, H), H)
        idx_d = torch.from_numpy(idx).cuda()
        wt_d = torch.from_numpy(wt).cuda()
        err_a = torch.zeros(1, dtype=torch.int32, device="cuda")
        err_b = torch.zeros(1, dtype=torch.int32, device="cuda")
        y_ref = q.moe_qgemv_combine(gud, dnd, idx_d, wt_d, dev16(x), dev16(r), err_flag=err_a)
        y_na = q.moe_qgemv_combine_noalloc(gud, dnd, idx_d, wt_d, dev16(x), dev16(r),
                                           err_flag=err_b)
        torch.cuda.synchronize()
        _, _, tol, _ = oracle.moe_qgemv_combine((gu.codes, gu.scales, gu.biases),
                                                (dn.codes, dn.scales, dn.biases), idx, wt, x, r)
        check(y_na, y_ref.double().cpu().numpy(), tol, f"noalloc call {call}")
        assert int(err_a.item()) == int(err_b.item()) == 0


def test_noalloc_bad_index_flag_and_size_limit():
    E, H, I = 5, 1024, 1024
    gu, dn = synth.moe_experts(302, 0, E, hidden=H, inter=I)
    gud, dnd = dev_weight(gu), dev_weight(dn)
    x = synth.activation(synth.rng(302, 0, 10), H)
    idx = torch.tensor([0, 7, 2, -1], dtype=torch.int32, device="cuda")
    wt = torch.tensor([0.4, 0.3, 0.2, 0.1], dtype=torch.float32, device="cuda")
    err_a = torch.zeros(1, dtype=torch.int32, device="cuda")
    err_b = torch.zeros(1, dtype=torch.int32, device="cuda")
    y_ref = q.moe_qgemv_combine(gud, dnd, idx, wt, dev16(x), dev16(x), err_flag=err_a)
    y_na = q.moe_qgemv_combine_noalloc(gud, dnd, idx, wt, dev16(x), dev16(x), err_flag=err_b)
    torch.cuda.synchronize()
    assert int(err_a.item()) == 1 and int(err_b.item()) == 1
    _, _, tol, _ = oracle.moe_qgemv_combine((gu.codes, gu.scales, gu.biases),
                                            (dn.codes, dn.scales, dn.biases),
                                            idx.cpu().numpy(), wt.cpu().numpy(), x, x)
    check(y_na, y_ref.double().cpu().numpy(), tol, "noalloc with bad indices")
    # top_k * I beyond the scratch array is refused before any launch
    cap = q.noalloc_max_scratch_bytes() // 4
    too_big_i = (cap // 4 + 64) // 64 * 64
    st = q.lib.moe_qgemv_combine_noalloc(gud[0].data_ptr(), gud[1].data_ptr(), gud[2].data_ptr(),
                                         dnd[0].data_ptr(), dnd[1].data_ptr(), dnd[2].data_ptr(),
                                         E, H, too_big_i, idx.data_ptr(), wt.data_ptr(), 4,
                                         dev16(x).data_ptr(), None, dev16(x).data_ptr(), None,
                                         None)
    assert st == -6
    assert q.device_status() == 0
