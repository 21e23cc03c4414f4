"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/qgemv.h declares, and rejects bad arguments with the
documented status before touching the device.  Plus the byte accounting."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "qgemv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def q():
    import __graft_entry__
    __graft_entry__.build()
    import bit_group_quantized_qgemv_gb300 as mod
    return mod


def test_header_lists_the_boundary():
    names = header_functions()
    for n in ["qgemv_w4g64", "qgemv_w2g64", "rmsnorm_qgemv", "swiglu_qgemv",
              "moe_qgemv_combine", "qgemv_moe_workspace_bytes", "qgemv_strerror",
              "decode_attention_seq1", "qgemv_device_status",
              "qgemv_selftest_wait_timeout", "qgemv_decode_stack", "qgemv_lm_head_argmax",
              "qgemv_argmax_scratch_bytes", "qgemv_moe_router", "qgemv_residual_rmsnorm",
              "qgemv_sample_topk", "qgemv_lm_head_sample", "qgemv_lut4"]:
        assert n in names


def test_library_exports_every_declared_symbol(q):
    raw = ctypes.CDLL(q._binding._build.LIB)
    for name in header_functions():
        assert hasattr(raw, name), name
    assert set(header_functions()) <= set(q.EXPORTED)


def _fake_ptr(v=0x10000):
    return ctypes.c_void_p(v)


def test_null_pointer_status(q):
    L = q.lib
    assert L.qgemv_w4g64(None, _fake_ptr(), _fake_ptr(), _fake_ptr(), _fake_ptr(),
                         1, 4, 64, None, None) == -2
    assert L.qgemv_w2g64(_fake_ptr(), _fake_ptr(), _fake_ptr(), None, _fake_ptr(),
                         1, 4, 64, None, None) == -2
    assert L.rmsnorm_qgemv(_fake_ptr(), _fake_ptr(), _fake_ptr(), _fake_ptr(), None, 1e-5,
                           _fake_ptr(), 4, 64, None) == -2
    assert L.moe_qgemv_combine(*[_fake_ptr()] * 6, 8, 64, 64, None, _fake_ptr(), 4,
                               _fake_ptr(), None, _fake_ptr(), _fake_ptr(), None, None) == -2


@pytest.mark.parametrize("M,N,K", [(0, 4, 64), (9, 4, 64), (1, 0, 64), (1, 4, 0),
                                   (1, 4, 96), (1, 4, 32), (1, -1, 64)])
def test_bad_shape_status(q, M, N, K):
    p = _fake_ptr()
    assert q.lib.qgemv_w4g64(p, p, p, p, p, M, N, K, None, None) == -1
    assert q.lib.qgemv_w2g64(p, p, p, p, p, M, N, K, None, None) == -1
    assert q.lib.qgemv_w8g64(p, p, p, p, p, M, N, K, None, None) == -1


def test_bad_scalar_status(q):
    p = _fake_ptr()
    assert q.lib.rmsnorm_qgemv(p, p, p, p, p, 0.0, p, 4, 64, None) == -1
    assert q.lib.rmsnorm_qgemv(p, p, p, p, p, -1.0, p, 4, 64, None) == -1
    assert q.lib.rmsnorm_qgemv(p, p, p, p, p, float("nan"), p, 4, 64, None) == -1
    assert q.lib.swiglu_qgemv(p, p, p, p, p, p, p, p, 0.0, p, 4, 64, None) == -1
    for top_k in (0, 9):
        assert q.lib.moe_qgemv_combine(p, p, p, p, p, p, 8, 64, 64, p, p, top_k, p, None, p,
                                       p, None, None) == -1
    assert q.lib.moe_qgemv_combine(p, p, p, p, p, p, 0, 64, 64, p, p, 4, p, None, p, p,
                                   None, None) == -1
    assert q.lib.decode_attention_seq1(p, p, 6, 4, 128, None) == -1
    for limit in (0, 1000001):
        assert q.lib.qgemv_selftest_wait_timeout(limit, None) == -1
    for N, K in ((0, 1024), (8, 96), (8, 0)):
        assert q.lib.qgemv_lm_head_argmax(p, p, p, p, p, N, K, p, p, None) == -1


def test_residual_rmsnorm_host_checks(q):
    p, odd = _fake_ptr(), _fake_ptr(0x10001)
    L = q.lib
    assert L.qgemv_residual_rmsnorm(p, None, p, 1e-5, 0, None, p, None) == -1
    assert L.qgemv_residual_rmsnorm(p, None, p, 0.0, 64, None, p, None) == -1
    assert L.qgemv_residual_rmsnorm(None, None, p, 1e-5, 64, None, p, None) == -2
    assert L.qgemv_residual_rmsnorm(p, p, p, 1e-5, 64, None, p, None) == -2   # h needed
    assert L.qgemv_residual_rmsnorm(p, None, p, 1e-5, 64, None, None, None) == -2
    assert L.qgemv_residual_rmsnorm(p, odd, p, 1e-5, 64, p, p, None) == -3


def test_moe_router_host_checks(q):
    p = _fake_ptr()
    L = q.lib
    for E, H, k, sh in ((0, 1024, 4, 0), (512, 96, 4, 0), (512, 1024, 0, 0), (512, 1024, 9, 0),
                        (3, 1024, 4, -1), (512, 1024, 4, 512), (512, 1024, 4, -2)):
        assert L.qgemv_moe_router(p, p, p, p, E, H, k, sh, p, p, p, None) == -1
    for i in (0, 1, 2, 3, 8, 9, 10):
        args = [p, p, p, p, 512, 1024, 4, 0, p, p, p]
        args[i] = None
        assert L.qgemv_moe_router(*args, None) == -2
    two = _fake_ptr(0x10002)
    assert L.qgemv_moe_router(p, p, p, p, 512, 1024, 4, 0, p, two, p, None) == -3


def test_lm_head_argmax_host_checks(q):
    p, two, four = _fake_ptr(), _fake_ptr(0x10002), _fake_ptr(0x10004)
    L = q.lib
    for i in range(7):
        args = [p] * 5 + [8, 64] + [p, p]
        args[[0, 1, 2, 3, 4, 7, 8][i]] = None
        assert L.qgemv_lm_head_argmax(*args, None) == -2
    assert L.qgemv_lm_head_argmax(p, p, p, p, p, 8, 64, four, p, None) == -3   # scratch: 8 B
    assert L.qgemv_lm_head_argmax(p, p, p, p, p, 8, 64, p, two, None) == -3    # token: 4 B
    assert q.argmax_scratch_bytes() == 16


def test_sample_topk_host_checks(q):
    p, two = _fake_ptr(), _fake_ptr(0x10002)
    L = q.lib
    inf, nan = float("inf"), float("nan")
    for N, k, T in ((0, 1, 1.0), (786433, 1, 1.0), (100, 0, 1.0), (100, 101, 1.0),
                    (5000, 1025, 1.0), (100, 5, 0.0), (100, 5, -1.0), (100, 5, inf),
                    (100, 5, nan)):
        assert L.qgemv_sample_topk(p, N, k, T, p, p, None, None, None) == -1
        assert L.qgemv_lm_head_sample(p, p, p, p, p, N, 64, k, T, p, p, None, None, None) == -1
    for i in (0, 4, 5):                      # logits, u, token are required
        args = [p, 100, 5, 1.0, p, p, p, p]
        args[i] = None
        assert L.qgemv_sample_topk(*args, None) == -2
    for i in (0, 1, 2, 3, 4, 9, 10):         # + the weight and x
        args = [p, p, p, p, p, 100, 64, 5, 1.0, p, p, p, p]
        args[i] = None
        assert L.qgemv_lm_head_sample(*args, None) == -2
    assert L.qgemv_lm_head_sample(p, p, p, p, p, 100, 96, 5, 1.0, p, p, None, None, None) == -1
    for i in (4, 5, 6, 7):                   # u, token, topk_idx, topk_prob: 4 B
        args = [p, 100, 5, 1.0, p, p, p, p]
        args[i] = two
        assert L.qgemv_sample_topk(*args, None) == -3
    assert L.qgemv_sample_topk(_fake_ptr(0x10001), 100, 5, 1.0, p, p, None, None, None) == -3


def test_lut4_host_checks(q):
    p, eight = _fake_ptr(), _fake_ptr(0x10008)
    L = q.lib
    for N, K, nl, R in ((0, 64, 1, 1), (8, 96, 8, 1), (8, 32, 8, 1), (8, 16448, 8, 1),
                        (8, 64, 8, 0), (8, 64, 0, 8), (9, 64, 4, 2), (8, 64, 1, 7)):
        assert L.qgemv_lut4(p, p, nl, R, p, p, N, K, None, None) == -1
    for i in (0, 1, 4, 5):                  # codes, lut, x, y are required
        args = [p, p, 8, 1, p, p, 8, 64, None]
        args[i] = None
        assert L.qgemv_lut4(*args, None) == -2
    for i in (0, 1, 4):                     # codes, lut, x: 16 bytes
        args = [p, p, 8, 1, p, p, 8, 64, None]
        args[i] = eight
        assert L.qgemv_lut4(*args, None) == -3
    assert L.qgemv_lut4(p, p, 8, 1, p, _fake_ptr(0x10001), 8, 64, None, None) == -3


def test_noalloc_status_precedence(q):
    """The allocation-free MoE entry point checks NULL pointers, then shapes,
    then the scratch capacity, all before touching the device."""
    p = _fake_ptr()
    f = q.lib.moe_qgemv_combine_noalloc
    big_i = (q.noalloc_max_scratch_bytes() // 4 // 4 + 64) // 64 * 64   # top_k = 4 overflows
    # NULL with an oversized I: ENULL, not ESCRATCH
    assert f(p, p, p, p, p, p, 8, 64, big_i, None, p, 4, p, None, p, None, None) == -2
    assert f(p, p, p, p, p, p, 8, 64, big_i, p, p, 4, p, None, None, None, None) == -2
    # a bad shape with an oversized I: EINVAL, not ESCRATCH
    assert f(p, p, p, p, p, p, 8, 64, big_i + 32, p, p, 4, p, None, p, None, None) == -1
    assert f(p, p, p, p, p, p, 0, 64, big_i, p, p, 4, p, None, p, None, None) == -1
    assert f(p, p, p, p, p, p, 8, 96, 64, p, p, 4, p, None, p, None, None) == -1
    assert f(p, p, p, p, p, p, 8, 64, 64, p, p, 9, p, None, p, None, None) == -1
    # valid shapes beyond the scratch: ESCRATCH
    assert f(p, p, p, p, p, p, 8, 64, big_i, p, p, 4, p, None, p, None, None) == -6


def test_misaligned_status(q):
    p, odd = _fake_ptr(), _fake_ptr(0x10001)
    two = _fake_ptr(0x10002)
    assert q.lib.qgemv_w4g64(two, p, p, p, p, 1, 4, 64, None, None) == -3   # codes need 4 B
    assert q.lib.qgemv_w4g64(p, odd, p, p, p, 1, 4, 64, None, None) == -3
    assert q.lib.qgemv_w4g64(p, p, p, p, p, 1, 4, 64, odd, None) == -3       # residual
    assert q.lib.moe_qgemv_combine(p, p, p, p, p, p, 8, 64, 64, p, p, 4, p, None, p,
                                   two, None, None) == -3                    # workspace


def test_workspace_bytes_and_strerror(q):
    assert q.moe_workspace_bytes(4, 1024) == 4 * 1024 * 4
    assert q.moe_workspace_bytes(0, 1024) == 0
    for s in (0, -1, -2, -3, -4, -5, -6):
        assert q.strerror(s) and q.strerror(s) != "unknown status"
    assert q.strerror(-99) == "unknown status"


def test_no_device_reports_edevice(q):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    p = _fake_ptr()
    assert q.lib.qgemv_w4g64(p, p, p, p, p, 1, 4, 64, None, None) == -5


def test_expert_byte_accounting_pins_group64_fp16():
    """The hada.io page (topic 27758, "SSD Expert Streaming") gives about
    6.75 MB per expert for hidden 4096 and 4-bit experts: 4096 x 2048 + 1024 x
    4096 weights at 0.5625 B/weight is exactly 6.75 MiB."""
    from bit_group_quantized_qgemv_gb300 import accounting as acc
    assert acc.expert_bytes(4096, 1024, 4) == 7077888
    assert acc.expert_bytes(4096, 1024, 4) == int(6.75 * 2**20)
    # 8B layer total from the matvec shapes
    assert sum(acc.weight_bytes(n, k, 4) for n, k in
               [(6144, 4096), (4096, 4096), (2 * 14336, 4096), (4096, 14336)]) == 122683392


def _plan(q, bits, M, N, K, sms=152, aligned16=True):
    return q.plan_gemv(bits, M, N, K, sms, aligned16)


def test_gemv_routing_by_batch_and_shape(q):
    """qgemv_plan_gemv (host-only) pins the routing of qgemv_w4g64 / w2g64 /
    w8g64: M = 1 streams; M >= 3 and short M = 2 ops take the tensor cores;
    long M = 2 ops the CUDA-core small-batch kernel; 8-bit batches and
    misaligned operands the generic kernel."""
    assert _plan(q, 4, 1, 4096, 4096)["path"] == "stream"
    assert _plan(q, 4, 1, 4096, 4096, aligned16=False)["path"] == "generic"
    assert _plan(q, 4, 4, 4096, 4096, aligned16=False)["path"] == "generic"
    # M = 2: tensor cores only for K <= 4096 and at most 128 KB of weights per SM
    assert _plan(q, 4, 2, 4096, 4096)["path"] == "mma"
    assert _plan(q, 4, 2, 1024, 1024)["path"] == "mma"
    assert _plan(q, 4, 2, 14336, 4096)["path"] == "batch"   # 217 KB per SM
    assert _plan(q, 4, 2, 4096, 14336)["path"] == "batch"
    assert _plan(q, 2, 2, 4096, 4096)["path"] == "mma"
    for M in (3, 4, 5, 8):
        for K in (4096, 14336):
            p = _plan(q, 4, M, 4096, K)
            assert p["path"] == "mma" and p["passes"] == 1, (M, K, p)
            assert p["m_pad"] == (4 if M <= 4 else 8)
    assert _plan(q, 8, 4, 4096, 4096)["path"] == "generic"
    # K not a multiple of 512 (tensor cores) nor of 1024 (CUDA-core small batch)
    assert _plan(q, 4, 3, 300, 1088)["path"] == "generic"


def test_gemv_tensor_core_cluster_and_stage_plan(q):
    """The tensor-core plan: K split four ways when a whole row's staged
    activations exceed 96 KB, chunks of at most 4096 k (the longest that
    divides the CTA's k range), a ring of at least two stages, all within the
    227 KB of shared memory a block may take."""
    cases = {  # (bits, M, K): (cluster, chunk_k)
        (4, 4, 4096): (1, 4096), (4, 8, 4096): (1, 4096), (4, 4, 8192): (1, 4096),
        (4, 8, 8192): (4, 2048), (4, 3, 14336): (4, 3584), (4, 8, 14336): (4, 3584),
        (4, 4, 16384): (4, 4096), (4, 8, 32768): (4, 4096), (2, 8, 14336): (4, 3584),
        (4, 4, 1024): (1, 1024),
    }
    for (bits, M, K), (cl, kc) in cases.items():
        p = _plan(q, bits, M, 4096, K)
        assert p["path"] == "mma", (bits, M, K, p)
        assert (p["cluster"], p["chunk_k"]) == (cl, kc), (bits, M, K, p)
        assert (K // cl) % kc == 0 and kc % 512 == 0
        assert 2 <= p["stages"] <= 16
        assert p["smem_bytes"] <= 227 * 1024
        # staged activations per CTA (fragments + group sums) stay within 132 KB
        mp = p["m_pad"]
        assert 2 * mp * (K // cl) + (K // cl) // 2 <= 132 * 1024
    # too long to hold even split four ways, and past the CUDA-core small
    # batch's K <= 16384: the generic kernel
    assert _plan(q, 4, 8, 4096, 65536)["path"] == "generic"


def test_gemv_plan_arguments(q):
    out = q._binding.GemvPlan()
    L = q.lib
    assert L.qgemv_plan_gemv(4, 4, 4096, 4096, 152, 1, None) == -2
    for args in [(3, 4, 4096, 4096, 152), (4, 0, 4096, 4096, 152), (4, 9, 4096, 4096, 152),
                 (4, 4, 0, 4096, 152), (4, 4, 4096, 100, 152), (4, 4, 4096, 4096, 0)]:
        assert L.qgemv_plan_gemv(*args, 1, ctypes.byref(out)) == -1, args
    assert L.qgemv_plan_gemv(4, 4, 4096, 4096, 152, 1, ctypes.byref(out)) == 0
