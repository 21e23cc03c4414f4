"""GB300-native dequant-fused quantized GEMV (4/2-bit, group 64, planar).

The kernels live in ``libqgemv.so`` (CUDA C++ for sm_103a, built in-tree by
``bit_group_quantized_qgemv_gb300.build``); ``include/qgemv.h`` declares its C
ABI.  This package is the thin Python binding over that ABI.
"""
from ._binding import (  # noqa: F401
    EXPORTED,
    QgemvError,
    StackLayer,
    StackShape,
    decode_attention_seq1,
    decode_stack,
    decode_stack_workspace_bytes,
    stack_layers,
    stack_shape,
    device_status,
    last_cuda_error,
    lib,
    lm_head_argmax,
    lm_head_sample,
    argmax_scratch_bytes,
    plan_gemv,
    moe_qgemv_combine,
    moe_qgemv_combine_traced,
    moe_router,
    moe_qgemv_combine_noalloc,
    noalloc_max_scratch_bytes,
    moe_workspace_bytes,
    qgemv_w2g64,
    qgemv_w4g64,
    qgemv_w8g64,
    qgemv_lut4,
    residual_rmsnorm,
    rmsnorm_qgemv,
    sample_topk,
    selftest_wait_timeout,
    strerror,
    swiglu_qgemv,
    version,
)
