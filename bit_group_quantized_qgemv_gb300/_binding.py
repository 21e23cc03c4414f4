"""ctypes binding of libqgemv.so: argument marshalling only.

Each function takes torch tensors that already live on the GPU, passes their
device pointers and shapes to the C ABI of the same name (include/qgemv.h)
on the current torch stream, and raises ``QgemvError`` on a non-zero status.
Every step of the computation runs in the library's CUDA kernels; there is
no fallback: if the library cannot be loaded, importing fails loudly.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float

_SIGS = {
    "qgemv_w4g64": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "qgemv_w2g64": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "qgemv_w8g64": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "rmsnorm_qgemv": (_I, [_P, _P, _P, _P, _P, _F, _P, _I, _I, _P]),
    "swiglu_qgemv": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _F, _P, _I, _I, _P]),
    "moe_qgemv_combine": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _I, _P, _P,
                               _P, _P, _P, _P]),
    "moe_qgemv_combine_traced": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _I, _P, _P,
                                      _P, _P, _P, _P, _I, ctypes.POINTER(_I), _P]),
    "qgemv_moe_workspace_bytes": (ctypes.c_size_t, [_I, _I]),
    "moe_qgemv_combine_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _I, _P, _P,
                                       _P, _P, _P]),
    "qgemv_noalloc_max_scratch": (ctypes.c_size_t, []),
    "decode_attention_seq1": (_I, [_P, _P, _I, _I, _I, _P]),
    "qgemv_decode_stack_workspace_bytes": (ctypes.c_size_t, [_P]),
    "qgemv_decode_stack": (_I, [_P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "qgemv_strerror": (ctypes.c_char_p, [_I]),
    "qgemv_last_cuda_error": (_I, []),
    "qgemv_device_status": (_I, [ctypes.POINTER(ctypes.c_uint)]),
    "qgemv_version": (_I, []),
    "qgemv_selftest_wait_timeout": (_I, [ctypes.c_uint, ctypes.c_void_p]),
    "qgemv_lm_head_argmax": (_I, [_P, _P, _P, _P, _P, _I, _I, _P, _P, _P]),
    "qgemv_argmax_scratch_bytes": (ctypes.c_size_t, []),
    "qgemv_moe_router": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P]),
    "qgemv_residual_rmsnorm": (_I, [_P, _P, _P, _F, _I, _P, _P, _P]),
    "qgemv_sample_topk": (_I, [_P, _I, _I, _F, _P, _P, _P, _P, _P]),
    "qgemv_lut4": (_I, [_P, _P, _I, _I, _P, _P, _I, _I, _P, _P]),
    "qgemv_lm_head_sample": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _F, _P, _P, _P, _P, _P]),
    "qgemv_plan_gemv": (_I, [_I, _I, _I, _I, _I, _I, _P]),
}


class GemvPlan(ctypes.Structure):
    """qgemv_gemv_plan (include/qgemv.h)."""
    _fields_ = [(n, ctypes.c_int) for n in
                ("path", "passes", "m_pad", "cluster", "chunk_k", "stages", "smem_bytes")]


#: QGEMV_PATH_* of include/qgemv.h, by value.
GEMV_PATHS = ("generic", "stream", "mma", "mma_passes", "batch", "batch_passes")

#: Names the C header declares (the binding exposes each one).
EXPORTED = tuple(_SIGS)


class QgemvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({strerror(status)})")


def _load():
    path = os.environ.get("QGEMV_LIB") or _build.LIB
    if not os.path.exists(path):
        raise ImportError(
            f"libqgemv.so not found at {path}; build it first with "
            "`python -m bit_group_quantized_qgemv_gb300.build` (needs nvcc)")
    handle = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    return handle


lib = _load()


def strerror(status: int) -> str:
    return lib.qgemv_strerror(int(status)).decode()


def _check(status: int, what: str):
    if status != 0:
        raise QgemvError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _cuda(t, dtypes, name):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


_CODES = (torch.int32, getattr(torch, "uint32", torch.int32))
_F16 = (torch.float16,)


def _weight(w, name):
    codes, scales, biases = w
    return (_cuda(codes, _CODES, name + ".codes"), _cuda(scales, _F16, name + ".scales"),
            _cuda(biases, _F16, name + ".biases"))


def _plain(fn, bits, w, x, y, residual, stream):
    codes, scales, biases = _weight(w, "w")
    x = _cuda(x, _F16, "x")
    N = codes.shape[-2]
    K = codes.shape[-1] * 32 // bits
    M = 1 if x.dim() == 1 else x.shape[0]
    if y is None:
        y = torch.empty((N,) if x.dim() == 1 else (M, N), dtype=torch.float16, device=x.device)
    _cuda(y, _F16, "y")
    _cuda(residual, _F16, "residual")
    st = fn(_ptr(codes), _ptr(scales), _ptr(biases), _ptr(x), _ptr(y), M, N, K,
            _ptr(residual), _stream(stream))
    _check(st, fn.__name__)
    return y


def qgemv_w4g64(w, x, y=None, residual=None, stream=None):
    """y = W x (+ residual) for a 4-bit g64 weight w = (codes, scales, biases)."""
    return _plain(lib.qgemv_w4g64, 4, w, x, y, residual, stream)


def qgemv_w2g64(w, x, y=None, residual=None, stream=None):
    """y = W x (+ residual) for a 2-bit g64 weight w = (codes, scales, biases)."""
    return _plain(lib.qgemv_w2g64, 2, w, x, y, residual, stream)


def residual_rmsnorm(x, gamma, residual=None, eps=1e-5, h=None, xn=None, stream=None):
    """qgemv_residual_rmsnorm: h = x + residual (fp16; x itself when residual
    is None), xn = RMSNorm(h) * gamma (fp16).  Returns (h, xn)."""
    x = _cuda(x, _F16, "x")
    gamma = _cuda(gamma, _F16, "gamma")
    _cuda(residual, _F16, "residual")
    K = x.shape[-1]
    if residual is not None and h is None:
        h = torch.empty(K, dtype=torch.float16, device=x.device)
    if xn is None:
        xn = torch.empty(K, dtype=torch.float16, device=x.device)
    st = lib.qgemv_residual_rmsnorm(_ptr(x), _ptr(residual), _ptr(gamma), float(eps), K, _ptr(h),
                                    _ptr(xn), _stream(stream))
    _check(st, "qgemv_residual_rmsnorm")
    return (h if residual is not None else x), xn


def moe_router(w, x, top_k=4, shared=0, logits=None, idx=None, wt=None, stream=None):
    """MoE routing on the GPU (qgemv_moe_router): logits = Wr x (4-bit g64),
    idx = shared expert + top routed experts, wt = softmax of their logits.
    Returns (idx int32 [top_k], wt float32 [top_k], logits fp16 [E])."""
    codes, scales, biases = _weight(w, "w")
    x = _cuda(x, _F16, "x")
    E = codes.shape[-2]
    H = codes.shape[-1] * 8
    if logits is None:
        logits = torch.empty(E, dtype=torch.float16, device=x.device)
    if idx is None:
        idx = torch.empty(top_k, dtype=torch.int32, device=x.device)
    if wt is None:
        wt = torch.empty(top_k, dtype=torch.float32, device=x.device)
    _cuda(logits, _F16, "logits")
    _cuda(idx, (torch.int32,), "idx")
    _cuda(wt, (torch.float32,), "wt")
    st = lib.qgemv_moe_router(_ptr(codes), _ptr(scales), _ptr(biases), _ptr(x), E, H, int(top_k),
                              int(shared), _ptr(logits), _ptr(idx), _ptr(wt), _stream(stream))
    _check(st, "qgemv_moe_router")
    return idx, wt, logits


def argmax_scratch_bytes() -> int:
    return int(lib.qgemv_argmax_scratch_bytes())


def plan_gemv(bits, M, N, K, sms, aligned16=True):
    """The kernels qgemv_w4g64 / w2g64 / w8g64 take for a shape
    (qgemv_plan_gemv; host-only): a dict with the path name and its plan."""
    out = GemvPlan()
    _check(lib.qgemv_plan_gemv(int(bits), int(M), int(N), int(K), int(sms), int(bool(aligned16)),
                               ctypes.byref(out)), "qgemv_plan_gemv")
    d = {n: getattr(out, n) for n, _ in GemvPlan._fields_}
    d["path"] = GEMV_PATHS[d["path"]]
    return d


def lm_head_argmax(w, x, logits=None, scratch=None, token=None, stream=None):
    """Greedy lm_head (qgemv_lm_head_argmax): logits = W x (4-bit g64) and
    token = the lowest index of the largest logit, both on the device.
    `scratch` (uint8, argmax_scratch_bytes(), zero before first use; left
    zero) may be kept across calls; a fresh zeroed one is made if None.
    Returns (token int32 [1], logits fp16 [N])."""
    codes, scales, biases = _weight(w, "w")
    x = _cuda(x, _F16, "x")
    N = codes.shape[-2]
    K = codes.shape[-1] * 8  # 4-bit: 8 codes per 32-bit word
    if logits is None:
        logits = torch.empty(N, dtype=torch.float16, device=x.device)
    if scratch is None:
        scratch = torch.zeros(argmax_scratch_bytes(), dtype=torch.uint8, device=x.device)
    if token is None:
        token = torch.empty(1, dtype=torch.int32, device=x.device)
    _cuda(logits, _F16, "logits")
    _cuda(token, (torch.int32,), "token")
    st = lib.qgemv_lm_head_argmax(_ptr(codes), _ptr(scales), _ptr(biases), _ptr(x), _ptr(logits),
                                  N, K, _ptr(scratch), _ptr(token), _stream(stream))
    _check(st, "qgemv_lm_head_argmax")
    return token, logits


def _sample_outputs(device, top_k, u, token, want_topk, topk_idx, topk_prob):
    u = _cuda(u, (torch.float32,), "u")
    if token is None:
        token = torch.empty(1, dtype=torch.int32, device=device)
    _cuda(token, (torch.int32,), "token")
    if want_topk:
        if topk_idx is None:
            topk_idx = torch.empty(top_k, dtype=torch.int32, device=device)
        if topk_prob is None:
            topk_prob = torch.empty(top_k, dtype=torch.float32, device=device)
    _cuda(topk_idx, (torch.int32,), "topk_idx")
    _cuda(topk_prob, (torch.float32,), "topk_prob")
    return u, token, topk_idx, topk_prob


def sample_topk(logits, top_k, temperature, u, token=None, want_topk=False, topk_idx=None,
                topk_prob=None, stream=None):
    """Top-k sampling on the device (qgemv_sample_topk) from fp16 logits [N];
    u: fp32 [1] on the device (the caller's random number in [0, 1)).
    Returns (token int32 [1], topk_idx int32 [top_k] or None, topk_prob fp32
    [top_k] or None); the candidate outputs are made when want_topk."""
    logits = _cuda(logits, _F16, "logits")
    u, token, topk_idx, topk_prob = _sample_outputs(logits.device, top_k, u, token, want_topk,
                                                    topk_idx, topk_prob)
    st = lib.qgemv_sample_topk(_ptr(logits), logits.numel(), int(top_k), float(temperature),
                               _ptr(u), _ptr(token), _ptr(topk_idx), _ptr(topk_prob),
                               _stream(stream))
    _check(st, "qgemv_sample_topk")
    return token, topk_idx, topk_prob


def lm_head_sample(w, x, top_k, temperature, u, logits=None, token=None, want_topk=False,
                   topk_idx=None, topk_prob=None, stream=None):
    """lm_head matvec (4-bit g64) then top-k sampling (qgemv_lm_head_sample).
    Returns (token, logits, topk_idx, topk_prob) as sample_topk."""
    codes, scales, biases = _weight(w, "w")
    x = _cuda(x, _F16, "x")
    N = codes.shape[-2]
    K = codes.shape[-1] * 8  # 4-bit: 8 codes per 32-bit word
    if logits is None:
        logits = torch.empty(N, dtype=torch.float16, device=x.device)
    _cuda(logits, _F16, "logits")
    u, token, topk_idx, topk_prob = _sample_outputs(x.device, top_k, u, token, want_topk,
                                                    topk_idx, topk_prob)
    st = lib.qgemv_lm_head_sample(_ptr(codes), _ptr(scales), _ptr(biases), _ptr(x),
                                  _ptr(logits), N, K, int(top_k), float(temperature), _ptr(u),
                                  _ptr(token), _ptr(topk_idx), _ptr(topk_prob), _stream(stream))
    _check(st, "qgemv_lm_head_sample")
    return token, logits, topk_idx, topk_prob


def qgemv_lut4(codes, lut, x, rows_per_lut=1, y=None, residual=None, stream=None):
    """LUT / palettised 4-bit GEMV (qgemv_lut4): y[n] = sum_k
    lut[n // rows_per_lut][q[n][k]] x[k] (+ residual[n]).  codes: int32/uint32
    view [N][K/8] on the device; lut: fp16 [n_luts][16]; x: fp16 [K]."""
    codes = _cuda(codes, _CODES, "codes")
    lut = _cuda(lut, _F16, "lut")
    x = _cuda(x, _F16, "x")
    if lut.dim() != 2 or lut.shape[1] != 16:
        raise ValueError("lut must be fp16 [n_luts][16]")
    N, K = codes.shape[-2], codes.shape[-1] * 8
    if y is None:
        y = torch.empty(N, dtype=torch.float16, device=x.device)
    _cuda(y, _F16, "y")
    residual = _cuda(residual, _F16, "residual")
    st = lib.qgemv_lut4(_ptr(codes), _ptr(lut), lut.shape[0], int(rows_per_lut), _ptr(x), _ptr(y),
                        N, K, _ptr(residual), _stream(stream))
    _check(st, "qgemv_lut4")
    return y


def qgemv_w8g64(w, x, y=None, residual=None, stream=None):
    """y = W x (+ residual) for an 8-bit g64 weight w = (codes, scales, biases)."""
    return _plain(lib.qgemv_w8g64, 8, w, x, y, residual, stream)


def rmsnorm_qgemv(w, x, norm_weight, eps=1e-5, y=None, stream=None):
    codes, scales, biases = _weight(w, "w")
    x = _cuda(x, _F16, "x")
    _cuda(norm_weight, _F16, "norm_weight")
    N, K = codes.shape[-2], codes.shape[-1] * 8
    if y is None:
        y = torch.empty(N, dtype=torch.float16, device=x.device)
    st = lib.rmsnorm_qgemv(_ptr(codes), _ptr(scales), _ptr(biases), _ptr(x), _ptr(norm_weight),
                           float(eps), _ptr(y), N, K, _stream(stream))
    _check(st, "rmsnorm_qgemv")
    return y


def swiglu_qgemv(gate, up, x, norm_weight=None, eps=1e-5, h=None, stream=None):
    gc, gs, gb = _weight(gate, "gate")
    uc, us, ub = _weight(up, "up")
    x = _cuda(x, _F16, "x")
    _cuda(norm_weight, _F16, "norm_weight")
    I, K = gc.shape[-2], gc.shape[-1] * 8
    if h is None:
        h = torch.empty(I, dtype=torch.float16, device=x.device)
    st = lib.swiglu_qgemv(_ptr(gc), _ptr(gs), _ptr(gb), _ptr(uc), _ptr(us), _ptr(ub), _ptr(x),
                          _ptr(norm_weight), float(eps), _ptr(h), I, K, _stream(stream))
    _check(st, "swiglu_qgemv")
    return h


def moe_workspace_bytes(top_k: int, inter: int) -> int:
    return int(lib.qgemv_moe_workspace_bytes(int(top_k), int(inter)))


def moe_qgemv_combine(gu, dn, expert_idx, expert_w, x, residual=None, y=None, workspace=None,
                      err_flag=None, stream=None):
    """gu = (codes [E][2I][H/8], scales, biases), dn = (codes [E][H][I/8], ...)."""
    gc, gs, gb = _weight(gu, "gu")
    dc, ds, db = _weight(dn, "dn")
    _cuda(expert_idx, (torch.int32,), "expert_idx")
    _cuda(expert_w, (torch.float32,), "expert_w")
    x = _cuda(x, _F16, "x")
    _cuda(residual, _F16, "residual")
    E, I2, H8 = gc.shape
    I, H = I2 // 2, H8 * 8
    top_k = expert_idx.numel()
    if y is None:
        y = torch.empty(H, dtype=torch.float16, device=x.device)
    if workspace is None:
        workspace = torch.empty(top_k * I, dtype=torch.float32, device=x.device)
    _cuda(workspace, (torch.float32,), "workspace")
    _cuda(err_flag, (torch.int32,), "err_flag")
    st = lib.moe_qgemv_combine(_ptr(gc), _ptr(gs), _ptr(gb), _ptr(dc), _ptr(ds), _ptr(db), E, H,
                               I, _ptr(expert_idx), _ptr(expert_w), top_k, _ptr(x),
                               _ptr(residual), _ptr(y), _ptr(workspace), _ptr(err_flag),
                               _stream(stream))
    _check(st, "moe_qgemv_combine")
    return y


def moe_qgemv_combine_traced(gu, dn, expert_idx, expert_w, x, residual=None, trace_ctas=256,
                             err_flag=None, stream=None):
    """moe_qgemv_combine that also returns what each CTA of its two kernels
    read and used: (y, trace uint32 [2][trace_ctas][top_k][4], ctas launched
    per phase).  Trace records: idx read, weight bits read, expert used (-1:
    skipped), weight bits used (0: skipped)."""
    gc, gs, gb = _weight(gu, "gu")
    dc, ds, db = _weight(dn, "dn")
    _cuda(expert_idx, (torch.int32,), "expert_idx")
    _cuda(expert_w, (torch.float32,), "expert_w")
    x = _cuda(x, _F16, "x")
    _cuda(residual, _F16, "residual")
    E, I2, H8 = gc.shape
    I, H = I2 // 2, H8 * 8
    top_k = expert_idx.numel()
    y = torch.empty(H, dtype=torch.float16, device=x.device)
    workspace = torch.empty(top_k * I, dtype=torch.float32, device=x.device)
    trace = torch.full((2, trace_ctas, top_k, 4), -1, dtype=torch.int32, device=x.device)
    _cuda(err_flag, (torch.int32,), "err_flag")
    launched = (_I * 2)(0, 0)
    st = lib.moe_qgemv_combine_traced(_ptr(gc), _ptr(gs), _ptr(gb), _ptr(dc), _ptr(ds), _ptr(db),
                                      E, H, I, _ptr(expert_idx), _ptr(expert_w), top_k, _ptr(x),
                                      _ptr(residual), _ptr(y), _ptr(workspace), _ptr(err_flag),
                                      _ptr(trace), trace_ctas, launched, _stream(stream))
    _check(st, "moe_qgemv_combine_traced")
    return y, trace, (int(launched[0]), int(launched[1]))


def moe_qgemv_combine_noalloc(gu, dn, expert_idx, expert_w, x, residual=None, y=None,
                              err_flag=None, stream=None):
    """moe_qgemv_combine without a workspace: the library's fixed scratch array
    stands in for it (see include/qgemv.h for its size limit and sharing)."""
    gc, gs, gb = _weight(gu, "gu")
    dc, ds, db = _weight(dn, "dn")
    _cuda(expert_idx, (torch.int32,), "expert_idx")
    _cuda(expert_w, (torch.float32,), "expert_w")
    x = _cuda(x, _F16, "x")
    _cuda(residual, _F16, "residual")
    E, I2, H8 = gc.shape
    I, H = I2 // 2, H8 * 8
    if y is None:
        y = torch.empty(H, dtype=torch.float16, device=x.device)
    _cuda(err_flag, (torch.int32,), "err_flag")
    st = lib.moe_qgemv_combine_noalloc(_ptr(gc), _ptr(gs), _ptr(gb), _ptr(dc), _ptr(ds),
                                       _ptr(db), E, H, I, _ptr(expert_idx), _ptr(expert_w),
                                       expert_idx.numel(), _ptr(x), _ptr(residual), _ptr(y),
                                       _ptr(err_flag), _stream(stream))
    _check(st, "moe_qgemv_combine_noalloc")
    return y


def noalloc_max_scratch_bytes() -> int:
    return int(lib.qgemv_noalloc_max_scratch())


def decode_attention_seq1(qkv, n_q, n_kv, head_dim, out=None, stream=None):
    qkv = _cuda(qkv, _F16, "qkv")
    if out is None:
        out = torch.empty(n_q * head_dim, dtype=torch.float16, device=qkv.device)
    st = lib.decode_attention_seq1(_ptr(qkv), _ptr(out), int(n_q), int(n_kv), int(head_dim),
                                   _stream(stream))
    _check(st, "decode_attention_seq1")
    return out


_LAYER_FIELDS = ["qkv_codes", "qkv_scales", "qkv_biases", "attn_norm", "o_codes", "o_scales",
                 "o_biases", "mlp_norm", "gate_codes", "gate_scales", "gate_biases", "up_codes",
                 "up_scales", "up_biases", "down_codes", "down_scales", "down_biases"]


class StackLayer(ctypes.Structure):
    """qgemv_stack_layer: device pointers of one layer."""
    _fields_ = [(f, ctypes.c_void_p) for f in _LAYER_FIELDS]


class StackShape(ctypes.Structure):
    """qgemv_stack_shape."""
    _fields_ = [("hidden", _I), ("n_q", _I), ("n_kv", _I), ("head_dim", _I), ("inter", _I),
                ("n_layers", _I), ("eps", _F)]


def stack_shape(hidden, n_q, n_kv, head_dim, inter, n_layers, eps=1e-5) -> StackShape:
    return StackShape(hidden, n_q, n_kv, head_dim, inter, n_layers, eps)


def decode_stack_workspace_bytes(shape: StackShape) -> int:
    return int(lib.qgemv_decode_stack_workspace_bytes(ctypes.byref(shape)))


def stack_layers(layers):
    """Descriptors for a list of layers, each a dict with weight triples
    'qkv', 'o', 'gate', 'up', 'down' and fp16 vectors 'attn_norm',
    'mlp_norm' (CUDA tensors)."""
    arr = (StackLayer * len(layers))()
    for i, L in enumerate(layers):
        d = arr[i]
        for name in ("qkv", "o", "gate", "up", "down"):
            c, sc, b = _weight(L[name], name)
            setattr(d, name + "_codes", c.data_ptr())
            setattr(d, name + "_scales", sc.data_ptr())
            setattr(d, name + "_biases", b.data_ptr())
        d.attn_norm = _cuda(L["attn_norm"], _F16, "attn_norm").data_ptr()
        d.mlp_norm = _cuda(L["mlp_norm"], _F16, "mlp_norm").data_ptr()
    return arr


def decode_stack(layers, shape: StackShape, x, y=None, workspace=None, stream=None):
    """One token through the layer stack in one call (qgemv_decode_stack).
    `layers` is a list of layer dicts or a prebuilt stack_layers() array."""
    arr = layers if isinstance(layers, ctypes.Array) else stack_layers(layers)
    x = _cuda(x, _F16, "x")
    if y is None:
        y = torch.empty(shape.hidden, dtype=torch.float16, device=x.device)
    nbytes = decode_stack_workspace_bytes(shape)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
    st = lib.qgemv_decode_stack(arr, ctypes.byref(shape), _ptr(x), _ptr(y), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "qgemv_decode_stack")
    return y


def device_status() -> int:
    """Read and clear the device-side status word (synchronises the device)."""
    flags = ctypes.c_uint(0)
    _check(lib.qgemv_device_status(ctypes.byref(flags)), "qgemv_device_status")
    return int(flags.value)


def selftest_wait_timeout(limit_us: int = 2000, stream=None) -> None:
    """Enqueue the bounded-wait self-test (qgemv_selftest_wait_timeout): a
    wait that nothing satisfies gives up after limit_us and sets bit 0 of
    the device status word."""
    _check(lib.qgemv_selftest_wait_timeout(int(limit_us), _stream(stream)),
           "qgemv_selftest_wait_timeout")


def last_cuda_error() -> int:
    return int(lib.qgemv_last_cuda_error())


def version() -> int:
    return int(lib.qgemv_version())
