"""fp64 CPU oracle for the dequant-fused quantized GEMV and its fusions.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` are the only callers.  The oracle shares
no code with the CUDA path (``bit_group_quantized_qgemv_gb300``), and neither
imports the other.

The arithmetic lives in ``qgemv_oracle.c`` (plain C, fp64, index-order sums,
one round-to-nearest-even rounding per fp16 output).  This module compiles it
with gcc on first use and wraps each function with numpy-friendly helpers.
fp16 arrays are passed as their IEEE binary16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qgemv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_P = ctypes.c_void_p
_I = ctypes.c_int
_D = ctypes.c_double

_SIGS = {
    "oracle_half_to_double": (_D, [ctypes.c_uint16]),
    "oracle_double_to_half": (ctypes.c_uint16, [_D]),
    "oracle_code": (_I, [_P, _I, _I]),
    "oracle_set_threads": (None, [_I]),
    "oracle_get_threads": (_I, []),
    "oracle_silu": (_D, [_D]),
    "oracle_matvec_f64": (None, [_I, _P, _P, _P, _I, _I, _P, _P, _P]),
    "oracle_qgemv": (None, [_I, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P]),
    "oracle_rmsnorm": (None, [_P, _P, _I, _D, _P]),
    "oracle_rmsnorm_qgemv": (None, [_P, _P, _P, _P, _P, _D, _I, _I, _P, _P, _P]),
    "oracle_swiglu_qgemv": (None, [_P, _P, _P, _P, _P, _P, _P, _P, _D, _I, _I,
                                   _P, _P, _P]),
    "oracle_moe_qgemv_combine": (None, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P,
                                        _P, _I, _P, _P, _P, _P, _P, _P]),
    "oracle_lut_qgemv": (None, [_P, _P, _I, _P, _P, _I, _I, _P, _P, _P]),
}


def lib():
    """Load (building if needed) the oracle shared library.

    ``QGEMV_ORACLE_LIB`` may name a prebuilt library to load instead; the
    mutation tests use it to run the pins against deliberately broken copies.
    """
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("QGEMV_ORACLE_LIB") or build()
            handle = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _u32(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint32, a.dtype
    return a


def _f16bits(a):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return a


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


def threads() -> int:
    return int(lib().oracle_get_threads())


def half_to_double(bits: int) -> float:
    return float(lib().oracle_half_to_double(int(bits)))


def double_to_half(v: float) -> int:
    return int(lib().oracle_double_to_half(float(v)))


def silu(z: float) -> float:
    return float(lib().oracle_silu(float(z)))


def code(row_words, bits: int, k: int) -> int:
    row = _u32(row_words)
    return int(lib().oracle_code(_ptr(row), int(bits), int(k)))


def matvec_f64(bits, codes, scales, biases, x64):
    """y = W x for an fp64 x; returns (y, sum|w||x|)."""
    codes, scales, biases = _u32(codes), _f16bits(scales), _f16bits(biases)
    N = codes.shape[0]
    x64 = np.ascontiguousarray(x64, dtype=np.float64)
    K = x64.shape[-1]
    y = np.empty(N, np.float64)
    ab = np.empty(N, np.float64)
    lib().oracle_matvec_f64(bits, _ptr(codes), _ptr(scales), _ptr(biases), N, K,
                            _ptr(x64), _ptr(y), _ptr(ab))
    return y, ab


def qgemv(bits, codes, scales, biases, x, residual=None):
    """Plain quantized GEMV.  x: fp16 [M][K] (or [K]); residual fp16 [M][N].

    Returns (y64, y16, bound) with y16 as float16, shapes [M][N] (or [N]).
    """
    codes, scales, biases = _u32(codes), _f16bits(scales), _f16bits(biases)
    xb = _f16bits(x)
    squeeze = xb.ndim == 1
    xb = xb.reshape(-1, xb.shape[-1])
    M, K = xb.shape
    N = codes.shape[0]
    rb = None if residual is None else _f16bits(residual).reshape(M, N)
    y64 = np.empty((M, N), np.float64)
    y16 = np.empty((M, N), np.uint16)
    bound = np.empty((M, N), np.float64)
    lib().oracle_qgemv(bits, _ptr(codes), _ptr(scales), _ptr(biases), _ptr(xb),
                       _ptr(rb), M, N, K, _ptr(y64), _ptr(y16), _ptr(bound))
    y16 = y16.view(np.float16)
    if squeeze:
        return y64[0], y16[0], bound[0]
    return y64, y16, bound


def lut_qgemv(codes, lut, rows_per_lut, x, residual=None):
    """LUT / palettised 4-bit GEMV (INFERENCE_RESEARCH.md section 3, item 4:
    4-bit indices and a 16-entry fp16 table, Core ML style):
    y[n] = sum_k lut[n // rows_per_lut][q[n][k]] x[k] (+ residual[n]).
    codes uint32 [N][K/8]; lut fp16 [ceil(N / rows_per_lut)][16]; x fp16
    [K].  Returns (y64, y16 as float16, bound = sum |w||x| + |residual|)."""
    codes = _u32(codes)
    lb = _f16bits(lut).reshape(-1, 16)
    xb = _f16bits(x).reshape(-1)
    N, K = codes.shape[0], xb.shape[0]
    assert codes.shape[1] * 8 == K and lb.shape[0] * rows_per_lut >= N
    rb = None if residual is None else _f16bits(residual).reshape(N)
    y64 = np.empty(N, np.float64)
    y16 = np.empty(N, np.uint16)
    bound = np.empty(N, np.float64)
    lib().oracle_lut_qgemv(_ptr(codes), _ptr(lb), int(rows_per_lut), _ptr(xb), _ptr(rb), N, K,
                           _ptr(y64), _ptr(y16), _ptr(bound))
    return y64, y16.view(np.float16), bound


def rmsnorm(x, gamma, eps):
    xb, gb = _f16bits(x), _f16bits(gamma)
    K = xb.shape[-1]
    out = np.empty(K, np.float64)
    lib().oracle_rmsnorm(_ptr(xb), _ptr(gb), K, float(eps), _ptr(out))
    return out


def rmsnorm_qgemv(codes, scales, biases, x, gamma, eps):
    codes, scales, biases = _u32(codes), _f16bits(scales), _f16bits(biases)
    xb, gb = _f16bits(x), _f16bits(gamma)
    N, K = codes.shape[0], xb.shape[-1]
    y64 = np.empty(N, np.float64)
    y16 = np.empty(N, np.uint16)
    bound = np.empty(N, np.float64)
    lib().oracle_rmsnorm_qgemv(_ptr(codes), _ptr(scales), _ptr(biases), _ptr(xb),
                               _ptr(gb), float(eps), N, K, _ptr(y64), _ptr(y16),
                               _ptr(bound))
    return y64, y16.view(np.float16), bound


def swiglu_qgemv(gate, up, x, gamma=None, eps=1e-5):
    """gate/up: (codes, scales, biases) triples.  Returns (h64, h16, tol)."""
    gc, gs, gb = _u32(gate[0]), _f16bits(gate[1]), _f16bits(gate[2])
    uc, us, ub = _u32(up[0]), _f16bits(up[1]), _f16bits(up[2])
    xb = _f16bits(x)
    gm = _f16bits(gamma)
    I, K = gc.shape[0], xb.shape[-1]
    h64 = np.empty(I, np.float64)
    h16 = np.empty(I, np.uint16)
    tol = np.empty(I, np.float64)
    lib().oracle_swiglu_qgemv(_ptr(gc), _ptr(gs), _ptr(gb), _ptr(uc), _ptr(us),
                              _ptr(ub), _ptr(xb), _ptr(gm), float(eps), I, K,
                              _ptr(h64), _ptr(h16), _ptr(tol))
    return h64, h16.view(np.float16), tol


def moe_qgemv_combine(gu, dn, idx, wt, x, residual):
    """gu = (codes [E][2I][H/8], scales [E][2I][H/64], biases ...),
    dn = (codes [E][H][I/8], scales [E][H][I/64], biases ...).

    Returns (y64, y16, tol, err_flag).
    """
    gc, gs, gb = _u32(gu[0]), _f16bits(gu[1]), _f16bits(gu[2])
    dc, ds, db = _u32(dn[0]), _f16bits(dn[1]), _f16bits(dn[2])
    E = gc.shape[0]
    I = gc.shape[1] // 2
    H = dc.shape[1]
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    wt = np.ascontiguousarray(wt, dtype=np.float32)
    xb, rb = _f16bits(x), _f16bits(residual)
    y64 = np.empty(H, np.float64)
    y16 = np.empty(H, np.uint16)
    tol = np.empty(H, np.float64)
    err = ctypes.c_int(0)
    lib().oracle_moe_qgemv_combine(_ptr(gc), _ptr(gs), _ptr(gb), _ptr(dc),
                                   _ptr(ds), _ptr(db), E, H, I, _ptr(idx),
                                   _ptr(wt), idx.shape[0], _ptr(xb), _ptr(rb),
                                   _ptr(y64), _ptr(y16), _ptr(tol),
                                   ctypes.addressof(err))
    return y64, y16.view(np.float16), tol, int(err.value)


def moe_route(logits, top_k: int, shared: int = 0):
    """MoE routing of one token from its router logits (the hada.io page,
    topic 27758, "Architecture du modele": K = 4 active experts of 512, one
    of them shared; which experts and with what weights is the reading the
    tests use): the shared expert (when ``shared`` >= 0), then the routed
    experts with the largest logits, one at a time, the lower index winning
    a tie, until ``top_k`` are chosen; the weights are the softmax of the
    chosen logits, in fp64.  ``logits``: fp16 [E] (the selection is decided
    on these values).  Returns (idx int32 [top_k] in choice order, weights
    float64 [top_k])."""
    lv = [float(v) for v in np.asarray(logits, np.float16).astype(np.float64)]
    chosen = [int(shared)] if shared >= 0 else []
    while len(chosen) < top_k:
        best = -1
        for e in range(len(lv)):
            if e in chosen:
                continue
            if best < 0 or lv[e] > lv[best]:  # strict: the lower index keeps a tie
                best = e
        chosen.append(best)
    sel = [lv[e] for e in chosen]
    m = max(sel)
    ex = [float(np.exp(v - m)) for v in sel]
    tot = sum(ex)
    return np.array(chosen, np.int32), np.array([v / tot for v in ex], np.float64)


def lm_head_sample(logits, top_k: int, temperature: float, u: float):
    """Top-k sampling of the next token from its logits (INFERENCE_RESEARCH.md
    section 1: lm_head and top-k sampling on the GPU, only the token read
    back; the random number u in [0, 1) is an input): the top_k largest fp16
    logits, ties to the lower index, in decreasing order; weights
    p_j = exp((l_j - l_0) / temperature) in fp64; the token is the first
    candidate whose cumulative weight exceeds u * sum(p).  Returns (token,
    candidates int64 [top_k], cumulative weights / sum float64 [top_k])."""
    lv = np.asarray(logits, np.float16).astype(np.float64)
    cand = np.argsort(-lv, kind="stable")[:top_k]      # a library sort as the selection step
    p = np.exp((lv[cand] - lv[cand[0]]) / float(temperature))
    cum = np.cumsum(p) / p.sum()
    j = int(np.argmax(cum > float(u))) if np.any(cum > float(u)) else top_k - 1
    return int(cand[j]), cand.astype(np.int64), cum
