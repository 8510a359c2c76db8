"""Plain fp64 CPU oracle for the epilogue-fusion hot path (ctypes over oracle.c).

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline / reference legs are the only callers.  The product path
(the CUDA library and its Python binding) never imports this package, and this
package imports nothing from the product.

Every function takes host numpy arrays holding the exact input bits (bf16 and
fp16 as ``uint16`` words, fp32 as ``float32``) and returns float64 results.
The arithmetic lives in ``oracle.c``; each C function cites the page and
section it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

EPI_NONE, EPI_FUSED, EPI_CHAIN = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (no CUDA involved).

    ``-ffp-contract=off`` keeps a*b+c as two rounded double operations on
    every host (aarch64 gcc would otherwise fuse them).
    """
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-D_GNU_SOURCE", "-ffp-contract=off", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # ORACLE_LIB lets the oracle's mutation test load a deliberately
            # broken build of oracle.c; nothing else sets it.
            lib = ctypes.CDLL(os.environ.get("ORACLE_LIB") or build())
            d, i, i64, vp = ctypes.c_double, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
            lib.oracle_pack_filter.argtypes = [vp, vp, i, i, i, i]
            lib.oracle_pack_filter.restype = None
            lib.oracle_conv2d_bn_silu.argtypes = [vp, vp, vp, vp] + [i] * 12 + [vp, i]
            lib.oracle_conv2d_bn_silu.restype = None
            lib.oracle_conv2d_bn_silu_points.argtypes = [vp, vp, vp, vp] + [i] * 12 + [vp, i64, vp, i]
            lib.oracle_conv2d_bn_silu_points.restype = None
            lib.oracle_bias_gelu.argtypes = [vp, vp, i64, i64, i, vp, i]
            lib.oracle_bias_gelu.restype = None
            lib.oracle_bias_gelu_rowsum.argtypes = [vp, vp, i64, i64, i, vp, vp, i]
            lib.oracle_bias_gelu_rowsum.restype = None
            lib.oracle_residual_layernorm.argtypes = [vp, vp, vp, vp, i64, i64, d, i, vp, vp, i]
            lib.oracle_residual_layernorm.restype = None
            for name in ("oracle_f16_value", "oracle_bf16_value"):
                getattr(lib, name).argtypes = [ctypes.c_uint16]
                getattr(lib, name).restype = d
            for name in ("oracle_round_to_f16", "oracle_round_to_bf16", "oracle_gelu", "oracle_silu"):
                getattr(lib, name).argtypes = [d]
                getattr(lib, name).restype = d
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def out_dim(size: int, k: int, stride: int, pad: int) -> int:
    return (size + 2 * pad - k) // stride + 1


def pack_filter(w_oihw: np.ndarray) -> np.ndarray:
    """OIHW -> OHWI permutation of bf16 words (uint16)."""
    w = _c(w_oihw, np.uint16)
    co, ci, kh, kw = w.shape
    out = np.empty((co, kh, kw, ci), np.uint16)
    _load().oracle_pack_filter(_ptr(w), _ptr(out), co, ci, kh, kw)
    return out


def conv2d_bn_silu(x_nhwc, w_oihw, scale, bias, stride=(1, 1), pad=(0, 0),
                   epilogue=EPI_FUSED, nthreads=None) -> np.ndarray:
    """Every output of conv -> scale/bias -> SiLU; x NHWC bf16 words, w OIHW bf16 words."""
    x = _c(x_nhwc, np.uint16)
    w = _c(w_oihw, np.uint16)
    sc = _c(scale, np.float32)
    bi = _c(bias, np.float32)
    n, h, wd, ci = x.shape
    co, ci2, kh, kw = w.shape
    assert ci == ci2 and sc.shape == (co,) and bi.shape == (co,)
    ho, wo = out_dim(h, kh, stride[0], pad[0]), out_dim(wd, kw, stride[1], pad[1])
    y = np.empty((n, ho, wo, co), np.float64)
    _load().oracle_conv2d_bn_silu(_ptr(x), _ptr(w), _ptr(sc), _ptr(bi), n, h, wd, ci, co, kh, kw,
                                  stride[0], stride[1], pad[0], pad[1], int(epilogue), _ptr(y),
                                  nthreads or default_threads())
    return y


def conv2d_bn_silu_points(x_nhwc, w_oihw, scale, bias, points, stride=(1, 1), pad=(0, 0),
                          epilogue=EPI_FUSED, nthreads=None) -> np.ndarray:
    """Selected outputs, ``points`` = flat indices into the NHWC output [N][Ho][Wo][C_out]."""
    x = _c(x_nhwc, np.uint16)
    w = _c(w_oihw, np.uint16)
    sc = _c(scale, np.float32)
    bi = _c(bias, np.float32)
    p = _c(np.asarray(points, np.int64), np.int64)
    n, h, wd, ci = x.shape
    co, ci2, kh, kw = w.shape
    assert ci == ci2
    y = np.empty(p.shape[0], np.float64)
    _load().oracle_conv2d_bn_silu_points(_ptr(x), _ptr(w), _ptr(sc), _ptr(bi), n, h, wd, ci, co, kh, kw,
                                         stride[0], stride[1], pad[0], pad[1], int(epilogue),
                                         _ptr(p), p.shape[0], _ptr(y), nthreads or default_threads())
    return y


def bias_gelu(x_f16, bias_f16, materialize=False, nthreads=None) -> np.ndarray:
    """y = GELU_erf(x + bias[col]) in fp64; x fp16 [rows, cols], bias fp16 [cols]."""
    x = _c(np.asarray(x_f16).view(np.uint16), np.uint16)
    b = _c(np.asarray(bias_f16).view(np.uint16), np.uint16)
    rows, cols = x.shape
    assert b.shape == (cols,)
    y = np.empty((rows, cols), np.float64)
    _load().oracle_bias_gelu(_ptr(x), _ptr(b), rows, cols, int(materialize), _ptr(y),
                             nthreads or default_threads())
    return y


def bias_gelu_rowsum(x_f16, bias_f16, materialize=False, want_y=True, nthreads=None):
    """(y, rowsum): GELU_erf(x + bias) and the sum of each row of it, in fp64."""
    x = _c(np.asarray(x_f16).view(np.uint16), np.uint16)
    b = _c(np.asarray(bias_f16).view(np.uint16), np.uint16)
    rows, cols = x.shape
    y = np.empty((rows, cols), np.float64) if want_y else None
    rs = np.empty(rows, np.float64)
    _load().oracle_bias_gelu_rowsum(_ptr(x), _ptr(b), rows, cols, int(materialize),
                                    _ptr(y) if y is not None else None, _ptr(rs),
                                    nthreads or default_threads())
    return y, rs


def residual_layernorm(act_f16, res_f16, gamma, beta, eps=1e-5, materialize=False,
                       want_stats=False, nthreads=None):
    """y = LayerNorm(act + res) * gamma + beta in fp64 (two-pass statistics)."""
    a = _c(np.asarray(act_f16).view(np.uint16), np.uint16)
    r = _c(np.asarray(res_f16).view(np.uint16), np.uint16)
    g = _c(gamma, np.float32)
    be = _c(beta, np.float32)
    rows, hidden = a.shape
    assert r.shape == a.shape and g.shape == (hidden,) and be.shape == (hidden,)
    y = np.empty((rows, hidden), np.float64)
    st = np.empty((rows, 2), np.float64) if want_stats else None
    _load().oracle_residual_layernorm(_ptr(a), _ptr(r), _ptr(g), _ptr(be), rows, hidden, float(eps),
                                      int(materialize), _ptr(y), _ptr(st) if st is not None else None,
                                      nthreads or default_threads())
    return (y, st) if want_stats else y


# scalar helpers, for the oracle's own pins
def f16_value(h: int) -> float:
    return _load().oracle_f16_value(h)


def bf16_value(b: int) -> float:
    return _load().oracle_bf16_value(b)


def round_to_f16(v: float) -> float:
    return _load().oracle_round_to_f16(v)


def round_to_bf16(v: float) -> float:
    return _load().oracle_round_to_bf16(v)


def gelu(s: float) -> float:
    return _load().oracle_gelu(s)


def silu(v: float) -> float:
    return _load().oracle_silu(v)
