"""Thin ctypes binding of libtf_epilogue.so (include/tf_epilogue.h).

Argument marshalling only: every function has the C entry point's name and
arguments, turns tensors into device pointers and streams into cudaStream_t
handles, and raises TfError on a non-zero status.  All computation happens
in the library's CUDA kernels; there is no other code path.  If the library
has not been built this module fails loudly at import.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtf_epilogue.so")

TF_OK, TF_ERR_INVALID_ARG, TF_ERR_UNSUPPORTED, TF_ERR_CUDA, TF_ERR_TIMEOUT = 0, 1, 2, 3, 4
(TF_CONV_AUTO, TF_CONV_DIRECT, TF_CONV_TILED, TF_CONV_UMMA, TF_CONV_UMMA_PAIR, TF_CONV_UMMA_PAIR_WIDE,
 TF_CONV_UMMA_WIDE) = -1, 0, 1, 2, 3, 4, 5
TF_LN_AUTO, TF_LN_WARP, TF_LN_CTA, TF_LN_CLUSTER = -1, 0, 1, 2
TF_DEVERR_PRODUCER_WAIT, TF_DEVERR_MMA_WAIT, TF_DEVERR_EPILOGUE_WAIT = 0x1, 0x2, 0x4
TF_DEVERR_DRAIN_WAIT, TF_DEVERR_PROBE_WAIT, TF_DEVERR_EXCHANGE_WAIT = 0x8, 0x10, 0x20
TF_DEVERR_PAIR_TMEM, TF_DEVERR_SMEM_ALIGN = 0x40, 0x80


class TfError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


class tf_conv_shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("N", "H", "W", "C_in", "C_out", "KH", "KW", "stride_h", "stride_w", "pad_h", "pad_w")]


if not os.path.exists(LIB_PATH):
    raise ImportError(f"libtf_epilogue.so is not built ({LIB_PATH}); run __graft_entry__.build() "
                      "or python -m gemm_conv_epilogues_gb300.build")

_lib = ctypes.CDLL(LIB_PATH)
_vp, _i, _i64, _u64, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float
_SIGS = {
    "tf_status_string": ([_i], ctypes.c_char_p),
    "tf_pack_filter_nhwc": ([_vp, _vp, _i, _i, _i, _i, _vp], _i),
    "tf_conv2d_bn_silu": ([_vp, _vp, _vp, _vp, _vp, ctypes.POINTER(tf_conv_shape), _vp], _i),
    "tf_conv2d_bn_silu_variant": ([_vp, _vp, _vp, _vp, _vp, ctypes.POINTER(tf_conv_shape), _i, _vp], _i),
    "tf_conv2d_bn_silu_select": ([ctypes.POINTER(tf_conv_shape)], _i),
    "tf_conv2d_bn_silu_workspace_size": ([ctypes.POINTER(tf_conv_shape)], _i64),
    "tf_conv2d_bn_silu_ws": ([_vp, _vp, _vp, _vp, _vp, ctypes.POINTER(tf_conv_shape), _vp, _i64, _vp], _i),
    "tf_conv2d_bn_silu_static_ws": ([_vp, _vp, _vp, _vp, _vp, ctypes.POINTER(tf_conv_shape), _vp], _i),
    "tf_bias_gelu": ([_vp, _vp, _vp, _i64, _i64, _vp], _i),
    "tf_bias_gelu_rowsum": ([_vp, _vp, _vp, _vp, _i64, _i64, _vp], _i),
    "tf_unfused_rowsum": ([_vp, _vp, _i64, _i64, _vp], _i),
    "tf_residual_layernorm": ([_vp, _vp, _vp, _vp, _vp, _i64, _i64, _f, _vp], _i),
    "tf_residual_layernorm_variant": ([_vp, _vp, _vp, _vp, _vp, _i64, _i64, _f, _i, _vp], _i),
    "tf_residual_layernorm_select": ([_i64], _i),
    "tf_unfused_conv2d": ([_vp, _vp, _vp, ctypes.POINTER(tf_conv_shape), _i, _vp], _i),
    "tf_unfused_bn": ([_vp, _vp, _vp, _vp, _i64, _i64, _vp], _i),
    "tf_unfused_silu": ([_vp, _vp, _i64, _vp], _i),
    "tf_unfused_bias_add": ([_vp, _vp, _vp, _i64, _i64, _vp], _i),
    "tf_unfused_gelu": ([_vp, _vp, _i64, _vp], _i),
    "tf_unfused_residual_add": ([_vp, _vp, _vp, _i64, _vp], _i),
    "tf_unfused_layernorm": ([_vp, _vp, _i64, _i64, _f, _vp], _i),
    "tf_unfused_affine": ([_vp, _vp, _vp, _vp, _i64, _i64, _vp], _i),
    "tf_set_wait_limit_ns": ([_u64], None),
    "tf_get_wait_limit_ns": ([], _u64),
    "tf_read_device_error": ([ctypes.POINTER(ctypes.c_uint32)], _i),
    "tf_wait_probe": ([_u64, _vp], _i),
    "tf_launch_count": ([], _u64),
}
for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res


def lib() -> ctypes.CDLL:
    return _lib


def status_string(status: int) -> str:
    return _lib.tf_status_string(int(status)).decode()


def _ptr(t):
    """Device address of a tensor (or an int address, or None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise TypeError("tf_* entry points take device tensors")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str, check: bool) -> int:
    if check and rc != TF_OK:
        raise TfError(rc, where)
    return rc


def conv_shape(N, H, W, C_in, C_out, KH, KW, stride=(1, 1), pad=(0, 0)) -> tf_conv_shape:
    return tf_conv_shape(N, H, W, C_in, C_out, KH, KW, stride[0], stride[1], pad[0], pad[1])


def tf_pack_filter_nhwc(w_oihw, w_ohwi, C_out, C_in, KH, KW, stream=None, check=True):
    return _check(_lib.tf_pack_filter_nhwc(_ptr(w_oihw), _ptr(w_ohwi), C_out, C_in, KH, KW, _stream(stream)),
                  "tf_pack_filter_nhwc", check)


def tf_conv2d_bn_silu(x, w_ohwi, scale, bias, y, shape, stream=None, check=True):
    return _check(_lib.tf_conv2d_bn_silu(_ptr(x), _ptr(w_ohwi), _ptr(scale), _ptr(bias), _ptr(y),
                                         ctypes.byref(shape), _stream(stream)), "tf_conv2d_bn_silu", check)


def tf_conv2d_bn_silu_variant(x, w_ohwi, scale, bias, y, shape, variant, stream=None, check=True):
    return _check(_lib.tf_conv2d_bn_silu_variant(_ptr(x), _ptr(w_ohwi), _ptr(scale), _ptr(bias), _ptr(y),
                                                 ctypes.byref(shape), int(variant), _stream(stream)),
                  "tf_conv2d_bn_silu_variant", check)


def tf_conv2d_bn_silu_select(shape) -> int:
    return _lib.tf_conv2d_bn_silu_select(ctypes.byref(shape))


def tf_conv2d_bn_silu_workspace_size(shape) -> int:
    return int(_lib.tf_conv2d_bn_silu_workspace_size(ctypes.byref(shape)))


def tf_conv2d_bn_silu_ws(x, w_ohwi, scale, bias, y, shape, workspace, workspace_bytes, stream=None, check=True):
    return _check(_lib.tf_conv2d_bn_silu_ws(_ptr(x), _ptr(w_ohwi), _ptr(scale), _ptr(bias), _ptr(y),
                                            ctypes.byref(shape), _ptr(workspace), int(workspace_bytes),
                                            _stream(stream)), "tf_conv2d_bn_silu_ws", check)


def tf_conv2d_bn_silu_static_ws(x, w_ohwi, scale, bias, y, shape, stream=None, check=True):
    """tf_conv2d_bn_silu_ws without a workspace argument, for callers that cannot
    allocate device memory: the split-K partials use the library's one 8 MiB
    static device array (calls that overlap on the GPU race on it)."""
    return _check(_lib.tf_conv2d_bn_silu_static_ws(_ptr(x), _ptr(w_ohwi), _ptr(scale), _ptr(bias), _ptr(y),
                                                   ctypes.byref(shape), _stream(stream)),
                  "tf_conv2d_bn_silu_static_ws", check)


def tf_bias_gelu(x, bias, y, rows, cols, stream=None, check=True):
    return _check(_lib.tf_bias_gelu(_ptr(x), _ptr(bias), _ptr(y), rows, cols, _stream(stream)),
                  "tf_bias_gelu", check)


def tf_bias_gelu_rowsum(x, bias, y, rowsum, rows, cols, stream=None, check=True):
    return _check(_lib.tf_bias_gelu_rowsum(_ptr(x), _ptr(bias), _ptr(y), _ptr(rowsum), rows, cols, _stream(stream)),
                  "tf_bias_gelu_rowsum", check)


def tf_unfused_rowsum(y, rowsum, rows, cols, stream=None, check=True):
    return _check(_lib.tf_unfused_rowsum(_ptr(y), _ptr(rowsum), rows, cols, _stream(stream)),
                  "tf_unfused_rowsum", check)


def tf_residual_layernorm(act, res, gamma, beta, y, rows, hidden, eps, stream=None, check=True):
    return _check(_lib.tf_residual_layernorm(_ptr(act), _ptr(res), _ptr(gamma), _ptr(beta), _ptr(y), rows,
                                             hidden, float(eps), _stream(stream)), "tf_residual_layernorm", check)


def tf_residual_layernorm_variant(act, res, gamma, beta, y, rows, hidden, eps, variant, stream=None, check=True):
    return _check(_lib.tf_residual_layernorm_variant(_ptr(act), _ptr(res), _ptr(gamma), _ptr(beta), _ptr(y), rows,
                                                     hidden, float(eps), int(variant), _stream(stream)),
                  "tf_residual_layernorm_variant", check)


def tf_residual_layernorm_select(hidden) -> int:
    return _lib.tf_residual_layernorm_select(int(hidden))


def tf_unfused_conv2d(x, w_ohwi, t1, shape, variant=TF_CONV_AUTO, stream=None, check=True):
    return _check(_lib.tf_unfused_conv2d(_ptr(x), _ptr(w_ohwi), _ptr(t1), ctypes.byref(shape), int(variant),
                                         _stream(stream)), "tf_unfused_conv2d", check)


def tf_unfused_bn(t1, scale, bias, t2, M, C, stream=None, check=True):
    return _check(_lib.tf_unfused_bn(_ptr(t1), _ptr(scale), _ptr(bias), _ptr(t2), M, C, _stream(stream)),
                  "tf_unfused_bn", check)


def tf_unfused_silu(t2, y, n, stream=None, check=True):
    return _check(_lib.tf_unfused_silu(_ptr(t2), _ptr(y), n, _stream(stream)), "tf_unfused_silu", check)


def tf_unfused_bias_add(x, bias, t, rows, cols, stream=None, check=True):
    return _check(_lib.tf_unfused_bias_add(_ptr(x), _ptr(bias), _ptr(t), rows, cols, _stream(stream)),
                  "tf_unfused_bias_add", check)


def tf_unfused_gelu(t, y, n, stream=None, check=True):
    return _check(_lib.tf_unfused_gelu(_ptr(t), _ptr(y), n, _stream(stream)), "tf_unfused_gelu", check)


def tf_unfused_residual_add(act, res, s, n, stream=None, check=True):
    return _check(_lib.tf_unfused_residual_add(_ptr(act), _ptr(res), _ptr(s), n, _stream(stream)),
                  "tf_unfused_residual_add", check)


def tf_unfused_layernorm(s, nrm, rows, hidden, eps, stream=None, check=True):
    return _check(_lib.tf_unfused_layernorm(_ptr(s), _ptr(nrm), rows, hidden, float(eps), _stream(stream)),
                  "tf_unfused_layernorm", check)


def tf_unfused_affine(nrm, gamma, beta, y, rows, hidden, stream=None, check=True):
    return _check(_lib.tf_unfused_affine(_ptr(nrm), _ptr(gamma), _ptr(beta), _ptr(y), rows, hidden,
                                         _stream(stream)), "tf_unfused_affine", check)


def tf_set_wait_limit_ns(limit_ns: int) -> None:
    _lib.tf_set_wait_limit_ns(int(limit_ns))


def tf_get_wait_limit_ns() -> int:
    return int(_lib.tf_get_wait_limit_ns())


def tf_launch_count() -> int:
    """Kernels the library has launched in this process so far."""
    return int(_lib.tf_launch_count())


def tf_read_device_error():
    """(status, word): synchronises the device, reads and clears the error word."""
    w = ctypes.c_uint32(0)
    rc = _lib.tf_read_device_error(ctypes.byref(w))
    return rc, int(w.value)


def tf_wait_probe(limit_ns, stream=None, check=True):
    return _check(_lib.tf_wait_probe(int(limit_ns), _stream(stream)), "tf_wait_probe", check)
