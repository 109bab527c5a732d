"""Python binding of libqmm (include/qmm.h): block-quantized matmul on GB300.

Every function has the name of the C entry point it calls and only marshals
arguments: tensors become device pointers, the stream defaults to torch's
current stream, and a non-OK status raises ``QmmError``. All computation runs
in the CUDA kernels of ``libqmm.so``; there is no fallback. If the library
has not been built, importing this package raises ``ImportError``.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqmm.so")

QMM_TYPE_Q4_0, QMM_TYPE_Q4_K, QMM_TYPE_Q8_0, QMM_TYPE_Q8_K, QMM_TYPE_W4A16, QMM_TYPE_Q6_K = 0, 1, 2, 3, 4, 5
QMM_OK = 0
STATUS = {0: "QMM_OK", 1: "QMM_ERR_ARG", 2: "QMM_ERR_UNSUPPORTED", 3: "QMM_ERR_CUDA",
          4: "QMM_ERR_TIMEOUT", 5: "QMM_ERR_NOMEM", 6: "QMM_ERR_WORKSPACE"}


class QmmError(RuntimeError):
    def __init__(self, func: str, status: int, message: str):
        super().__init__(f"{func}: {STATUS.get(status, status)}: {message}")
        self.status = status


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python -c 'import __graft_entry__ as g; g.build()'`")

_lib = ctypes.CDLL(LIB_PATH)
_vp, _i64, _i32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
_SIGS = {
    "qmm_block_bytes": (_sz, [_i32]),
    "qmm_block_elems": (_i32, [_i32]),
    "qmm_packed_bytes": (_sz, [_i32, _i64, _i64]),
    "qmm_workspace_bytes": (_sz, [_i32, _i64, _i64]),
    "qmm_quantize_row_q8": (_i32, [_i32, _vp, _vp, _i64, _i64, _vp]),
    "qmm_quantize_weights": (_i32, [_i32, _vp, _vp, _i64, _i64, _vp]),
    "qmm_repack_weights": (_i32, [_i32, _vp, _vp, _i64, _i64, _vp]),
    "qmm_unrepack_weights": (_i32, [_i32, _vp, _vp, _i64, _i64, _vp]),
    "qmm_mul_mat": (_i32, [_i32, _vp, _i64, _i64, _vp, _i64, _vp, _vp]),
    "qmm_mul_mat_ws": (_i32, [_i32, _vp, _i64, _i64, _vp, _i64, _vp, _vp, _sz, _vp]),
    "qmm_host_call_bytes": (_sz, [_i32, _i64, _i64, _i64]),
    "qmm_mul_mat_host": (_i32, [_i32, _vp, _i64, _i64, _vp, _i64, _vp, _vp, _sz, ctypes.c_uint, _vp]),
    "qmm_mul_mat_q8": (_i32, [_i32, _vp, _i64, _i64, _vp, _i64, _vp, _vp]),
    "qmm_mul_mat_multi": (_i32, [_i32, _i32, ctypes.POINTER(_vp), ctypes.POINTER(_i64), _i64, _vp,
                                 _i64, ctypes.POINTER(_vp), _vp]),
    "qmm_quantize_activations": (_i32, [_i32, _vp, _i64, _i64, _vp, _sz, _vp]),
    "qmm_mul_mat_prepared": (_i32, [_i32, _vp, _i64, _i64, _vp, _sz, _i64, _vp, _vp]),
    "qmm_mul_mat_static": (_i32, [_i32, _vp, _i64, _i64, _vp, _i64, _vp, _vp]),
    "qmm_debug_block_sums": (_i32, [_i32, _vp, _i64, _i64, _vp, _i64, _vp, _vp]),
    "qmm_w4a16": (_i32, [_vp, _vp, _vp, _i64, _vp, _vp, _i64, _i64, _i64, _vp]),
    "qmm_w4a16_lut": (_i32, [_vp, _vp, _vp, _i64, _vp, _vp, _i64, _i64, _i64, _vp]),
    "qmm_w4a16_unpack_zeros": (_i32, [_vp, _vp, _i64, _i64, _vp]),
    "qmm_debug_wait_timeout": (_i32, [_i64, _vp]),
    "qmm_debug_peak": (_i32, [_i32, _i64, ctypes.POINTER(ctypes.c_double), _vp]),
    "qmm_status_string": (ctypes.c_char_p, [_i32]),
    "qmm_last_error": (ctypes.c_char_p, []),
    "qmm_check_device_error": (_i32, [_vp]),
    "qmm_kernel_launch_count": (ctypes.c_uint64, []),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_SIGS)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("libqmm takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libqmm takes contiguous tensors")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(func: str, status: int):
    if status != QMM_OK:
        raise QmmError(func, status, _lib.qmm_last_error().decode(errors="replace"))


# ---------------------------------------------------------------- sizes
def qmm_block_bytes(t: int) -> int:
    return int(_lib.qmm_block_bytes(t))


def qmm_block_elems(t: int) -> int:
    return int(_lib.qmm_block_elems(t))


def qmm_packed_bytes(wt: int, N: int, K: int) -> int:
    return int(_lib.qmm_packed_bytes(wt, N, K))


def qmm_workspace_bytes(wt: int, M: int, K: int) -> int:
    return int(_lib.qmm_workspace_bytes(wt, M, K))


def row_bytes(t: int, K: int) -> int:
    return qmm_block_bytes(t) * (K // qmm_block_elems(t))


# ---------------------------------------------------------------- calls
def qmm_quantize_row_q8(vt: int, X, Xq, M: int, K: int, stream=None):
    _check("qmm_quantize_row_q8",
           _lib.qmm_quantize_row_q8(vt, _ptr(X), _ptr(Xq), M, K, _stream(stream)))


def qmm_quantize_weights(wt: int, W, Wq, N: int, K: int, stream=None):
    _check("qmm_quantize_weights",
           _lib.qmm_quantize_weights(wt, _ptr(W), _ptr(Wq), N, K, _stream(stream)))


def qmm_repack_weights(wt: int, W_canon, W_packed, N: int, K: int, stream=None):
    _check("qmm_repack_weights",
           _lib.qmm_repack_weights(wt, _ptr(W_canon), _ptr(W_packed), N, K, _stream(stream)))


def qmm_unrepack_weights(wt: int, W_packed, W_canon, N: int, K: int, stream=None):
    _check("qmm_unrepack_weights",
           _lib.qmm_unrepack_weights(wt, _ptr(W_packed), _ptr(W_canon), N, K, _stream(stream)))


def qmm_mul_mat(wt: int, W_packed, N: int, K: int, X, M: int, Y, stream=None):
    _check("qmm_mul_mat",
           _lib.qmm_mul_mat(wt, _ptr(W_packed), N, K, _ptr(X), M, _ptr(Y), _stream(stream)))


def qmm_mul_mat_q8(wt: int, W_packed, N: int, K: int, Xq, M: int, Y, stream=None):
    """Y = Xq W^T from canonical Q8 activation blocks (qmm_quantize_row_q8)."""
    _check("qmm_mul_mat_q8",
           _lib.qmm_mul_mat_q8(wt, _ptr(W_packed), N, K, _ptr(Xq), M, _ptr(Y), _stream(stream)))


def qmm_mul_mat_multi(wt: int, W_packed: list, N: list, K: int, X, M: int, Y: list, stream=None):
    """Y[i] = X W_packed[i]^T for every i, X quantized once, one decode launch."""
    n = len(W_packed)
    if not (len(N) == n == len(Y)):
        raise ValueError("W_packed, N and Y must have the same length")
    w = (_vp * n)(*[_ptr(t) for t in W_packed])
    nn = (_i64 * n)(*N)
    y = (_vp * n)(*[_ptr(t) for t in Y])
    _check("qmm_mul_mat_multi", _lib.qmm_mul_mat_multi(wt, n, w, nn, K, _ptr(X), M, y, _stream(stream)))


def qmm_mul_mat_ws(wt: int, W_packed, N: int, K: int, X, M: int, Y, workspace, ws_bytes: int,
                   stream=None):
    _check("qmm_mul_mat_ws",
           _lib.qmm_mul_mat_ws(wt, _ptr(W_packed), N, K, _ptr(X), M, _ptr(Y), _ptr(workspace),
                               ws_bytes, _stream(stream)))


def _host_ptr(t):
    if isinstance(t, int):
        return t
    if t.is_cuda:
        raise ValueError("qmm_mul_mat_host takes host tensors for X and Y")
    if not t.is_contiguous():
        raise ValueError("libqmm takes contiguous tensors")
    return t.data_ptr()


def qmm_host_call_bytes(wt: int, M: int, N: int, K: int) -> int:
    return int(_lib.qmm_host_call_bytes(wt, M, N, K))


QMM_HOST_MAPPED = 1


def qmm_mul_mat_host(wt: int, W_packed, N: int, K: int, X_host, M: int, Y_host, device_buf,
                     buf_bytes: int, stream=None, flags: int = 0):
    _check("qmm_mul_mat_host",
           _lib.qmm_mul_mat_host(wt, _ptr(W_packed), N, K, _host_ptr(X_host), M, _host_ptr(Y_host),
                                 _ptr(device_buf), buf_bytes, flags, _stream(stream)))


def qmm_quantize_activations(wt: int, X, M: int, K: int, workspace, ws_bytes: int, stream=None):
    _check("qmm_quantize_activations",
           _lib.qmm_quantize_activations(wt, _ptr(X), M, K, _ptr(workspace), ws_bytes,
                                         _stream(stream)))


def qmm_mul_mat_prepared(wt: int, W_packed, N: int, K: int, workspace, ws_bytes: int, M: int, Y,
                         stream=None):
    _check("qmm_mul_mat_prepared",
           _lib.qmm_mul_mat_prepared(wt, _ptr(W_packed), N, K, _ptr(workspace), ws_bytes, M,
                                     _ptr(Y), _stream(stream)))


def qmm_mul_mat_static(wt: int, W_packed, N: int, K: int, X, M: int, Y, stream=None):
    """qmm_mul_mat without any allocation: the activation scratch is a fixed
    4 MiB device array inside libqmm (see include/qmm.h)."""
    _check("qmm_mul_mat_static",
           _lib.qmm_mul_mat_static(wt, _ptr(W_packed), N, K, _ptr(X), M, _ptr(Y),
                                   _stream(stream)))


def qmm_debug_block_sums(wt: int, W_packed, N: int, K: int, Xq, M: int, out, stream=None):
    _check("qmm_debug_block_sums",
           _lib.qmm_debug_block_sums(wt, _ptr(W_packed), N, K, _ptr(Xq), M, _ptr(out),
                                     _stream(stream)))


def qmm_w4a16(W_packed, scales, zeros, G: int, A, C, M: int, N: int, K: int, stream=None):
    """C [M, N] fp16 = A [M, K] fp16 x W^T for packed W4A16 weights (scales fp16
    and zeros uint8 [N, K/G]); see include/qmm.h."""
    _check("qmm_w4a16",
           _lib.qmm_w4a16(_ptr(W_packed), _ptr(scales), _ptr(zeros), G, _ptr(A), _ptr(C), M, N, K,
                          _stream(stream)))


def qmm_w4a16_lut(W_packed, scales, lut, G: int, A, C, M: int, N: int, K: int, stream=None):
    """C [M, N] fp16 = A [M, K] fp16 x W^T with W = s LUT(q): packed codes,
    scales fp16 [N, K/G], a 16-entry fp16 code table; see include/qmm.h."""
    _check("qmm_w4a16_lut",
           _lib.qmm_w4a16_lut(_ptr(W_packed), _ptr(scales), _ptr(lut), G, _ptr(A), _ptr(C), M, N, K,
                              _stream(stream)))


def qmm_w4a16_unpack_zeros(zeros_packed, zeros, N: int, ngroups: int, stream=None):
    """uint8 zeros [N, ngroups] from zero points packed 8 per uint32 word
    ([N, ceil(ngroups/8)]); see include/qmm.h."""
    _check("qmm_w4a16_unpack_zeros",
           _lib.qmm_w4a16_unpack_zeros(_ptr(zeros_packed), _ptr(zeros), N, ngroups, _stream(stream)))


QMM_PEAK_MMA_S8, QMM_PEAK_MMA_F16, QMM_PEAK_TC_SS_128, QMM_PEAK_TC_TS_128, QMM_PEAK_TC_SS_256, \
    QMM_PEAK_TC_TS_256 = range(6)


def qmm_debug_peak(which: int, iters: int, stream=None) -> float:
    """Launch tensor-core microbenchmark `which` on the stream; returns the
    operations (2 per multiply-add) the launch performs."""
    ops = ctypes.c_double(0.0)
    _check("qmm_debug_peak", _lib.qmm_debug_peak(which, iters, ctypes.byref(ops), _stream(stream)))
    return ops.value


def qmm_debug_wait_timeout(limit_cycles: int, stream=None):
    """One CTA waits, bounded by limit_cycles, on a barrier nothing completes:
    the next qmm_check_device_error reports QMM_ERR_TIMEOUT."""
    _check("qmm_debug_wait_timeout", _lib.qmm_debug_wait_timeout(limit_cycles, _stream(stream)))


def qmm_status_string(status: int) -> str:
    return _lib.qmm_status_string(status).decode()


def qmm_last_error() -> str:
    return _lib.qmm_last_error().decode(errors="replace")


def qmm_check_device_error(stream=None):
    _check("qmm_check_device_error", _lib.qmm_check_device_error(_stream(stream)))


def qmm_kernel_launch_count() -> int:
    return int(_lib.qmm_kernel_launch_count())


# ---------------------------------------------------------------- conveniences
def empty_blocks(t: int, rows: int, K: int, device="cuda") -> torch.Tensor:
    """A uint8 device buffer for `rows` rows of canonical blocks of type t."""
    return torch.empty(rows * row_bytes(t, K), dtype=torch.uint8, device=device)


def empty_packed(wt: int, N: int, K: int, device="cuda") -> torch.Tensor:
    return torch.empty(qmm_packed_bytes(wt, N, K), dtype=torch.uint8, device=device)
