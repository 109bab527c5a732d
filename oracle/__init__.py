"""Python view of the plain-C CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product library
never imports, links or calls it, and it never imports the product library.

The C code is compiled in-tree with gcc (``build()``) into ``liboracle.so`` and
called through ctypes. Arrays are numpy; every function here only marshals
arguments, all arithmetic is in ``oracle.c`` (see that file for the page and
section each routine follows).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")

Q4_0, Q4_K, Q8_0, Q8_K, Q6_K = 0, 1, 2, 3, 5
BLOCK_BYTES = {Q4_0: 18, Q4_K: 144, Q8_0: 34, Q8_K: 292, Q6_K: 210}
BLOCK_ELEMS = {Q4_0: 32, Q4_K: 256, Q8_0: 32, Q8_K: 256, Q6_K: 256}
ACT_TYPE = {Q4_0: Q8_0, Q4_K: Q8_K, Q6_K: Q8_K}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain C, no fused multiply-add)."""
    fresh = os.path.exists(_LIB) and all(
        os.path.getmtime(_LIB) >= os.path.getmtime(p) for p in (_SRC, _HDR))
    if fresh and not force:
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            # QMM_ORACLE_LIB points at an alternative build of oracle.c (the
            # mutation tests load deliberately broken copies this way)
            path = os.environ.get("QMM_ORACLE_LIB") or build()
            L = ctypes.CDLL(path)
            vp, i64, f32p, f64p = ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
            L.orc_block_bytes.restype = ctypes.c_size_t
            L.orc_block_bytes.argtypes = [ctypes.c_int]
            L.orc_block_elems.restype = ctypes.c_int
            L.orc_block_elems.argtypes = [ctypes.c_int]
            L.orc_fp32_to_fp16.restype = ctypes.c_uint16
            L.orc_fp32_to_fp16.argtypes = [ctypes.c_float]
            L.orc_fp64_to_fp16.restype = ctypes.c_uint16
            L.orc_fp64_to_fp16.argtypes = [ctypes.c_double]
            L.orc_fp16_to_fp32.restype = ctypes.c_float
            L.orc_fp16_to_fp32.argtypes = [ctypes.c_uint16]
            L.orc_get_scale_min_k4.argtypes = [ctypes.c_int, vp, vp, vp]
            L.orc_set_scale_min_k4.argtypes = [ctypes.c_int, vp, ctypes.c_uint8, ctypes.c_uint8]
            L.orc_quantize_rows.argtypes = [ctypes.c_int, f32p, vp, i64, i64, ctypes.c_int]
            L.orc_dequantize_row.argtypes = [ctypes.c_int, vp, f32p, i64]
            L.orc_dequantize_row_f64.argtypes = [ctypes.c_int, vp, f64p, i64]
            L.orc_vec_dot_q4_0_q8_0.restype = ctypes.c_float
            L.orc_vec_dot_q4_0_q8_0.argtypes = [i64, vp, vp]
            L.orc_vec_dot_q4_K_q8_K.restype = ctypes.c_float
            L.orc_vec_dot_q4_K_q8_K.argtypes = [i64, vp, vp]
            L.orc_vec_dot_q6_K_q8_K.restype = ctypes.c_float
            L.orc_vec_dot_q6_K_q8_K.argtypes = [i64, vp, vp]
            L.orc_vec_dot_f64.restype = ctypes.c_double
            L.orc_vec_dot_f64.argtypes = [ctypes.c_int, i64, vp, vp]
            L.orc_block_sums_q4_0.argtypes = [i64, vp, vp, vp]
            L.orc_block_sums_q4_K.argtypes = [i64, vp, vp, vp, vp, vp]
            L.orc_block_sums_q6_K.argtypes = [i64, vp, vp, vp, vp]
            L.orc_mul_mat_q8.argtypes = [ctypes.c_int, vp, i64, i64, vp, i64, vp, i64,
                                         f32p, f64p, f64p, ctypes.c_int]
            L.orc_w4a16_pack.argtypes = [vp, vp, i64, i64]
            L.orc_w4a16_unpack.argtypes = [vp, vp, i64, i64]
            L.orc_w4a16_unpack_zeros.argtypes = [vp, vp, i64, i64]
            L.orc_w4a16_matmul.argtypes = [vp, vp, vp, i64, vp, i64, i64, i64, vp, i64,
                                           vp, f64p, f64p, ctypes.c_int]
            L.orc_w4a16_lut_matmul.argtypes = [vp, vp, vp, i64, vp, i64, i64, i64, vp, i64,
                                               vp, f64p, f64p, ctypes.c_int]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# ---------------------------------------------------------------- scalars
def fp32_to_fp16(x: float) -> int:
    return int(lib().orc_fp32_to_fp16(float(x)))


def fp64_to_fp16(x: float) -> int:
    return int(lib().orc_fp64_to_fp16(float(x)))


def fp16_to_fp32(h: int) -> float:
    return float(lib().orc_fp16_to_fp32(int(h)))


def block_bytes(t: int) -> int:
    return int(lib().orc_block_bytes(t))


def row_bytes(t: int, k: int) -> int:
    return BLOCK_BYTES[t] * (k // BLOCK_ELEMS[t])


# ---------------------------------------------------------------- Q4_K scales
def get_scale_min_k4(j: int, scales: np.ndarray):
    s = np.zeros(1, np.uint8)
    m = np.zeros(1, np.uint8)
    sc = _c(scales, np.uint8)
    lib().orc_get_scale_min_k4(j, _ptr(sc), _ptr(s), _ptr(m))
    return int(s[0]), int(m[0])


def set_scale_min_k4(j: int, scales: np.ndarray, s: int, m: int) -> np.ndarray:
    sc = _c(scales, np.uint8).copy()
    lib().orc_set_scale_min_k4(j, _ptr(sc), s, m)
    return sc


# ---------------------------------------------------------------- quantize
def quantize(t: int, x: np.ndarray, nthreads: int = 1) -> np.ndarray:
    """Quantize a [rows, k] fp32 matrix into canonical blocks -> uint8 [rows, row_bytes]."""
    x = _c(x, np.float32)
    if x.ndim == 1:
        x = x[None, :]
    rows, k = x.shape
    assert k % BLOCK_ELEMS[t] == 0
    out = np.zeros((rows, row_bytes(t, k)), np.uint8)
    lib().orc_quantize_rows(t, _ptr(x), _ptr(out), rows, k, nthreads)
    return out


def dequantize(t: int, blocks: np.ndarray, k: int, f64: bool = False) -> np.ndarray:
    b = _c(blocks, np.uint8).reshape(-1, row_bytes(t, k))
    out = np.zeros((b.shape[0], k), np.float64 if f64 else np.float32)
    for r in range(b.shape[0]):
        if f64:
            lib().orc_dequantize_row_f64(t, _ptr(b[r]), _ptr(out[r]), k)
        else:
            lib().orc_dequantize_row(t, _ptr(b[r]), _ptr(out[r]), k)
    return out


# ---------------------------------------------------------------- dots
def vec_dot(wt: int, k: int, w_row: np.ndarray, a_row: np.ndarray) -> float:
    w = _c(w_row, np.uint8)
    a = _c(a_row, np.uint8)
    if wt == Q4_0:
        return float(lib().orc_vec_dot_q4_0_q8_0(k, _ptr(w), _ptr(a)))
    if wt == Q6_K:
        return float(lib().orc_vec_dot_q6_K_q8_K(k, _ptr(w), _ptr(a)))
    return float(lib().orc_vec_dot_q4_K_q8_K(k, _ptr(w), _ptr(a)))


def vec_dot_f64(wt: int, k: int, w_row: np.ndarray, a_row: np.ndarray) -> float:
    w = _c(w_row, np.uint8)
    a = _c(a_row, np.uint8)
    return float(lib().orc_vec_dot_f64(wt, k, _ptr(w), _ptr(a)))


def block_sums(wt: int, k: int, w_row: np.ndarray, a_row: np.ndarray):
    """Per-block integer sums of one (weight row, activation row) pair.

    Q4_0: returns isum [k/32]. Q4_K: returns (S [k/256, 8], isum [k/256], msum [k/256]).
    Q6_K: returns (S [k/256, 16], isum [k/256]).
    """
    w = _c(w_row, np.uint8)
    a = _c(a_row, np.uint8)
    if wt == Q4_0:
        isum = np.zeros(k // 32, np.int32)
        lib().orc_block_sums_q4_0(k, _ptr(w), _ptr(a), _ptr(isum))
        return isum
    if wt == Q6_K:
        S = np.zeros((k // 256, 16), np.int32)
        isum = np.zeros(k // 256, np.int32)
        lib().orc_block_sums_q6_K(k, _ptr(w), _ptr(a), _ptr(S), _ptr(isum))
        return S, isum
    S = np.zeros((k // 256, 8), np.int32)
    isum = np.zeros(k // 256, np.int32)
    msum = np.zeros(k // 256, np.int32)
    lib().orc_block_sums_q4_K(k, _ptr(w), _ptr(a), _ptr(S), _ptr(isum), _ptr(msum))
    return S, isum, msum


def mul_mat_q8(wt: int, W: np.ndarray, N: int, K: int, Xq: np.ndarray, M: int,
               rows=None, nthreads: int = 1, want=("y32", "y64", "den")):
    """Y[m, n] over already-quantized activations; returns dict of [M, nrows] arrays."""
    W = _c(W, np.uint8)
    Xq = _c(Xq, np.uint8)
    r = None if rows is None else _c(rows, np.int64)
    nrows = N if r is None else r.shape[0]
    y32 = np.zeros((M, nrows), np.float32) if "y32" in want else None
    y64 = np.zeros((M, nrows), np.float64) if "y64" in want else None
    den = np.zeros((M, nrows), np.float64) if "den" in want else None
    lib().orc_mul_mat_q8(wt, _ptr(W), N, K, _ptr(Xq), M, _ptr(r), nrows,
                         _ptr(y32), _ptr(y64), _ptr(den), nthreads)
    out = {}
    if y32 is not None:
        out["y32"] = y32
    if y64 is not None:
        out["y64"] = y64
    if den is not None:
        out["den"] = den
    return out


def mul_mat(wt: int, W: np.ndarray, N: int, K: int, X: np.ndarray, rows=None,
            nthreads: int = 1, want=("y32", "y64", "den")):
    """Full method: quantize the fp32 activations X [M, K], then mul_mat_q8."""
    X = _c(X, np.float32)
    M = X.shape[0]
    Xq = quantize(ACT_TYPE[wt], X, nthreads)
    res = mul_mat_q8(wt, W, N, K, Xq, M, rows=rows, nthreads=nthreads, want=want)
    res["xq"] = Xq
    return res


# ---------------------------------------------------------------- W4A16
def w4a16_pack(q: np.ndarray) -> np.ndarray:
    q = _c(q, np.uint8)
    N, K = q.shape
    out = np.zeros((N, K // 8), np.uint32)
    lib().orc_w4a16_pack(_ptr(q), _ptr(out), N, K)
    return out


def w4a16_unpack(qweight: np.ndarray, K: int) -> np.ndarray:
    qw = _c(qweight, np.uint32)
    N = qw.shape[0]
    out = np.zeros((N, K), np.uint8)
    lib().orc_w4a16_unpack(_ptr(qw), _ptr(out), N, K)
    return out


def w4a16_unpack_zeros(zp: np.ndarray, ng: int) -> np.ndarray:
    """Zero points packed 8 per uint32 word like the codes, [N, ceil(ng/8)]
    -> uint8 [N, ng]."""
    w = _c(zp, np.uint32)
    N = w.shape[0]
    assert w.shape[1] == (ng + 7) // 8
    out = np.zeros((N, ng), np.uint8)
    lib().orc_w4a16_unpack_zeros(_ptr(w), _ptr(out), N, ng)
    return out


def w4a16_matmul(qweight, scales16, zeros, G: int, A16, rows=None, nthreads: int = 1):
    """C [M, nrows]: fp16 bits of the exact (fp64) result, the fp64 value and den."""
    qw = _c(qweight, np.uint32)
    s = _c(scales16, np.uint16)
    z = _c(zeros, np.uint8)
    A = _c(A16, np.uint16)
    M, K = A.shape
    N = qw.shape[0]
    r = None if rows is None else _c(rows, np.int64)
    nrows = N if r is None else r.shape[0]
    c16 = np.zeros((M, nrows), np.uint16)
    c64 = np.zeros((M, nrows), np.float64)
    den = np.zeros((M, nrows), np.float64)
    lib().orc_w4a16_matmul(_ptr(qw), _ptr(s), _ptr(z), G, _ptr(A), M, N, K, _ptr(r), nrows,
                           _ptr(c16), _ptr(c64), _ptr(den), nthreads)
    return {"c16": c16, "c64": c64, "den": den}


def w4a16_lut_matmul(qweight, scales16, lut16, G: int, A16, rows=None, nthreads: int = 1):
    """C [M, nrows] with W-hat = s * LUT(q): fp16 bits of the fp64 result, the
    fp64 value and den."""
    qw = _c(qweight, np.uint32)
    s = _c(scales16, np.uint16)
    lut = _c(lut16, np.uint16)
    assert lut.shape == (16,)
    A = _c(A16, np.uint16)
    M, K = A.shape
    N = qw.shape[0]
    r = None if rows is None else _c(rows, np.int64)
    nrows = N if r is None else r.shape[0]
    c16 = np.zeros((M, nrows), np.uint16)
    c64 = np.zeros((M, nrows), np.float64)
    den = np.zeros((M, nrows), np.float64)
    lib().orc_w4a16_lut_matmul(_ptr(qw), _ptr(s), _ptr(lut), G, _ptr(A), M, N, K, _ptr(r), nrows,
                               _ptr(c16), _ptr(c64), _ptr(den), nthreads)
    return {"c16": c16, "c64": c64, "den": den}
