"""The C-ABI boundary on the CPU: libqmm.so loads, exports every entry point
include/qmm.h declares, and its host-side logic (sizes, validation, status
strings) works without a GPU. No compute call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qmm.h")


@pytest.fixture(scope="module")
def lib(built_lib):
    L = ctypes.CDLL(built_lib)
    L.qmm_packed_bytes.restype = ctypes.c_size_t
    L.qmm_packed_bytes.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64]
    L.qmm_workspace_bytes.restype = ctypes.c_size_t
    L.qmm_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64]
    L.qmm_block_bytes.restype = ctypes.c_size_t
    L.qmm_status_string.restype = ctypes.c_char_p
    L.qmm_last_error.restype = ctypes.c_char_p
    return L


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qmm_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), f"libqmm.so does not export {n}"


def test_binding_names_match_header(built_lib):
    import block_quantized_matmul_q4_gb300 as q
    for n in declared_functions():
        assert n in q.EXPORTED and callable(getattr(q, n)), n


def test_block_sizes(lib):
    assert [lib.qmm_block_bytes(t) for t in range(4)] == [18, 144, 34, 292]
    assert [lib.qmm_block_elems(t) for t in range(4)] == [32, 256, 32, 256]
    assert lib.qmm_block_bytes(5) == 210 and lib.qmm_block_elems(5) == 256  # Q6_K
    assert lib.qmm_block_bytes(7) == 0


def test_packed_and_workspace_sizes(lib):
    # rows padded to a multiple of 8, block bytes unchanged by the repack
    assert lib.qmm_packed_bytes(1, 4096, 4096) == 4096 * 16 * 144
    assert lib.qmm_packed_bytes(1, 13, 512) == 16 * 2 * 144
    assert lib.qmm_packed_bytes(0, 256, 1024) == 256 * 32 * 18
    assert lib.qmm_packed_bytes(1, 10, 100) == 0  # K not a multiple of 256
    assert lib.qmm_packed_bytes(3, 10, 256) == 0  # activation type is not a weight type
    assert lib.qmm_packed_bytes(5, 13, 512) == 16 * 2 * 210  # Q6_K: 8-row records of 1680 B
    assert lib.qmm_packed_bytes(5, 8, 300) == 0
    assert lib.qmm_workspace_bytes(5, 40, 4096) >= 40 * 4096 + 40 * 16 * 4 + 40 * 16 * 16 * 2
    ws = lib.qmm_workspace_bytes(1, 16, 4096)
    assert ws >= 16 * 4096 + 16 * 16 * 4 + 16 * 16 * 16 * 2
    assert lib.qmm_workspace_bytes(0, 1, 1000) == 0


def test_validation_without_gpu(lib):
    vp = ctypes.c_void_p
    f = lib.qmm_mul_mat
    f.argtypes = [ctypes.c_int, vp, ctypes.c_int64, ctypes.c_int64, vp, ctypes.c_int64, vp, vp]
    assert f(2, None, 8, 256, None, 1, None, None) == 1          # Q8_0 is not a weight type
    assert f(1, None, 8, 100, None, 1, None, None) == 1          # K % 256 != 0
    assert f(1, None, 8, 256, None, 1, None, None) == 1          # null pointers
    assert f(1, 16, 8, 256, 32, -1, 48, None) == 1                # M < 0
    assert f(1, 8, 8, 256, 32, 1, 48, None) == 1                  # W not 16-byte aligned
    assert f(1, None, 8, 256, None, 0, None, None) == 0           # M == 0 is a no-op
    assert b"multiple" in lib.qmm_last_error() or lib.qmm_last_error() == b""
    g = lib.qmm_quantize_row_q8
    g.argtypes = [ctypes.c_int, vp, vp, ctypes.c_int64, ctypes.c_int64, vp]
    assert g(0, 16, 16, 1, 256, None) == 1                        # Q4_0 is not an activation type
    assert g(3, 16, 16, 1, 255, None) == 1
    assert lib.qmm_status_string(4) == b"QMM_ERR_TIMEOUT"
    assert lib.qmm_status_string(99) == b"QMM_ERR_UNKNOWN"


def test_type_ids_agree(built_lib):
    """The qmm_type values in include/qmm.h, the binding's constants and the
    oracle's type ids name the same formats."""
    import block_quantized_matmul_q4_gb300 as q
    import oracle
    text = open(HEADER).read()
    ids = {n: int(v) for n, v in re.findall(r"\b(QMM_TYPE_[A-Z0-9_]+)\s*=\s*(\d+)", text)}
    assert ids == {"QMM_TYPE_Q4_0": 0, "QMM_TYPE_Q4_K": 1, "QMM_TYPE_Q8_0": 2, "QMM_TYPE_Q8_K": 3,
                   "QMM_TYPE_W4A16": 4, "QMM_TYPE_Q6_K": 5}
    for name, v in ids.items():
        assert getattr(q, name) == v
    for name in ("Q4_0", "Q4_K", "Q8_0", "Q8_K", "Q6_K"):
        assert getattr(oracle, name) == ids["QMM_TYPE_" + name]
        assert oracle.BLOCK_BYTES[getattr(oracle, name)] == ctypes.CDLL(built_lib).qmm_block_bytes(
            ids["QMM_TYPE_" + name])


def test_host_call_bytes(lib):
    """qmm_mul_mat_host's device buffer: X, then Y (each rounded up to 16
    bytes), then the workspace of qmm_mul_mat_ws; 0 for invalid shapes."""
    f = lib.qmm_host_call_bytes
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
    r16 = lambda n: (n + 15) // 16 * 16
    for wt, M, N, K in [(1, 1, 4096, 4096), (0, 3, 40, 4096), (5, 20, 11008, 4096), (1, 1, 5, 256)]:
        assert f(wt, M, N, K) == r16(M * K * 4) + r16(M * N * 4) + lib.qmm_workspace_bytes(wt, M, K)
    assert f(1, 1, 10, 100) == 0  # K not a multiple of 256
    assert f(3, 1, 10, 256) == 0  # not a weight type


def test_repack_overlap_rejected(lib):
    """qmm_repack_weights refuses overlapping canonical and packed buffers
    before it launches anything. (Buffers that only the packed side's tile
    padding would make overlap are accepted: the Q6_K N = 300 case of
    test_gpu_parity.test_mul_mat_host_buffers allocates such a pair.)"""
    f = lib.qmm_repack_weights
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
    src = 1 << 20
    assert f(5, src, src + 16, 300, 2048, None) == 1  # QMM_ERR_ARG
    assert "overlap" in lib.qmm_last_error().decode()


def test_host_call_rejects_unknown_flags(lib):
    """qmm_mul_mat_host checks its flags (only QMM_HOST_MAPPED = 1 exists)
    before any CUDA call."""
    f = lib.qmm_mul_mat_host
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint, ctypes.c_void_p]
    p = 1 << 20
    assert f(1, p, 8, 256, p, 1, p, p, 1 << 30, 2, None) == 1
    assert "flags" in lib.qmm_last_error().decode()
