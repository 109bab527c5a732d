"""qmm_mul_mat_static, the entry point for callers that cannot allocate device
memory (a serving loop with a frozen allocator, a runtime that gives the
library no allocator, a step that must never block in cudaMalloc). It keeps
its activation scratch in a fixed array inside libqmm; this checks, through
the C ABI, that two calls in a row give what qmm_mul_mat gives, within the
same 1e-3 * sum|w a| bound the other GPU tests use, and that oversized
requests are refused. Collected last so that a failure here does not stop the
rest of a stop-at-first-failure run."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantized_matmul_q4_gb300 as q
    return q


def setup(q, orc, wt, N, K, seed):
    w = wl.weights(seed, N, K, 0.02, row_offset_std=0.005).numpy()
    Wc = orc.quantize(wt, w)
    Wp = q.empty_packed(wt, N, K)
    q.qmm_repack_weights(wt, torch.from_numpy(Wc).cuda(), Wp, N, K)
    return Wc, Wp


def test_static_scratch_matches_mul_mat(q, orc):
    lib = ctypes.CDLL(q.LIB_PATH)
    f = lib.qmm_mul_mat_static
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    f.argtypes = [ctypes.c_int, vp, i64, i64, vp, i64, vp, vp]
    f.restype = ctypes.c_int
    stream = torch.cuda.current_stream().cuda_stream
    # two calls in a row, of different shapes and types, sharing the scratch
    cases = [(q.QMM_TYPE_Q4_K, 72, 4096, 16, 21), (q.QMM_TYPE_Q4_0, 40, 1024, 3, 22)]
    outs = []
    for wt, N, K, M, seed in cases:
        Wc, Wp = setup(q, orc, wt, N, K, seed)
        x = wl.activations(seed, M, K).numpy()
        X = torch.from_numpy(x).cuda()
        Y = torch.full((M, N), float("nan"), device="cuda")
        st = f(wt, Wp.data_ptr(), N, K, X.data_ptr(), M, Y.data_ptr(), stream)
        assert st == 0, q.qmm_last_error()
        outs.append((wt, Wc, Wp, N, K, M, x, X, Y))
    for wt, Wc, Wp, N, K, M, x, X, Y in outs:
        Yref = torch.empty(M, N, device="cuda")
        q.qmm_mul_mat(wt, Wp, N, K, X, M, Yref)
        torch.cuda.synchronize()
        den = orc.mul_mat(wt, Wc, N, K, x, want=("den",))["den"]
        err = np.abs(Y.cpu().numpy().astype(np.float64) - Yref.cpu().numpy())
        assert np.all(np.isfinite(Y.cpu().numpy()))
        assert np.all(err <= 1e-3 * den + 1e-30), f"type {wt}: worst {np.max(err / den):.3e}"
    q.qmm_check_device_error()


def test_static_scratch_refuses_oversized(q):
    lib = ctypes.CDLL(q.LIB_PATH)
    f = lib.qmm_mul_mat_static
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    f.argtypes = [ctypes.c_int, vp, i64, i64, vp, i64, vp, vp]
    f.restype = ctypes.c_int
    K, M = 4096, 1024  # 4.7 MB of quantized activations > 4 MiB of scratch
    assert q.qmm_workspace_bytes(q.QMM_TYPE_Q4_K, M, K) > 4 << 20
    buf = torch.empty(16, device="cuda")
    st = f(q.QMM_TYPE_Q4_K, buf.data_ptr(), 8, K, buf.data_ptr(), M, buf.data_ptr(),
           torch.cuda.current_stream().cuda_stream)
    assert st == 6  # QMM_ERR_WORKSPACE, nothing launched
    assert "scratch" in q.qmm_last_error()
    torch.cuda.synchronize()
