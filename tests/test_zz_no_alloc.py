"""qmm_mul_mat_static, the entry point for callers that cannot allocate device
memory (a serving loop with a frozen allocator, a runtime that gives the
library no allocator, a step that must never block in cudaMalloc). It keeps
its activation scratch in a fixed array inside libqmm. Through the C ABI,
several calls in a row share that array, each in a different layout than the
one before (the tensor-core GEMVs' activation images, the Q8_K and Q8_0
planar codes of the one-token GEMV, a call split into two launches); each result is checked
against the oracle's fp64 result and against qmm_mul_mat's (the existing
entry point), within the same 1e-3 * sum|w a| bound the other GPU tests use,
and bit for bit against qmm_mul_mat_ws where that call runs the same
kernels. Oversized requests are refused. Collected last so that a failure
here does not stop the rest of a stop-at-first-failure run."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu
TOL = 1e-3


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantized_matmul_q4_gb300 as q
    return q


def static_fn(q):
    lib = ctypes.CDLL(q.LIB_PATH)
    f = lib.qmm_mul_mat_static
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    f.argtypes = [ctypes.c_int, vp, i64, i64, vp, i64, vp, vp]
    f.restype = ctypes.c_int
    return f


def check_rel(y, ref, den, what):
    y = np.asarray(y, dtype=np.float64)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y - ref)
    worst = np.max(np.where(den > 0, err / np.where(den > 0, den, 1.0), 0.0))
    assert np.all(err <= TOL * den), f"{what}: worst normalised error {worst:.3e}"


def test_static_scratch_matches_oracle_and_mul_mat(q, orc):
    f = static_fn(q)
    stream = torch.cuda.current_stream().cuda_stream
    Q4_0, Q4_K, Q6_K = q.QMM_TYPE_Q4_0, q.QMM_TYPE_Q4_K, q.QMM_TYPE_Q6_K
    # (type, N, K, M, seed, same kernels as qmm_mul_mat_ws): in call order
    cases = [(Q4_K, 72, 4096, 16, 21, True),    # activation images, one launch
             (Q4_0, 40, 4096, 3, 22, True),     # Q4_0 tensor-core image
             (Q4_K, 72, 4096, 20, 23, False),   # images, two launches (16 + 4); mul_mat: GEMM
             (Q6_K, 40, 2048, 5, 24, True),     # Q6_K tensor-core image
             (Q6_K, 40, 16384, 1, 25, True),    # Q8_K planar (one token above the fused limit)
             (Q4_0, 24, 16384, 1, 26, True),    # Q8_0 planar
             (Q4_K, 72, 4096, 16, 21, True)]    # the first call again, after the others
    outs = []
    for wt, N, K, M, seed, same in cases:
        w = wl.weights(seed, N, K, 0.02, row_offset_std=0.0 if wt == Q4_0 else 0.005).numpy()
        Wc = orc.quantize(wt, w)
        Wp = q.empty_packed(wt, N, K)
        q.qmm_repack_weights(wt, torch.from_numpy(Wc).cuda(), Wp, N, K)
        x = wl.activations(seed, M, K).numpy()
        X = torch.from_numpy(x).cuda()
        Y = torch.full((M, N), float("nan"), device="cuda")
        st = f(wt, Wp.data_ptr(), N, K, X.data_ptr(), M, Y.data_ptr(), stream)
        assert st == 0, q.qmm_last_error()
        outs.append((wt, Wc, Wp, N, K, M, x, X, Y, same))
    q.qmm_check_device_error()
    for wt, Wc, Wp, N, K, M, x, X, Y, same in outs:
        what = f"type {wt} N={N} K={K} M={M}"
        ref = orc.mul_mat(wt, Wc, N, K, x, nthreads=orc.default_threads())
        y = Y.cpu().numpy()
        check_rel(y, ref["y64"], ref["den"], what + " vs oracle")
        Yref = torch.empty(M, N, device="cuda")
        q.qmm_mul_mat(wt, Wp, N, K, X, M, Yref)
        q.qmm_check_device_error()
        err = np.abs(y.astype(np.float64) - Yref.cpu().numpy())
        assert np.all(err <= TOL * ref["den"]), what + " vs qmm_mul_mat"
        if same:
            ws_bytes = q.qmm_workspace_bytes(wt, M, K)
            ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
            Yws = torch.empty(M, N, device="cuda")
            q.qmm_mul_mat_ws(wt, Wp, N, K, X, M, Yws, ws, ws_bytes)
            q.qmm_check_device_error()
            assert torch.equal(Y, Yws), what + " vs qmm_mul_mat_ws (same kernels)"
    # the repeated call gives the same bits as the first
    assert torch.equal(outs[0][8], outs[-1][8])


def test_static_scratch_refuses_oversized(q):
    f = static_fn(q)
    K, M = 4096, 1024  # 4.7 MB of quantized activations > 4 MiB of scratch
    buf = torch.empty(16, device="cuda")
    st = f(q.QMM_TYPE_Q4_K, buf.data_ptr(), 8, K, buf.data_ptr(), M, buf.data_ptr(),
           torch.cuda.current_stream().cuda_stream)
    assert st == 6  # QMM_ERR_WORKSPACE, nothing launched
    assert "scratch" in q.qmm_last_error()
    torch.cuda.synchronize()
