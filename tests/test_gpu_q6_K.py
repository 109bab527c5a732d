"""GPU parity of the Q6_K path (page 1, "更低的比特: Q6_K 与 Q2_K 的取舍":
6-bit codes in ql/qh, 16 int8 group scales, fp16 d, no min) against the CPU
oracle: the GPU weight quantizer, the repack and the per-group integer sums
bit-exact; mul_mat outputs within |Y - Y_ref| <= 1e-3 sum_k |w_k a_k| of the
oracle's fp64 result on the same quantized operands."""
import numpy as np
import pytest
import torch

import workloads as wl
from test_gpu_parity import check_close, dev, edge_rows, host, run_mul_mat

pytestmark = pytest.mark.gpu

Q6_K = 5


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantized_matmul_q4_gb300 as q
    return q


def weights(seed, N, K):
    return wl.weights(seed, N, K, 0.02, row_offset_std=0.005, outlier_frac=1e-3).numpy()


@pytest.mark.parametrize("N,K", [(13, 512), (64, 4096), (3, 256)])
def test_q6_K_weight_quantizer_bit_exact(q, orc, N, K):
    w = np.concatenate([weights(40, N, K), edge_rows(K, 40)])
    Wq = q.empty_blocks(Q6_K, w.shape[0], K)
    q.qmm_quantize_weights(Q6_K, dev(w), Wq, w.shape[0], K)
    got = host(Wq).reshape(w.shape[0], -1)
    assert np.array_equal(got, orc.quantize(Q6_K, w))


@pytest.mark.parametrize("N,K,M", [(13, 512, 2), (9, 4352, 1), (21, 768, 3), (8, 256, 1)])
def test_q6_K_repack_roundtrip_and_group_sums(q, orc, N, K, M):
    Wc = orc.quantize(Q6_K, weights(41, N, K))
    Xq = orc.quantize(orc.Q8_K, wl.activations(41, M, K).numpy())
    Wp = q.empty_packed(Q6_K, N, K)
    q.qmm_repack_weights(Q6_K, dev(Wc), Wp, N, K)
    back = q.empty_blocks(Q6_K, N, K)
    q.qmm_unrepack_weights(Q6_K, Wp, back, N, K)
    assert np.array_equal(host(back).reshape(N, -1), Wc)
    nsb = K // 256
    out = torch.empty(M * N * nsb * 17, dtype=torch.int32, device="cuda")
    q.qmm_debug_block_sums(Q6_K, Wp, N, K, dev(Xq), M, out)
    got = host(out).reshape(M, N, nsb, 17)
    for m in range(M):
        for n in range(N):
            S, isum = orc.block_sums(Q6_K, K, Wc[n], Xq[m])
            assert np.array_equal(got[m, n, :, :16], S)
            assert np.array_equal(got[m, n, :, 16], isum)


@pytest.mark.parametrize("N,K,M", [
    (256, 1024, 1),       # fused quantizer, one launch
    (13, 512, 3), (37, 4352, 5), (64, 4096, 16),
    (16, 1024, 17),       # two 16-token launches
    (40, 2304, 40),       # three launches on the planar workspace
    (8, 256, 1), (10000, 256, 2),   # many tile pairs per CTA
    (24, 65536, 2)])      # activations read from global memory in place
def test_q6_K_mul_mat_against_oracle(q, orc, N, K, M):
    Wc = orc.quantize(Q6_K, weights(42, N, K), nthreads=orc.default_threads())
    x = wl.activations(42, M, K).numpy()
    y = run_mul_mat(q, Q6_K, Wc, N, K, x)
    ref = orc.mul_mat(Q6_K, Wc, N, K, x, nthreads=orc.default_threads())
    check_close(y, ref["y64"], ref["den"], f"Q6_K N={N} K={K} M={M}")
    check_close(ref["y32"], ref["y64"], ref["den"], "oracle fp32")


def test_q6_K_4096_square(q, orc):
    """The 4096 x 4096 decode shape, every output element."""
    N = K = 4096
    Wc = orc.quantize(Q6_K, weights(43, N, K), nthreads=orc.default_threads())
    for M in (1, 4):
        x = wl.activations(43, M, K).numpy()
        y = run_mul_mat(q, Q6_K, Wc, N, K, x)
        ref = orc.mul_mat(Q6_K, Wc, N, K, x, nthreads=orc.default_threads())
        check_close(y, ref["y64"], ref["den"], f"Q6_K 4096^2 M={M}")


def test_q6_K_edge_inputs(q, orc):
    K = 512
    w = edge_rows(K, 44)
    x = np.concatenate([edge_rows(K, 45), wl.activations(45, 2, K).numpy()])
    Wc = orc.quantize(Q6_K, w)
    y = run_mul_mat(q, Q6_K, Wc, w.shape[0], K, x)
    ref = orc.mul_mat(Q6_K, Wc, w.shape[0], K, x)
    check_close(y, ref["y64"], ref["den"], "Q6_K edge rows")


@pytest.mark.parametrize("N,K,M", [(40, 4096, 1), (24, 8192, 8), (200, 1536, 40)])
def test_q6_K_prepared_ws_static_q8(q, orc, N, K, M):
    """Every entry point on Q6_K weights: prepared (workspace read twice),
    one-call with a workspace, the allocation-free variant and canonical Q8_K
    input all give the same bits as qmm_mul_mat."""
    Wc = orc.quantize(Q6_K, weights(46, N, K))
    x = wl.activations(46, M, K).numpy()
    Wp = q.empty_packed(Q6_K, N, K)
    q.qmm_repack_weights(Q6_K, dev(Wc), Wp, N, K)
    X = dev(x)
    Y0 = torch.empty(M, N, device="cuda")
    q.qmm_mul_mat(Q6_K, Wp, N, K, X, M, Y0)
    ref = orc.mul_mat(Q6_K, Wc, N, K, x, nthreads=orc.default_threads())
    check_close(host(Y0), ref["y64"], ref["den"], f"Q6_K mul_mat M={M}")
    ws_bytes = q.qmm_workspace_bytes(Q6_K, M, K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    q.qmm_quantize_activations(Q6_K, X, M, K, ws, ws_bytes)
    Y1 = torch.empty(M, N, device="cuda")
    Y2 = torch.empty(M, N, device="cuda")
    q.qmm_mul_mat_prepared(Q6_K, Wp, N, K, ws, ws_bytes, M, Y1)
    q.qmm_mul_mat_prepared(Q6_K, Wp, N, K, ws, ws_bytes, M, Y2)
    assert torch.equal(Y1, Y2)
    check_close(host(Y1), ref["y64"], ref["den"], f"Q6_K prepared M={M}")
    Y3 = torch.empty(M, N, device="cuda")
    q.qmm_mul_mat_ws(Q6_K, Wp, N, K, X, M, Y3, ws, ws_bytes)
    check_close(host(Y3), ref["y64"], ref["den"], f"Q6_K ws M={M}")
    Y4 = torch.empty(M, N, device="cuda")
    q.qmm_mul_mat_static(Q6_K, Wp, N, K, X, M, Y4)
    if M <= 8:
        assert torch.equal(Y4, Y3)
    else:  # the static variant stays on the scalar GEMV; the others run the GEMM
        check_close(host(Y4), ref["y64"], ref["den"], f"Q6_K static M={M}")
    Xq = q.empty_blocks(orc.Q8_K, M, K)
    q.qmm_quantize_row_q8(orc.Q8_K, X, Xq, M, K)
    Y5 = torch.empty(M, N, device="cuda")
    q.qmm_mul_mat_q8(Q6_K, Wp, N, K, Xq, M, Y5)
    assert torch.equal(Y5, Y3), "mul_mat_q8 differs from the workspace path"
    q.qmm_check_device_error()


@pytest.mark.parametrize("N,K,M", [(128, 256, 17), (200, 512, 300), (136, 2304, 129),
                                   (1000, 4096, 300)])   # stream-K: tiles split across CTAs
def test_q6_K_prefill_gemm(q, orc, N, K, M):
    """More than 16 tokens: the fp16-operand tcgen05 GEMM on the Q6_K records
    (weights fp16(fp16(d s_j) q), activations fp16(d_a y)), within R16."""
    Wc = orc.quantize(Q6_K, weights(49, N, K), nthreads=orc.default_threads())
    x = wl.activations(49, M, K).numpy()
    y = run_mul_mat(q, Q6_K, Wc, N, K, x)
    ref = orc.mul_mat(Q6_K, Wc, N, K, x, nthreads=orc.default_threads())
    check_close(y, ref["y64"], ref["den"], f"Q6_K prefill N={N} K={K} M={M}")
    q.qmm_check_device_error()


@pytest.mark.parametrize("Ns,K,M", [((96, 40, 37), 4096, 1), ((64, 0, 24), 2304, 5),
                                    ((200, 56), 1024, 40)])
def test_q6_K_mul_mat_multi(q, orc, Ns, K, M):
    x = wl.activations(47, M, K).numpy()
    X = dev(x)
    Wcs, Wps, Ys = [], [], []
    for i, N in enumerate(Ns):
        Wc = orc.quantize(Q6_K, weights(48 + i, max(N, 1), K))[:N]
        Wp = q.empty_packed(Q6_K, max(N, 1), K)
        if N:
            q.qmm_repack_weights(Q6_K, dev(Wc), Wp, N, K)
        Wcs.append(Wc)
        Wps.append(Wp)
        Ys.append(torch.full((max(M * N, 1),), float("nan"), device="cuda"))
    q.qmm_mul_mat_multi(Q6_K, Wps, list(Ns), K, X, M, Ys)
    for N, Wc, Wp, Y in zip(Ns, Wcs, Wps, Ys):
        if N == 0:
            assert torch.isnan(Y).all()
            continue
        Y1 = torch.empty(M * N, device="cuda")
        q.qmm_mul_mat(Q6_K, Wp, N, K, X, M, Y1)
        assert torch.equal(Y, Y1), f"N={N}: multi differs from a single call"
        ref = orc.mul_mat(Q6_K, Wc, N, K, x, nthreads=orc.default_threads())
        check_close(host(Y).reshape(M, N), ref["y64"], ref["den"], f"Q6_K multi N={N}")
    q.qmm_check_device_error()
