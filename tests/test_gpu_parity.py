"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bar (from the method's own contract): quantized blocks, the repack round trip
and per-block integer sums are bit-exact; fp32 outputs satisfy
|Y_gpu - Y_ref| <= 1e-3 * sum_k |w_k a_k| element by element, with Y_ref the
oracle's fp64 result on the same quantized operands.
"""
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


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def gpu_quantize_q8(q, vt, x):
    M, K = x.shape
    X = dev(x.astype(np.float32))
    Xq = q.empty_blocks(vt, M, K)
    q.qmm_quantize_row_q8(vt, X, Xq, M, K)
    return host(Xq).reshape(M, -1)


def gpu_quantize_w(q, wt, w):
    N, K = w.shape
    Wq = q.empty_blocks(wt, N, K)
    q.qmm_quantize_weights(wt, dev(w.astype(np.float32)), Wq, N, K)
    return Wq


def edge_rows(K, seed):
    rows = [np.zeros(K), np.full(K, 0.37), np.full(K, -2.5),
            wl.normal_flat(seed, 90, K).numpy() * 1e-30,
            wl.normal_flat(seed, 91, K).numpy() * 1e4,
            -np.abs(wl.normal_flat(seed, 92, K).numpy()),
            np.where(np.arange(K) % 3 == 0, -0.0, 0.0)]
    spike = np.zeros(K)
    spike[K // 3] = -5.0
    rows.append(spike)
    return np.stack(rows).astype(np.float32)


def check_close(y, ref, den, what):
    """Relative bar with no absolute slack: where sum_k |w_k a_k| is 0 the
    output must be exactly 0."""
    err = np.abs(y.astype(np.float64) - ref)
    bad = err > TOL * den
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    worst = np.max(np.where(den > 0, err / np.where(den > 0, den, 1.0), 0.0))
    assert not bad.any(), f"{what}: {bad.sum()} outputs off; worst normalised error {worst:.3e}"


# ------------------------------------------------------------------ quantizers
@pytest.mark.parametrize("vt,M,K", [(2, 1, 1024), (2, 5, 96), (2, 16, 4096),
                                    (3, 1, 256), (3, 3, 4352), (3, 17, 4096)])
def test_activation_quantizer_bit_exact(q, orc, vt, M, K):
    x = wl.activations(7, M, K, hot_frac=0.01).numpy()
    x = np.concatenate([x, edge_rows(K, 7)])
    got = gpu_quantize_q8(q, vt, x)
    assert np.array_equal(got, orc.quantize(vt, x))


@pytest.mark.parametrize("wt,N,K", [(0, 256, 1024), (0, 13, 96), (1, 13, 512), (1, 64, 4096)])
def test_weight_quantizer_bit_exact(q, orc, wt, N, K):
    w = wl.weights(8, N, K, 0.02, row_offset_std=0.005, outlier_frac=1e-3).numpy()
    w = np.concatenate([w, edge_rows(K, 8)])
    got = host(gpu_quantize_w(q, wt, w)).reshape(w.shape[0], -1)
    assert np.array_equal(got, orc.quantize(wt, w))


# ------------------------------------------------------------------ layout + sums
@pytest.mark.parametrize("wt,N,K,M", [(0, 13, 96, 3), (0, 21, 4160, 2), (1, 13, 512, 2),
                                      (1, 9, 4352, 1)])
def test_repack_roundtrip_and_block_sums(q, orc, wt, N, K, M):
    w = wl.weights(9, N, K, 0.02, row_offset_std=0.005).numpy()
    x = wl.activations(9, M, K).numpy()
    Wc = orc.quantize(wt, w)
    Xq = orc.quantize(orc.ACT_TYPE[wt], x)
    Wp = q.empty_packed(wt, N, K)
    q.qmm_repack_weights(wt, dev(Wc), Wp, N, K)
    back = q.empty_blocks(wt, N, K)
    q.qmm_unrepack_weights(wt, Wp, back, N, K)
    assert np.array_equal(host(back).reshape(N, -1), Wc)
    per = 10 if wt == 1 else 1
    nblk = K // (256 if wt == 1 else 32)
    out = torch.empty(M * N * nblk * per, dtype=torch.int32, device="cuda")
    q.qmm_debug_block_sums(wt, Wp, N, K, dev(Xq), M, out)
    got = host(out).reshape(M, N, nblk, per)
    for m in range(M):
        for n in range(N):
            if wt == 0:
                assert np.array_equal(got[m, n, :, 0], orc.block_sums(0, K, Wc[n], Xq[m]))
            else:
                S, isum, msum = orc.block_sums(1, K, Wc[n], Xq[m])
                assert np.array_equal(got[m, n, :, :8], S)
                assert np.array_equal(got[m, n, :, 8], isum)
                assert np.array_equal(got[m, n, :, 9], msum)


# ------------------------------------------------------------------ mul_mat
def run_mul_mat(q, wt, Wc, N, K, x, guard=64):
    """qmm_mul_mat on canonical blocks Wc and fp32 x; returns Y [M, N] and
    checks that the guard words after Y are untouched."""
    M = x.shape[0]
    Wp = q.empty_packed(wt, N, K)
    q.qmm_repack_weights(wt, dev(Wc) if isinstance(Wc, np.ndarray) else Wc, Wp, N, K)
    Y = torch.full((M * N + guard,), float("nan"), dtype=torch.float32, device="cuda")
    Y[M * N:] = 12345.0
    q.qmm_mul_mat(wt, Wp, N, K, dev(x.astype(np.float32)), M, Y)
    y = host(Y)
    assert np.all(y[M * N:] == 12345.0), "write past the end of Y"
    return y[:M * N].reshape(M, N)


@pytest.mark.parametrize("wt,N,K,M", [
    (0, 256, 1024, 1),    # Q4_0 x Q8_0 GEMV, 256 x 1024, M = 1
    (0, 13, 96, 3), (0, 37, 4160, 5), (0, 64, 1024, 16), (0, 24, 512, 33),
    (1, 13, 512, 1), (1, 37, 4352, 5), (1, 64, 4096, 16), (1, 16, 1024, 17), (1, 8, 256, 1)])
def test_mul_mat_against_oracle(q, orc, wt, N, K, M):
    w = wl.weights(10, N, K, 0.02, row_offset_std=0.005 if wt == 1 else 0.0).numpy()
    x = wl.activations(10, M, K).numpy()
    Wc = orc.quantize(wt, w)
    y = run_mul_mat(q, wt, Wc, N, K, x)
    ref = orc.mul_mat(wt, Wc, N, K, x, nthreads=orc.default_threads())
    check_close(y, ref["y64"], ref["den"], f"wt={wt} N={N} K={K} M={M}")
    # the fp32 oracle itself sits inside the same bound
    check_close(ref["y32"], ref["y64"], ref["den"], "oracle fp32")


@pytest.mark.parametrize("wt,N,K,M", [(1, 40, 4096, 1), (1, 40, 4096, 4), (1, 24, 8192, 8),
                                      (1, 16, 4096, 16), (0, 40, 1024, 1), (0, 24, 4096, 16),
                                      (1, 200, 4096, 40), (0, 136, 8192, 33)])  # prefill GEMMs
def test_mul_mat_prepared(q, orc, wt, N, K, M):
    """The two halves (quantize into a workspace, GEMV or GEMM on it):
    activations bulk-copied into shared memory when they fit, read in place
    otherwise; the prefill GEMMs take stream-K scratch of their own."""
    w = wl.weights(13, N, K, 0.02, row_offset_std=0.005).numpy()
    x = wl.activations(13, M, K).numpy()
    Wc = orc.quantize(wt, w)
    Wp = q.empty_packed(wt, N, K)
    q.qmm_repack_weights(wt, dev(Wc), Wp, N, K)
    ws_bytes = q.qmm_workspace_bytes(wt, M, K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    q.qmm_quantize_activations(wt, dev(x), M, K, ws, ws_bytes)
    Y1 = torch.empty(M, N, device="cuda")
    Y2 = torch.empty(M, N, device="cuda")
    q.qmm_mul_mat_prepared(wt, Wp, N, K, ws, ws_bytes, M, Y1)
    q.qmm_mul_mat_prepared(wt, Wp, N, K, ws, ws_bytes, M, Y2)  # workspace is read-only
    ref = orc.mul_mat(wt, Wc, N, K, x)
    check_close(host(Y1), ref["y64"], ref["den"], f"prepared wt={wt} K={K} M={M}")
    assert torch.equal(Y1, Y2)
    # the one-call path gives the same codes, so the same fp32 sums per row
    Y3 = torch.empty(M, N, device="cuda")
    q.qmm_mul_mat_ws(wt, Wp, N, K, dev(x), M, Y3, ws, ws_bytes)
    check_close(host(Y3), ref["y64"], ref["den"], f"one-call wt={wt} K={K} M={M}")


@pytest.mark.parametrize("N,K,M", [
    (10000, 256, 3),     # 625 tile pairs: several pairs per CTA
    (8, 2304, 9),        # one tile (no second tile in the pair), 9 super-blocks, two n8 token tiles
    (40, 4096, 2), (200, 1536, 16), (72, 8192, 12),
    (24, 65536, 3),      # one token per launch fits shared memory: three launches, planar workspace
    (8, 1048576, 2)])    # no token fits: the scalar GEMV reads the workspace in place
def test_q4_K_decode_tensor_core_shapes(q, orc, N, K, M):
    """Q4_K decode with M >= 2 runs on mma.sync (integer-valued fp16
    operands); shapes that exercise its work split, token tiles, launch
    chunking and the fallback."""
    w = wl.weights(14, N, K, 0.02, row_offset_std=0.005).numpy()
    x = wl.activations(14, M, K).numpy()
    Wc = orc.quantize(1, w, nthreads=orc.default_threads())
    y = run_mul_mat(q, 1, Wc, N, K, x)
    ref = orc.mul_mat(1, Wc, N, K, x, nthreads=orc.default_threads())
    check_close(y, ref["y64"], ref["den"], f"N={N} K={K} M={M}")


def test_mul_mat_edge_inputs(q, orc):
    for wt, K in ((0, 256), (1, 256)):
        w = edge_rows(K, 11)
        x = np.concatenate([edge_rows(K, 12), wl.activations(12, 2, K).numpy()])
        N = w.shape[0]
        Wc = orc.quantize(wt, w)
        y = run_mul_mat(q, wt, Wc, N, K, x)
        ref = orc.mul_mat(wt, Wc, N, K, x)
        check_close(y, ref["y64"], ref["den"], f"edge wt={wt}")
        assert np.all(y[:, 0] == 0) and np.all(y[0, :] == 0)  # zero weights / activations


def test_mul_mat_empty_and_workspace_errors(q):
    Wp = q.empty_packed(1, 8, 256)
    Y = torch.zeros(8, device="cuda")
    X = torch.zeros(1, 256, device="cuda")
    q.qmm_mul_mat(1, Wp, 8, 256, X, 0, Y)  # M == 0: nothing to do
    with pytest.raises(q.QmmError) as e:
        q.qmm_mul_mat_ws(1, Wp, 8, 256, X, 1, Y, torch.empty(16, dtype=torch.uint8, device="cuda"), 16)
    assert e.value.status == 6
    with pytest.raises(q.QmmError) as e:
        q.qmm_mul_mat(3, Wp, 8, 256, X, 1, Y)
    assert e.value.status == 1
    q.qmm_check_device_error()


# ------------------------------------------------------------------ full sizes
@pytest.mark.parametrize("M", wl.GEMV_Q4_K_M_SWEEP)
def test_q4_K_4096_full_size(q, orc, M):
    """Q4_K x Q8_K GEMV, N = K = 4096, every output of the M sweep."""
    L = wl.GEMV_Q4_K_4096
    w = wl.weights(0, L.N, L.K, L.wstd, row_offset_std=L.row_offset_std).numpy()
    x = wl.activations(0, M, L.K).numpy()
    Wc = orc.quantize(1, w, nthreads=orc.default_threads())
    y = run_mul_mat(q, 1, Wc, L.N, L.K, x)
    ref = orc.mul_mat(1, Wc, L.N, L.K, x, nthreads=orc.default_threads())
    check_close(y, ref["y64"], ref["den"], f"4096x4096 M={M}")


def test_q4_K_4096_graph_launch(q, orc):
    """The launch configuration of the benchmark: quantizer + GEMV with a
    caller workspace, captured once in a CUDA graph and replayed."""
    L = wl.GEMV_Q4_K_4096
    w = wl.weights(0, L.N, L.K, L.wstd, row_offset_std=L.row_offset_std, device="cuda")
    x = wl.activations(0, 1, L.K, device="cuda")
    Wq = q.empty_blocks(1, L.N, L.K)
    q.qmm_quantize_weights(1, w, Wq, L.N, L.K)
    Wp = q.empty_packed(1, L.N, L.K)
    q.qmm_repack_weights(1, Wq, Wp, L.N, L.K)
    ws_bytes = q.qmm_workspace_bytes(1, 1, L.K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    Y = torch.zeros(L.N, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    q.qmm_mul_mat_ws(1, Wp, L.N, L.K, x, 1, Y, ws, ws_bytes, s)  # warm-up before capture
    torch.cuda.synchronize()
    Y.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        q.qmm_mul_mat_ws(1, Wp, L.N, L.K, x, 1, Y, ws, ws_bytes)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    rows = np.r_[0:8, 1000:1008, L.N - 8:L.N]
    assert torch.isfinite(Y).all()
    Wc = host(Wq).reshape(L.N, -1)
    assert np.array_equal(Wc[rows], orc.quantize(1, w[torch.as_tensor(rows, device="cuda")].cpu().numpy()))
    ref = orc.mul_mat(1, Wc, L.N, L.K, x.cpu().numpy(), rows=rows)
    check_close(host(Y)[rows][None, :], ref["y64"], ref["den"], "graph replay")


def test_70B_layer_sampled_rows(q, orc):
    """70B-shaped decode layer (7 Q4_K projections, M = 1): weights generated
    and quantized on the GPU at full size; sampled rows checked bit-exact
    (blocks) and within tolerance (outputs) against the oracle, which
    quantizes those rows itself from the same fp32 inputs."""
    for i, L in enumerate(wl.LAYER_70B):
        w = wl.weights(100 + i, L.N, L.K, L.wstd, outlier_frac=L.outlier_frac, device="cuda")
        x = wl.activations(100 + i, 1, L.K, hot_frac=wl.LAYER_70B_HOT_FRAC, device="cuda")
        Wq = q.empty_blocks(1, L.N, L.K)
        q.qmm_quantize_weights(1, w, Wq, L.N, L.K)
        Wp = q.empty_packed(1, L.N, L.K)
        q.qmm_repack_weights(1, Wq, Wp, L.N, L.K)
        del Wq
        Y = torch.empty(L.N, device="cuda")
        q.qmm_mul_mat(1, Wp, L.N, L.K, x, 1, Y)
        rows = np.unique(np.r_[0:4, L.N - 4:L.N, np.linspace(0, L.N - 1, 40).astype(np.int64)])
        w_rows = w[torch.as_tensor(rows, device="cuda")].cpu().numpy()
        Wc_rows = orc.quantize(1, w_rows)
        back = q.empty_blocks(1, L.N, L.K)
        q.qmm_unrepack_weights(1, Wp, back, L.N, L.K)
        assert np.array_equal(host(back).reshape(L.N, -1)[rows], Wc_rows), L.name
        ref = orc.mul_mat(1, Wc_rows, len(rows), L.K, x.cpu().numpy())
        check_close(host(Y)[rows][None, :], ref["y64"], ref["den"], L.name)
        del w, Wp, back
        torch.cuda.empty_cache()


# ------------------------------------------------------------------ several projections, one launch
@pytest.mark.parametrize("wt,Ns,K,M", [
    (1, (96, 40, 37), 4096, 1),        # scalar GEMV, quantizer fused
    (1, (96, 40, 37), 4096, 2),        # tensor-core GEMV, quantizer fused
    (1, (200, 16, 8, 56), 2304, 5),    # tensor-core GEMV on the activation image
    (1, (64, 0, 24), 8192, 1),         # a matrix with no rows is skipped
    (0, (64, 40, 13), 1024, 1), (0, (64, 40), 4160, 3),
    (1, (48, 32), 1024, 40), (0, (40, 24), 1024, 33),  # prefill GEMM per matrix
    (1, (1000, 300), 4096, 300), (0, (1000, 300), 2048, 200)])  # ... with split tiles
def test_mul_mat_multi(q, orc, wt, Ns, K, M):
    """qmm_mul_mat_multi: Y_i = X W_i^T for all i from one quantization of X
    (and one decode launch); each Y_i equals a qmm_mul_mat call bit for bit
    and the oracle within tolerance."""
    x = wl.activations(15, M, K).numpy()
    X = dev(x)
    Wcs, Wps, Ys = [], [], []
    for i, N in enumerate(Ns):
        w = wl.weights(30 + i, max(N, 1), K, 0.02, row_offset_std=0.005 if wt == 1 else 0.0).numpy()[:N]
        Wc = orc.quantize(wt, w) if N else np.zeros((0, K // (256 if wt == 1 else 32) * (144 if wt == 1 else 18)), np.uint8)
        Wp = q.empty_packed(wt, max(N, 1), K)
        if N:
            q.qmm_repack_weights(wt, dev(Wc), Wp, N, K)
        Wcs.append(Wc)
        Wps.append(Wp)
        Ys.append(torch.full((max(M * N, 1),), float("nan"), device="cuda"))
    q.qmm_mul_mat_multi(wt, Wps, list(Ns), K, X, M, Ys)
    for N, Wc, Wp, Y in zip(Ns, Wcs, Wps, Ys):
        if N == 0:
            assert torch.isnan(Y).all()  # untouched
            continue
        Y1 = torch.empty(M * N, device="cuda")
        q.qmm_mul_mat(wt, Wp, N, K, X, M, Y1)
        assert torch.equal(Y, Y1), f"N={N}: multi differs from a single call"
        ref = orc.mul_mat(wt, Wc, N, K, x, nthreads=orc.default_threads())
        check_close(host(Y).reshape(M, N), ref["y64"], ref["den"], f"multi wt={wt} N={N} M={M}")
    with pytest.raises(q.QmmError) as e:
        q.qmm_mul_mat_multi(wt, Wps * 5, list(Ns) * 5, K, X, M, Ys * 5)  # more than 8
    assert e.value.status == 1
    q.qmm_check_device_error()


# ------------------------------------------------------------------ canonical Q8 input
@pytest.mark.parametrize("wt,N,K,M", [(1, 40, 4096, 1), (1, 37, 2304, 2), (1, 64, 4096, 7),
                                      (1, 24, 65536, 2), (1, 48, 1024, 33), (0, 40, 1024, 1),
                                      (0, 13, 4160, 5), (0, 40, 1024, 40)])
def test_mul_mat_q8(q, orc, wt, N, K, M):
    """qmm_mul_mat_q8 on the canonical blocks of qmm_quantize_row_q8 equals
    qmm_mul_mat on the fp32 input bit for bit (same codes, scales and sums,
    same kernels), and so the oracle within tolerance; blocks written by the
    oracle itself give the same result."""
    vt = 3 if wt == 1 else 2
    w = wl.weights(16, N, K, 0.02, row_offset_std=0.005 if wt == 1 else 0.0).numpy()
    x = wl.activations(16, M, K).numpy()
    Wc = orc.quantize(wt, w)
    Wp = q.empty_packed(wt, N, K)
    q.qmm_repack_weights(wt, dev(Wc), Wp, N, K)
    X = dev(x)
    Xq = q.empty_blocks(vt, M, K)
    q.qmm_quantize_row_q8(vt, X, Xq, M, K)
    Y = torch.full((M, N), float("nan"), device="cuda")
    q.qmm_mul_mat_q8(wt, Wp, N, K, Xq, M, Y)
    Yref = torch.empty(M, N, device="cuda")
    q.qmm_mul_mat(wt, Wp, N, K, X, M, Yref)
    assert torch.equal(Y, Yref), "mul_mat_q8 differs from mul_mat"
    ref = orc.mul_mat(wt, Wc, N, K, x, nthreads=orc.default_threads())
    check_close(host(Y), ref["y64"], ref["den"], f"q8 wt={wt} N={N} K={K} M={M}")
    Xo = dev(orc.quantize(vt, x))  # the oracle's own blocks
    Y2 = torch.empty(M, N, device="cuda")
    q.qmm_mul_mat_q8(wt, Wp, N, K, Xo, M, Y2)
    assert torch.equal(Y2, Y)
    q.qmm_check_device_error()


# ------------------------------------------------------------------ failure detection
def test_bounded_wait_times_out_and_context_survives(q, orc):
    """A device-side wait that nothing completes gives up after its bound,
    records QMM_ERR_TIMEOUT in the device error word (reported once, then
    cleared) and the context keeps working: no fault, no hang."""
    q.qmm_check_device_error()  # start clean
    q.qmm_debug_wait_timeout(2_000_000)  # about 1 ms of SM clocks
    with pytest.raises(q.QmmError) as e:
        q.qmm_check_device_error()
    assert e.value.status == 4
    q.qmm_check_device_error()  # cleared
    with pytest.raises(q.QmmError) as e:
        q.qmm_debug_wait_timeout(0)
    assert e.value.status == 1
    # the same context still computes
    N, K, M = 24, 512, 1
    w = wl.weights(17, N, K, 0.02, row_offset_std=0.005).numpy()
    x = wl.activations(17, M, K).numpy()
    Wc = orc.quantize(1, w)
    y = run_mul_mat(q, 1, Wc, N, K, x)
    ref = orc.mul_mat(1, Wc, N, K, x)
    check_close(y, ref["y64"], ref["den"], "after a timed-out wait")
    q.qmm_check_device_error()


@pytest.mark.parametrize("wt", [0, 1])
def test_prepared_shared_workspace_two_streams(q, orc, wt):
    """Prefill GEMMs on two streams at once from one read-only workspace:
    each call's split tiles go through scratch of its own, so both results
    equal the single-stream one bit for bit."""
    N, K, M = 1000, 4096, 300
    w = wl.weights(16, N, K, 0.02).numpy()
    x = wl.activations(16, M, K).numpy()
    Wc = orc.quantize(wt, w, nthreads=orc.default_threads())
    Wp = q.empty_packed(wt, N, K)
    q.qmm_repack_weights(wt, dev(Wc), Wp, N, K)
    ws_bytes = q.qmm_workspace_bytes(wt, M, K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    q.qmm_quantize_activations(wt, dev(x), M, K, ws, ws_bytes)
    Y0 = torch.empty(M, N, device="cuda")
    q.qmm_mul_mat_prepared(wt, Wp, N, K, ws, ws_bytes, M, Y0)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    Ys = [torch.full((M, N), float("nan"), device="cuda") for _ in range(6)]
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    for i, Y in enumerate(Ys):
        st = s1 if i % 2 == 0 else s2
        q.qmm_mul_mat_prepared(wt, Wp, N, K, ws, ws_bytes, M, Y, st.cuda_stream)
    torch.cuda.synchronize()
    q.qmm_check_device_error()
    for Y in Ys:
        assert torch.equal(Y.view(torch.int32), Y0.view(torch.int32))


@pytest.mark.parametrize("wt,N,K,M", [(1, 4096, 4096, 1), (0, 40, 4096, 3), (5, 300, 2048, 20)])
@pytest.mark.parametrize("pinned,flags", [(True, 0), (True, 1), (False, 0)])
def test_mul_mat_host_buffers(q, wt, N, K, M, pinned, flags):
    """qmm_mul_mat_host (X from and Y to host memory, one call; with
    QMM_HOST_MAPPED the kernels pull X and store Y through the mapped pinned
    buffers) gives the bits of qmm_mul_mat on device copies of the same X."""
    w = wl.weights(60, N, K, 0.02, row_offset_std=0.0 if wt == 0 else 0.005, device="cuda")
    Wq = torch.empty(N * (K // (32 if wt == 0 else 256)) * q.qmm_block_bytes(wt), dtype=torch.uint8, device="cuda")
    q.qmm_quantize_weights(wt, w, Wq, N, K)
    Wp = q.empty_packed(wt, N, K)
    q.qmm_repack_weights(wt, Wq, Wp, N, K)
    x = wl.activations(60, M, K)
    Xh = x.pin_memory() if pinned else x.clone()
    Yh = torch.full((M, N), float("nan"))
    Yh = Yh.pin_memory() if pinned else Yh
    nbytes = q.qmm_host_call_bytes(wt, M, N, K)
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    q.qmm_mul_mat_host(wt, Wp, N, K, Xh, M, Yh, buf, nbytes, stream, flags)
    stream.synchronize()
    q.qmm_check_device_error()
    Yd = torch.empty(M, N, device="cuda")
    q.qmm_mul_mat(wt, Wp, N, K, x.cuda(), M, Yd)
    assert torch.equal(Yh, Yd.cpu())
    with pytest.raises(q.QmmError) as e:
        q.qmm_mul_mat_host(wt, Wp, N, K, Xh, M, Yh, buf, nbytes - 16, stream, flags)
    assert e.value.status == 6
