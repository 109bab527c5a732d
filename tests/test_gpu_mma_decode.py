"""GPU parity of the tensor-core decode GEMVs for Q6_K and Q4_0 (M = 2..16
tokens per launch): integer-valued fp16 operands on mma.sync, every block's
integer sum exact, through the C ABI against the oracle.

Bars: |Y_gpu - Y_fp64| <= 1e-3 sum_k |w_k a_k| element by element (as every
GPU parity test), and, where one block (Q4_0) or one super-block (Q6_K)
carries a token's whole product, Y bit for bit equal to the factored form
fp32(d_a fp32(d_w isum)) of the oracle's exact integer block sums."""
import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu
TOL = 1e-3
Q4_0, Q4_K, Q6_K = 0, 1, 5


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantized_matmul_q4_gb300 as q
    return q


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check(y, ref, den, what):
    y = np.asarray(y, dtype=np.float64)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y - ref)
    worst = np.max(np.where(den > 0, err / np.where(den > 0, den, 1.0), 0.0))
    assert np.all(err <= TOL * den), f"{what}: worst normalised error {worst:.3e}"


def packed(q, orc, wt, w, N, K):
    Wc = orc.quantize(wt, w, nthreads=orc.default_threads())
    Wp = q.empty_packed(wt, N, K)
    q.qmm_repack_weights(wt, dev(Wc), Wp, N, K)
    return Wc, Wp


@pytest.mark.parametrize("wt", [Q6_K, Q4_0])
@pytest.mark.parametrize("N,K,M", [
    (10000, 256, 3),   # 625 tile pairs: several pairs per CTA; one unit per row
    (8, 2304, 9),      # one tile (no second tile in the pair), 9 units, two n8 token tiles
    (37, 4352, 5),     # odd tile count, 17 units (a partial last stage)
    (40, 4096, 2), (200, 1536, 16),
    (72, 8192, 12),    # 8 tokens per launch fit shared memory: two launches, one image each
    (24, 65536, 3)])   # no token fits: the scalar GEMV
def test_mma_decode_shapes(q, orc, wt, N, K, M):
    w = wl.weights(50, N, K, 0.02, row_offset_std=0.0 if wt == Q4_0 else 0.005).numpy()
    x = wl.activations(50, M, K).numpy()
    Wc, Wp = packed(q, orc, wt, w, N, K)
    Y = torch.full((M * N + 32,), 12345.0, device="cuda")
    q.qmm_mul_mat(wt, Wp, N, K, dev(x), M, Y)
    q.qmm_check_device_error()
    y = Y.cpu().numpy()
    assert np.all(y[M * N:] == 12345.0), "write past the end of Y"
    ref = orc.mul_mat(wt, Wc, N, K, x, nthreads=orc.default_threads())
    check(y[:M * N].reshape(M, N), ref["y64"], ref["den"], f"wt={wt} N={N} K={K} M={M}")


@pytest.mark.parametrize("wt,M", [(Q6_K, 3), (Q6_K, 5), (Q6_K, 8), (Q4_0, 2), (Q4_0, 5), (Q4_0, 8)])
def test_mma_decode_block_arithmetic_exact(q, orc, wt, M):
    """Each token's activations nonzero in one block only (Q4_0: block m % 8
    of 8; Q6_K: the one super-block of K = 256): the output is the factored
    form of that block's integer sum, bit for bit. (Q6_K at two tokens and a
    K this small takes the dp4a GEMV with its fused quantizer, whose lanes
    add partial products, so its first tensor-core case is three tokens.)"""
    N, K = 40, 256
    w = wl.weights(51, N, K, 0.02, row_offset_std=0.0 if wt == Q4_0 else 0.005).numpy()
    x = wl.activations(51, M, K).numpy()
    if wt == Q4_0:
        for m in range(M):
            keep = np.zeros(K, dtype=bool)
            keep[32 * (m % 8):32 * (m % 8) + 32] = True
            x[m, ~keep] = 0.0
    Wc, Wp = packed(q, orc, wt, w, N, K)
    Y = torch.empty(M, N, device="cuda")
    q.qmm_mul_mat(wt, Wp, N, K, dev(x), M, Y)
    q.qmm_check_device_error()
    y = Y.cpu().numpy()
    act = orc.ACT_TYPE[wt]
    Xq = orc.quantize(act, x)
    f32 = np.float32
    for m in range(M):
        for n in range(N):
            if wt == Q6_K:
                _, isum = orc.block_sums(Q6_K, K, Wc[n], Xq[m])
                dw = Wc[n][208:210].view(np.float16)[0]
                da = Xq[m][0:4].view(np.float32)[0]
                want = f32(da) * (f32(dw) * f32(int(np.asarray(isum).ravel()[0])))
            else:
                b = m % 8
                isum = np.asarray(orc.block_sums(Q4_0, K, Wc[n], Xq[m])).ravel()[b]
                dw = Wc[n][18 * b:18 * b + 2].view(np.float16)[0]
                da = Xq[m][34 * b:34 * b + 2].view(np.float16)[0]
                want = f32(da) * (f32(dw) * f32(int(isum)))
            assert y[m, n] == want, f"wt={wt} m={m} n={n}: {y[m, n]!r} != {want!r}"


@pytest.mark.parametrize("wt,N,K,M", [(Q6_K, 40, 4096, 4), (Q4_0, 37, 2304, 6), (Q4_0, 24, 8192, 16)])
def test_mma_decode_prepared_and_q8(q, orc, wt, N, K, M):
    """The image written by qmm_quantize_activations (read-only for two
    calls), and the one imported from the caller's canonical Q8 blocks by
    qmm_mul_mat_q8: the same codes, so the same output bits."""
    w = wl.weights(52, N, K, 0.02, row_offset_std=0.0 if wt == Q4_0 else 0.005).numpy()
    x = wl.activations(52, M, K).numpy()
    Wc, Wp = packed(q, orc, wt, w, N, K)
    ws_bytes = q.qmm_workspace_bytes(wt, M, K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    q.qmm_quantize_activations(wt, dev(x), M, K, ws, ws_bytes)
    Y1 = torch.empty(M, N, device="cuda")
    Y2 = torch.empty(M, N, device="cuda")
    q.qmm_mul_mat_prepared(wt, Wp, N, K, ws, ws_bytes, M, Y1)
    q.qmm_mul_mat_prepared(wt, Wp, N, K, ws, ws_bytes, M, Y2)
    Xq = orc.quantize(orc.ACT_TYPE[wt], x)
    Y3 = torch.empty(M, N, device="cuda")
    q.qmm_mul_mat_q8(wt, Wp, N, K, dev(Xq), M, Y3)
    q.qmm_check_device_error()
    ref = orc.mul_mat(wt, Wc, N, K, x, nthreads=orc.default_threads())
    check(Y1.cpu().numpy(), ref["y64"], ref["den"], f"prepared wt={wt}")
    assert torch.equal(Y1, Y2)
    assert torch.equal(Y1, Y3), "image from canonical Q8 blocks differs"


@pytest.mark.parametrize("wt,K,M", [(Q4_K, 28672, 9), (Q4_K, 28672, 16), (Q6_K, 8192, 12), (Q4_0, 8192, 16)])
def test_large_k_decode_batch(q, orc, wt, K, M):
    """A decode batch whose K is too large for the tensor-core GEMV to hold
    it in one or two launches (Q4_K: fewer than three) takes the GEMM; the
    output is checked against the oracle like any other, through every entry
    point that dispatches on it (mul_mat, the workspace call, prepared)."""
    N = 40
    w = wl.weights(53, N, K, 0.02, row_offset_std=0.0 if wt == Q4_0 else 0.005).numpy()
    x = wl.activations(53, M, K).numpy()
    Wc, Wp = packed(q, orc, wt, w, N, K)
    ref = orc.mul_mat(wt, Wc, N, K, x, nthreads=orc.default_threads())
    X = dev(x)
    Y1 = torch.full((M, N), float("nan"), device="cuda")
    q.qmm_mul_mat(wt, Wp, N, K, X, M, Y1)
    ws_bytes = q.qmm_workspace_bytes(wt, M, K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    Y2 = torch.full((M, N), float("nan"), device="cuda")
    q.qmm_mul_mat_ws(wt, Wp, N, K, X, M, Y2, ws, ws_bytes)
    Y3 = torch.full((M, N), float("nan"), device="cuda")
    q.qmm_quantize_activations(wt, X, M, K, ws, ws_bytes)
    q.qmm_mul_mat_prepared(wt, Wp, N, K, ws, ws_bytes, M, Y3)
    q.qmm_check_device_error()
    for Y, what in ((Y1, "mul_mat"), (Y2, "mul_mat_ws"), (Y3, "prepared")):
        check(Y.cpu().numpy(), ref["y64"], ref["den"], f"{what} wt={wt} K={K} M={M}")
    assert torch.equal(Y1, Y2)
