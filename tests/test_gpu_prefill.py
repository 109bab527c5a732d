"""GPU parity of the prefill path (more than 16 tokens): the prefill
quantizers and the tcgen05 GEMMs, whose operands are the weights rounded once
to fp16 and the activations 2^e d_a y rounded once to fp16 (a power of two
2^e per token, taken off in the epilogue), through
the C ABI, against the oracle.
Bar: |Y_gpu - Y_fp64| <= 1e-3 * sum_k |w_k a_k| per element, no absolute
slack (an output whose sum is 0 must be exactly 0)."""
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


def check(y, ref, den, what):
    err = np.abs(y.astype(np.float64) - ref)
    assert np.all(np.isfinite(y)), f"{what}: non-finite"
    bad = err > TOL * den
    worst = np.max(np.where(den > 0, err / np.where(den > 0, den, 1.0), 0.0))
    assert not bad.any(), f"{what}: {bad.sum()} off, worst {worst:.3e}"


def packed(q, orc, w, N, K, wt=None):
    wt = q.QMM_TYPE_Q4_K if wt is None else wt
    Wc = orc.quantize(wt, w, nthreads=orc.default_threads())
    Wp = q.empty_packed(wt, N, K)
    q.qmm_repack_weights(wt, torch.from_numpy(Wc).cuda(), Wp, N, K)
    return Wc, Wp


@pytest.mark.parametrize("N,K,M", [(128, 256, 17), (200, 512, 300), (384, 1024, 256),
                                   (136, 2304, 129), (64, 256, 64),
                                   (128, 16384, 40),   # one tile over 64 CTAs (stream-K pieces)
                                   (1000, 4096, 300)])  # CTA ranges straddling tiles
def test_prefill_gemm_small(q, orc, N, K, M):
    w = wl.weights(30, N, K, 0.02, row_offset_std=0.005).numpy()
    x = wl.activations(30, M, K).numpy()
    Wc, Wp = packed(q, orc, w, N, K)
    Y = torch.full((M * N + 64,), float("nan"), device="cuda")
    Y[M * N:] = 777.0
    q.qmm_mul_mat(q.QMM_TYPE_Q4_K, Wp, N, K, torch.from_numpy(x).cuda(), M, Y)
    q.qmm_check_device_error()
    y = Y.cpu().numpy()
    assert np.all(y[M * N:] == 777.0), "write past the end of Y"
    ref = orc.mul_mat(q.QMM_TYPE_Q4_K, Wc, N, K, x, nthreads=orc.default_threads())
    check(y[:M * N].reshape(M, N), ref["y64"], ref["den"], f"N={N} K={K} M={M}")


@pytest.mark.parametrize("shape", wl.PREFILL_SHAPES, ids=lambda L: L.name)
@pytest.mark.parametrize("M", wl.PREFILL_M)
def test_prefill_full_size_sampled(q, orc, shape, M):
    """Prefill shapes at full size (M in {512, 2048}, 11008x4096 and
    4096x11008), weights quantized on the GPU; sampled rows checked against
    the oracle, which quantizes those rows itself from the same fp32."""
    L = shape
    w = wl.weights(31, L.N, L.K, L.wstd, row_offset_std=L.row_offset_std, device="cuda")
    x = wl.activations(31, M, L.K, device="cuda")
    Wq = q.empty_blocks(q.QMM_TYPE_Q4_K, L.N, L.K)
    q.qmm_quantize_weights(q.QMM_TYPE_Q4_K, w, Wq, L.N, L.K)
    Wp = q.empty_packed(q.QMM_TYPE_Q4_K, L.N, L.K)
    q.qmm_repack_weights(q.QMM_TYPE_Q4_K, Wq, Wp, L.N, L.K)
    Y = torch.full((M, L.N), float("nan"), device="cuda")
    q.qmm_mul_mat(q.QMM_TYPE_Q4_K, Wp, L.N, L.K, x, M, Y)
    q.qmm_check_device_error()
    assert bool(torch.isfinite(Y).all()), "non-finite (or unwritten) outputs"
    rows = np.unique(np.r_[0:3, 127:130, L.N - 3:L.N, np.linspace(0, L.N - 1, 24).astype(np.int64)])
    w_rows = w[torch.as_tensor(rows, device="cuda")].cpu().numpy()
    Wc_rows = orc.quantize(q.QMM_TYPE_Q4_K, w_rows)
    assert np.array_equal(Wq.view(L.N, -1)[torch.as_tensor(rows, device="cuda")].cpu().numpy(),
                          Wc_rows)
    ref = orc.mul_mat(q.QMM_TYPE_Q4_K, Wc_rows, len(rows), L.K, x.cpu().numpy(),
                      nthreads=orc.default_threads())
    check(Y[:, torch.as_tensor(rows, device="cuda")].cpu().numpy(), ref["y64"], ref["den"],
          f"{L.name} M={M}")


@pytest.mark.parametrize("N,K,M", [(128, 256, 17), (200, 512, 300), (136, 2304, 129), (64, 96, 40),
                                   (300, 1056, 130),
                                   (128, 16384, 40),   # one tile over 64 CTAs (stream-K pieces)
                                   (1000, 4096, 300),  # CTA ranges straddling tiles
                                   (72, 8224, 20)])    # ragged last round in every piece
def test_prefill_q4_0_small(q, orc, N, K, M):
    """Q4_0 prefill GEMM: ragged N, M and K (K a multiple of 32 only)."""
    wt = q.QMM_TYPE_Q4_0
    w = wl.weights(32, N, K, 0.02).numpy()
    x = wl.activations(32, M, K).numpy()
    Wc, Wp = packed(q, orc, w, N, K, wt)
    Y = torch.full((M * N + 64,), float("nan"), device="cuda")
    Y[M * N:] = 777.0
    q.qmm_mul_mat(wt, Wp, N, K, torch.from_numpy(x).cuda(), M, Y)
    q.qmm_check_device_error()
    y = Y.cpu().numpy()
    assert np.all(y[M * N:] == 777.0), "write past the end of Y"
    ref = orc.mul_mat(wt, Wc, N, K, x, nthreads=orc.default_threads())
    check(y[:M * N].reshape(M, N), ref["y64"], ref["den"], f"Q4_0 N={N} K={K} M={M}")


@pytest.mark.parametrize("shape", wl.PREFILL_SHAPES, ids=lambda L: L.name)
@pytest.mark.parametrize("M", wl.PREFILL_M)
def test_prefill_q4_0_full_size_sampled(q, orc, shape, M):
    """Q4_0 prefill at full size (M in {512, 2048}): weights quantized on the
    GPU, every output finite, sampled rows checked against the oracle."""
    L, wt = shape, q.QMM_TYPE_Q4_0
    w = wl.weights(33, L.N, L.K, L.wstd, device="cuda")
    x = wl.activations(33, M, L.K, device="cuda")
    Wq = q.empty_blocks(wt, L.N, L.K)
    q.qmm_quantize_weights(wt, w, Wq, L.N, L.K)
    Wp = q.empty_packed(wt, L.N, L.K)
    q.qmm_repack_weights(wt, Wq, Wp, L.N, L.K)
    Y = torch.full((M, L.N), float("nan"), device="cuda")
    q.qmm_mul_mat(wt, Wp, L.N, L.K, x, M, Y)
    q.qmm_check_device_error()
    assert bool(torch.isfinite(Y).all()), "non-finite (or unwritten) outputs"
    rows = np.unique(np.r_[0:3, 127:130, L.N - 3:L.N, np.linspace(0, L.N - 1, 24).astype(np.int64)])
    Wc_rows = Wq.view(L.N, -1)[torch.as_tensor(rows, device="cuda")].cpu().numpy()
    ref = orc.mul_mat(wt, Wc_rows, len(rows), L.K, x.cpu().numpy(), nthreads=orc.default_threads())
    check(Y[:, torch.as_tensor(rows, device="cuda")].cpu().numpy(), ref["y64"], ref["den"],
          f"Q4_0 {L.name} M={M}")


@pytest.mark.parametrize("wt_name", ["Q4_K", "Q4_0", "Q6_K"])
def test_stream_k_deterministic(q, orc, wt_name):
    """Split tiles are summed in a fixed order: two calls give the same bits."""
    wt = getattr(q, "QMM_TYPE_" + wt_name)
    N, K, M = 1000, 4096, 300
    w = wl.weights(34, N, K, 0.02).numpy()
    x = torch.from_numpy(wl.activations(34, M, K).numpy()).cuda()
    _, Wp = packed(q, orc, w, N, K, wt)
    Y1 = torch.empty(M, N, device="cuda")
    Y2 = torch.full((M, N), float("nan"), device="cuda")
    q.qmm_mul_mat(wt, Wp, N, K, x, M, Y1)
    q.qmm_mul_mat(wt, Wp, N, K, x, M, Y2)
    q.qmm_check_device_error()
    assert torch.equal(Y1.view(torch.int32), Y2.view(torch.int32))


def dequant_f64(orc, t, blocks, K):
    """Rows of canonical blocks -> fp64 values, by the oracle's dequantizer."""
    return torch.from_numpy(orc.dequantize(t, blocks, K, f64=True))


@pytest.mark.parametrize("wt_name", ["Q4_K", "Q4_0", "Q6_K"])
@pytest.mark.parametrize("shape", wl.PREFILL_SHAPES, ids=lambda L: L.name)
def test_prefill_full_output(q, orc, wt_name, shape):
    """Every element of a full-size prefill output (M = 512: the stream-K
    grid and its fixup on 11008 x 4096, one CTA per tile on 4096 x 11008)
    against sum_k w_k a_k in fp64 over the oracle's dequantized weights and
    activations (the factored sums the kernels use equal that product up to
    fp64 rounding). The first weight rows and tokens are the edge-case rows
    (tiny, huge and out-of-fp16-range activations, symmetric sub-blocks,
    zeros, spikes), the rest the workload's distributions. Bar: 1e-3 sum_k
    |w_k a_k| per element, exact zeros where that sum is 0."""
    wt, L, M = getattr(q, "QMM_TYPE_" + wt_name), shape, 512
    w = wl.weights(35, L.N, L.K, L.wstd, row_offset_std=L.row_offset_std if wt_name != "Q4_0" else 0.0,
                   device="cuda")
    x = wl.activations(35, M, L.K, device="cuda")
    we, xe = wl.edge_weight_rows(35, L.K, device="cuda"), wl.edge_activation_rows(35, L.K, device="cuda")
    w[:we.shape[0]] = we
    x[:xe.shape[0]] = xe
    Wq = q.empty_blocks(wt, L.N, L.K)
    q.qmm_quantize_weights(wt, w, Wq, L.N, L.K)
    Wp = q.empty_packed(wt, L.N, L.K)
    q.qmm_repack_weights(wt, Wq, Wp, L.N, L.K)
    Y = torch.full((M, L.N), float("nan"), device="cuda")
    q.qmm_mul_mat(wt, Wp, L.N, L.K, x, M, Y)
    q.qmm_check_device_error()
    act = orc.ACT_TYPE[wt]
    Wd = dequant_f64(orc, wt, Wq.view(L.N, -1).cpu().numpy(), L.K).cuda()
    Xd = dequant_f64(orc, act, orc.quantize(act, x.cpu().numpy(), nthreads=orc.default_threads()), L.K).cuda()
    ref = Xd @ Wd.T
    den = Xd.abs() @ Wd.abs().T
    err = (Y.double() - ref).abs()
    assert torch.isfinite(Y).all(), "non-finite output"
    bad = err > TOL * den
    worst = float(torch.where(den > 0, err / torch.where(den > 0, den, 1.0), 0.0).max())
    assert not bad.any(), f"{int(bad.sum())} off, worst {worst:.3e}"
