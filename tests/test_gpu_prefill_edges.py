"""GPU parity of the prefill GEMMs (the tcgen05 kernels that take fp16
operands) on the inputs that stress their rounding: activations at 1e-30,
1e-6, 1e-3, 1e4 and above fp16's range, six decades inside one token,
all-positive and all-negative tokens, spikes and zeros; weight rows at 1e-30,
1e-3 and 1e2, rows with a large min term, sub-blocks symmetric about zero
(where d s_j q and dmin m_j nearly cancel), zero rows and spikes.

Every case runs through qmm_quantize_activations + qmm_mul_mat_prepared,
which take the prefill GEMM from 17 tokens on (every format),
whatever K; where qmm_mul_mat takes it too, through qmm_mul_mat as well.
Bar, element by element: |Y_gpu - Y_fp64| <= 1e-3 sum_k |w_k a_k|, with no
absolute slack: where that sum is 0 the output must be exactly 0.
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


def check_rel(y, ref, den, what):
    y = np.asarray(y, dtype=np.float64)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y - ref)
    bad = err > TOL * den
    worst = np.max(np.where(den > 0, err / np.where(den > 0, den, 1.0), 0.0))
    assert not bad.any(), f"{what}: {int(bad.sum())} outputs off; worst normalised error {worst:.3e}"
    print(f"{what}: worst normalised error {worst:.3e}")
    return worst


def inputs(N, K, M, seed, offset):
    """Edge rows first, then seeded N(0, 0.02) (+ row offset) weights and
    N(0, 1) activations up to N and M."""
    we = wl.edge_weight_rows(seed, K)
    xe = wl.edge_activation_rows(seed, K)
    w = torch.cat([we, wl.weights(seed, N - we.shape[0], K, 0.02, row_offset_std=offset)])
    x = torch.cat([xe, wl.activations(seed, M - xe.shape[0], K)])
    return w.numpy(), x.numpy()


GEMM_MIN_M = {"Q4_K": 17, "Q4_0": 17, "Q6_K": 17}


@pytest.mark.parametrize("wt_name", ["Q4_K", "Q6_K", "Q4_0"])
@pytest.mark.parametrize("N,K,M", [(150, 256, 40),     # one super-block: nothing averages out
                                   (150, 1024, 40),
                                   (136, 2304, 20)])
def test_prefill_edge_inputs(q, orc, wt_name, N, K, M):
    wt = getattr(q, "QMM_TYPE_" + wt_name)
    assert M >= GEMM_MIN_M[wt_name]
    w, x = inputs(N, K, M, 40 + K, 0.0 if wt_name == "Q4_0" else 0.005)
    Wc = orc.quantize(wt, w, nthreads=orc.default_threads())
    Wp = q.empty_packed(wt, N, K)
    q.qmm_repack_weights(wt, torch.from_numpy(Wc).cuda(), Wp, N, K)
    X = torch.from_numpy(x).cuda()
    ref = orc.mul_mat(wt, Wc, N, K, x, nthreads=orc.default_threads())
    # the prefill GEMM, whatever K
    ws_bytes = q.qmm_workspace_bytes(wt, M, K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    q.qmm_quantize_activations(wt, X, M, K, ws, ws_bytes)
    Y = torch.full((M, N), float("nan"), device="cuda")
    q.qmm_mul_mat_prepared(wt, Wp, N, K, ws, ws_bytes, M, Y)
    q.qmm_check_device_error()
    check_rel(Y.cpu().numpy(), ref["y64"], ref["den"], f"{wt_name} prepared N={N} K={K} M={M}")
    # the one-call entry point (the GEMM too, unless the fused decode GEMV
    # takes these sizes)
    Y2 = torch.full((M, N), float("nan"), device="cuda")
    q.qmm_mul_mat(wt, Wp, N, K, X, M, Y2)
    q.qmm_check_device_error()
    check_rel(Y2.cpu().numpy(), ref["y64"], ref["den"], f"{wt_name} mul_mat N={N} K={K} M={M}")
    # zero weight row / zero token give exact zeros
    assert torch.all(Y[:, 0] == 0) and torch.all(Y[0, :] == 0)


@pytest.mark.parametrize("wt_name", ["Q4_K", "Q6_K", "Q4_0"])
def test_prefill_edge_inputs_q8(q, orc, wt_name):
    """The same operand built from the caller's canonical Q8 blocks
    (qmm_mul_mat_q8): the per-token prescale comes from the blocks' scales."""
    wt = getattr(q, "QMM_TYPE_" + wt_name)
    N, K, M = 150, 1024, 40
    w, x = inputs(N, K, M, 47, 0.0 if wt_name == "Q4_0" else 0.005)
    Wc = orc.quantize(wt, w, nthreads=orc.default_threads())
    Wp = q.empty_packed(wt, N, K)
    q.qmm_repack_weights(wt, torch.from_numpy(Wc).cuda(), Wp, N, K)
    Xq = orc.quantize(orc.ACT_TYPE[wt], x)
    Y = torch.full((M, N), float("nan"), device="cuda")
    q.qmm_mul_mat_q8(wt, Wp, N, K, torch.from_numpy(Xq).cuda(), M, Y)
    q.qmm_check_device_error()
    ref = orc.mul_mat(wt, Wc, N, K, x, nthreads=orc.default_threads())
    check_rel(Y.cpu().numpy(), ref["y64"], ref["den"], f"{wt_name} q8 N={N} K={K} M={M}")
