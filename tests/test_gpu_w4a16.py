"""GPU parity of the W4A16 path (page 3: C = A (s (q - z))^T per group),
through the C ABI, against the oracle's exact (fp64) result.

Bar per element: |C_gpu - C_fp64| <= 1e-3 * sum_k |A[m,k] w[n,k]| + half an
fp16 ulp of |C_fp64| (C is returned in fp16) + 2^-24 (the fp16 subnormal
step). The repack is a bit permutation, checked bit-exact by a round trip."""
import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu
TOL = 1e-3
W = 4  # qmm type id of W4A16


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantized_matmul_q4_gb300 as q
    assert q.QMM_TYPE_W4A16 == W
    return q


def check(c16, ref, den, what):
    c = c16.astype(np.float64)
    assert np.all(np.isfinite(c)), f"{what}: non-finite"
    err = np.abs(c - ref)
    bound = TOL * den + np.abs(ref) * 2.0 ** -11 + 2.0 ** -24
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} off, worst "
                           f"{np.max(err / np.maximum(den, 1e-30)):.3e} of den")


def pack_torch(qcodes: torch.Tensor) -> torch.Tensor:
    """Canonical qweight [N, K/8] int32 from codes [N, K] (element 8c + i in
    bits 4i of word c), for inputs built on the device."""
    N, K = qcodes.shape
    v = qcodes.view(N, K // 8, 8).to(torch.int64)
    word = torch.zeros(N, K // 8, dtype=torch.int64, device=qcodes.device)
    for i in range(8):
        word |= v[:, :, i] << (4 * i)
    return (word - ((word >> 31) << 32)).to(torch.int32).contiguous()


def packed_from_canon(q, qweight_dev, N, K):
    Wp = torch.empty(q.qmm_packed_bytes(W, N, K), dtype=torch.uint8, device="cuda")
    q.qmm_repack_weights(W, qweight_dev, Wp, N, K)
    return Wp


def run(q, Wp, s16, z, G, A16, M, N, K):
    C = torch.full((M * N + 32,), float("nan"), dtype=torch.float16, device="cuda")
    C[M * N:] = 77.0
    q.qmm_w4a16(Wp, s16, z, G, A16, C, M, N, K)
    q.qmm_check_device_error()
    c = C.cpu()
    assert torch.all(c[M * N:] == 77.0), "write past the end of C"
    return c[:M * N].view(M, N).numpy()


def test_repack_round_trip(q):
    N, K = 37, 1024
    g = torch.Generator().manual_seed(5)
    canon = torch.randint(-2 ** 31, 2 ** 31 - 1, (N, K // 8), generator=g, dtype=torch.int64)
    canon = canon.to(torch.int32).cuda()
    Wp = packed_from_canon(q, canon, N, K)
    back = torch.empty_like(canon)
    q.qmm_unrepack_weights(W, Wp, back, N, K)
    torch.cuda.synchronize()
    assert torch.equal(back, canon)
    assert Wp.numel() == (N + 15) // 16 * 16 * K // 2
    assert not torch.equal(Wp.view(torch.int32)[:N * K // 8], canon.view(-1)), "repack is the identity"


@pytest.mark.parametrize("N,K,G,M", [(64, 256, 128, 1), (100, 512, 128, 5), (48, 1024, 256, 16),
                                     (33, 384, 128, 9), (16, 128, 128, 3), (40, 512, 128, 8),
                                     (24, 640, 128, 12), (40, 512, 128, 17), (64, 256, 128, 40),
                                     (100, 384, 128, 130), (200, 640, 128, 33), (48, 1024, 256, 200),
                                     (136, 1152, 384, 257),
                                     (128, 8192, 128, 40),    # one tile over 32 CTAs (stream-K pieces)
                                     (1000, 4096, 128, 300),  # CTA ranges straddling tiles
                                     (40, 2304, 128, 9),      # K-major decode: a partial K chunk, a partial tile
                                     (10000, 1024, 128, 16),  # K-major decode: more tiles per CTA than one group
                                     (64, 4096, 128, 4)])     # decode with A read in place (too large to stage)
def test_w4a16_small(q, orc, N, K, G, M):
    qc, s16, z, A16 = wl.w4a16_inputs(40, N, K, G, M)
    qweight = orc.w4a16_pack(qc.numpy())
    Wp = packed_from_canon(q, torch.from_numpy(qweight.view(np.int32)).cuda(), N, K)
    c = run(q, Wp, s16.cuda(), z.cuda(), G, A16.cuda(), M, N, K)
    ref = orc.w4a16_matmul(qweight, s16.view(torch.int16).numpy().view(np.uint16), z.numpy(), G,
                           A16.view(torch.int16).numpy().view(np.uint16),
                           nthreads=orc.default_threads())
    check(c, ref["c64"], ref["den"], f"N={N} K={K} G={G} M={M}")


@pytest.mark.parametrize("M", wl.W4A16_M)
def test_w4a16_full_size_sampled(q, orc, M):
    """N = K = 8192, G = 128 at M in {1, 16, 256}: inputs generated on the
    device, every output row computed, 48 sampled rows checked."""
    N = K = wl.W4A16_N
    G = wl.W4A16_G
    qc, s16, z, A16 = wl.w4a16_inputs(41, N, K, G, M, device="cuda")
    qweight = pack_torch(qc)
    del qc
    Wp = packed_from_canon(q, qweight, N, K)
    c = run(q, Wp, s16, z, G, A16, M, N, K)
    rows = np.random.default_rng(7).choice(N, 48, replace=False)
    rows[:2] = (0, N - 1)
    ref = orc.w4a16_matmul(qweight.cpu().numpy().view(np.uint32), s16.cpu().view(torch.int16).numpy()
                           .view(np.uint16), z.cpu().numpy(), G,
                           A16.cpu().view(torch.int16).numpy().view(np.uint16), rows=rows,
                           nthreads=orc.default_threads())
    check(c[:, rows], ref["c64"], ref["den"], f"8192x8192 M={M}")


@pytest.mark.parametrize("N,K,G,M", [(48, 1024, 128, 1), (100, 512, 128, 5), (40, 2304, 128, 9),
                                     (64, 4096, 128, 4), (64, 256, 128, 40), (1000, 4096, 128, 300)])
def test_w4a16_degenerate_weights(q, orc, N, K, G, M):
    """The method's degenerate weights on every path (decode with staged and
    in-place activations, K-major decode, GEMM, stream-K GEMM): q = z
    everywhere (w = 0, so C must be exactly 0: no residue of the zero-point
    arithmetic), then one nonzero weight per row at a row-dependent position
    (C[m, n] = s d A[m, k_n]: a misplaced code, scale, zero or activation
    element lands in the wrong output or multiplies the wrong A)."""
    _, s16, z, A16 = wl.w4a16_inputs(46, N, K, G, M)
    zk = z.repeat_interleave(G, dim=1).numpy()  # [N, K]: every code equal to its group's zero
    s_d, z_d, A_d = s16.cuda(), z.cuda(), A16.cuda()
    Wz = packed_from_canon(q, torch.from_numpy(orc.w4a16_pack(zk).view(np.int32)).cuda(), N, K)
    c = run(q, Wz, s_d, z_d, G, A_d, M, N, K)
    assert np.all(c == 0), f"w = 0 gave {np.count_nonzero(c)} nonzero outputs"
    n = np.arange(N)
    k = (n * 7919 + 13) % K
    one = zk.copy()
    one[n, k] = (zk[n, k] + 1 + n % 15) % 16  # q - z != 0 (mod 16), varied per row
    qweight = orc.w4a16_pack(one)
    Wp = packed_from_canon(q, torch.from_numpy(qweight.view(np.int32)).cuda(), N, K)
    c = run(q, Wp, s_d, z_d, G, A_d, M, N, K)
    ref = orc.w4a16_matmul(qweight, s16.view(torch.int16).numpy().view(np.uint16), z.numpy(), G,
                           A16.view(torch.int16).numpy().view(np.uint16),
                           nthreads=orc.default_threads())
    assert np.all(ref["den"] > 0)
    check(c, ref["c64"], ref["den"], f"one-hot N={N} K={K} G={G} M={M}")


def test_w4a16_errors(q):
    N, K, G, M = 16, 256, 128, 2
    Wp = torch.zeros(N * K // 2, dtype=torch.uint8, device="cuda")
    s = torch.ones(N, K // G, dtype=torch.float16, device="cuda")
    z = torch.zeros(N, K // G, dtype=torch.uint8, device="cuda")
    A = torch.zeros(M, K, dtype=torch.float16, device="cuda")
    C = torch.zeros(M, N, dtype=torch.float16, device="cuda")
    with pytest.raises(q.QmmError) as e:
        q.qmm_w4a16(Wp, s, z, 64, A, C, M, N, K)  # G % 128 != 0
    assert e.value.status == 2
    with pytest.raises(q.QmmError) as e:
        q.qmm_w4a16(Wp, s, z, 96, A, C, M, N, K)  # K % G != 0
    assert e.value.status == 1
    with pytest.raises(q.QmmError) as e:
        q.qmm_w4a16(Wp, s, z, G, A.view(-1)[1:].data_ptr(), C, M, N, K)  # misaligned A
    assert e.value.status == 1
    q.qmm_w4a16(Wp, s, z, G, A, C, 0, N, K)  # M == 0: no-op
    q.qmm_w4a16(Wp, s, z, G, A, C, M, 0, K)  # N == 0: no-op
    q.qmm_check_device_error()


@pytest.mark.parametrize("M", [256, 512])
def test_w4a16_full_output(q, orc, M):
    """Every element of the 8192 x 8192, G = 128 layer (M = 256: one CTA per
    tile; M = 512: the stream-K grid and its fixup) against sum_k A w in fp64
    with w = s (q - z) from the oracle's unpacking of the same codes.
    Bar as test_w4a16_small."""
    N = K = wl.W4A16_N
    G = wl.W4A16_G
    qc, s16, z, A16 = wl.w4a16_inputs(42, N, K, G, M, device="cuda")
    qweight = pack_torch(qc)
    del qc
    Wp = packed_from_canon(q, qweight, N, K)
    c = run(q, Wp, s16, z, G, A16, M, N, K)
    codes = torch.from_numpy(orc.w4a16_unpack(qweight.cpu().numpy().view(np.uint32), K).astype(np.float64)).cuda()
    sz = s16.double().repeat_interleave(G, dim=1)
    zz = z.double().repeat_interleave(G, dim=1)
    w = sz * (codes - zz)
    del codes, sz, zz
    a = A16.double()
    ref = (a @ w.T).cpu().numpy()
    den = (a.abs() @ w.abs().T).cpu().numpy()
    check(c, ref, den, f"8192x8192 M={M} full")


@pytest.mark.parametrize("N,ng", [(37, 3), (64, 8), (100, 9), (8192, 64)])
def test_w4a16_unpack_zeros(q, orc, N, ng):
    """Packed zero points unpacked on the GPU equal the oracle's reading bit
    for bit, and a W4A16 call on them equals the call on the original
    zeros."""
    g = torch.Generator().manual_seed(N * 131 + ng)
    words = (ng + 7) // 8
    zp = torch.randint(-2 ** 31, 2 ** 31 - 1, (N, words), generator=g, dtype=torch.int64).to(torch.int32)
    z = torch.empty(N, ng, dtype=torch.uint8, device="cuda")
    q.qmm_w4a16_unpack_zeros(zp.cuda(), z, N, ng)
    torch.cuda.synchronize()
    ref = orc.w4a16_unpack_zeros(zp.numpy().view(np.uint32), ng)
    assert np.array_equal(z.cpu().numpy(), ref)
    if N <= 100:
        G = 128
        K = ng * G
        qc, s16, _, A16 = wl.w4a16_inputs(43, N, K, G, 5)
        qweight = orc.w4a16_pack(qc.numpy())
        Wp = packed_from_canon(q, torch.from_numpy(qweight.view(np.int32)).cuda(), N, K)
        c1 = run(q, Wp, s16.cuda(), z, G, A16.cuda(), 5, N, K)
        c2 = run(q, Wp, s16.cuda(), torch.from_numpy(ref).cuda(), G, A16.cuda(), 5, N, K)
        assert np.array_equal(c1.view(np.uint16), c2.view(np.uint16))


def test_w4a16_unpack_zeros_errors(q):
    z = torch.empty(4, 4, dtype=torch.uint8, device="cuda")
    zp = torch.zeros(4, 1, dtype=torch.int32, device="cuda")
    with pytest.raises(q.QmmError):
        q.qmm_w4a16_unpack_zeros(zp, z, 4, 0)
    q.qmm_w4a16_unpack_zeros(zp, z, 0, 4)  # N == 0: no-op


# ------------------------------------------------------------------ code table (NF4-like)
def run_lut(q, Wp, s16, lut16, G, A16, M, N, K):
    C = torch.full((M * N + 32,), float("nan"), dtype=torch.float16, device="cuda")
    C[M * N:] = 77.0
    q.qmm_w4a16_lut(Wp, s16, lut16, G, A16, C, M, N, K)
    q.qmm_check_device_error()
    c = C.cpu()
    assert torch.all(c[M * N:] == 77.0), "write past the end of C"
    return c[:M * N].view(M, N).numpy()


@pytest.mark.parametrize("N,K,G,M", [(64, 256, 128, 1), (100, 512, 128, 5), (48, 1024, 256, 16),
                                     (33, 384, 128, 9), (40, 512, 128, 17), (200, 640, 128, 33),
                                     (136, 1152, 384, 257), (1000, 4096, 128, 300), (40, 2304, 128, 9)])
def test_w4a16_lut_small(q, orc, N, K, G, M):
    """W-hat = s LUT(q) with the NF4-like table: decode (M <= 16) and the
    tensor-core GEMM (M > 16, stream-K when tiles outnumber SMs)."""
    qc, s16, _, A16 = wl.w4a16_inputs(43, N, K, G, M)
    lut = wl.nf4_like_table()
    qweight = orc.w4a16_pack(qc.numpy())
    Wp = packed_from_canon(q, torch.from_numpy(qweight.view(np.int32)).cuda(), N, K)
    c = run_lut(q, Wp, s16.cuda(), lut.cuda(), G, A16.cuda(), M, N, K)
    ref = orc.w4a16_lut_matmul(qweight, s16.view(torch.int16).numpy().view(np.uint16),
                               lut.view(torch.int16).numpy().view(np.uint16), G,
                               A16.view(torch.int16).numpy().view(np.uint16),
                               nthreads=orc.default_threads())
    check(c, ref["c64"], ref["den"], f"lut N={N} K={K} G={G} M={M}")


@pytest.mark.parametrize("M", [1, 16, 256])
def test_w4a16_lut_equals_zero_point_form(q, M):
    """The table LUT(q) = q - 8 gives the zero-point kernels' bits with every
    zero point 8 (same exact products, same sums)."""
    N = K = 2048
    G = 128
    qc, s16, _, A16 = wl.w4a16_inputs(44, N, K, G, M, device="cuda")
    Wp = packed_from_canon(q, pack_torch(qc), N, K)
    z = torch.full((N, K // G), 8, dtype=torch.uint8, device="cuda")
    lut = (torch.arange(16) - 8).to(torch.float16).cuda()
    a = run(q, Wp, s16, z, G, A16, M, N, K)
    b = run_lut(q, Wp, s16, lut, G, A16, M, N, K)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


@pytest.mark.parametrize("M", wl.W4A16_M)
def test_w4a16_lut_full_size_sampled(q, orc, M):
    """N = K = 8192, G = 128, the NF4-like table, at M in {1, 16, 256}: 48
    sampled rows against the oracle."""
    N = K = wl.W4A16_N
    G = wl.W4A16_G
    qc, s16, _, A16 = wl.w4a16_inputs(45, N, K, G, M, device="cuda")
    qweight = pack_torch(qc)
    del qc
    Wp = packed_from_canon(q, qweight, N, K)
    lut = wl.nf4_like_table()
    c = run_lut(q, Wp, s16, lut.cuda(), G, A16, M, N, K)
    rows = np.random.default_rng(8).choice(N, 48, replace=False)
    rows[:2] = (0, N - 1)
    ref = orc.w4a16_lut_matmul(qweight.cpu().numpy().view(np.uint32),
                               s16.cpu().view(torch.int16).numpy().view(np.uint16),
                               lut.view(torch.int16).numpy().view(np.uint16), G,
                               A16.cpu().view(torch.int16).numpy().view(np.uint16), rows=rows,
                               nthreads=orc.default_threads())
    check(c[:, rows], ref["c64"], ref["den"], f"lut 8192x8192 M={M}")


def test_w4a16_lut_errors(q):
    N, K, G, M = 16, 256, 128, 2
    Wp = torch.zeros(N * K // 2, dtype=torch.uint8, device="cuda")
    s = torch.ones(N, K // G, dtype=torch.float16, device="cuda")
    lut = torch.zeros(16, dtype=torch.float16, device="cuda")
    A = torch.zeros(M, K, dtype=torch.float16, device="cuda")
    C = torch.zeros(M, N, dtype=torch.float16, device="cuda")
    with pytest.raises(q.QmmError) as e:
        q.qmm_w4a16_lut(Wp, s, None, G, A, C, M, N, K)  # no table
    assert e.value.status == 1
    with pytest.raises(q.QmmError) as e:
        q.qmm_w4a16_lut(Wp, s, lut, 64, A, C, M, N, K)  # G % 128 != 0
    assert e.value.status == 2
    q.qmm_w4a16_lut(Wp, s, lut, G, A, C, 0, N, K)  # M == 0: no-op
    q.qmm_check_device_error()
