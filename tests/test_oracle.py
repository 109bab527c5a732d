"""Pins of the CPU oracle against facts the pages print and mathematics fixes.

Every check here is independent of the oracle's own code path: numpy's IEEE
float16 conversion, numpy matmul in float64, hand-derived bytes from the pages'
layout rules (tests/golden), brute force over the 16 possible codes, one-hot
probes, closed-form bounds and invariants. A plausible mistake in the oracle
(dropped min term, wrong nibble order, wrong scale packing, wrong sign or
index, transposed output) fails at least one of them.
"""
import json
import os

import numpy as np
import pytest
import torch

import workloads as wl

GOLD = os.path.join(os.path.dirname(__file__), "golden")

DT_Q4_0 = np.dtype([("d", "<u2"), ("qs", "u1", 16)])
DT_Q8_0 = np.dtype([("d", "<u2"), ("qs", "i1", 32)])
DT_Q4_K = np.dtype([("d", "<u2"), ("dmin", "<u2"), ("scales", "u1", 12), ("qs", "u1", 128)])
DT_Q8_K = np.dtype([("d", "<f4"), ("qs", "i1", 256), ("bsums", "<i2", 16)])
DT_Q6_K = np.dtype([("ql", "u1", 128), ("qh", "u1", 64), ("scales", "i1", 16), ("d", "<u2")])


def h2f(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float32)


def f2h(x):
    return np.asarray(x, np.float32).astype(np.float16).view(np.uint16)


def rng_normal(seed, stream, shape, std=1.0):
    n = int(np.prod(shape))
    return wl.normal_flat(seed, stream, n, std=std).numpy().reshape(shape)


# --------------------------------------------------------------- sizes
def test_block_sizes_and_bits_per_weight(orc):
    # The page's byte counts and bits/weight: 2+16=18 B (4.5 bpw), 2+32=34 B
    # (8.5), 2+2+12+128=144 B (4.5), 4+256+32=292 B (9.125).
    assert [orc.block_bytes(t) for t in (orc.Q4_0, orc.Q4_K, orc.Q8_0, orc.Q8_K)] == [18, 144, 34, 292]
    assert [orc.block_bytes(t) * 8 / orc.BLOCK_ELEMS[t] for t in (0, 1, 2, 3)] == [4.5, 4.5, 8.5, 9.125]
    assert DT_Q4_0.itemsize == 18 and DT_Q8_0.itemsize == 34
    assert DT_Q4_K.itemsize == 144 and DT_Q8_K.itemsize == 292
    # Q6_K: 128 + 64 + 16 + 2 = 210 B per 256 elements = 6.5625 bpw
    assert orc.block_bytes(orc.Q6_K) == 210 and DT_Q6_K.itemsize == 210
    assert orc.block_bytes(orc.Q6_K) * 8 / orc.BLOCK_ELEMS[orc.Q6_K] == 6.5625


# --------------------------------------------------------------- fp16
def test_fp16_decode_exhaustive(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([orc.fp16_to_fp32(int(b)) for b in bits], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_fp16_encode_matches_ieee(orc):
    rs = np.random.RandomState(0)
    vals = [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -24, 2.0 ** -25,
            2.0 ** -25 * 1.0000001, 2.0 ** -26, 6.1035156e-05, 6.0975552e-05, 1e-30, -1e-30,
            float("inf"), -float("inf")]
    # exact midpoints between adjacent halves (ties to even) in the normal and subnormal range
    h = np.arange(0, 0x7BFF, 37, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    vals += list(((lo + hi) / 2).astype(np.float32))
    np.seterr(over="ignore")
    vals += list((rs.randn(4000) * np.exp2(rs.uniform(-30, 17, 4000))).astype(np.float32))
    for v in vals:
        v32 = np.float32(v)
        assert orc.fp32_to_fp16(float(v32)) == int(np.array(v32).astype(np.float16).view(np.uint16)), v
    for v in list(rs.randn(2000) * np.exp2(rs.uniform(-30, 17, 2000))) + [2.0 ** -25, 65520.0]:
        assert orc.fp64_to_fp16(float(v)) == int(np.array(v, np.float64).astype(np.float16).view(np.uint16)), v
    assert orc.fp32_to_fp16(float("nan")) & 0x7C00 == 0x7C00


# --------------------------------------------------------------- Q4_K scale packing
def test_scale_min_k4_golden(orc):
    g = json.load(open(os.path.join(GOLD, "scale_min_k4.json")))
    packed = np.array(g["packed"], np.uint8)
    for j in range(8):
        assert orc.get_scale_min_k4(j, packed) == (g["scales"][j], g["mins"][j])
    built = np.zeros(12, np.uint8)
    for j in range(8):
        built = orc.set_scale_min_k4(j, built, g["scales"][j], g["mins"][j])
    assert built.tolist() == g["packed"]


def test_scale_min_k4_exhaustive(orc):
    rs = np.random.RandomState(1)
    for j in range(8):
        for s in range(64):
            base = rs.randint(0, 256, 12).astype(np.uint8)
            before = [orc.get_scale_min_k4(i, base) for i in range(8)]
            for m in range(64):
                b = orc.set_scale_min_k4(j, base, s, m)
                assert orc.get_scale_min_k4(j, b) == (s, m)
                if m in (0, 37, 63):
                    for i in range(8):
                        if i != j:
                            assert orc.get_scale_min_k4(i, b) == before[i]


# --------------------------------------------------------------- Q4_0
def test_q4_0_layout(orc):
    # d = -x_max/8 with x_max = -8 gives d = 1 and codes q = x + 8 exactly.
    q = np.array([(7 * i + 3) % 16 for i in range(32)], np.int64)
    q[5] = 0
    q[q == 0] = 0
    x = (q - 8).astype(np.float32)
    assert np.abs(x).max() == 8 and x[np.argmax(np.abs(x))] == -8
    blk = orc.quantize(orc.Q4_0, x).view(DT_Q4_0)[0, 0]
    assert blk["d"] == 0x3C00  # fp16(1.0)
    # reading of the page's "32 nibbles in 16 bytes": low nibble of byte l is
    # element l, high nibble is element l + 16
    expect = [int(q[l]) | (int(q[l + 16]) << 4) for l in range(16)]
    assert blk["qs"].tolist() == expect


def _q4_0_blocks(orc, x):
    return orc.quantize(orc.Q4_0, x).view(DT_Q4_0).reshape(x.shape[0], -1)


def test_q4_0_quantize_invariants(orc):
    x = rng_normal(0, 50, (64, 256), std=0.02)
    x[3, 40] = 0.5    # outlier, positive
    x[7, 100] = -0.7  # outlier, negative
    blocks = _q4_0_blocks(orc, x)
    for r in range(x.shape[0]):
        for b in range(x.shape[1] // 32):
            xb = x[r, 32 * b:32 * b + 32].astype(np.float64)
            blk = blocks[r, b]
            i_max = int(np.argmax(np.abs(xb)))      # first index of the largest |x|
            x_max = xb[i_max]
            assert blk["d"] == f2h(np.float32(x_max) / np.float32(-8.0))
            codes = np.array([int(blk["qs"][l]) & 15 for l in range(16)] + [int(blk["qs"][l]) >> 4 for l in range(16)], np.int64)
            assert codes[i_max] == 0          # the extreme element maps to code 0
            d = x_max / -8.0
            t = xb / d + 8.0                  # the real-valued code
            # brute force over the 16 codes: q is the nearest code, the only
            # exception being t = 16 (x = -x_max), clamped to 15
            for i in range(32):
                best = np.argmin(np.abs(t[i] - np.arange(16)))
                if abs(abs(t[i] - np.floor(t[i])) - 0.5) < 1e-4:
                    continue  # tie within rounding of fp32 reciprocal
                assert codes[i] == best, (r, b, i, t[i])
            # reconstruction error <= |d|/2 (with the stored fp16 d)
            d16 = float(h2f(blk["d"]))
            w = d16 * (codes - 8)
            ok = t < 15.5
            assert np.all(np.abs(w - xb)[ok] <= abs(d16) / 2 + abs(d - d16) * 8 + 1e-9)


def test_q4_0_zero_and_constant_blocks(orc):
    x = np.zeros((1, 64), np.float32)
    x[0, 32:] = 0.25
    blk = _q4_0_blocks(orc, x)[0]
    # d = -0/8 is a (negative) zero in IEEE arithmetic; all codes are 8
    assert h2f(blk[0]["d"]) == 0 and np.all(blk[0]["qs"] == 0x88)
    # constant block: x_max = 0.25, d = -1/32, x/d + 8 = 0 -> code 0 everywhere
    assert blk[1]["d"] == f2h(-0.25 / 8) and np.all(blk[1]["qs"] == 0)


# --------------------------------------------------------------- Q8_0 / Q8_K
def test_q8_0_invariants(orc):
    x = rng_normal(0, 51, (16, 512))
    x[2, 7] = 40.0
    blocks = orc.quantize(orc.Q8_0, x).view(DT_Q8_0).reshape(16, -1)
    for r in range(16):
        for b in range(16):
            xb = x[r, 32 * b:32 * b + 32]
            blk = blocks[r, b]
            amax = np.float32(np.abs(xb).max())
            d32 = amax / np.float32(127.0)
            assert blk["d"] == f2h(d32)
            q = blk["qs"].astype(np.int64)
            assert np.all(np.abs(q) <= 127)
            i = int(np.argmax(np.abs(xb)))
            assert q[i] == np.sign(xb[i]) * 127
            assert np.all(np.abs(xb / np.float64(d32) - q) <= 0.5 + 1e-5)


def test_q8_K_invariants(orc):
    x = rng_normal(0, 52, (8, 1024))
    x[1, 9] = -30.0
    blocks = orc.quantize(orc.Q8_K, x).view(DT_Q8_K).reshape(8, -1)
    for r in range(8):
        for b in range(4):
            xb = x[r, 256 * b:256 * b + 256]
            blk = blocks[r, b]
            d32 = np.float32(np.abs(xb).max()) / np.float32(127.0)
            assert blk["d"] == d32
            q = blk["qs"].astype(np.int64)
            assert np.all(np.abs(q) <= 127)
            assert np.all(np.abs(xb / np.float64(d32) - q) <= 0.5 + 1e-5)
            # bsums: the sum of each run of 16 codes
            assert blk["bsums"].tolist() == q.reshape(16, 16).sum(1).tolist()
    z = orc.quantize(orc.Q8_K, np.zeros((1, 256), np.float32)).view(DT_Q8_K)[0, 0]
    assert z["d"] == 0 and not z["qs"].any() and not z["bsums"].any()


# --------------------------------------------------------------- Q4_K
def test_q4_K_layout(orc):
    # all x >= 0 so mins are 0; each sub-block holds a 15 so its range is 945
    # and d = 945/15/63 = 1, s_j = 63, codes q = x / 63 exactly.
    q = np.array([(5 * i + 1) % 16 for i in range(256)], np.int64)
    for j in range(8):
        q[32 * j + 3] = 15
    x = (63 * q).astype(np.float32)
    blk = orc.quantize(orc.Q4_K, x).view(DT_Q4_K)[0, 0]
    assert blk["d"] == 0x3C00 and blk["dmin"] == 0
    for j in range(8):
        assert orc.get_scale_min_k4(j, blk["scales"]) == (63, 0)
    # the page's packing loop: per 64 elements, byte l holds element l (low
    # nibble) and element l + 32 (high nibble)
    expect = [int(q[64 * c + l]) | (int(q[64 * c + 32 + l]) << 4) for c in range(4) for l in range(32)]
    assert blk["qs"].tolist() == expect


def _q4_K_fields(blk):
    s = np.zeros(8, np.int64)
    m = np.zeros(8, np.int64)
    sc = blk["scales"].astype(np.int64)
    for j in range(8):
        if j < 4:
            s[j], m[j] = sc[j] & 63, sc[j + 4] & 63
        else:
            s[j] = (sc[j + 4] & 15) | ((sc[j - 4] >> 6) << 4)
            m[j] = (sc[j + 4] >> 4) | ((sc[j] >> 6) << 4)
    qs = blk["qs"].astype(np.int64)
    codes = np.zeros(256, np.int64)
    for c in range(4):
        codes[64 * c:64 * c + 32] = qs[32 * c:32 * c + 32] & 15
        codes[64 * c + 32:64 * c + 64] = qs[32 * c:32 * c + 32] >> 4
    return s, m, codes


def test_q4_K_reconstruction_bound(orc):
    rows = 32
    x = wl.weights(0, rows, 1024, 0.02, row_offset_std=0.005, outlier_frac=2e-3).numpy()
    x[4, :256] = -np.abs(x[4, :256])  # an all-negative super-block
    blocks = orc.quantize(orc.Q4_K, x).view(DT_Q4_K).reshape(rows, -1)
    for r in range(rows):
        for b in range(4):
            xb = x[r, 256 * b:256 * b + 256].astype(np.float64)
            blk = blocks[r, b]
            s, m, codes = _q4_K_fields(blk)
            assert codes.max() <= 15 and s.max() <= 63 and m.max() <= 63
            d16, dm16 = float(h2f(blk["d"])), float(h2f(blk["dmin"]))
            w = d16 * s[np.arange(256) // 32] * codes - dm16 * m[np.arange(256) // 32]
            # every element lies within half a step of the sub-block's grid,
            # plus the error of storing d, dmin in fp16 and the 6-bit scale/min
            for j in range(8):
                sl = slice(32 * j, 32 * j + 32)
                lo = min(0.0, xb[sl].min())
                hi = xb[sl].max()
                step = d16 * s[j]
                err = np.abs(w[sl] - xb[sl])
                # grid error: half a step; scale/min quantization error: up to
                # 15 * (half a 6-bit scale step of d) + half a min step of dmin
                bound = step / 2 + 15 * d16 * 0.5 + dm16 * 0.5 + 1e-6 + 0.01 * (hi - lo)
                assert np.all(err <= bound), (r, b, j, err.max(), bound)
            # the reconstructed row tracks the input closely on average
            assert np.sqrt(np.mean((w - xb) ** 2)) < 0.2 * np.std(xb) + 1e-6


def test_q4_K_nibble_order_by_dequantize(orc):
    # each element must come back in its own position: sub-block j is a ramp
    # at level 0.1 j, so an element placed in another sub-block or another
    # half of its own ramp lands at least two grid steps (0.1) away, while a
    # correct round trip stays within about half a step (0.05 / 2 here).
    x = np.concatenate([np.linspace(j * 0.1, j * 0.1 + 0.05, 32) for j in range(8)]).astype(np.float32)
    w = orc.dequantize(orc.Q4_K, orc.quantize(orc.Q4_K, x), 256)[0]
    assert np.max(np.abs(w - x)) < 0.03


# --------------------------------------------------------------- dot products
def _q4_K_block(d, dmin, s, m, codes):
    blk = np.zeros(1, DT_Q4_K)
    blk["d"] = f2h(d)
    blk["dmin"] = f2h(dmin)
    sc = np.zeros(12, np.uint8)
    for j in range(8):
        if j < 4:
            sc[j] |= s[j]
            sc[j + 4] |= m[j]
        else:
            sc[j + 4] = (s[j] & 15) | ((m[j] & 15) << 4)
            sc[j - 4] |= (s[j] >> 4) << 6
            sc[j] |= (m[j] >> 4) << 6
    blk["scales"] = sc
    qs = np.zeros(128, np.uint8)
    for c in range(4):
        for l in range(32):
            qs[32 * c + l] = codes[64 * c + l] | (codes[64 * c + 32 + l] << 4)
    blk["qs"] = qs
    return blk.view(np.uint8)


def _q8_K_block(d, y):
    blk = np.zeros(1, DT_Q8_K)
    blk["d"] = d
    blk["qs"] = y
    blk["bsums"] = np.asarray(y, np.int64).reshape(16, 16).sum(1)
    return blk.view(np.uint8)


def test_worked_example(orc):
    g = json.load(open(os.path.join(GOLD, "worked_example_q4_K.json")))
    W, A, E = g["weights"], g["activations"], g["expected"]
    s = [W["s_j"]] + [0] * 7
    m = [W["m_j"]] + [0] * 7
    codes = np.zeros(256, np.int64)
    codes[:32] = W["q"]
    y = np.zeros(256, np.int64)
    y[:32] = A["y"]
    wb = _q4_K_block(W["d"], W["dmin"], s, m, codes)
    ab = _q8_K_block(A["d_a"], y)
    S, isum, msum = orc.block_sums(orc.Q4_K, 256, wb, ab)
    assert S[0, 0] == E["sum_q_y"]
    assert isum[0] == W["s_j"] * E["sum_q_y"]
    assert msum[0] == W["m_j"] * E["sum_y"]
    d_a = float(np.float32(A["d_a"]))
    tol = 32 * 16 * abs(E["dot"]) * 2.0 ** -23
    assert abs(orc.vec_dot(orc.Q4_K, 256, wb, ab) - E["dot"]) <= tol + abs(d_a - A["d_a"]) * 2000
    assert abs(orc.vec_dot_f64(orc.Q4_K, 256, wb, ab) - E["dot"]) <= abs(d_a - A["d_a"]) * 2000 + 1e-12
    # dequantize-then-multiply, as the page does first: w = 5.75, a = 0.2
    w = orc.dequantize(orc.Q4_K, wb, 256)[0]
    a = orc.dequantize(orc.Q8_K, ab, 256)[0]
    assert np.all(w[:32] == E["w_elem"])
    assert np.allclose(a[:32], E["a_elem"], rtol=1e-6)
    assert abs(float(np.dot(w.astype(np.float64), a.astype(np.float64))) - E["dot"]) < 1e-5


def test_factored_form_equals_bruteforce_fp64(orc):
    for wt, K in ((orc.Q4_0, 96), (orc.Q4_0, 512), (orc.Q4_K, 256), (orc.Q4_K, 512),
                  (orc.Q6_K, 256), (orc.Q6_K, 768)):
        w = wl.weights(3, 4, K, 0.02, row_offset_std=0.005).numpy()
        x = rng_normal(3, 60, (3, K))
        Wq = orc.quantize(wt, w)
        Xq = orc.quantize(orc.ACT_TYPE[wt], x)
        wd = orc.dequantize(wt, Wq, K, f64=True)
        ad = orc.dequantize(orc.ACT_TYPE[wt], Xq, K, f64=True)
        for n in range(4):
            for mm in range(3):
                ref = float(np.dot(wd[n], ad[mm]))
                den = float(np.sum(np.abs(wd[n] * ad[mm])))
                f64 = orc.vec_dot_f64(wt, K, Wq[n], Xq[mm])
                f32 = orc.vec_dot(wt, K, Wq[n], Xq[mm])
                assert abs(f64 - ref) <= 1e-12 * den
                assert abs(f32 - ref) <= 1e-5 * den


def test_block_sums_onehot_probe(orc):
    # an activation that is 1 at one position reads back that position's code
    K = 256
    w = wl.weights(4, 1, K, 0.02, row_offset_std=0.005).numpy()
    wq = orc.quantize(orc.Q4_K, w)[0]
    s, m, codes = _q4_K_fields(wq.view(DT_Q4_K)[0])
    for p in range(0, K, 7):
        y = np.zeros(K, np.int64)
        y[p] = 1
        S, isum, msum = orc.block_sums(orc.Q4_K, K, wq, _q8_K_block(1.0, y))
        assert S[0, p // 32] == codes[p] and S[0].sum() == codes[p]
        assert isum[0] == s[p // 32] * codes[p] and msum[0] == m[p // 32]
    w0 = rng_normal(4, 61, (1, 64), std=0.02)
    wq0 = orc.quantize(orc.Q4_0, w0)[0]
    blk = wq0.view(DT_Q4_0)
    for p in range(64):
        y = np.zeros(64, np.int64)
        y[p] = 1
        ab = np.zeros(2, DT_Q8_0)
        ab["d"] = 0x3C00
        ab["qs"] = y.reshape(2, 32)
        isum = orc.block_sums(orc.Q4_0, 64, wq0, ab.view(np.uint8))
        l = p % 32
        byte = int(blk[p // 32]["qs"][l % 16])
        code = (byte & 15) if l < 16 else (byte >> 4)
        assert isum[p // 32] == code - 8 and isum.sum() == code - 8


def test_integer_sum_bounds():
    # int32 accumulators cannot overflow: |isum| <= 8 * 63 * 32 * 15 * 127 for
    # Q4_K, |msum| <= 8 * 63 * 2 * 16 * 127, |Q4_0 isum| <= 32 * 8 * 127.
    assert 8 * 63 * 32 * 15 * 127 == 30_723_840 < 2 ** 31
    assert 8 * 63 * 2 * 16 * 127 < 2 ** 31 and 32 * 8 * 127 < 2 ** 31


def test_mul_mat_q8_against_numpy(orc):
    for wt, N, K, M in ((orc.Q4_0, 7, 96, 3), (orc.Q4_K, 5, 512, 2), (orc.Q4_K, 1, 256, 1),
                        (orc.Q6_K, 6, 512, 3)):
        w = wl.weights(5, N, K, 0.02, row_offset_std=0.005).numpy()
        x = rng_normal(5, 62, (M, K))
        Wq = orc.quantize(wt, w)
        res = orc.mul_mat(wt, Wq, N, K, x)
        wd = orc.dequantize(wt, Wq, K, f64=True)
        ad = orc.dequantize(orc.ACT_TYPE[wt], res["xq"], K, f64=True)
        ref = ad @ wd.T                     # [M, N]: output index m * N + n
        den = np.abs(ad) @ np.abs(wd).T
        assert res["y64"].shape == (M, N)
        assert np.all(np.abs(res["y64"] - ref) <= 1e-12 * den + 1e-300)
        assert np.allclose(res["den"], den, rtol=1e-12)
        assert np.all(np.abs(res["y32"] - ref) <= 1e-5 * den + 1e-30)
        rows = [N - 1, 0]
        sub = orc.mul_mat_q8(wt, Wq, N, K, res["xq"], M, rows=rows)
        assert np.array_equal(sub["y32"], res["y32"][:, rows])


# --------------------------------------------------------------- Q6_K
def _q6_K_golden():
    g = json.load(open(os.path.join(GOLD, "q6_K_layout.json")))
    q = np.full(256, g["codes_default"], np.int64)
    for e, v in g["codes"].items():
        q[int(e)] = v
    return g, q


def test_q6_K_golden_pack(orc):
    # x = d s_j q exactly (d = 2^-10); each group holds a -32, so the scale
    # rule gives back d and s_j, and the bytes must be the hand-derived ones
    g, q = _q6_K_golden()
    s = np.array(g["scales"], np.int64)
    x = (g["d"] * s[np.arange(256) // 16] * q).astype(np.float32)
    blk = orc.quantize(orc.Q6_K, x).view(DT_Q6_K)[0, 0]
    assert int(blk["d"]) == g["d_bits"]
    assert blk["scales"].tolist() == g["scales"]
    ql = np.zeros(128, np.int64)
    for i, v in g["ql_nonzero"].items():
        ql[int(i)] = v
    qh = np.full(64, 0xAA, np.int64)
    for i, v in g["qh_not_0xAA"].items():
        qh[int(i)] = v
    assert blk["ql"].tolist() == ql.tolist()
    assert blk["qh"].tolist() == qh.tolist()


def test_q6_K_golden_dequantize(orc):
    # the golden bytes, built by hand, read back as the hand-computed values
    g, q = _q6_K_golden()
    blk = np.zeros(1, DT_Q6_K)
    blk["d"] = g["d_bits"]
    blk["scales"] = g["scales"]
    ql = np.zeros(128, np.uint8)
    for i, v in g["ql_nonzero"].items():
        ql[int(i)] = v
    qh = np.full(64, 0xAA, np.uint8)
    for i, v in g["qh_not_0xAA"].items():
        qh[int(i)] = v
    blk["ql"] = ql
    blk["qh"] = qh
    for f64 in (False, True):
        w = orc.dequantize(orc.Q6_K, blk.view(np.uint8), 256, f64=f64)[0]
        for e, v in g["dequantized"].items():
            assert w[int(e)] == v, (e, w[int(e)], v)
        s = np.array(g["scales"], np.int64)
        assert np.array_equal(w, g["d"] * s[np.arange(256) // 16] * q)


def test_q6_K_reconstruction_bound(orc):
    rows = 16
    x = wl.weights(7, rows, 1024, 0.02, row_offset_std=0.005, outlier_frac=2e-3).numpy()
    x[3, :256] = -np.abs(x[3, :256])  # an all-negative super-block
    x[5, 256:272] = 0.0               # an all-zero group
    blocks = orc.quantize(orc.Q6_K, x).view(DT_Q6_K).reshape(rows, -1)
    w = orc.dequantize(orc.Q6_K, orc.quantize(orc.Q6_K, x), 1024, f64=True)
    for r in range(rows):
        for b in range(4):
            blk = blocks[r, b]
            d16 = float(h2f(blk["d"]))
            s = blk["scales"].astype(np.int64)
            assert np.abs(s).max() == 127 or d16 == 0.0  # the largest group sets d
            for j in range(16):
                sl = slice(256 * b + 16 * j, 256 * b + 16 * j + 16)
                xs = x[r, sl].astype(np.float64)
                sc = np.abs(xs).max() / 32.0           # |sc_j|
                D = d16 * abs(s[j])
                err = np.abs(w[r, sl] - xs)
                # half a grid step, plus up to 32 x the scale's own error
                # (fp16 d, 8-bit s_j), plus one step where +32 clamps to 31
                bound = D + 32 * abs(sc - D) + 1e-9
                assert np.all(err <= bound), (r, b, j, err.max(), bound)
        assert np.sqrt(np.mean((w[r] - x[r]) ** 2)) < 0.05 * np.std(x[r]) + 1e-9
    assert np.all(w[5, 256:272] == 0.0)


def test_q6_K_block_sums_onehot_probe(orc):
    # a one-hot activation reads back the code at that position, in its group
    K = 256
    g, q = _q6_K_golden()
    s = np.array(g["scales"], np.int64)
    x = (g["d"] * s[np.arange(256) // 16] * q).astype(np.float32)
    wq = orc.quantize(orc.Q6_K, x)[0]
    for p in range(K):
        y = np.zeros(K, np.int64)
        y[p] = 1
        S, isum = orc.block_sums(orc.Q6_K, K, wq, _q8_K_block(1.0, y))
        assert S[0, p // 16] == q[p] and S[0].sum() == q[p]
        assert isum[0] == s[p // 16] * q[p]
    # all-ones activation: S_j is the sum of group j's codes
    S, isum = orc.block_sums(orc.Q6_K, K, wq, _q8_K_block(1.0, np.ones(K, np.int64)))
    assert S[0].tolist() == q.reshape(16, 16).sum(1).tolist()


def test_q6_K_integer_sum_bound():
    # |S_j| <= 16 * 32 * 127 and |isum| <= 16 * 127 * that: int32 holds it
    assert 16 * 127 * (16 * 32 * 127) == 132_128_768 < 2 ** 31


# --------------------------------------------------------------- W4A16
def test_w4a16_pack_golden(orc):
    g = json.load(open(os.path.join(GOLD, "w4a16_pack.json")))
    for case in g["cases"]:
        q = np.array([case["q"]], np.uint8)
        u = orc.w4a16_pack(q)
        assert int(u[0, 0]) == case["u"]
        assert orc.w4a16_unpack(u, 8).tolist() == [case["q"]]


def test_w4a16_zeros_pack_golden(orc):
    """Packed zero points (8 per word, like the codes) read back from
    hand-derived words, rows whose group count is not a multiple of 8
    included."""
    g = json.load(open(os.path.join(GOLD, "w4a16_zeros_pack.json")))
    for case in g["cases"]:
        words = np.array([case["words"]], np.uint32)
        assert orc.w4a16_unpack_zeros(words, len(case["z"])).tolist() == [case["z"]]


def test_w4a16_pack_roundtrip(orc):
    q, _, _, _ = wl.w4a16_inputs(0, 8, 256, 128, 1)
    qn = q.numpy()
    assert np.array_equal(orc.w4a16_unpack(orc.w4a16_pack(qn), 256), qn)


def test_w4a16_matmul_against_numpy(orc):
    N, K, G, M = 6, 512, 128, 3
    q, s, z, A = wl.w4a16_inputs(1, N, K, G, M)
    qn, sn, zn, An = q.numpy(), s.numpy(), z.numpy(), A.numpy()
    res = orc.w4a16_matmul(orc.w4a16_pack(qn), sn.view(np.uint16), zn, G, An.view(np.uint16))
    g = np.arange(K) // G
    What = sn.astype(np.float64)[:, g] * (qn.astype(np.float64) - zn.astype(np.float64)[:, g])
    ref = An.astype(np.float64) @ What.T
    den = np.abs(An.astype(np.float64)) @ np.abs(What).T
    assert np.all(np.abs(res["c64"] - ref) <= 1e-12 * den)
    assert np.array_equal(res["c16"], ref.astype(np.float16).view(np.uint16))
    assert np.allclose(res["den"], den, rtol=1e-12)


def test_w4a16_lut_reduces_to_zero_point(orc):
    # the table LUT(q) = q - 8 is the zero-point form with every z = 8: the
    # same products in fp64, so identical results
    N, K, G, M = 7, 512, 128, 3
    q, s, z, A = wl.w4a16_inputs(2, N, K, G, M)
    qw = orc.w4a16_pack(q.numpy())
    s16, A16 = s.numpy().view(np.uint16), A.numpy().view(np.uint16)
    lut = (np.arange(16) - 8).astype(np.float16).view(np.uint16)
    a = orc.w4a16_lut_matmul(qw, s16, lut, G, A16)
    b = orc.w4a16_matmul(qw, s16, np.full((N, K // G), 8, np.uint8), G, A16)
    for key in ("c16", "c64", "den"):
        assert np.array_equal(a[key], b[key]), key


def test_w4a16_lut_onehot_and_relabel(orc):
    N, K, G = 5, 256, 128
    q, s, _, _ = wl.w4a16_inputs(3, N, K, G, 1)
    qn = q.numpy()
    lut = wl.nf4_like_table().numpy()
    qw = orc.w4a16_pack(qn)
    s16 = s.numpy().view(np.uint16)
    # a one-hot activation reads back s[n, k / G] * LUT[q[n, k]] for every row
    for k in (0, 1, 7, 127, 128, 200, 255):
        A = np.zeros((1, K), np.float16)
        A[0, k] = 1.0
        c = orc.w4a16_lut_matmul(qw, s16, lut.view(np.uint16), G, A.view(np.uint16))["c64"][0]
        expect = s.numpy()[:, k // G].astype(np.float64) * lut[qn[:, k]].astype(np.float64)
        assert np.array_equal(c, expect), k
    # relabelling the codes and permuting the table alike changes nothing
    A = wl.w4a16_inputs(3, N, K, G, 4)[3].numpy().view(np.uint16)
    perm = np.array([(7 * i + 3) % 16 for i in range(16)])
    lut2 = np.zeros(16, np.float16)
    lut2[perm] = lut
    a = orc.w4a16_lut_matmul(qw, s16, lut.view(np.uint16), G, A)
    b = orc.w4a16_lut_matmul(orc.w4a16_pack(perm[qn].astype(np.uint8)), s16, lut2.view(np.uint16), G, A)
    assert np.array_equal(a["c64"], b["c64"])


def test_nf4_like_table_is_sorted_and_symmetric():
    t = wl.nf4_like_table().numpy().astype(np.float64)
    assert np.all(np.diff(t) > 0) and t[0] == -1.0 and t[-1] == 1.0
    assert np.array_equal(t, -t[::-1])


# --------------------------------------------------------------- edge cases
@pytest.mark.parametrize("scale", [0.0, 1e-30, 1e-3, 1.0, 1e4])
def test_edge_magnitudes(orc, scale):
    for wt in (orc.Q4_0, orc.Q4_K):
        K = 256
        w = (wl.weights(6, 3, K, 1.0).numpy() * scale).astype(np.float32)
        x = (rng_normal(6, 63, (1, K)) * max(scale, 1e-30)).astype(np.float32)
        Wq = orc.quantize(wt, w)
        res = orc.mul_mat(wt, Wq, 3, K, x)
        assert np.all(np.isfinite(res["y32"]))
        assert np.all(np.abs(res["y32"] - res["y64"]) <= 1e-5 * res["den"] + 1e-37)
        if scale == 0.0:
            assert not res["y32"].any()


def test_q6_K_exact_blocks_round_trip(orc):
    # blocks built from exact values: d = 2^e, int8 scales with |s| = 127 in
    # some group, a -32 in every group (the code of largest magnitude), so the
    # scale rule must return exactly these d, s_j and codes -- for many
    # random draws, sign patterns and exponents
    rng = np.random.default_rng(11)
    for trial in range(60):
        e = int(rng.integers(-14, 0))
        s = rng.integers(1, 128, 16) * rng.choice([-1, 1], 16)
        s[int(rng.integers(0, 16))] = 127 * int(rng.choice([-1, 1]))
        q = rng.integers(-31, 32, 256)
        for j in range(16):
            q[16 * j + int(rng.integers(0, 16))] = -32
        x = (2.0 ** e * s[np.arange(256) // 16] * q).astype(np.float32)
        raw = orc.quantize(orc.Q6_K, x)
        blk = raw.view(DT_Q6_K)[0, 0]
        assert float(h2f(blk["d"])) == 2.0 ** e, trial
        assert blk["scales"].tolist() == s.tolist(), trial
        w = orc.dequantize(orc.Q6_K, raw, 256)[0]
        assert np.array_equal(w, x), trial
