"""Seeded synthetic inputs for the quantized matmul workloads.

This module is the one thing the oracle side and the CUDA side share: it draws
random numbers and shapes them into the workloads' fp32/fp16/uint inputs. It
holds none of the method's arithmetic (no quantization, packing or dot
products).

Generator: a counter-based stream. Element i of stream (seed, stream_id) is a
32-bit hash of its counter, ``lowbias32`` (Chris Wellons, "hash-prospector",
2018: x ^= x >> 16; x *= 0x7feb352d; x ^= x >> 15; x *= 0x846ca68b;
x ^= x >> 16), applied to ``counter + key`` and again after xor with a second
key derived from (seed, stream_id). Uniforms are (h + 0.5) / 2^32; normals use
Box-Muller (sqrt(-2 ln u1) cos(2 pi u2), one normal per two uniforms) in
float64, then rounded to float32. Everything is int64/float64 torch arithmetic
with no overflow, so the same numbers come out on any device; counters make
any slice (a set of rows) reproducible on its own.

Workload shapes follow the pages' examples: a 70B-class layer (q/k/v/o,
gate/up/down projections), 4096x4096 and 11008x4096 linear layers, and a
W4A16 8192x8192 layer with group size 128.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

_M32 = 0xFFFFFFFF
_CHUNK = 1 << 24


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2^32 for 0 <= x < 2^32 without int64 overflow."""
    lo = x & 0xFFFF
    hi = x >> 16
    return (lo * c + (((hi * c) & 0xFFFF) << 16)) & _M32


def _lowbias32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _lowbias32_int(x: int) -> int:
    x &= _M32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & _M32
    x ^= x >> 15
    x = (x * 0x846CA68B) & _M32
    x ^= x >> 16
    return x


def _keys(seed: int, stream: int):
    s = (seed * 1000 + stream) & _M32
    k1 = _lowbias32_int(s ^ 0x9E3779B9)
    k2 = _lowbias32_int(k1 ^ 0x85EBCA6B ^ (s * 0x27D4EB2F & _M32))
    return k1, k2


def bits32(seed: int, stream: int, start: int, n: int, device="cpu") -> torch.Tensor:
    """n 32-bit hashes (as int64) for counters start .. start+n-1 (< 2^32)."""
    assert 0 <= start and start + n <= (1 << 32)
    k1, k2 = _keys(seed, stream)
    c = torch.arange(start, start + n, dtype=torch.int64, device=device)
    h = _lowbias32((c + k1) & _M32)
    return _lowbias32(h ^ k2)


def uniform(seed: int, stream: int, n: int, start: int = 0, device="cpu") -> torch.Tensor:
    """float64 uniforms in (0, 1)."""
    return (bits32(seed, stream, start, n, device).to(torch.float64) + 0.5) * (1.0 / 4294967296.0)


def normal_flat(seed: int, stream: int, n: int, start: int = 0, device="cpu",
                std: float = 1.0) -> torch.Tensor:
    """float32 normals for element indices start .. start+n-1 of the stream."""
    out = torch.empty(n, dtype=torch.float32, device=device)
    for off in range(0, n, _CHUNK):
        cnt = min(_CHUNK, n - off)
        u = uniform(seed, stream, 2 * cnt, 2 * (start + off), device)
        u1, u2 = u[0::2], u[1::2]
        z = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)
        out[off:off + cnt] = (z * std).to(torch.float32)
    return out


def normal_rows(seed: int, stream: int, n_rows: int, k: int, rows=None, device="cpu",
                std: float = 1.0) -> torch.Tensor:
    """[len(rows) or n_rows, k] normals of an [n_rows, k] matrix (row r = counters r*k..)."""
    if rows is None:
        return normal_flat(seed, stream, n_rows * k, 0, device, std).view(n_rows, k)
    out = torch.empty(len(rows), k, dtype=torch.float32, device=device)
    for i, r in enumerate(rows):
        out[i] = normal_flat(seed, stream, k, int(r) * k, device, std)
    return out


def uniform_int(seed: int, stream: int, n: int, lo: int, hi: int, start: int = 0,
                device="cpu") -> torch.Tensor:
    """int64 uniform integers in [lo, hi] (inclusive)."""
    b = bits32(seed, stream, start, n, device)
    return lo + ((b * (hi - lo + 1)) >> 32)


# ------------------------------------------------------------------ recipes
# Stream ids per tensor (one stream per tensor, as seed*1000 + id).
S_W, S_ROWOFF, S_X, S_OUTPOS, S_OUTSIGN, S_HOTCH, S_Q, S_SCALE, S_ZERO, S_A = range(10)


def weights(seed: int, N: int, K: int, std: float, row_offset_std: float = 0.0,
            outlier_frac: float = 0.0, outlier_sigma: float = 8.0, rows=None,
            device="cpu") -> torch.Tensor:
    """fp32 weights [N, K] (or only the listed rows): N(0, std), plus a per-row
    offset N(0, row_offset_std) added to every element of the row, plus a
    seeded set of outlier elements set to +-outlier_sigma*std (random sign)."""
    idx = torch.arange(N, dtype=torch.int64) if rows is None else \
        torch.as_tensor([int(r) for r in rows], dtype=torch.int64)
    out = torch.empty(idx.numel(), K, dtype=torch.float32, device=device)
    off = normal_flat(seed, S_ROWOFF, N, 0, device, row_offset_std) if row_offset_std > 0 else None
    thr = int(outlier_frac * 4294967296.0)
    big = outlier_sigma * std
    # contiguous runs of rows are generated together (counters are row-major)
    step = max(1, _CHUNK // K)
    i = 0
    while i < idx.numel():
        j = i + 1
        while j < idx.numel() and j - i < step and int(idx[j]) == int(idx[j - 1]) + 1:
            j += 1
        r0, nr = int(idx[i]), j - i
        w = normal_flat(seed, S_W, nr * K, r0 * K, device, std).view(nr, K)
        if off is not None:
            w += off[r0:r0 + nr, None]
        if thr > 0:
            pos = (bits32(seed, S_OUTPOS, r0 * K, nr * K, device) < thr).view(nr, K)
            sgn = (bits32(seed, S_OUTSIGN, r0 * K, nr * K, device) & 1).view(nr, K)
            val = torch.where(sgn == 1, big, -big).to(torch.float32)
            w = torch.where(pos, val, w)
        out[i:j] = w
        i = j
    return out


def activations(seed: int, M: int, K: int, hot_frac: float = 0.0, hot_scale: float = 20.0,
                device="cpu") -> torch.Tensor:
    """fp32 activations [M, K] ~ N(0, 1); a seeded set of hot_frac of the
    channels k (the same for every token) is scaled by hot_scale."""
    x = normal_rows(seed, S_X, M, K, device=device)
    if hot_frac > 0.0:
        thr = int(hot_frac * 4294967296.0)
        hot = bits32(seed, S_HOTCH, 0, K, device) < thr
        x = torch.where(hot[None, :], x * hot_scale, x)
    return x


S_EDGE = 20  # first stream id of the edge-case rows


def edge_activation_rows(seed: int, K: int, device="cpu") -> torch.Tensor:
    """fp32 activation rows [14, K] with the magnitudes and shapes that stress
    a quantized product: zeros, constants, N(0, 1) scaled by 1e-30, 1e-6,
    1e-3, 1e4 and 3e5 (above fp16's largest value), all positive (as after a
    SiLU) and all negative, a lone spike, a normal row with one element x 1e4,
    a row whose first 32 elements are x 1e3 and the rest x 1e-3 (six decades
    inside one token), and a +-0 pattern."""
    n = lambda i, std=1.0: normal_flat(seed, S_EDGE + i, K, 0, device, std)
    rows = [torch.zeros(K, device=device), torch.full((K,), 0.37, device=device),
            torch.full((K,), -2.5, device=device),
            n(0, 1e-30), n(1, 1e-6), n(2, 1e-3), n(3, 1e4), n(4, 3e5),
            n(5).abs(), -n(6).abs()]
    spike = torch.zeros(K, device=device)
    spike[K // 3] = -5.0
    rows.append(spike)
    hot = n(7).clone()
    hot[(2 * K) // 5] *= 1e4
    rows.append(hot)
    wide = n(8) * 1e-3
    wide[:32] = n(9)[:32] * 1e3
    rows.append(wide)
    rows.append(torch.where(torch.arange(K, device=device) % 3 == 0, -0.0, 0.0))
    return torch.stack(rows).to(torch.float32)


def edge_weight_rows(seed: int, K: int, device="cpu") -> torch.Tensor:
    """fp32 weight rows [10, K]: zeros, a negative constant, N(0, 0.02) scaled
    by 1e-30, N(0, 1e-3), N(0, 1e2), N(0, 0.02) - 0.5 (every element
    negative: a large min term), two rows whose every 32-element sub-block is
    symmetric about zero (elements 16..31 the negatives of 0..15: the min term
    and the code term nearly cancel), a lone spike and |N(0, 0.02)| + 0.01."""
    n = lambda i, std=0.02: normal_flat(seed, S_EDGE + 10 + i, K, 0, device, std)
    sym = n(3).view(-1, 2, 16)
    sym = torch.stack([sym[:, 0], -sym[:, 0]], dim=1).reshape(K)
    sym2 = n(4, 0.05).view(-1, 2, 16)
    sym2 = torch.stack([sym2[:, 0], -sym2[:, 0]], dim=1).reshape(K) + 0.001
    spike = torch.zeros(K, device=device)
    spike[K // 2 + 1] = 0.3
    rows = [torch.zeros(K, device=device), torch.full((K,), -0.013, device=device),
            n(0) * 1e-30, n(1, 1e-3), n(2, 1e2), n(5) - 0.5, sym, sym2, spike,
            n(6).abs() + 0.01]
    return torch.stack(rows).to(torch.float32)


@dataclass(frozen=True)
class Linear:
    """One projection of a workload: weight [N, K], activations [M, K]."""
    name: str
    N: int
    K: int
    wstd: float
    row_offset_std: float = 0.0
    outlier_frac: float = 0.0


# Q4_0 x Q8_0 GEMV, M=1, 256 x 1024, W ~ N(0, 0.02), X ~ N(0, 1).
GEMV_Q4_0_SMALL = Linear("q4_0_256x1024", 256, 1024, 0.02)
# Q4_K x Q8_K GEMV, 4096 x 4096, W ~ N(0, 0.02) + per-row offset N(0, 0.005).
GEMV_Q4_K_4096 = Linear("q4_K_4096x4096", 4096, 4096, 0.02, row_offset_std=0.005)
GEMV_Q4_K_M_SWEEP = (1, 2, 4, 8, 16)
# 70B-class decoder layer, Q4_K, M=1: W ~ N(0, 0.015) with 0.1% outliers at 8 sigma;
# activations N(0, 1) with 1% of the channels scaled x20.
LAYER_70B = (
    Linear("q_proj", 8192, 8192, 0.015, outlier_frac=1e-3),
    Linear("k_proj", 1024, 8192, 0.015, outlier_frac=1e-3),
    Linear("v_proj", 1024, 8192, 0.015, outlier_frac=1e-3),
    Linear("o_proj", 8192, 8192, 0.015, outlier_frac=1e-3),
    Linear("gate_proj", 28672, 8192, 0.015, outlier_frac=1e-3),
    Linear("up_proj", 28672, 8192, 0.015, outlier_frac=1e-3),
    Linear("down_proj", 8192, 28672, 0.015, outlier_frac=1e-3),
)
LAYER_70B_HOT_FRAC = 0.01
# Prefill GEMM shapes: M in {512, 2048}, N x K in {11008 x 4096, 4096 x 11008}.
PREFILL_SHAPES = (Linear("up_11008x4096", 11008, 4096, 0.02, row_offset_std=0.005),
                  Linear("down_4096x11008", 4096, 11008, 0.02, row_offset_std=0.005))
PREFILL_M = (512, 2048)
# W4A16: N = K = 8192, G = 128, M in {1, 16, 256}.
W4A16_N = W4A16_K = 8192
W4A16_G = 128
W4A16_M = (1, 16, 256)


def nf4_like_table() -> torch.Tensor:
    """A 16-entry code table for the non-uniform W4A16 form (W-hat = s LUT(q)):
    the standard normal's quantiles at probabilities (i + 1/2) / 16, scaled so
    the largest magnitude is 1, as fp16. Equal-probability levels, so codes of
    normally distributed weights are uniform over 0..15 (the q recipe of
    w4a16_inputs). An input table, not the method: any 16 values will do."""
    from statistics import NormalDist
    lv = [NormalDist().inv_cdf((i + 0.5) / 16) for i in range(16)]
    m = max(abs(v) for v in lv)
    return torch.tensor([v / m for v in lv], dtype=torch.float32).to(torch.float16)


def w4a16_inputs(seed: int, N: int, K: int, G: int, M: int, rows=None, device="cpu"):
    """q [N, K] uint8 ~ U{0..15}; s [N, K/G] fp16 ~ U(0.005, 0.02); z [N, K/G]
    uint8 ~ U{0..15}; A [M, K] fp16 ~ N(0, 1). Returns (q, s16, z, A16)."""
    ng = K // G
    idx = list(range(N)) if rows is None else [int(r) for r in rows]
    qs, ss, zs = [], [], []
    if rows is None:
        q = uniform_int(seed, S_Q, N * K, 0, 15, 0, device).view(N, K)
        s = 0.005 + 0.015 * uniform(seed, S_SCALE, N * ng, 0, device).view(N, ng)
        z = uniform_int(seed, S_ZERO, N * ng, 0, 15, 0, device).view(N, ng)
    else:
        for n in idx:
            qs.append(uniform_int(seed, S_Q, K, 0, 15, n * K, device))
            ss.append(0.005 + 0.015 * uniform(seed, S_SCALE, ng, n * ng, device))
            zs.append(uniform_int(seed, S_ZERO, ng, 0, 15, n * ng, device))
        q, s, z = torch.stack(qs), torch.stack(ss), torch.stack(zs)
    A = normal_rows(seed, S_A, M, K, device=device).to(torch.float16)
    return q.to(torch.uint8), s.to(torch.float16), z.to(torch.uint8), A
