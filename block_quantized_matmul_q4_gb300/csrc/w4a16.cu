// w4a16.cu -- the W4A16 group-asymmetric path of page 3 ("BitBLAS 完全拆解",
// "从数学表达式到真实存储" and "位级打包"):
//   C[m, n] = sum_k A[m, k] * s[n, g] * (q[n, k] - z[n, g]),  g = k / G,
// with A and C fp16, q 4-bit codes (8 per uint32 word, element 8c + i in
// bits 4i of word c), s fp16 and z uint8 per (row, group); or, for
// non-uniform codes like NF4 (same section), W-hat = s LUT(q) with a
// 16-entry fp16 table and no zero point.
//
// Layout (qmm_repack_weights, QMM_TYPE_W4A16): rows in tiles of 16 (the
// last one padded with zero rows); a tile is stored step by step, each
// 128-element step as its 16 rows x 16 words (1 KB contiguous), so a CTA
// streams long contiguous runs. Within every word the nibbles are
// interleaved -- even elements in the low 16 bits, odd ones in the high 16
// bits (slots 0..7 hold elements 0,2,4,6,1,3,5,7) -- so one lop3 turns a
// word into fp16 pairs (k, k+1) laid out as the tensor-core operands want
// them (page 3, "Ladder": lay the bits out offline for the decoder), and no
// kernel permutes the activations.
//
// Decode (M <= 16): mma.sync m16n8k16, weights as the A operand (16 rows per
// warp), tokens as B (8 per MMA). q - z is exact in fp16 (1024 + q minus
// 1024 + z, or the x16 form through one fp16 FMA), the products are exact in
// the fp32 accumulator, and each 128-element step of a group is scaled by s
// in fp32. Decode reads every weight once, so it is bound by HBM: each CTA
// takes a contiguous range of 16-row tiles, and a producer warp streams
// them through a 5-stage shared-memory ring (one 16 KB bulk copy of 16
// steps per stage, so 80 KB in flight per CTA; 64-byte rows, so the
// consumers' 16-byte reads hit distinct banks), together with each tile's
// scales and zeros (two slots) and, when small, all activations. Eight
// consumer warps split each stage's K, then reduce per tile; every load in
// their loop is from shared memory.
#include "tc.cuh"

namespace qmm {
namespace {

constexpr int kStepK = 128;  // elements per warp step: 16 words = 64 bytes per row
constexpr int kDecodeWarps = 8;
constexpr int kDecodeThreads = (kDecodeWarps + 1) * 32;  // + producer warp
constexpr int kRowsPerTile = 16;
constexpr int kStepsPerStage = 16;  // 2048 elements per stage
constexpr int kDStages = 5;
constexpr int kDStageBytes = kStepsPerStage * kRowsPerTile * 64;  // 16 KB: [step][row][64 B]
constexpr size_t kActStageMax = 16 * 1024;  // activations staged in shared memory up to this
constexpr int kSzSlots = 2;                // tiles whose scales and zeros are staged at once

__device__ __forceinline__ uint32_t lop_or(uint32_t x, uint32_t mask) {
    uint32_t d;  // (x & mask) | 0x64006400
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(x), "r"(mask), "r"(0x64006400u));
    return d;
}
__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// (q - z) for the 8 codes of one packed word as four fp16 pairs:
// p01 = (k0, k1), p23 = (k2, k3), p45 = (k4, k5), p67 = (k6, k7), minus z.
// zz = two copies of fp16(1024 + z); zh = two copies of fp16(-64 - z).
struct Zero2 {
    uint32_t zz, zh;
};
__device__ __forceinline__ Zero2 make_zero2(uint32_t z) {
    // z <= 15: fp16 1024 + z is 0x6400 + z, fp16 -(64 + z) is 0xD400 + 16 z
    return Zero2{0x64006400u + z * 0x00010001u, 0xD400D400u + z * 0x00100010u};
}
__device__ __forceinline__ void dequant_word(uint32_t w, const Zero2 &z, uint32_t &p01,
                                             uint32_t &p23, uint32_t &p45, uint32_t &p67) {
    constexpr uint32_t kSixteenth = 0x2C002C00u;  // fp16 1/16 twice
    const uint32_t v = w >> 8;
    p01 = hsub2_u(lop_or(w, 0x000F000Fu), z.zz);
    p23 = hfma2_u(lop_or(w, 0x00F000F0u), kSixteenth, z.zh);
    p45 = hsub2_u(lop_or(v, 0x000F000Fu), z.zz);
    p67 = hfma2_u(lop_or(v, 0x00F000F0u), kSixteenth, z.zh);
}

// LUT(q) for the 8 codes of one packed word as the same four fp16 pairs.
// Slots j and j + 4 hold the pair (k, k + 1) = (2j, 2j + 1): one byte
// index q_k | q_k+1 << 4 per pair (two per word in t, two in t2) into the
// 256-entry pair table tbl[i] = (LUT[i & 15], LUT[i >> 4]). Values of the
// table are exact fp16, so the MMA products stay exact in fp32.
__device__ __forceinline__ void lut_word(uint32_t w, const uint32_t *tbl, uint32_t &p01,
                                         uint32_t &p23, uint32_t &p45, uint32_t &p67) {
    const uint32_t t = (w & 0x0F0Fu) | ((w >> 12) & 0xF0F0u);          // pairs (0,1), (4,5)
    const uint32_t t2 = ((w >> 4) & 0x0F0Fu) | ((w >> 16) & 0xF0F0u);  // pairs (2,3), (6,7)
    p01 = tbl[t & 0xFF];
    p45 = tbl[(t >> 8) & 0xFF];
    p23 = tbl[t2 & 0xFF];
    p67 = tbl[(t2 >> 8) & 0xFF];
}

__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kDecodeWarps * 32) : "memory");
}

struct DecodeArgs {
    const uint8_t *W;  // packed, tile-major
    const __half *S;   // [N][K/G]
    const uint8_t *Z;  // [N][K/G]; unused with a table
    const __half *lut; // 16 fp16 code values (W-hat = s LUT(q)), or null
    const __half *A;   // [M][K]
    __half *C;         // [M][N]
    int64_t M, N, K, G;
    int ng, spg;  // groups per row, 128-element steps per group
    unsigned *err;
    uint32_t act_bytes;  // > 0: all of A staged in shared memory (M * K * 2 bytes);
                         // 0: A is read from global memory (L2) in place
};

// What one thread needs for one step besides the weights: its 32 activation
// elements of token t/4 (and t/4 + 8 for the second N tile), the scales of
// rows r0, r1 and their zeros as the fp16 constants of dequant_word.
template <int NT, bool kLut>
struct Operands {
    uint4 x[NT][4];
    float s0, s1;
    Zero2 z0, z1;
};

// xq[nt]: this thread's 32 activation elements of the step (shared or global
// memory, generic addressing).
template <int NT, bool kLut>
__device__ __forceinline__ void load_ops(const DecodeArgs &a, const __half *const (&xq)[NT],
                                         const __half *s_r0, const __half *s_r1,
                                         const uint8_t *z_r0, const uint8_t *z_r1, int st,
                                         Operands<NT, kLut> &P) {
    const int g = a.spg == 1 ? st : st / a.spg;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) P.x[nt][q] = *reinterpret_cast<const uint4 *>(xq[nt] + 8 * q);
    P.s0 = __half2float(s_r0[g * kRowsPerTile]);
    P.s1 = __half2float(s_r1[g * kRowsPerTile]);
    if (!kLut) {
        P.z0 = make_zero2(z_r0[g * kRowsPerTile]);
        P.z1 = make_zero2(z_r1[g * kRowsPerTile]);
    }
}

// One 128-element step of rows r0, r1 against tokens t/4 (+8): 8 (or 16)
// MMAs on exact q - z, scaled by s once in fp32. Two accumulator chains
// (even and odd words) halve the dependent MMA latency.
template <int NT, bool kLut>
__device__ __forceinline__ void step_mma(const Operands<NT, kLut> &P, const uint32_t *tbl,
                                         const uint8_t *wrow, int tok, int j, float (&tot)[NT][4]) {
    const uint4 wv0 = *reinterpret_cast<const uint4 *>(wrow + tok * 64 + 16 * j);
    const uint4 wv1 = *reinterpret_cast<const uint4 *>(wrow + (tok + 8) * 64 + 16 * j);
    const uint32_t w0[4] = {wv0.x, wv0.y, wv0.z, wv0.w};
    const uint32_t w1[4] = {wv1.x, wv1.y, wv1.z, wv1.w};
    float acc[2][NT][4];
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[c][nt][i] = 0.0f;
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        // (q - z) pairs of row r0 (u*) and row r1 (v*) for this word
        uint32_t u01, u23, u45, u67, v01, v23, v45, v67;
        if (kLut) {
            lut_word(w0[wi], tbl, u01, u23, u45, u67);
            lut_word(w1[wi], tbl, v01, v23, v45, v67);
        } else {
            dequant_word(w0[wi], P.z0, u01, u23, u45, u67);
            dequant_word(w1[wi], P.z1, v01, v23, v45, v67);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint4 xv = P.x[nt][wi];
            // MMA 2wi takes elements 8wi + 0..3 of each thread's 32 as the
            // fragment columns 2j, 2j+1, 2j+8, 2j+9; MMA 2wi + 1 elements
            // 8wi + 4..7. A (rows r0, r1) and B (token t/4) agree, so the
            // step's sum is unchanged.
            mma_16816(acc[wi & 1][nt], u01, v01, u23, v23, xv.x, xv.y);
            mma_16816(acc[wi & 1][nt], u45, v45, u67, v67, xv.z, xv.w);
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        tot[nt][0] = fmaf(P.s0, acc[0][nt][0] + acc[1][nt][0], tot[nt][0]);
        tot[nt][1] = fmaf(P.s0, acc[0][nt][1] + acc[1][nt][1], tot[nt][1]);
        tot[nt][2] = fmaf(P.s1, acc[0][nt][2] + acc[1][nt][2], tot[nt][2]);
        tot[nt][3] = fmaf(P.s1, acc[0][nt][3] + acc[1][nt][3], tot[nt][3]);
    }
}

template <int NT, bool kLut>
__global__ void __launch_bounds__(kDecodeThreads, NT == 1 ? 2 : 1)
    w4a16_decode_kernel(const DecodeArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ float red[kDecodeWarps][NT][4][32];
    __shared__ uint32_t pair_tbl[kLut ? 256 : 1];  // (LUT[i & 15], LUT[i >> 4]) as fp16 pairs
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ntiles = (a.N + kRowsPerTile - 1) / kRowsPerTile;
    const int64_t tb = (int64_t)blockIdx.x * ntiles / gridDim.x;
    const int64_t te = ((int64_t)blockIdx.x + 1) * ntiles / gridDim.x;
    const int64_t nsteps = a.K / kStepK;
    constexpr int sps = kStepsPerStage, S = kDStages;
    const int64_t spt = (nsteps + sps - 1) / sps;  // stages per tile
    // a tile's scales (16 rows x ng fp16) and zeros (16 x ng bytes), contiguous
    // in global memory and in its shared-memory slot
    const uint32_t s_bytes = (uint32_t)kRowsPerTile * (uint32_t)a.ng * 2u;
    const uint32_t z_bytes = kLut ? 0u : (uint32_t)kRowsPerTile * (uint32_t)a.ng;
    const uint32_t sz_slot = s_bytes + z_bytes;  // multiple of 32
    constexpr uint32_t ring_bytes = (uint32_t)S * kDStageBytes;

    // shared memory: weight ring | activations | scale/zero slots | barriers
    __half *x_sm = reinterpret_cast<__half *>(smem + ring_bytes);
    uint8_t *sz_sm = smem + ring_bytes + a.act_bytes;
    // the current tile's scales and zeros transposed to [group][16 rows], so
    // that the 8 rows a warp reads at once sit in neighbouring banks
    __half *s_tr = reinterpret_cast<__half *>(sz_sm + kSzSlots * sz_slot);
    uint8_t *z_tr = reinterpret_cast<uint8_t *>(s_tr) + s_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(z_tr + z_bytes);
    uint64_t *empty = full + kDStages;
    uint64_t *szfull = empty + kDStages;
    uint64_t *szempty = szfull + kSzSlots;
    uint64_t *actb = szempty + kSzSlots;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), kDecodeWarps);
        }
        for (int i = 0; i < kSzSlots; ++i) {
            mbar_init(smem_u32(&szfull[i]), 1);
            mbar_init(smem_u32(&szempty[i]), kDecodeWarps);
        }
        mbar_init(smem_u32(actb), 1);
        fence_barrier_init();
    }
    if (kLut) {
        // the table is weight data, like the scales: ready before the launch
        for (int i = threadIdx.x; i < 256; i += kDecodeThreads)
            pair_tbl[i] = (uint32_t)__half_as_ushort(a.lut[i & 15]) |
                          ((uint32_t)__half_as_ushort(a.lut[i >> 4]) << 16);
    }
    __syncthreads();

    if (warp == kDecodeWarps) {
        // ------------------------------------------------------------ producer
        // Per tile: its scales and zeros, then its weight stages; the ring
        // holds five stages, so every CTA keeps 80 KB of weights in flight.
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();  // every weight is read once
            if (a.act_bytes) {
                pdl_wait();  // the activations may come from the preceding kernel
                mbar_arrive_expect_tx(smem_u32(actb), a.act_bytes);
                bulk_g2s(smem_u32(x_sm), a.A, a.act_bytes, smem_u32(actb), policy_evict_last());
            }
            int64_t it = 0;
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int64_t tile = tb; tile < te && ok; ++tile) {
                const int64_t ti = tile - tb;
                const int zs = (int)(ti % kSzSlots);
                ok = mbar_wait(smem_u32(&szempty[zs]), (uint32_t)(((ti / kSzSlots) & 1) ^ 1), a.err);
                if (!ok) break;
                {
                    // the tile's rows of scales and zeros: the 16-byte multiple by
                    // bulk copy, a short tail (a partial last tile) by this thread
                    // before its arrival publishes the slot
                    const int64_t rows = a.N - tile * kRowsPerTile < kRowsPerTile
                                             ? a.N - tile * kRowsPerTile : kRowsPerTile;
                    const uint32_t sb = (uint32_t)rows * (uint32_t)a.ng * 2u;
                    const uint32_t zb = kLut ? 0u : (uint32_t)rows * (uint32_t)a.ng;
                    const uint32_t sb16 = sb & ~15u, zb16 = zb & ~15u;
                    const uint8_t *ssrc = reinterpret_cast<const uint8_t *>(a.S + tile * kRowsPerTile * a.ng);
                    const uint8_t *zsrc = kLut ? nullptr : a.Z + tile * kRowsPerTile * a.ng;
                    uint8_t *dst = sz_sm + zs * sz_slot;
                    for (uint32_t b = sb16; b < sb; ++b) dst[b] = ssrc[b];
                    for (uint32_t b = zb16; b < zb; ++b) dst[s_bytes + b] = zsrc[b];
                    const uint32_t bar = smem_u32(&szfull[zs]);
                    mbar_arrive_expect_tx(bar, sb16 + zb16);
                    if (sb16) bulk_g2s(smem_u32(dst), ssrc, sb16, bar, pol);
                    if (zb16) bulk_g2s(smem_u32(dst + s_bytes), zsrc, zb16, bar, pol);
                }
                for (int64_t sg = 0; sg < spt; ++sg, ++it) {
                    ok = mbar_wait(smem_u32(&empty[s]), ph ^ 1u, a.err);
                    if (!ok) break;
                    const int64_t step0 = sg * sps;
                    const int64_t nst = nsteps - step0 < sps ? nsteps - step0 : sps;
                    const uint32_t bar = smem_u32(&full[s]);
                    // steps past K are not copied (and never read)
                    mbar_arrive_expect_tx(bar, (uint32_t)nst * 1024u);
                    bulk_g2s(smem_u32(smem + (size_t)s * kDStageBytes), a.W + (tile * nsteps + step0) * 1024,
                             (uint32_t)nst * 1024u, bar, pol);
                    if (++s == S) s = 0, ph ^= 1u;
                }
            }
            // drain: nothing may still be landing when the CTA exits
            for (int64_t k = it > S ? it - S : 0; k < it; ++k)
                mbar_wait(smem_u32(&full[k % S]), (uint32_t)((k / S) & 1), a.err);
            const int64_t nt_issued = te - tb;
            for (int64_t k = nt_issued > kSzSlots ? nt_issued - kSzSlots : 0; k < nt_issued; ++k)
                mbar_wait(smem_u32(&szfull[k % kSzSlots]), (uint32_t)((k / kSzSlots) & 1), a.err);
            if (a.act_bytes) mbar_wait(smem_u32(actb), 0, a.err);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // After a timed-out wait a warp stops waiting but keeps its place in the
    // per-tile barriers (results are garbage, the error word says so), so no
    // warp can be left waiting for another.
    const int j = lane & 3, tok = lane >> 2;
    bool ok = true;
    const __half *xs = a.A;
    if (a.act_bytes) {
        ok = mbar_wait(smem_u32(actb), 0, a.err);
        xs = x_sm;
    } else {
        pdl_wait();  // the activations may come from the preceding kernel
    }
    // tokens past M read a valid token's activations (they only feed outputs
    // that are never stored)
    int mt[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mt[nt] = nt * 8 + tok < a.M ? nt * 8 + tok : (int)a.M - 1;
    int64_t it = 0;
    int s = 0;
    uint32_t ph = 0;
    constexpr int kps = sps / kDecodeWarps;  // this warp's steps per stage
    for (int64_t tile = tb; tile < te; ++tile) {
        const int64_t ti = tile - tb;
        const int zs = (int)(ti % kSzSlots);
        if (ok) ok = mbar_wait(smem_u32(&szfull[zs]), (uint32_t)((ti / kSzSlots) & 1), a.err);
        const int64_t r0 = tile * kRowsPerTile + tok, r1 = r0 + 8;
        // Rows past N (zero weights) and tokens past M read valid addresses
        // (clamped tokens, stale scale slots); they only feed outputs that are
        // never stored, so no load needs a predicate.
        {
            const __half *s_all = reinterpret_cast<const __half *>(sz_sm + zs * sz_slot);
            const uint8_t *z_all = sz_sm + zs * sz_slot + s_bytes;
            for (int i = threadIdx.x; i < kRowsPerTile * a.ng; i += kDecodeWarps * 32) {
                const int r = i / a.ng, g = i - r * a.ng;
                s_tr[g * kRowsPerTile + r] = s_all[i];
                if (!kLut) z_tr[g * kRowsPerTile + r] = z_all[i];
            }
            consumers_sync();
            if (lane == 0) mbar_arrive(smem_u32(&szempty[zs]));  // slot free again
        }
        // scales / zeros of rows r0, r1 for group g at index g * 16 (stride 16)
        const __half *s_r0 = s_tr + tok, *s_r1 = s_tr + tok + 8;
        const uint8_t *z_r0 = z_tr + tok, *z_r1 = z_tr + tok + 8;
        float tot[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) tot[nt][i] = 0.0f;
        // This warp's steps are warp + 8k, k = 0 .. nk-1, two per stage. While
        // it computes step k it has the operands of step k + 1 in flight (two
        // register sets, alternating).
        const int nk = warp < nsteps ? (int)((nsteps - 1 - warp) / kDecodeWarps) + 1 : 0;
        Operands<NT, kLut> P[2];
        auto ops = [&](int k, Operands<NT, kLut> &Q) {
            const int64_t st = warp + (int64_t)k * kDecodeWarps;
            const __half *xq[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) xq[nt] = xs + (int64_t)mt[nt] * a.K + st * kStepK + 32 * j;
            load_ops<NT, kLut>(a, xq, s_r0, s_r1, z_r0, z_r1, (int)st, Q);
        };
        if (nk > 0) ops(0, P[0]);
        for (int64_t sg = 0; sg < spt; ++sg, ++it) {
            if (ok) ok = mbar_wait(smem_u32(&full[s]), ph, a.err);
            const uint8_t *stage = smem + (size_t)s * kDStageBytes;
#pragma unroll
            for (int h = 0; h < kps; ++h) {
                const int k = (int)sg * kps + h;
                if (k < nk) {
                    if (k + 1 < nk) ops(k + 1, P[(h + 1) & 1]);
                    step_mma<NT, kLut>(P[h & 1], pair_tbl, stage + (warp + h * kDecodeWarps) * 1024, tok, j,
                                       tot);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
            if (++s == S) s = 0, ph ^= 1u;
        }
        // reduce the consumer warps' partial sums of this tile
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) red[warp][nt][i][lane] = tot[nt][i];
        consumers_sync();
        if (warp < NT) {
            const int nt = warp;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float sum = 0.0f;
#pragma unroll
                for (int w = 0; w < kDecodeWarps; ++w) sum += red[w][nt][i][lane];
                // c0, c1: row t/4, tokens 2j, 2j+1; c2, c3: row t/4 + 8
                const int64_t n = (i < 2) ? r0 : r1;
                const int64_t m = nt * 8 + 2 * j + (i & 1);
                if (n < a.N && m < a.M) a.C[m * a.N + n] = __float2half_rn(sum);
            }
        }
        consumers_sync();
    }
}

// ------------------------------------------------------------------ repack
// Nibble slot p of a packed word holds element kPackOrder[p] of the word.
__device__ __forceinline__ uint32_t pack_word(uint32_t c) {
    uint32_t p = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t slot = (i & 1) ? 4 + (i >> 1) : (i >> 1);
        p |= ((c >> (4 * i)) & 15u) << (4 * slot);
    }
    return p;
}
__device__ __forceinline__ uint32_t unpack_word(uint32_t p) {
    uint32_t c = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t slot = (i & 1) ? 4 + (i >> 1) : (i >> 1);
        c |= ((p >> (4 * slot)) & 15u) << (4 * i);
    }
    return c;
}
// Word index in the packed buffer of word c of row n (K/8 words per row).
__host__ __device__ __forceinline__ int64_t packed_index(int64_t n, int64_t c, int64_t nsteps) {
    const int64_t t = n / kRowsPerTile, r = n % kRowsPerTile;
    const int64_t st = c / (kStepK / 8), w = c % (kStepK / 8);
    return ((t * nsteps + st) * kRowsPerTile + r) * (kStepK / 8) + w;
}
// One thread per packed word (padding rows included): forward reads the
// canonical word (or writes zero for a padding row), inverse writes it back.
__global__ void w4a16_repack_kernel(const uint32_t *__restrict__ src, uint32_t *__restrict__ dst,
                                    int64_t N, int64_t K, bool inverse) {
    const int64_t kw = K / 8, nsteps = K / kStepK;
    const int64_t npad = (N + kRowsPerTile - 1) / kRowsPerTile * kRowsPerTile;
    const int64_t total = npad * kw;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / kw, c = i % kw;
        const int64_t pi = packed_index(n, c, nsteps);
        if (!inverse)
            dst[pi] = n < N ? pack_word(src[n * kw + c]) : 0u;
        else if (n < N)
            dst[n * kw + c] = unpack_word(src[pi]);
    }
}

}  // namespace

cudaError_t launch_w4a16_repack(bool inverse, const void *src, void *dst, int64_t N, int64_t K,
                                cudaStream_t s) {
    const int64_t nwords = (N + kRowsPerTile - 1) / kRowsPerTile * kRowsPerTile * (K / 8);
    int64_t grid = (nwords + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    w4a16_repack_kernel<<<(int)grid, 256, 0, s>>>(static_cast<const uint32_t *>(src),
                                                  static_cast<uint32_t *>(dst), N, K, inverse);
    count_launch();
    return cudaGetLastError();
}

template <int NT, bool kLut>
cudaError_t launch_decode_nt(const DecodeArgs &a, int64_t grid, size_t smem, cudaStream_t s) {
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(w4a16_decode_kernel<NT, kLut>), (int)smem);
    if (e != cudaSuccess) return e;
    w4a16_decode_kernel<NT, kLut><<<(unsigned)grid, kDecodeThreads, smem, s>>>(a);
    return cudaSuccess;
}

cudaError_t launch_w4a16_decode(const void *W, const __half *S, const uint8_t *Z, const __half *lut,
                                int64_t G, const __half *A, __half *C, int64_t M, int64_t N, int64_t K,
                                cudaStream_t s) {
    DecodeArgs a;
    a.W = static_cast<const uint8_t *>(W);
    a.S = S;
    a.Z = Z;
    a.lut = lut;
    a.A = A;
    a.C = C;
    a.M = M;
    a.N = N;
    a.K = K;
    a.G = G;
    a.ng = (int)(K / G);
    a.spg = (int)(G / kStepK);
    a.err = device_error_word();
    const int64_t ntiles = (N + kRowsPerTile - 1) / kRowsPerTile;
    // all of A in shared memory when it is small (one bulk copy per CTA)
    const size_t act = (size_t)M * K * 2;
    a.act_bytes = act <= kActStageMax ? (uint32_t)act : 0u;
    const size_t sz = (size_t)(kSzSlots + 1) * kRowsPerTile * a.ng * 3;
    const size_t bars = (2 * kDStages + 2 * kSzSlots + 1) * 8;
    const int64_t grid = balanced_grid(ntiles, (M <= 8 ? 2 : 1) * (int64_t)sm_count());
    const size_t smem = (size_t)kDStages * kDStageBytes + a.act_bytes + sz + bars;
    cudaError_t e;
    if (M <= 8)
        e = lut ? launch_decode_nt<1, true>(a, grid, smem, s) : launch_decode_nt<1, false>(a, grid, smem, s);
    else
        e = lut ? launch_decode_nt<2, true>(a, grid, smem, s) : launch_decode_nt<2, false>(a, grid, smem, s);
    if (e != cudaSuccess) return e;
    count_launch();
    return cudaGetLastError();
}

// Zero points packed 8 per word like the codes ([N][ceil(ng/8)] words,
// group g of row n at bits 4 (g mod 8) of word g / 8) -> uint8 [N][ng], the
// layout the W4A16 kernels read; once, at load time, like the repack.
__global__ void __launch_bounds__(256) w4a16_unpack_zeros_kernel(const uint32_t *__restrict__ zp,
                                                                 uint8_t *__restrict__ z, int64_t N,
                                                                 int64_t ng) {
    const int64_t words = (ng + 7) / 8, total = N * ng;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / ng, g = i - n * ng;
        z[i] = (uint8_t)((zp[n * words + g / 8] >> (4 * (g % 8))) & 15u);
    }
}

cudaError_t launch_w4a16_unpack_zeros(const uint32_t *zp, uint8_t *z, int64_t N, int64_t ng,
                                      cudaStream_t s) {
    const int64_t total = N * ng;
    int64_t grid = (total + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    w4a16_unpack_zeros_kernel<<<(unsigned)grid, 256, 0, s>>>(zp, z, N, ng);
    count_launch();
    return cudaGetLastError();
}

}  // namespace qmm
