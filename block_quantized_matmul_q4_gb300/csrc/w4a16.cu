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
// consumers' 16-byte reads hit distinct banks) from the kernel's first
// instruction (programmatic dependent launch: the weights never depend on
// the preceding kernel), together with each tile's scales and zeros, row by
// row into one of two shared-memory slots whose rows are padded by 16 bytes
// (the 8 rows a warp reads at once fall in distinct banks). Small
// activations are staged in shared memory by the consumers once the
// preceding kernel is done, in rows of 64 elements padded to 144 bytes (the
// four 64-byte slices the lanes of a step read fall in distinct banks).
// Eight consumer warps split each stage's K, then reduce per tile; every
// operand of a step is loaded one step ahead.
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

// A register-only operation: not volatile, so the compiler may interleave
// independent MMAs with the loads and conversions around them.
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm(
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
    uint32_t act_bytes;  // kStagedA: A in shared memory, padded (actpad_bytes)
};

// Activations staged in shared memory: rows of 64 elements (128 B) padded to
// 144 B, so the four 64-byte slices the lanes j = 0..3 of a step read sit in
// distinct banks.
constexpr uint32_t kActRow = 64, kActRowBytes = 144;
__host__ __device__ inline uint32_t actpad_bytes(int64_t M, int64_t K) {
    return (uint32_t)((M * K / kActRow) * kActRowBytes);
}
// Scales and zeros of a tile in shared memory, row by row with 16 bytes of
// padding per row, so the 8 rows a warp reads at once sit in distinct banks
// (rows of ng fp16 scales, then rows of ng zero bytes; ng % 16 == 0).
__host__ __device__ inline uint32_t sz_stride_s(int ng) { return (uint32_t)ng * 2u + 16u; }
__host__ __device__ inline uint32_t sz_stride_z(int ng) { return (uint32_t)ng + 16u; }
__host__ __device__ inline uint32_t sz_slot_bytes(int ng, bool lut) {
    return kRowsPerTile * (sz_stride_s(ng) + (lut ? 0u : sz_stride_z(ng)));
}
constexpr int kSzSlots = 2;

// What one thread needs for one step besides the weights: its 32 activation
// elements of token t/4 (and t/4 + 8 for the second N tile), the scales of
// rows r0, r1 and their zeros as the fp16 constants of dequant_word.
template <int NT>
struct Operands {
    uint4 x[NT][4];
    float s0, s1;
    Zero2 z0, z1;
};

// One 128-element step of rows r0, r1 against tokens t/4 (+8): 8 (or 16)
// MMAs on exact q - z (or LUT(q)) into two accumulator chains (even and odd
// words, halving the dependent MMA latency), then scaled by s once in fp32.
template <int NT, bool kLut>
__device__ __forceinline__ void step_mma(const Operands<NT> &P, const uint32_t *tbl, uint4 wv0, uint4 wv1,
                                         float (&tot)[NT][4]) {
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

// The decode kernel. kStagedA: all of A sits in shared memory (copied in by
// the consumers into the padded layout), else it is read in place from
// global memory (L2). kSzSmem: the producer copies each tile's scales and
// zeros into one of two shared-memory slots (padded rows), else the
// consumers read them from global memory. The producer streams the CTA's
// tiles stage by stage from its first instruction on (the weights do not
// depend on the preceding kernel, which may still be running: programmatic
// dependent launch). Every operand of a step is loaded one step ahead.
template <int NT, bool kLut, bool kStagedA, bool kSzSmem>
__global__ void __launch_bounds__(kDecodeThreads, NT == 1 ? 2 : 1) w4a16_decode_kernel(const DecodeArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ float red[kDecodeWarps][NT][4][32];
    __shared__ uint32_t pair_tbl[kLut ? 256 : 1];  // (LUT[i & 15], LUT[i >> 4]) as fp16 pairs
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ntiles = (a.N + kRowsPerTile - 1) / kRowsPerTile;
    const int64_t tb = (int64_t)blockIdx.x * ntiles / gridDim.x;
    const int64_t te = ((int64_t)blockIdx.x + 1) * ntiles / gridDim.x;
    const int nsteps = (int)(a.K / kStepK);
    constexpr int sps = kStepsPerStage, S = kDStages;
    const int spt = (nsteps + sps - 1) / sps;  // stages per tile
    constexpr uint32_t ring_bytes = (uint32_t)S * kDStageBytes;
    const uint32_t ss = sz_stride_s(a.ng), zs = sz_stride_z(a.ng), slot_bytes = sz_slot_bytes(a.ng, kLut);

    // shared memory: weight ring | activations (kStagedA) | scale/zero slots (kSzSmem) | barriers
    const uint32_t act_sm = smem_u32(smem) + ring_bytes;
    const uint32_t sz_sm = act_sm + (kStagedA ? a.act_bytes : 0u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + ring_bytes + (kStagedA ? a.act_bytes : 0u) +
                                                  (kSzSmem ? kSzSlots * slot_bytes : 0u));
    uint64_t *empty = full + kDStages;
    uint64_t *szfull = empty + kDStages;
    uint64_t *szempty = szfull + kSzSlots;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), kDecodeWarps);
        }
        for (int i = 0; i < kSzSlots; ++i) {
            mbar_init(smem_u32(&szfull[i]), 1);
            mbar_init(smem_u32(&szempty[i]), kDecodeWarps);
        }
        fence_barrier_init();
        pdl_launch_dependents();  // the next kernel may start streaming its weights
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
        // Per tile: its scales and zeros (kSzSmem), then its weight stages;
        // the ring holds five 16 KB stages, so every CTA keeps 80 KB of
        // weights in flight.
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();  // every weight is read once
            int64_t it = 0;
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int64_t tile = tb; tile < te && ok; ++tile) {
                if (kSzSmem) {
                    const int64_t ti = tile - tb;
                    const int zsl = (int)(ti % kSzSlots);
                    ok = mbar_wait(smem_u32(&szempty[zsl]), (uint32_t)(((ti / kSzSlots) & 1) ^ 1), a.err);
                    if (!ok) break;
                    const int rows = (int)(a.N - tile * kRowsPerTile < kRowsPerTile ? a.N - tile * kRowsPerTile
                                                                                   : kRowsPerTile);
                    const uint32_t sb = (uint32_t)a.ng * 2u, zb = (uint32_t)a.ng;
                    const uint32_t bar = smem_u32(&szfull[zsl]);
                    const uint32_t dst = sz_sm + (uint32_t)zsl * slot_bytes;
                    mbar_arrive_expect_tx(bar, (uint32_t)rows * (sb + (kLut ? 0u : zb)));
                    for (int r = 0; r < rows; ++r) {
                        const int64_t n = tile * kRowsPerTile + r;
                        bulk_g2s(dst + r * ss, a.S + n * a.ng, sb, bar, pol);
                        if (!kLut) bulk_g2s(dst + kRowsPerTile * ss + r * zs, a.Z + n * a.ng, zb, bar, pol);
                    }
                }
                for (int sg = 0; sg < spt; ++sg, ++it) {
                    ok = mbar_wait(smem_u32(&empty[s]), ph ^ 1u, a.err);
                    if (!ok) break;
                    const int step0 = sg * sps;
                    const int nst = nsteps - step0 < sps ? nsteps - step0 : sps;
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
            if (kSzSmem) {
                const int64_t nt_issued = te - tb;
                for (int64_t k = nt_issued > kSzSlots ? nt_issued - kSzSlots : 0; k < nt_issued; ++k)
                    mbar_wait(smem_u32(&szfull[k % kSzSlots]), (uint32_t)((k / kSzSlots) & 1), a.err);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // After a timed-out wait a warp stops waiting but keeps its place in the
    // per-tile barriers (results are garbage, the error word says so), so no
    // warp can be left waiting for another.
    const int j = lane & 3, tok = lane >> 2;
    bool ok = true;
    pdl_wait();  // the activations may come from the preceding kernel
    if (kStagedA) {
        // A into the padded layout: 16 bytes per thread per pass
        const uint32_t nchunks = (uint32_t)(a.M * a.K / 8);
        for (uint32_t c = threadIdx.x; c < nchunks; c += kDecodeWarps * 32) {
            const uint4 v = ldg_nc128(a.A + 8 * (size_t)c);
            const uint32_t e = 8u * c;
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(act_sm + (e / kActRow) * kActRowBytes +
                                                                          (e % kActRow) * 2u),
                         "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                         : "memory");
        }
        consumers_sync();
    }
    // tokens past M read a valid token's activations (they only feed outputs
    // that are never stored)
    uint32_t xrow[NT];  // kStagedA: padded row of element tok_row * K + 32 j; else its element offset
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const uint32_t e0 = (uint32_t)((nt * 8 + tok < a.M ? nt * 8 + tok : a.M - 1) * a.K) + 32u * j;
        xrow[nt] = kStagedA ? act_sm + (e0 / kActRow) * kActRowBytes + (e0 % kActRow) * 2u : e0;
    }
    int64_t it = 0;
    int s = 0;
    uint32_t ph = 0;
    constexpr int kps = sps / kDecodeWarps;  // this warp's steps per stage
    const int nk = warp < nsteps ? (nsteps - 1 - warp) / kDecodeWarps + 1 : 0;
    for (int64_t tile = tb; tile < te; ++tile) {
        const int64_t ti = tile - tb;
        const int zsl = (int)(ti % kSzSlots);
        if (kSzSmem && ok) ok = mbar_wait(smem_u32(&szfull[zsl]), (uint32_t)((ti / kSzSlots) & 1), a.err);
        const int64_t r0 = tile * kRowsPerTile + tok, r1 = r0 + 8;
        // Rows past N (zero weights) read row N - 1's scales and zeros (or a
        // stale slot row); they only feed outputs that are never stored, so
        // no load needs a predicate.
        const int64_t rc0 = r0 < a.N ? r0 : a.N - 1, rc1 = r1 < a.N ? r1 : a.N - 1;
        const __half *s_r0 = a.S + rc0 * a.ng, *s_r1 = a.S + rc1 * a.ng;
        const uint8_t *z_r0 = kLut ? nullptr : a.Z + rc0 * a.ng;
        const uint8_t *z_r1 = kLut ? nullptr : a.Z + rc1 * a.ng;
        const uint32_t slot = sz_sm + (uint32_t)zsl * slot_bytes;
        const uint32_t ss0 = slot + tok * ss, ss1 = ss0 + 8 * ss;
        const uint32_t zs0 = slot + kRowsPerTile * ss + tok * zs, zs1 = zs0 + 8 * zs;
        float tot[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) tot[nt][i] = 0.0f;
        // This warp's steps are warp + 8k, k = 0 .. nk-1, two per stage. While
        // it computes step k it has the operands of step k + 1 in flight (two
        // register sets, alternating).
        Operands<NT> P[2];
        auto ops = [&](int k, Operands<NT> &Q) {
            const int st = warp + k * kDecodeWarps;
            const int g = a.spg == 1 ? st : st / a.spg;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (kStagedA) {
                    const uint32_t ad = xrow[nt] + (uint32_t)st * (2u * kActRowBytes);
#pragma unroll
                    for (int q = 0; q < 4; ++q) Q.x[nt][q] = lds128(ad + 16u * q);
                } else {
                    const uint32_t e = xrow[nt] + (uint32_t)st * kStepK;
#pragma unroll
                    for (int q = 0; q < 4; ++q) Q.x[nt][q] = ldg_nc128(a.A + e + 8 * q);
                }
            }
            if (kSzSmem) {
                uint32_t h0, h1;
                asm volatile("ld.shared.u16 %0, [%1];" : "=r"(h0) : "r"(ss0 + 2u * g));
                asm volatile("ld.shared.u16 %0, [%1];" : "=r"(h1) : "r"(ss1 + 2u * g));
                Q.s0 = __half2float(__ushort_as_half((unsigned short)h0));
                Q.s1 = __half2float(__ushort_as_half((unsigned short)h1));
                if (!kLut) {
                    uint32_t z0, z1;
                    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(z0) : "r"(zs0 + g));
                    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(z1) : "r"(zs1 + g));
                    Q.z0 = make_zero2(z0);
                    Q.z1 = make_zero2(z1);
                }
            } else {
                Q.s0 = __half2float(__ldg(s_r0 + g));
                Q.s1 = __half2float(__ldg(s_r1 + g));
                if (!kLut) {
                    Q.z0 = make_zero2(__ldg(z_r0 + g));
                    Q.z1 = make_zero2(__ldg(z_r1 + g));
                }
            }
        };
        if (nk > 0) ops(0, P[0]);
        for (int sg = 0; sg < spt; ++sg, ++it) {
            if (ok) ok = mbar_wait(smem_u32(&full[s]), ph, a.err);
            const uint32_t stage = smem_u32(smem) + (uint32_t)s * kDStageBytes + tok * 64u + 16u * j;
#pragma unroll
            for (int h = 0; h < kps; ++h) {
                const int k = sg * kps + h;
                if (k < nk) {
                    if (k + 1 < nk) ops(k + 1, P[(h + 1) & 1]);
                    const uint32_t w = stage + (uint32_t)(warp + h * kDecodeWarps) * 1024u;
                    step_mma<NT, kLut>(P[h & 1], pair_tbl, lds128(w), lds128(w + 512u), tot);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
            if (++s == S) s = 0, ph ^= 1u;
        }
        // this tile's scale/zero slot is free again
        __syncwarp();
        if (kSzSmem && lane == 0) mbar_arrive(smem_u32(&szempty[zsl]));
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

// K-major decode, for 9..16 tokens whose activations are too large for the
// staged layout (M K > 8192 elements; 16 tokens of K = 8192 are 256 KB). The kernel above would
// fetch every step's activation fragments from L2 once per tile, with the
// load latency on each step's critical path. Here a CTA takes up to
// kKmTiles of its tiles at a time, 16-step chunk of K by chunk: the
// producer bulk-copies the chunk of A ([M][2048] fp16, one copy per token
// into a row skewed by 16 bytes so that the eight tokens a step reads fall
// in different banks) into one of two shared-memory slots once, and all of
// those tiles' weight stages of that chunk read it. Each tile keeps its
// own partial sums (statically indexed), reduced across the consumer warps
// at the end. Scales and zeros are read from global memory for each (tile,
// chunk), ahead of the chunk's MMAs -- from shared memory where every row of
// them is a multiple of 16 bytes (kSzSmem: the producer copies the scales and
// zeros of a group's tiles into one slot each, as the kernel above does per
// tile), else from global memory.
constexpr int kKmTiles = 4;
constexpr int kKmASlots = 2;
constexpr int kKmStages = 4;  // weight stages (the A slots take the room of the fifth)
constexpr uint32_t kKmTokBytes = kStepsPerStage * kStepK * 2 + 16;  // one token's chunk, skewed
__host__ __device__ inline uint32_t km_slot_bytes(int64_t M) {
    return (uint32_t)(((uint64_t)M * kKmTokBytes + 127) & ~127ull);
}

template <bool kLut, bool kSzSmem>
__global__ void __launch_bounds__(kDecodeThreads, 1) w4a16_decode_kmajor_kernel(const DecodeArgs a) {
    constexpr int NT = 2;  // 9..16 tokens
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ float red[kDecodeWarps][NT][4][32];
    __shared__ uint32_t pair_tbl[kLut ? 256 : 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ntiles = (a.N + kRowsPerTile - 1) / kRowsPerTile;
    const int64_t tb = (int64_t)blockIdx.x * ntiles / gridDim.x;
    const int64_t te = ((int64_t)blockIdx.x + 1) * ntiles / gridDim.x;
    const int nsteps = (int)(a.K / kStepK);
    constexpr int sps = kStepsPerStage, S = kKmStages;
    const int spt = (nsteps + sps - 1) / sps;  // chunks of K
    constexpr uint32_t ring_bytes = (uint32_t)S * kDStageBytes;
    const uint32_t slot_bytes = km_slot_bytes(a.M);
    const uint32_t a_sm = smem_u32(smem) + ring_bytes;
    const uint32_t ss = sz_stride_s(a.ng), zs = sz_stride_z(a.ng), sz_bytes = sz_slot_bytes(a.ng, kLut);
    const uint32_t sz_sm = a_sm + kKmASlots * slot_bytes;  // kKmTiles scale/zero slots (kSzSmem)
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + ring_bytes + kKmASlots * slot_bytes +
                                                  (kSzSmem ? kKmTiles * sz_bytes : 0u));
    uint64_t *empty = full + S;
    uint64_t *afull = empty + S;
    uint64_t *aempty = afull + kKmASlots;
    uint64_t *szfull = aempty + kKmASlots;
    uint64_t *szempty = szfull + kKmTiles;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), kDecodeWarps);
        }
        for (int i = 0; i < kKmASlots; ++i) {
            mbar_init(smem_u32(&afull[i]), 1);
            mbar_init(smem_u32(&aempty[i]), kDecodeWarps);
        }
        for (int i = 0; i < kKmTiles; ++i) {
            mbar_init(smem_u32(&szfull[i]), 1);
            mbar_init(smem_u32(&szempty[i]), kDecodeWarps);
        }
        fence_barrier_init();
        pdl_launch_dependents();  // the next kernel may start streaming its weights
    }
    if (kLut) {
        for (int i = threadIdx.x; i < 256; i += kDecodeThreads)
            pair_tbl[i] = (uint32_t)__half_as_ushort(a.lut[i & 15]) |
                          ((uint32_t)__half_as_ushort(a.lut[i >> 4]) << 16);
    }
    __syncthreads();

    if (warp == kDecodeWarps) {
        // ------------------------------------------------------------ producer
        // Per group of tiles and chunk: the A chunk (after the first chunk's
        // weights, so that those stream before the wait for the preceding
        // kernel), then one weight stage per tile of the group.
        if (lane == 0) {
            const uint64_t pol = policy_evict_first(), pol_a = policy_evict_last();
            int64_t it = 0, ai = 0;
            int s = 0;
            uint32_t ph = 0;
            bool ok = true, released = false;
            auto a_chunk = [&](int sg) {
                if (!released) {
                    pdl_wait();  // A may be written by the preceding kernel
                    released = true;
                }
                const int as = (int)(ai % kKmASlots);
                ok = mbar_wait(smem_u32(&aempty[as]), (uint32_t)(((ai / kKmASlots) & 1) ^ 1), a.err);
                if (!ok) return;
                const int nst = nsteps - sg * sps < sps ? nsteps - sg * sps : sps;
                const uint32_t bar = smem_u32(&afull[as]);
                mbar_arrive_expect_tx(bar, (uint32_t)a.M * (uint32_t)nst * (kStepK * 2));
                for (int64_t m = 0; m < a.M; ++m)
                    bulk_g2s(a_sm + (uint32_t)as * slot_bytes + (uint32_t)m * kKmTokBytes,
                             a.A + m * a.K + (int64_t)sg * sps * kStepK, (uint32_t)nst * (kStepK * 2), bar, pol_a);
                ++ai;
            };
            int64_t gi = 0;  // groups issued
            for (int64_t g0 = tb; g0 < te && ok; g0 += kKmTiles, ++gi) {
                const int64_t g1 = te - g0 < kKmTiles ? te : g0 + kKmTiles;
                // the group's scales and zeros, one slot per tile (weight data:
                // ready before the launch, like the weights)
                for (int64_t tile = g0; kSzSmem && tile < g1 && ok; ++tile) {
                    const int ti = (int)(tile - g0);
                    ok = mbar_wait(smem_u32(&szempty[ti]), (uint32_t)((gi & 1) ^ 1), a.err);
                    if (!ok) break;
                    const int rows = (int)(a.N - tile * kRowsPerTile < kRowsPerTile ? a.N - tile * kRowsPerTile
                                                                                   : kRowsPerTile);
                    const uint32_t sb = (uint32_t)a.ng * 2u, zb = (uint32_t)a.ng;
                    const uint32_t bar = smem_u32(&szfull[ti]);
                    const uint32_t dst = sz_sm + (uint32_t)ti * sz_bytes;
                    mbar_arrive_expect_tx(bar, (uint32_t)rows * (sb + (kLut ? 0u : zb)));
                    for (int r = 0; r < rows; ++r) {
                        const int64_t n = tile * kRowsPerTile + r;
                        bulk_g2s(dst + r * ss, a.S + n * a.ng, sb, bar, pol);
                        if (!kLut) bulk_g2s(dst + kRowsPerTile * ss + r * zs, a.Z + n * a.ng, zb, bar, pol);
                    }
                }
                for (int sg = 0; sg < spt && ok; ++sg) {
                    if (released) a_chunk(sg);
                    const int nst = nsteps - sg * sps < sps ? nsteps - sg * sps : sps;
                    for (int64_t tile = g0; tile < g1 && ok; ++tile, ++it) {
                        ok = mbar_wait(smem_u32(&empty[s]), ph ^ 1u, a.err);
                        if (!ok) break;
                        const uint32_t bar = smem_u32(&full[s]);
                        mbar_arrive_expect_tx(bar, (uint32_t)nst * 1024u);
                        bulk_g2s(smem_u32(smem + (size_t)s * kDStageBytes), a.W + (tile * nsteps + sg * sps) * 1024,
                                 (uint32_t)nst * 1024u, bar, pol);
                        if (++s == S) s = 0, ph ^= 1u;
                    }
                    if (!released && ok) a_chunk(sg);  // the very first chunk
                }
            }
            // drain: nothing may still be landing when the CTA exits
            for (int64_t k = it > S ? it - S : 0; k < it; ++k)
                mbar_wait(smem_u32(&full[k % S]), (uint32_t)((k / S) & 1), a.err);
            for (int64_t k = ai > kKmASlots ? ai - kKmASlots : 0; k < ai; ++k)
                mbar_wait(smem_u32(&afull[k % kKmASlots]), (uint32_t)((k / kKmASlots) & 1), a.err);
            if (kSzSmem && gi > 0) {  // the last group's slots
                const int64_t glast = tb + (gi - 1) * kKmTiles;
                const int nlast = (int)(te - glast < kKmTiles ? te - glast : kKmTiles);
                for (int ti = 0; ti < nlast; ++ti)
                    mbar_wait(smem_u32(&szfull[ti]), (uint32_t)((gi - 1) & 1), a.err);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // A timed-out wait leaves `ok` false: the warp stops waiting but keeps its
    // place in the barriers (results are garbage, the error word says so).
    const int j = lane & 3, tok = lane >> 2;
    bool ok = true;
    pdl_wait();  // C is written below
    uint32_t xoff[NT];  // this lane's token row inside an A slot, at its 32 elements of a step
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        // tokens past M read a valid token's activations (their outputs are never stored)
        const int64_t m = nt * 8 + tok < a.M ? nt * 8 + tok : a.M - 1;
        xoff[nt] = (uint32_t)m * kKmTokBytes + 64u * j;
    }
    constexpr int kps = sps / kDecodeWarps;  // this warp's steps per chunk
    int64_t ai = 0, gi = 0;
    int s = 0;
    uint32_t ph = 0;
    for (int64_t g0 = tb; g0 < te; g0 += kKmTiles, ++gi) {
        const int ng_tiles = (int)(te - g0 < kKmTiles ? te - g0 : kKmTiles);
        if (kSzSmem) {
#pragma unroll
            for (int ti = 0; ti < kKmTiles; ++ti)
                if (ti < ng_tiles && ok) ok = mbar_wait(smem_u32(&szfull[ti]), (uint32_t)(gi & 1), a.err);
        }
        float tot[kKmTiles][NT][4];
#pragma unroll
        for (int ti = 0; ti < kKmTiles; ++ti)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) tot[ti][nt][i] = 0.0f;
        for (int sg = 0; sg < spt; ++sg, ++ai) {
            const int as = (int)(ai % kKmASlots);
            if (ok) ok = mbar_wait(smem_u32(&afull[as]), (uint32_t)((ai / kKmASlots) & 1), a.err);
            const uint32_t aslot = a_sm + (uint32_t)as * slot_bytes;
#pragma unroll
            for (int ti = 0; ti < kKmTiles; ++ti) {
                if (ti < ng_tiles) {
                    const int64_t tile = g0 + ti;
                    const int64_t r0 = tile * kRowsPerTile + tok, r1 = r0 + 8;
                    const int64_t rc0 = r0 < a.N ? r0 : a.N - 1, rc1 = r1 < a.N ? r1 : a.N - 1;
                    // this warp's steps of the chunk: their activations, scales, zeros
                    if (ok) ok = mbar_wait(smem_u32(&full[s]), ph, a.err);
                    const uint32_t stage = smem_u32(smem) + (uint32_t)s * kDStageBytes + tok * 64u + 16u * j;
                    // this warp's steps of the chunk, each with its activations,
                    // scales and zeros loaded just before its MMAs
#pragma unroll
                    for (int h = 0; h < kps; ++h) {
                        const int sl = warp + h * kDecodeWarps, st = sg * sps + sl;
                        if (st < nsteps) {
                            const int g = a.spg == 1 ? st : st / a.spg;
                            Operands<NT> P;
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    P.x[nt][q] = lds128(aslot + xoff[nt] + (uint32_t)sl * (kStepK * 2) + 16u * q);
                            if (kSzSmem) {
                                const uint32_t ss0 = sz_sm + (uint32_t)ti * sz_bytes + tok * ss, ss1 = ss0 + 8 * ss;
                                const uint32_t zs0 = sz_sm + (uint32_t)ti * sz_bytes + kRowsPerTile * ss + tok * zs;
                                uint32_t h0, h1;
                                asm volatile("ld.shared.u16 %0, [%1];" : "=r"(h0) : "r"(ss0 + 2u * g));
                                asm volatile("ld.shared.u16 %0, [%1];" : "=r"(h1) : "r"(ss1 + 2u * g));
                                P.s0 = __half2float(__ushort_as_half((unsigned short)h0));
                                P.s1 = __half2float(__ushort_as_half((unsigned short)h1));
                                if (!kLut) {
                                    uint32_t z0, z1;
                                    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(z0) : "r"(zs0 + g));
                                    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(z1) : "r"(zs0 + 8 * zs + g));
                                    P.z0 = make_zero2(z0);
                                    P.z1 = make_zero2(z1);
                                }
                            } else {
                                P.s0 = __half2float(__ldg(a.S + rc0 * a.ng + g));
                                P.s1 = __half2float(__ldg(a.S + rc1 * a.ng + g));
                                if (!kLut) {
                                    P.z0 = make_zero2(__ldg(a.Z + rc0 * a.ng + g));
                                    P.z1 = make_zero2(__ldg(a.Z + rc1 * a.ng + g));
                                }
                            }
                            const uint32_t w = stage + (uint32_t)sl * 1024u;
                            step_mma<NT, kLut>(P, pair_tbl, lds128(w), lds128(w + 512u), tot[ti]);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
                    if (++s == S) s = 0, ph ^= 1u;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&aempty[as]));  // the chunk's activations are read
        }
        // reduce the consumer warps' partial sums, tile by tile
#pragma unroll
        for (int ti = 0; ti < kKmTiles; ++ti) {
            if (ti < ng_tiles) {
                const int64_t tile = g0 + ti;
                const int64_t r0 = tile * kRowsPerTile + tok, r1 = r0 + 8;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) red[warp][nt][i][lane] = tot[ti][nt][i];
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
        if (kSzSmem) {  // the group's scale/zero slots are free again
            __syncwarp();
#pragma unroll
            for (int ti = 0; ti < kKmTiles; ++ti)
                if (ti < ng_tiles && lane == 0) mbar_arrive(smem_u32(&szempty[ti]));
        }
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

template <int NT, bool kLut, bool kStagedA, bool kSzSmem>
cudaError_t launch_decode_nt(const DecodeArgs &a, int64_t grid, size_t smem, cudaStream_t s) {
    auto fn = w4a16_decode_kernel<NT, kLut, kStagedA, kSzSmem>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(fn), (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kDecodeThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, a);
}

template <int NT, bool kLut>
cudaError_t launch_decode_m(const DecodeArgs &a, bool staged, bool szsmem, int64_t grid, size_t smem,
                            cudaStream_t s) {
    if (staged)
        return szsmem ? launch_decode_nt<NT, kLut, true, true>(a, grid, smem, s)
                      : launch_decode_nt<NT, kLut, true, false>(a, grid, smem, s);
    return szsmem ? launch_decode_nt<NT, kLut, false, true>(a, grid, smem, s)
                  : launch_decode_nt<NT, kLut, false, false>(a, grid, smem, s);
}

template <bool kLut, bool kSzSmem>
cudaError_t launch_decode_kmajor(const DecodeArgs &a, int64_t grid, size_t smem, cudaStream_t s) {
    auto fn = w4a16_decode_kmajor_kernel<kLut, kSzSmem>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(fn), (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kDecodeThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, a);
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
    // all of A in shared memory when it is small (padded rows); else, from
    // 9 tokens, the K-major kernel with A chunks in shared memory (8192^2, 16
    // tokens: 25.4 -> 19.6 us; with 8 or fewer, whose activation fragments are
    // fewer, reading them from L2 stays faster: 14.9 against 17.4 us at 8)
    const bool staged = (size_t)M * K * 2 <= kActStageMax;
    if (!staged && M > 8) {
        a.act_bytes = 0;
        const bool szk = a.ng % 16 == 0 && sz_slot_bytes(a.ng, lut != nullptr) <= 8192;
        const size_t smem = (size_t)kKmStages * kDStageBytes + kKmASlots * (size_t)km_slot_bytes(M) +
                            (szk ? (size_t)kKmTiles * sz_slot_bytes(a.ng, lut != nullptr) : 0) +
                            (2 * kKmStages + 2 * kKmASlots + 2 * kKmTiles) * 8;
        const int64_t grid = balanced_grid(ntiles, (int64_t)sm_count());
        const cudaError_t e = lut ? (szk ? launch_decode_kmajor<true, true>(a, grid, smem, s)
                                         : launch_decode_kmajor<true, false>(a, grid, smem, s))
                                  : (szk ? launch_decode_kmajor<false, true>(a, grid, smem, s)
                                         : launch_decode_kmajor<false, false>(a, grid, smem, s));
        count_launch();
        return e;
    }
    a.act_bytes = staged ? actpad_bytes(M, K) : 0u;
    // the tile's scales and zeros in shared memory when every row is a
    // multiple of 16 bytes and both slots fit beside the ring
    const bool szsmem = a.ng % 16 == 0 && sz_slot_bytes(a.ng, lut != nullptr) <= 16384;
    const size_t sz = szsmem ? (size_t)kSzSlots * sz_slot_bytes(a.ng, lut != nullptr) : 0;
    const size_t bars = (2 * kDStages + 2 * kSzSlots) * 8;
    const int64_t grid = balanced_grid(ntiles, (M <= 8 ? 2 : 1) * (int64_t)sm_count());
    const size_t smem = (size_t)kDStages * kDStageBytes + a.act_bytes + sz + bars;
    cudaError_t e;
    if (M <= 8)
        e = lut ? launch_decode_m<1, true>(a, staged, szsmem, grid, smem, s)
                : launch_decode_m<1, false>(a, staged, szsmem, grid, smem, s);
    else  // 9..16 tokens reach here only with the staged layout
        e = lut ? launch_decode_m<2, true>(a, true, szsmem, grid, smem, s)
                : launch_decode_m<2, false>(a, true, szsmem, grid, smem, s);
    count_launch();
    return e;
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
