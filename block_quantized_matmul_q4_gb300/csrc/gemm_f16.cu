// gemm_f16.cu -- tensor-core GEMMs whose weights are decoded to fp16 on the
// way into the operand (page 3, "BitBLAS 完全拆解": "边解码边计算"), for the
// formats whose scales cannot be taken out of the sum once per 256
// elements:
//   W4A16 (page 3, "从数学表达式到真实存储"): C = A w^T, w = fp16(s (q - z)),
//     A fp16 as given, C fp16.
//   Q4_0 prefill (page 1, "最基础的两块"): Y = a w^T, w = fp16(d_w (q - 8)),
//     a = fp16(d_a y) from the Q8_0 codes y of X (both sides carry a scale
//     per 32 elements, so no integer sum spans more than one MMA K step;
//     both operands are rounded once to fp16 instead), Y fp32.
//   Q4_K prefill (page 1, "K-quant", "6-bit 参数"): Y = a w^T, w =
//     fp16(d s_j q - dmin m_j) per sub-block of 32: the weight is formed in
//     fp32 (d s_j q is exact, one rounding for the difference) and rounded
//     once to fp16, so its error stays within 2^-11 |w| even where the two
//     terms nearly cancel; a = fp16(2^e d_a y) from the Q8_K codes y of X,
//     Y fp32.
//   Q6_K prefill (page 1, "更低的比特: Q6_K 与 Q2_K 的取舍"): Y = a w^T,
//     w = fp16(d s_j q) with q = u - 32 per group of 16 (d s_j q has at most
//     24 significant bits, so it is exact in fp32 and rounded once), a as
//     for Q4_K.
// In all, the codes are exact, every weight is its exact value rounded once
// to fp16 (relative error <= 2^-11), and every activation is 2^e d_a y
// rounded once to fp16, with a power of two 2^e per token that puts the
// token's largest block scale 2^e d_a in [2^7, 2^8) -- so its largest |a| is
// below 2^15 and its smaller ones stay in fp16's normal range for 28 more
// octaves, whatever the magnitude of X -- and that the epilogue takes off
// again (exact: a power of two). The MMA accumulates in fp32 over all of K.
//
// Tile = 128 weight rows (MMA M) x BN tokens (MMA N): BN = 256 above 128
// tokens (every decoded weight then serves 256 tokens), else 128. Up to one
// tile per SM the grid has one CTA per tile; with more, one CTA per SM walks
// a contiguous range of (tile, 256-element K round) units (stream-K): pieces
// of tiles that span two or more CTAs go to partial slots and a fixup
// kernel adds them (streamk.cu). With BN = 128 two TMEM accumulators let the
// MMAs of the next piece start while the epilogue drains the last one.
// 16 warps:
//   warp 0      activation producer: 16 KB stages, 2-D TMA tiles of BN
//               tokens by 64 (BN = 128, 128B swizzle) or 32 (BN = 256, 64B
//               swizzle) elements of K;
//   warp 1      MMA issuer (one thread) and TMEM owner;
//   warp 2      MMA waiter: the issuer's barrier waits, handed over per pair
//               of K chunks through a named barrier (a shared-memory access
//               by the issuing thread would drain the tensor pipe);
//   warps 3..10 converters, two sets of four: one weight row per thread
//               (its TMEM lane), fp16 weights built in registers and stored
//               into a TMEM operand ring with tcgen05.st;
//   warps 11..14 epilogue: one tcgen05.ld pass over the accumulator per
//               piece;
//   warp 15     weight producer: per 256 elements of K one weight stage (TMA
//               copies of the packed tiles of the CTA's 128 rows), as soon as
//               the converters free one.
// All mbarrier waits are bounded; on a timeout the CTA drains its copies and
// MMAs, frees its TMEM and returns with the device error word set.
#include <cstring>

#include "tc.cuh"

namespace qmm {
namespace {

enum Format { kW4A16 = 0, kQ40 = 1, kQ6K = 2, kQ4K = 3 };

constexpr int kBM = 128, kBK = 64;  // rows, K per chunk; the tile's token count BN is 128 or 256
constexpr int kSB = 256;            // K per pipeline round
constexpr int kChunks = kSB / kBK;  // 4
static_assert(kSB == kSkRound && kBM == kSkTile, "stream-K units");
constexpr int kGroups = 2;          // A handed over in pairs of chunks
constexpr int kARounds = 2;         // the A operand ring holds two rounds: converters run a round ahead
constexpr int kWStagesMax = 4;          // weight stages: 4 where shared memory allows, else 3
constexpr int kWBytesMax = 16 * kQ6Rec;  // largest weight stage: Q6_K, 16 records of 8 rows
constexpr int kConvWarps = 8, kEpiWarps = 4;
constexpr int kEpiWarp0 = 3 + kConvWarps, kWProdWarp = kEpiWarp0 + kEpiWarps;
constexpr int kThreads = (kWProdWarp + 1) * 32;
constexpr int kActRing = 128 * 1024;  // activation stages: 8 x 16 KB
constexpr int kOffAct = 0;
constexpr int kOffW = kOffAct + kActRing;
constexpr int kActStagesMax = 8;
constexpr int kNumBars = 2 * (kWStagesMax + kActStagesMax + kARounds * kGroups) + 5;  // + acc_full[2], acc_empty[2], done
constexpr uint32_t kTmemCols = 512;
// Epilogue output staging: 16 tokens x 128 rows (the C tile's 2-D TMA box),
// fp32 or fp16, double-buffered.
constexpr int kStageCols = 16;
constexpr int kStageBytes = kStageCols * kBM * 4;
constexpr uint32_t kARingCols = kBK / 2;

// Tile width BN (tokens): 128 with two TMEM accumulators, so the next
// piece's MMAs run while the epilogue drains the last one; or 256 with one
// (256 columns), so that every weight the converters decode serves twice as
// many tokens. Either way the accumulators take 256 columns and the A
// operand ring (two rounds of four 32-column chunks) the other 256. An
// activation stage is 16 KB either way: BN tokens x kActK elements of K (64
// with the 128-byte swizzle, or 32 with the 64-byte one), so that the ring
// always has eight stages and a stage is freed as soon as its own MMAs are
// done.
template <int BN>
struct Tile {
    static_assert(BN == 128 || BN == 256, "tile width");
    static constexpr int kAccs = BN == 128 ? 2 : 1;
    static constexpr int kActK = BN == 128 ? 64 : 32;
    static constexpr int kSlices = kBK / kActK;            // activation stages per 64-element chunk
    static constexpr int kActBytes = BN * kActK * 2;       // one activation stage
    static constexpr int kActStages = kActRing / kActBytes;
    static constexpr uint32_t kSwz = kActK == 64 ? 2 : 4;  // descriptor layout: 128- or 64-byte swizzle
    static constexpr uint32_t kSbo = 8 * kActK * 2;        // bytes per 8 rows
    static constexpr uint32_t kColARing = kAccs * BN;
    static_assert(kColARing + kARounds * kChunks * kARingCols <= kTmemCols, "TMEM budget");
    static_assert(kActStages <= kActStagesMax, "barriers");
};

// W4A16 packed tiles: 16 rows, steps of 128 elements (1 KB each).
constexpr int kW4StepK = 128, kW4Tile = 16;
// Q4_0 packed tiles: 8 rows; per tile [8][nb][16 B nibbles] then [nb][8] fp16.
constexpr int kQ4Tile = kTileRows;
constexpr int kQ4Blocks = kSB / QK4_0;  // blocks per stage: 8
constexpr int kQ4NibBytes = (kBM / kQ4Tile) * kQ4Blocks * kQ4Tile * 16;  // 16 KB

template <int F>
struct FmtInfo {
    static constexpr int kWBytes = F == kW4A16 ? (kBM / kW4Tile) * (kSB / kW4StepK) * 1024
                                   : F == kQ6K ? (kBM / kTileRows) * kQ6Rec
                                   : F == kQ4K ? (kBM / kTileRows) * kTileRows * B_Q4_K
                                               : kQ4NibBytes + (kBM / kQ4Tile) * kQ4Blocks * 16;
    static_assert(kWBytes <= kWBytesMax, "weight stage");
    // Shared memory: activation stages | weight stages (this format's size:
    // the unused rest of the SM's 228 KB stays L1, where the W4A16
    // converters' scale and zero reads hit) | W4A16 code table (256 fp16
    // pairs) or, for the other formats, the epilogue's token scales (up to
    // 256 floats) | the epilogue's two output staging blocks | barriers.
    static constexpr int kWStage = (kWBytes + 127) / 128 * 128;
    static constexpr int kFixed = kOffW + 1024 + 2 * kStageBytes + kNumBars * 8 + 16 + 1024;
    static constexpr int kWStages = kFixed + kWStagesMax * kWStage <= 227 * 1024 ? kWStagesMax : 3;
    static constexpr int kOffLut = kOffW + kWStages * kWStage;
    static constexpr int kOffStage = kOffLut + 1024;
    static constexpr int kOffBar = kOffStage + 2 * kStageBytes;
    static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

struct Args {
    const __half *S;   // W4A16: [N][ng]
    const uint8_t *Z;  // W4A16: [N][ng], unused with a table
    const __half *lut; // W4A16: 16 fp16 code values (W-hat = s LUT(q)), or null
    void *C;           // W4A16: fp16 [M][N]; Q4_0: fp32 [M][N]
    int64_t M, N, K;
    int ng, spg;  // W4A16: groups per row, 128-element steps per group
    unsigned *err;
    // stream-K: tile t = (row block t / mblocks, token block t % mblocks);
    // unit u = t * nsb + round; CTA c takes units [c U / G, (c+1) U / G)
    int64_t mblocks, units;
    float *part;  // split tiles: [CTA][slot 0: first tile, 1: last tile][BN cols][128 rows]
    const float *tok_scale;  // 2^-e per token (padded to 16), or null (W4A16)
    int c_tma;               // whole tiles go to C through tmap_c (rows of C 16-byte aligned), else plain stores
};

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
__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ void handoff_sync() { asm volatile("bar.sync 1, 64;" ::: "memory"); }
// the four epilogue warps
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

// fp16 scale * (q - zero) for the 8 codes of one word, as four pairs of
// (low 16 bits, high 16 bits) fields: fields at bits 0-3 | 16-19, 8-11 |
// 24-27 (via w >> 8), 4-7 | 20-23 and 12-15 | 28-31. zz = fp16(1024 + zero)
// twice, zh = fp16(-(64 + zero)) twice, ss = the scale twice. q - zero is
// exact (1024 + q minus 1024 + zero, or the x16 form through one FMA); the
// product with the scale is one rounding.
__device__ __forceinline__ void scaled_word(uint32_t w, uint32_t zz, uint32_t zh, uint32_t ss,
                                            uint32_t &f0, uint32_t &f8, uint32_t &f4,
                                            uint32_t &f12) {
    constexpr uint32_t kSixteenth = 0x2C002C00u;  // fp16 1/16 twice
    const uint32_t v = w >> 8;
    f0 = hmul2_u(hsub2_u(lop_or(w, 0x000F000Fu), zz), ss);
    f8 = hmul2_u(hsub2_u(lop_or(v, 0x000F000Fu), zz), ss);
    f4 = hmul2_u(hfma2_u(lop_or(w, 0x00F000F0u), kSixteenth, zh), ss);
    f12 = hmul2_u(hfma2_u(lop_or(v, 0x00F000F0u), kSixteenth, zh), ss);
}

// fp16 scale * LUT(q) for the 8 codes of one word (non-uniform codes, page
// 3: W-hat = s LUT(q)), the pairs (k0,k1), (k2,k3), (k4,k5), (k6,k7) in that
// order: slots j and j + 4 of the word hold elements 2j and 2j + 1, so one
// byte q_2j | q_2j+1 << 4 per pair indexes the table tbl[i] = (LUT[i & 15],
// LUT[i >> 4]). One rounding, the product with the scale.
__device__ __forceinline__ void lut_scaled_word(uint32_t w, const uint32_t *tbl, uint32_t ss,
                                                uint32_t &p01, uint32_t &p23, uint32_t &p45,
                                                uint32_t &p67) {
    const uint32_t t = (w & 0x0F0Fu) | ((w >> 12) & 0xF0F0u);          // pairs (0,1), (4,5)
    const uint32_t t2 = ((w >> 4) & 0x0F0Fu) | ((w >> 16) & 0xF0F0u);  // pairs (2,3), (6,7)
    p01 = hmul2_u(tbl[t & 0xFF], ss);
    p45 = hmul2_u(tbl[(t >> 8) & 0xFF], ss);
    p23 = hmul2_u(tbl[t2 & 0xFF], ss);
    p67 = hmul2_u(tbl[(t2 >> 8) & 0xFF], ss);
}

// Pairs of fp32 values (Blackwell's f32x2 arithmetic: one instruction for
// two lanes of work).
__device__ __forceinline__ uint64_t pack2(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ uint64_t f2(float lo, float hi) { return pack2(__float_as_uint(lo), __float_as_uint(hi)); }
__device__ __forceinline__ uint64_t add_f2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t mul_f2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma_f2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// fp32 pair -> fp16 pair (first value in the low half), round to nearest even.
__device__ __forceinline__ uint32_t h2_of_f2(uint64_t v) {
    uint32_t lo, hi, r;
    asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(__uint_as_float(hi)), "f"(__uint_as_float(lo)));
    return r;
}
// (x & mask) | 2^23's bit pattern: a field of x at bit p (p + width <= 23)
// becomes the float 2^23 + field 2^p, exactly.
__device__ __forceinline__ uint32_t magic23(uint32_t x, uint32_t mask) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(x), "r"(mask), "r"(0x4B000000u));
    return d;
}
constexpr float kTwo23 = 8388608.0f;

// The 4 Q6_K codes of one byte word u (bytes 0..3, stored u = q + 32) as two
// fp16 pairs (bytes 0, 1) and (2, 3) of d s_j q: byte b sits at bit p = 0,
// 8, 16 of u or 8 of u >> 16, its float 2^23 + u 2^p less 2^23 + 32 2^p is
// q 2^p exactly, and the product with (d s_j) 2^-p is exact (at most 24
// significant bits); one rounding, to fp16. s01 = (ds, ds 2^-8), s23 = (ds
// 2^-16, ds 2^-8).
__device__ __forceinline__ void q6k_pairs(uint32_t u, uint64_t s01, uint64_t s23, uint32_t &p01, uint32_t &p23) {
    const uint32_t v = u >> 16;
    const uint64_t f01 = pack2(magic23(u, 0x3Fu), magic23(u, 0x3F00u));
    const uint64_t f23 = pack2(magic23(u, 0x3F0000u), magic23(v, 0x3F00u));
    const uint64_t b01 = f2(-(kTwo23 + 32.0f), -(kTwo23 + 8192.0f));
    const uint64_t b23 = f2(-(kTwo23 + 2097152.0f), -(kTwo23 + 8192.0f));
    p01 = h2_of_f2(mul_f2(add_f2(f01, b01), s01));
    p23 = h2_of_f2(mul_f2(add_f2(f23, b23), s23));
}

// The 8 Q4_K codes of one word of qs bytes: the low nibbles are elements
// 0..3 of the low sub-block, the high nibbles elements 0..3 of the high one.
// Each becomes q 2^p exactly (its float 2^23 + q 2^p less 2^23; the nibble at
// bit p = 0, 8, 16 of w or 12 of w >> 12 for the low set, 4, 12 of w or 8,
// 16 of w >> 12 for the high set), then one fused multiply-add with
// (d s_j) 2^-p and -dmin m_j: the fp32 weight d s_j q - dmin m_j with one
// rounding, then rounded once to fp16. Output: fp16 pairs (0, 1), (2, 3) of
// each set. sl01 = (dsl, dsl 2^-8), sl23 = (dsl 2^-16, dsl 2^-12), sh01 =
// (dsh 2^-4, dsh 2^-12), sh23 = (dsh 2^-8, dsh 2^-16); nml, nmh = -dmin m_j
// twice.
__device__ __forceinline__ void q4k_word(uint32_t w, uint64_t sl01, uint64_t sl23, uint64_t nml, uint64_t sh01,
                                         uint64_t sh23, uint64_t nmh, uint32_t &l01, uint32_t &l23,
                                         uint32_t &h01, uint32_t &h23) {
    const uint32_t v = w >> 12;
    const uint64_t bias = f2(-kTwo23, -kTwo23);
    const uint64_t fl01 = pack2(magic23(w, 0xFu), magic23(w, 0xF00u));
    const uint64_t fl23 = pack2(magic23(w, 0xF0000u), magic23(v, 0xF000u));
    const uint64_t fh01 = pack2(magic23(w, 0xF0u), magic23(w, 0xF000u));
    const uint64_t fh23 = pack2(magic23(v, 0xF00u), magic23(v, 0xF0000u));
    l01 = h2_of_f2(fma_f2(add_f2(fl01, bias), sl01, nml));
    l23 = h2_of_f2(fma_f2(add_f2(fl23, bias), sl23, nml));
    h01 = h2_of_f2(fma_f2(add_f2(fh01, bias), sh01, nmh));
    h23 = h2_of_f2(fma_f2(add_f2(fh23, bias), sh23, nmh));
}

// Columns m0 .. m0+15 of output row n (C is [M][N]: fp16 for W4A16, fp32 for
// Q4_0); columns past M are skipped.
template <int F>
__device__ __forceinline__ void store_cols(const Args &a, int64_t m0, int64_t n, const float v[16]) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int64_t m = m0 + j;
        if (m < a.M) {
            if (F == kW4A16)
                static_cast<__half *>(a.C)[m * a.N + n] = __float2half_rn(v[j]);
            else
                static_cast<float *>(a.C)[m * a.N + n] = v[j];
        }
    }
}

// v[j] *= 2^-e of token j of the 16 at ts, in shared memory (the activation
// prescale taken off: exact, a power of two). ts is 16-byte aligned.
__device__ __forceinline__ void scale16_s(const float *ts, float v[16]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 t = reinterpret_cast<const float4 *>(ts)[i];
        v[4 * i] *= t.x;
        v[4 * i + 1] *= t.y;
        v[4 * i + 2] *= t.z;
        v[4 * i + 3] *= t.w;
    }
}

template <int F, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_f16_kernel(const Args a, const __grid_constant__ CUtensorMap tmap_w,
                    const __grid_constant__ CUtensorMap tmap_d,
                    const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_c) {
    constexpr int kWBytes = FmtInfo<F>::kWBytes, kWStages = FmtInfo<F>::kWStages;
    using T = Tile<BN>;
    constexpr int kActStages = T::kActStages, kActBytes = T::kActBytes, kAccs = T::kAccs;
    constexpr int kSlices = T::kSlices, kActK = T::kActK;
    constexpr uint32_t kColARing = T::kColARing;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t sbase = (raw_base + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw_base);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nsb = (a.K + kSB - 1) / kSB;
    // this CTA's units (stream-K): a contiguous range of (tile, round)
    const int64_t u0 = (int64_t)blockIdx.x * a.units / gridDim.x;
    const int64_t u1 = ((int64_t)blockIdx.x + 1) * a.units / gridDim.x;

    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + FmtInfo<F>::kOffBar);
    uint64_t *w_full = bar, *w_empty = w_full + kWStages;
    uint64_t *act_full = w_empty + kWStages, *act_empty = act_full + kActStages;
    // A ring slot group (round parity r, group g) = r * kGroups + g
    uint64_t *a_full = act_empty + kActStages, *a_empty = a_full + kARounds * kGroups;
    uint64_t *acc_full = a_empty + kARounds * kGroups, *acc_empty = acc_full + kAccs, *done = acc_empty + kAccs;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kWStages; ++i) {
            mbar_init(smem_u32(&w_full[i]), 1);
            mbar_init(smem_u32(&w_empty[i]), kConvWarps);
        }
        for (int i = 0; i < kActStages; ++i) {
            mbar_init(smem_u32(&act_full[i]), 1);
            mbar_init(smem_u32(&act_empty[i]), 1);
        }
        for (int i = 0; i < kARounds * kGroups; ++i) {
            mbar_init(smem_u32(&a_full[i]), kConvWarps);  // both sets, one chunk each
            mbar_init(smem_u32(&a_empty[i]), 1);
        }
        for (int i = 0; i < kAccs; ++i) {
            mbar_init(smem_u32(&acc_full[i]), 1);
            mbar_init(smem_u32(&acc_empty[i]), kEpiWarps);
        }
        mbar_init(smem_u32(done), 1);
        fence_barrier_init();
    }
    uint32_t *pair_tbl = reinterpret_cast<uint32_t *>(smem + FmtInfo<F>::kOffLut);
    if (F == kW4A16 && a.lut) {
        // the table is weight data, like the scales: ready before the launch
        for (int i = threadIdx.x; i < 256; i += kThreads)
            pair_tbl[i] = (uint32_t)__half_as_ushort(a.lut[i & 15]) |
                          ((uint32_t)__half_as_ushort(a.lut[i >> 4]) << 16);
    }
    __syncwarp();  // warps meet converged at every CTA barrier below
    if (warp == 1) tc::tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ activation producer
        if (lane == 0) {
            tc::prefetch_tensormap(&tmap_a);
            const uint64_t pol = policy_evict_last();  // A is reused by the other row blocks' CTAs
            pdl_wait();  // the activations may come from the preceding kernel
            int64_t issued_a = 0;
            bool ok = true;
            for (int64_t i = 0; i < u1 - u0 && ok; ++i) {
                const int64_t tile = (u0 + i) / nsb, sb = u0 + i - tile * nsb;
                const int64_t m0 = (tile % a.mblocks) * BN;
                // the round's activations: one stage per kActK elements of K
                // (stage sequence number (4 i + c) kSlices + slice); K past the
                // end and tokens past M read as zeros
                for (int q = 0; q < kChunks * kSlices && ok; ++q, ++issued_a) {
                    const int st = (int)(issued_a % kActStages);
                    ok = mbar_wait(smem_u32(&act_empty[st]), (uint32_t)(((issued_a / kActStages) & 1) ^ 1), a.err);
                    if (!ok) break;
                    const uint32_t abar = smem_u32(&act_full[st]);
                    mbar_arrive_expect_tx(abar, kActBytes);
                    tc::tma_load_2d(smem_u32(smem + kOffAct + st * kActBytes), &tmap_a,
                                    (int32_t)(sb * kSB + q * kActK), (int32_t)m0, abar, pol);
                }
            }
            for (int64_t k = issued_a > kActStages ? issued_a - kActStages : 0; k < issued_a; ++k)
                mbar_wait(smem_u32(&act_full[k % kActStages]), (uint32_t)((k / kActStages) & 1), a.err);
        }
        __syncwarp();  // lanes 1..31 wait here for the producer lane
    } else if (warp == kWProdWarp) {
        // ------------------------------------------------------------ weight producer
        // A warp of its own, so that weight stages go out as soon as the
        // converters free them, never queued behind activation chunks.
        if (lane == 0) {
            tc::prefetch_tensormap(&tmap_w);
            if (F == kQ40) tc::prefetch_tensormap(&tmap_d);
            const uint64_t pol = policy_evict_last();  // the other token blocks' CTAs read the same rows
            pdl_wait();
            int64_t issued_w = 0;
            for (int64_t i = 0; i < u1 - u0; ++i) {
                const int64_t tile = (u0 + i) / nsb, sb = u0 + i - tile * nsb;
                const int64_t n0 = (tile / a.mblocks) * kBM;
                const int ws = (int)(i % kWStages);
                if (!mbar_wait(smem_u32(&w_empty[ws]), (uint32_t)(((i / kWStages) & 1) ^ 1), a.err)) break;
                // rows past the last tile and K past the end read as zeros
                const uint32_t wbar = smem_u32(&w_full[ws]);
                uint8_t *wdst = smem + kOffW + ws * FmtInfo<F>::kWStage;
                mbar_arrive_expect_tx(wbar, kWBytes);
                if (F == kW4A16) {
                    // 8 tiles x 2 steps: [tile][step][16 rows x 64 B]
                    tc::tma_load_3d(smem_u32(wdst), &tmap_w, 0, (int32_t)(2 * sb),
                                    (int32_t)(n0 / kW4Tile), wbar, pol);
                } else if (F == kQ6K || F == kQ4K) {
                    // 16 records of 8 rows for super-block sb: [tile][8 x 210 or 144 B]
                    tc::tma_load_3d(smem_u32(wdst), &tmap_w, 0, (int32_t)sb, (int32_t)(n0 / kTileRows),
                                    wbar, pol);
                } else {
                    // 16 tiles x 8 blocks: nibbles [tile][block][8 rows][16 B],
                    // scales [tile][block][8 rows fp16]
                    tc::tma_load_4d(smem_u32(wdst), &tmap_w, 0, 0, (int32_t)(sb * kQ4Blocks),
                                    (int32_t)(n0 / kQ4Tile), wbar, pol);
                    tc::tma_load_3d(smem_u32(wdst + kQ4NibBytes), &tmap_d, 0, (int32_t)(sb * kQ4Blocks),
                                    (int32_t)(n0 / kQ4Tile), wbar, pol);
                }
                ++issued_w;
            }
            for (int64_t k = issued_w > kWStages ? issued_w - kWStages : 0; k < issued_w; ++k)
                mbar_wait(smem_u32(&w_full[k % kWStages]), (uint32_t)((k / kWStages) & 1), a.err);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Meets the waiter at the named barrier the same number of times
        // whatever happens; after a timeout the MMAs run on stale operands and
        // the error word reports it.
        constexpr uint32_t idesc = tc::idesc_f16_f32(kBM, BN);
        const uint64_t bdesc0 = tc::smem_desc(smem_u32(smem + kOffAct), T::kSbo, T::kSwz);
        int64_t i = 0;  // units done: the pipeline position
        int pc = 0;     // pieces done: accumulator pc % kAccs
        for (int64_t u = u0; u < u1; ++pc) {
            const int64_t tile = u / nsb;
            const int sb_begin = (int)(u - tile * nsb);
            const int sb_end = (int)(nsb < sb_begin + (u1 - u) ? nsb : sb_begin + (u1 - u));
            u += sb_end - sb_begin;
            const uint32_t dacc = tmem + (uint32_t)((pc % kAccs) * BN);
            for (int sb = sb_begin; sb < sb_end; ++sb, ++i) {
#pragma unroll 1
                for (int g = 0; g < kGroups; ++g) {
                    handoff_sync();
                    if (lane == 0) {
                        tc::fence_after_sync();
#pragma unroll
                        for (int h = 0; h < kChunks / kGroups; ++h) {
                            const int c = g * (kChunks / kGroups) + h;
                            const uint32_t acol =
                                tmem + kColARing + (uint32_t)((int)(i & 1) * kChunks + c) * kARingCols;
#pragma unroll
                            for (int sl = 0; sl < kSlices; ++sl) {
                                const int st = (int)(((i * kChunks + c) * kSlices + sl) % kActStages);
                                const uint64_t bdesc = bdesc0 + (uint64_t)((st * kActBytes) >> 4);
                                // K step of 16 fp16 = 32 bytes = 2 in the descriptor's address field
#pragma unroll
                                for (int kq = 0; kq < kActK / 16; ++kq) {
                                    const int kk = sl * (kActK / 16) + kq;
                                    tc::mma_f16_ta(dacc, acol + 8 * kk, bdesc + 2 * kq, idesc,
                                                   ((sb - sb_begin) | c | kk) != 0);
                                }
                                tc::commit(smem_u32(&act_empty[st]));  // the stage is free once these are done
                            }
                        }
                        tc::commit(smem_u32(&a_empty[(int)(i & 1) * kGroups + g]));
                    }
                    __syncwarp();
                }
            }
            if (lane == 0) tc::commit(smem_u32(&acc_full[pc % kAccs]));
            __syncwarp();
        }
        if (lane == 0) {
            tc::commit(smem_u32(done));
            mbar_wait(smem_u32(done), 0, a.err);  // no MMA may run when TMEM is freed
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------------ MMA waiter
        // Before a piece's first MMA: its accumulator has been read by the
        // epilogue (two pieces back); before each group: its operands.
        bool ok = true;
        int64_t i = 0;
        int pc = 0;
        for (int64_t u = u0; u < u1; ++pc) {
            const int64_t tile = u / nsb;
            const int sb_begin = (int)(u - tile * nsb);
            const int sb_end = (int)(nsb < sb_begin + (u1 - u) ? nsb : sb_begin + (u1 - u));
            u += sb_end - sb_begin;
            if (lane == 0 && ok)
                ok = mbar_wait(smem_u32(&acc_empty[pc % kAccs]), (uint32_t)(((pc / kAccs) & 1) ^ 1), a.err);
            for (int sb = sb_begin; sb < sb_end; ++sb, ++i) {
                const uint32_t par = (uint32_t)((i >> 1) & 1);  // slot group used every other round
                const int rg = (int)(i & 1) * kGroups;
#pragma unroll 1
                for (int g = 0; g < kGroups; ++g) {
                    // the group's two activation chunks, then its A operands
                    for (int h = 0; h < (kChunks / kGroups) * kSlices && ok; ++h) {
                        const int64_t ci = (i * kChunks + g * (kChunks / kGroups)) * kSlices + h;
                        if (lane == 0)
                            ok = mbar_wait(smem_u32(&act_full[ci % kActStages]), (uint32_t)((ci / kActStages) & 1),
                                           a.err);
                    }
                    if (lane == 0 && ok) ok = mbar_wait(smem_u32(&a_full[rg + g]), par, a.err);
                    __syncwarp();
                    handoff_sync();
                }
            }
        }
    } else if (warp < 3 + kConvWarps) {
        // ------------------------------------------------------------ converters
        const int ct = 32 * (warp & 3) + lane;  // weight row within the CTA = TMEM lane
        const uint32_t lane_addr = (uint32_t)(32 * (warp & 3)) << 16;
        const int set = (warp - 3) >> 2;  // chunk `set` of each group
        const int64_t nsteps = a.K / kW4StepK;
        bool ok = true;
        int64_t pos = 0;  // units done: the pipeline position
        for (int64_t u = u0; u < u1 && ok;) {
            const int64_t tile = u / nsb;
            const int sb_begin = (int)(u - tile * nsb);
            const int sb_end = (int)(nsb < sb_begin + (u1 - u) ? nsb : sb_begin + (u1 - u));
            u += sb_end - sb_begin;
            const int64_t n = (tile / a.mblocks) * kBM + ct;
            const int64_t nc = n < a.N ? n : a.N - 1;  // rows past N: zero codes, clamped scales
            for (int64_t sb = sb_begin; sb < sb_end && ok; ++sb, ++pos) {
                const int ws = (int)(pos % kWStages);
                const uint32_t par = (uint32_t)((pos >> 1) & 1);  // A ring slot group used every other round
                const int rg = (int)(pos & 1) * kGroups;
                ok = mbar_wait_warp(smem_u32(&w_full[ws]), (uint32_t)((pos / kWStages) & 1), a.err);
                if (!ok) break;
                const uint8_t *wst = smem + kOffW + ws * FmtInfo<F>::kWStage;
#pragma unroll 1
                for (int g = 0; g < kGroups && ok; ++g) {
                    const int c = g * (kChunks / kGroups) + set;  // chunk of this round
                    uint32_t lo[16], hi[16];  // TMEM columns 0..15 and 16..31 of the chunk
                    if (F == kW4A16) {
                        // chunk c = half (c & 1) of step 2 sb + (c >> 1); columns hold
                        // elements (2i, 2i + 1): the packed words put even elements
                        // in the low half, odd in the high half
                        const int sl = c >> 1;
                        int64_t step = 2 * sb + sl;
                        if (step >= nsteps) step = nsteps - 1;  // past K the activations are zero
                        const int grp = a.spg == 1 ? (int)step : (int)step / a.spg;
                        const uint32_t zv = a.lut ? 0u : (uint32_t)a.Z[nc * a.ng + grp];
                        const uint32_t sv = (uint32_t)__half_as_ushort(a.S[nc * a.ng + grp]);
                        const uint32_t zz = 0x64006400u + zv * 0x00010001u;  // fp16 1024 + z twice
                        const uint32_t zh = 0xD400D400u + zv * 0x00100010u;  // fp16 -(64 + z) twice
                        const uint32_t ss = sv | (sv << 16);
                        const uint8_t *src = wst + ((ct >> 4) * (kSB / kW4StepK) + sl) * 1024 + (ct & 15) * 64 +
                                             (c & 1) * 32;
                        const uint4 w0 = *reinterpret_cast<const uint4 *>(src);
                        const uint4 w1 = *reinterpret_cast<const uint4 *>(src + 16);
                        const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                        if (a.lut) {
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                lut_scaled_word(wv[i], pair_tbl, ss, lo[4 * i], lo[4 * i + 1], lo[4 * i + 2],
                                                lo[4 * i + 3]);
                                lut_scaled_word(wv[i + 4], pair_tbl, ss, hi[4 * i], hi[4 * i + 1],
                                                hi[4 * i + 2], hi[4 * i + 3]);
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                // W4A16 word: (k0,k1) at 0|16, (k2,k3) at 4|20, (k4,k5) at 8|24, (k6,k7) at 12|28
                                scaled_word(wv[i], zz, zh, ss, lo[4 * i], lo[4 * i + 2], lo[4 * i + 1],
                                            lo[4 * i + 3]);
                                scaled_word(wv[i + 4], zz, zh, ss, hi[4 * i], hi[4 * i + 2], hi[4 * i + 1],
                                            hi[4 * i + 3]);
                            }
                        }
                    } else if (F == kQ4K) {
                        // chunk c = sub-blocks 2c (low nibbles of qs bytes 32c ..
                        // 32c+31, chunk elements 0..31) and 2c + 1 (high nibbles,
                        // 32..63); their scales and mins are header field c
                        const uint8_t *blk = wst + (ct >> 3) * (kTileRows * B_Q4_K) + (ct & 7) * B_Q4_K;
                        const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
                        const uint4 qa = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * c);
                        const uint4 qb = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * c);
                        const uint32_t f = k4_field(hdr.y, hdr.z, hdr.w, c);
                        const float dw = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xFFFFu)));
                        const float dmw = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
                        // d s_j and dmin m_j of the low (h = 0) and high sub-block:
                        // exact in fp32 (11-bit by 6-bit significands)
                        float ds[2], dm[2];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            ds[h] = __fmul_rn(dw, (float)((f >> (12 * h)) & 63u));
                            dm[h] = __fmul_rn(dmw, (float)((f >> (12 * h + 6)) & 63u));
                        }
                        const uint64_t sl01 = f2(ds[0], ds[0] * 0x1p-8f), sl23 = f2(ds[0] * 0x1p-16f, ds[0] * 0x1p-12f);
                        const uint64_t sh01 = f2(ds[1] * 0x1p-4f, ds[1] * 0x1p-12f);
                        const uint64_t sh23 = f2(ds[1] * 0x1p-8f, ds[1] * 0x1p-16f);
                        const uint64_t nml = f2(-dm[0], -dm[0]), nmh = f2(-dm[1], -dm[1]);
                        const uint32_t qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
                        for (int w = 0; w < 8; ++w)
                            q4k_word(qv[w], sl01, sl23, nml, sh01, sh23, nmh, lo[2 * w], lo[2 * w + 1], hi[2 * w],
                                     hi[2 * w + 1]);
                    } else if (F == kQ6K) {
                        // chunk c = elements 64c .. 64c+63 of super-block sb: the
                        // low nibbles of ql bytes 32c .. 32c+31 are its elements
                        // 0..31, the high nibbles 32..63; their high bits are in
                        // the words of GEMV lanes 2c, 2c+1 (16 elements each), the
                        // scales of groups 4c + tl (low) and 4c + 2 + tl (high) in
                        // bytes 4c .. 4c+3 (tl = lane 2c + tl)
                        const uint8_t *rec = wst + (ct >> 3) * kQ6Rec;
                        const int r = ct & 7;
                        const uint8_t *row = rec + r * kQ6Codes;
                        const uint4 qa = *reinterpret_cast<const uint4 *>(row + 32 * c);
                        const uint4 qb = *reinterpret_cast<const uint4 *>(row + 32 * c + 16);
                        const uint4 hw = *reinterpret_cast<const uint4 *>(row + 128 + 16 * c);
                        const uint32_t sc4 = *reinterpret_cast<const uint32_t *>(rec + kQ6ScOff + 16 * r + 4 * c);
                        const float dw = __half2float(*reinterpret_cast<const __half *>(rec + kQ6DOff + 2 * r));
                        // (d s) 2^-p pairs, p as q6k_pairs takes them, for (tl 0, low),
                        // (tl 0, high), (tl 1, low), (tl 1, high); d s is exact in fp32
                        uint64_t s01[4], s23[4];
#pragma unroll
                        for (int b = 0; b < 4; ++b) {
                            const float v = __fmul_rn(dw, (float)(int)(int8_t)(uint8_t)(sc4 >> (8 * b)));
                            s01[b] = f2(v, v * 0x1p-8f);
                            s23[b] = f2(v * 0x1p-16f, v * 0x1p-8f);
                        }
                        const uint32_t qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
                        for (int w = 0; w < 8; ++w) {
                            const int tl = w >> 2, ww = w & 3;
                            const uint32_t ul = q6k_u(qv[w], tl ? hw.z : hw.x, ww);
                            const uint32_t uh = q6k_u(qv[w] >> 4, tl ? hw.w : hw.y, ww);
                            q6k_pairs(ul, s01[2 * tl], s23[2 * tl], lo[2 * w], lo[2 * w + 1]);
                            q6k_pairs(uh, s01[2 * tl + 1], s23[2 * tl + 1], hi[2 * w], hi[2 * w + 1]);
                        }
                    } else {
                        // chunk c = blocks 2c, 2c + 1 of the round. Byte l of a block
                        // holds elements l (low nibble) and l + 16 (high); word i
                        // gives columns 4i .. 4i+3 = (e4i, e4i+2), (e4i+1, e4i+3),
                        // (e16+4i, e18+4i), (e17+4i, e19+4i) -- the order the Q4_0
                        // prefill quantizer writes the activations of a block in.
                        constexpr uint32_t zz = 0x64086408u;  // fp16 1024 + 8 twice
                        constexpr uint32_t zh = 0xD480D480u;  // fp16 -(64 + 8) twice
                        const int tt = ct >> 3, r = ct & 7;
#pragma unroll
                        for (int b = 0; b < 2; ++b) {
                            const int blk = 2 * c + b;
                            const uint4 q = *reinterpret_cast<const uint4 *>(wst + tt * 1024 + blk * 128 + r * 16);
                            const uint32_t dv = *reinterpret_cast<const uint16_t *>(
                                wst + kQ4NibBytes + tt * (kQ4Blocks * 16) + blk * 16 + r * 2);
                            const uint32_t ss = dv | (dv << 16);
                            const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
                            uint32_t *out = b == 0 ? lo : hi;
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                scaled_word(wv[i], zz, zh, ss, out[4 * i], out[4 * i + 1], out[4 * i + 2],
                                            out[4 * i + 3]);
                        }
                    }
                    ok = mbar_wait_warp(smem_u32(&a_empty[rg + g]), par ^ 1, a.err);
                    if (!ok) break;
                    tc::fence_after_sync();
                    const uint32_t acol =
                        tmem + lane_addr + kColARing + (uint32_t)((int)(pos & 1) * kChunks + c) * kARingCols;
                    tc::tmem_st16(acol, lo);
                    tc::tmem_st16(acol + 16, hi);
                    tc::tmem_st_wait();
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&a_full[rg + g]));
                }
                __syncwarp();
                if (lane == 0 && ok) mbar_arrive(smem_u32(&w_empty[ws]));
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Per piece: the piece's token scales (2^-e per token) go to shared
        // memory while its MMAs run; then the accumulator is read back 32
        // columns per TMEM wait, and the accumulator is free for the piece
        // kAccs later. A whole tile goes to C 16 columns at a time through a
        // staging block in shared memory [16 tokens][128 rows] and a 2-D TMA
        // store (which leaves out rows past N and tokens past M): one thread
        // (the first epilogue lane) issues the stores, and a staging block is
        // rewritten once the store issued from it two blocks back has read it.
        // Where C's rows are not 16-byte aligned, whole tiles go to C by
        // plain stores. A part of a split tile goes to this CTA's partial
        // slot by plain stores (contiguous). After a timed-out wait the loop
        // still walks the pieces and blocks (and meets the other epilogue
        // warps at every barrier), without waits, TMEM loads or stores.
        const int quarter = warp & 3;  // TMEM lanes 32 * (warp % 4) ..
        const int nl = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const bool issuer = warp == kEpiWarp0 && lane == 0;
        float *ts_s = reinterpret_cast<float *>(smem + FmtInfo<F>::kOffLut);
        uint8_t *stage = smem + FmtInfo<F>::kOffStage;
        if (F != kW4A16) pdl_wait();  // the token scales come from the preceding kernel
        bool ok = true;
        int pc = 0;
        uint32_t blk = 0;  // staging blocks used so far: block blk is in buffer blk & 1
        for (int64_t u = u0; u < u1; ++pc) {
            const int64_t tile = u / nsb;
            const int sb_begin = (int)(u - tile * nsb);
            const int sb_end = (int)(nsb < sb_begin + (u1 - u) ? nsb : sb_begin + (u1 - u));
            u += sb_end - sb_begin;
            const int64_t n0 = (tile / a.mblocks) * kBM, m0 = (tile % a.mblocks) * BN;
            const int64_t n = n0 + nl;
            const uint32_t acc = tmem + lane_addr + (uint32_t)((pc % kAccs) * BN);
            // column groups holding tokens < M (warp-uniform): the rest is
            // padding; m0 + 16 ncg <= M rounded up to 16, the scales' length
            const int ncg = (int)((a.M - m0 < BN ? a.M - m0 + 15 : BN) / 16);
            if (F != kW4A16) {
                epi_sync();  // every epilogue warp is done with the last piece's scales
                for (int j = (warp - kEpiWarp0) * 32 + lane; j < ncg * 16; j += kEpiWarps * 32)
                    ts_s[j] = a.tok_scale[m0 + j];
                epi_sync();
            }
            if (ok) ok = mbar_wait_warp(smem_u32(&acc_full[pc % kAccs]), (uint32_t)((pc / kAccs) & 1), a.err);
            if (ok) tc::fence_after_sync();
            const bool whole = sb_begin == 0 && sb_end == nsb;
            const bool staged = whole && a.c_tma;
            // this CTA's partial slot for a part of a split tile: column j at j * kBM
            float *slot = whole ? nullptr : a.part + sk_slot(blockIdx.x, tile, a.units, gridDim.x, nsb, BN);
#pragma unroll 1
            for (int c32 = 0; c32 < ncg; c32 += 2) {
                // columns 16 c32 .. 16 c32 + 31 (below BN even where the
                // second half is past the last group); TMEM loads are
                // warp-collective and ok is warp-uniform
                float v[2][16];
                if (ok) {
                    tc::tmem_ld16(acc + (uint32_t)(c32 * 16), v[0]);
                    tc::tmem_ld16(acc + (uint32_t)(c32 * 16 + 16), v[1]);
                    tc::tmem_ld_wait();
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int c16 = c32 + h;
                    if (c16 >= ncg) break;
                    if (F != kW4A16 && ok) scale16_s(ts_s + c16 * 16, v[h]);
                    if (!staged) {
                        if (ok && whole && n < a.N) {
                            store_cols<F>(a, m0 + c16 * 16, n, v[h]);
                        } else if (ok && !whole) {
                            float *mine = slot + c16 * 16 * kBM + nl;
#pragma unroll
                            for (int j = 0; j < 16; ++j) mine[j * kBM] = v[h][j];
                        }
                        continue;
                    }
                    uint8_t *sb = stage + (blk & 1) * kStageBytes;
                    if (issuer) tc::bulk_wait_read<1>();  // the copy from this buffer two blocks back
                    epi_sync();
                    if (ok) {
                        if (F == kW4A16) {
                            __half *st = reinterpret_cast<__half *>(sb) + nl;
#pragma unroll
                            for (int j = 0; j < 16; ++j) st[j * kBM] = __float2half_rn(v[h][j]);
                        } else {
                            float *st = reinterpret_cast<float *>(sb) + nl;
#pragma unroll
                            for (int j = 0; j < 16; ++j) st[j * kBM] = v[h][j];
                        }
                    }
                    tc::fence_proxy_async();
                    epi_sync();
                    if (issuer && ok) {
                        tc::tma_store_2d(&tmap_c, (int32_t)n0, (int32_t)(m0 + c16 * 16), smem_u32(sb));
                        tc::bulk_commit();
                    }
                    ++blk;
                }
            }
            if (ok) {
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&acc_empty[pc % kAccs]));
            }
        }
        if (issuer) tc::bulk_wait_all();  // the copies' writes done before the CTA ends
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ prefill activations
// The fp16 activation operand a = fp16(2^e d_a y) [M][K], y the bit-exact Q8
// codes and d_a their block scale (Q8_0: the fp16 scale widened; Q8_K: fp32),
// with one power of two 2^e per token: e puts the token's largest block scale
// 2^e d_a in [2^7, 2^8), so |a| < 127 2^8 < 65504 and the token's smaller
// values keep fp16's full precision down to 2^-28 of its largest. 2^-e goes to
// the per-token scale array (after the operand in the workspace, padded with
// 1.0 to a multiple of 16 tokens) that the GEMM epilogue multiplies by.
// One CTA of 256 threads per token: max |x| (or max d) over the token first,
// then the blocks. The block scales are monotone in the block's max |x|, so
// the token's largest d_a is the scale of the token's max |x|.
constexpr int kActThreads = 256;

__device__ __forceinline__ int prescale_exp(float dmax) {
    const int ef = (int)((__float_as_uint(dmax) >> 23) & 0xFFu);
    if (!(dmax > 0.0f) || ef == 255) return 0;  // zero token, or not finite
    if (ef == 0) return 126;                    // subnormal scale
    return min(126, max(-126, 134 - ef));       // 2^e dmax in [2^7, 2^8)
}
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }
__host__ __device__ inline int64_t pad16(int64_t M) { return (M + 15) / 16 * 16; }

// Max of v >= +0 over the CTA; every thread gets it.
__device__ __forceinline__ float cta_max_nonneg(float v, float *red) {
    v = warp_max_nonneg(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = 0.0f;
#pragma unroll
    for (int i = 0; i < kActThreads / 32; ++i) r = fmaxf(r, red[i]);
    return r;
}

// max |x| over the token's K values (16-byte loads; K % 32 == 0).
__device__ __forceinline__ float token_amax(const float *__restrict__ x, int64_t K, float *red) {
    float a = 0.0f;
    for (int64_t i = threadIdx.x; i < K / 4; i += kActThreads) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(x) + i);
        a = fmaxf(fmaxf(a, fmaxf(fabsf(v.x), fabsf(v.y))), fmaxf(fabsf(v.z), fabsf(v.w)));
    }
    return cta_max_nonneg(a, red);
}

__device__ __forceinline__ void store_tok_scale(float *ts, int64_t M, int e) {
    if (threadIdx.x == 0) ts[blockIdx.x] = pow2f(-e);
    if (blockIdx.x == 0)
        for (int64_t i = M + threadIdx.x; i < pad16(M); i += kActThreads) ts[i] = 1.0f;
}

// Q4_0: X fp32 -> Q8_0 codes y and fp16 scale d per 32 (the arithmetic of
// the Q8_0 quantizer: amax / 127, codes rounded half away from zero), then
// a = fp16(2^e f32(d) y) written with the elements of each block permuted to
// the order the Q4_0 converter puts the weights in: element e (e' = e mod 16,
// i = e' / 4, r = e' mod 4) goes to position 8 i + 4 (e >= 16) + 2 (r mod 2)
// + r / 2. 4 lanes per block, 8 consecutive elements per lane (two 16-byte
// loads); the 4 elements 4i .. 4i+3 of a lane land at positions 8 i + 4 (e >=
// 16) + (0, 2, 1, 3), so each lane writes two 8-byte groups.
__global__ void __launch_bounds__(kActThreads) quantize_q4_0_prefill_kernel(const float *__restrict__ X,
                                                                            __half *__restrict__ out,
                                                                            float *__restrict__ ts,
                                                                            int64_t M, int64_t K) {
    pdl_launch_dependents();
    __shared__ float red[kActThreads / 32];
    const int64_t m = blockIdx.x, nb = K / QK4_0;
    const float *x = X + m * K;
    const float dmax = __half2float(__float2half_rn(__fdiv_rn(token_amax(x, K, red), 127.0f)));
    const int ex = prescale_exp(dmax);
    const float p2 = pow2f(ex);
    store_tok_scale(ts, M, ex);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, j = lane & 3;  // j: elements 8j .. 8j+7
    // positions of this lane's two groups: elements 8j + 4g .. 8j + 4g + 3
    const int e0 = 8 * j, base0 = 8 * ((e0 & 15) >> 2) + ((e0 >> 4) << 2);
    const int e1 = e0 + 4, base1 = 8 * ((e1 & 15) >> 2) + ((e1 >> 4) << 2);
    for (int64_t g = warp; g * 8 < nb; g += kActThreads / 32) {
        const int64_t b = g * 8 + (lane >> 2);
        const bool live = b < nb;
        float4 v0 = make_float4(0.0f, 0.0f, 0.0f, 0.0f), v1 = v0;
        if (live) {
            const float4 *src = reinterpret_cast<const float4 *>(x + b * QK4_0 + e0);
            v0 = src[0];
            v1 = src[1];
        }
        float a = fmaxf(fmaxf(fmaxf(fabsf(v0.x), fabsf(v0.y)), fmaxf(fabsf(v0.z), fabsf(v0.w))),
                        fmaxf(fmaxf(fabsf(v1.x), fabsf(v1.y)), fmaxf(fabsf(v1.z), fabsf(v1.w))));
        // max over the block's 4 lanes (non-negative floats order like their bits)
        uint32_t ab = __float_as_uint(a);
        ab = max(ab, __shfl_xor_sync(0xffffffffu, ab, 1));
        ab = max(ab, __shfl_xor_sync(0xffffffffu, ab, 2));
        const float d = __fdiv_rn(__uint_as_float(ab), 127.0f);
        const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
        const float sd = __fmul_rn(__half2float(__float2half_rn(d)), p2);  // exact
        auto val = [&](float xv) { return __float2half_rn(__fmul_rn(sd, int_as_exact_float(q8_code(xv, id)))); };
        if (live) {
            __half *dst = out + (m * nb + b) * QK4_0;
            const __half2 p0 = __halves2half2(val(v0.x), val(v0.z)), p1 = __halves2half2(val(v0.y), val(v0.w));
            const __half2 q0 = __halves2half2(val(v1.x), val(v1.z)), q1 = __halves2half2(val(v1.y), val(v1.w));
            *reinterpret_cast<uint2 *>(dst + base0) = make_uint2(h2_bits(p0), h2_bits(p1));
            *reinterpret_cast<uint2 *>(dst + base1) = make_uint2(h2_bits(q0), h2_bits(q1));
        }
    }
}

// The same operand from canonical Q8_0 blocks [M][nb] x 34 B, for
// qmm_mul_mat_q8: the token's largest |d| first, then one warp per block.
__global__ void __launch_bounds__(kActThreads) import_q8_0_prefill_kernel(const uint8_t *__restrict__ Xq,
                                                                          __half *__restrict__ out,
                                                                          float *__restrict__ ts,
                                                                          int64_t M, int64_t K) {
    pdl_launch_dependents();
    __shared__ float red[kActThreads / 32];
    const int64_t m = blockIdx.x, nb = K / QK4_0;
    const uint8_t *row = Xq + m * nb * B_Q8_0;
    float a = 0.0f;
    for (int64_t b = threadIdx.x; b < nb; b += kActThreads)
        a = fmaxf(a, fabsf(__half2float(*reinterpret_cast<const __half *>(row + b * B_Q8_0))));
    const int ex = prescale_exp(cta_max_nonneg(a, red));
    const float p2 = pow2f(ex);
    store_tok_scale(ts, M, ex);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = lane, ep = e & 15, i = ep >> 2, r = ep & 3;
    const int pos = 8 * i + ((e >> 4) << 2) + 2 * (r & 1) + (r >> 1);
    for (int64_t b = warp; b < nb; b += kActThreads / 32) {
        const uint8_t *blk = row + b * B_Q8_0;
        const int q = (int8_t)blk[2 + lane];
        const float sd = __fmul_rn(__half2float(*reinterpret_cast<const __half *>(blk)), p2);
        out[(m * nb + b) * QK4_0 + pos] = __float2half_rn(__fmul_rn(sd, (float)q));
    }
}

// Q4_K and Q6_K: X fp32 -> Q8_K codes y and fp32 scale d per 256 (the Q8_K
// quantizer's arithmetic: amax / 127, codes rounded half away from zero),
// then a = fp16(2^e d y) in natural order [M][K]. One warp per super-block,
// 8 consecutive elements per lane (two 16-byte loads, one 16-byte store).
__global__ void __launch_bounds__(kActThreads) quantize_q8_K_f16_kernel(const float *__restrict__ X,
                                                                        __half *__restrict__ out,
                                                                        float *__restrict__ ts, int64_t M,
                                                                        int64_t K) {
    pdl_launch_dependents();
    __shared__ float red[kActThreads / 32];
    const int64_t m = blockIdx.x, nsb = K / QK_K;
    const float *x = X + m * K;
    const int ex = prescale_exp(__fdiv_rn(token_amax(x, K, red), 127.0f));
    const float p2 = pow2f(ex);
    store_tok_scale(ts, M, ex);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t b = warp; b < nsb; b += kActThreads / 32) {
        const float4 *src = reinterpret_cast<const float4 *>(x + b * QK_K + 8 * lane);
        const float4 v0 = src[0], v1 = src[1];
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
        const float d = __fdiv_rn(warp_max_nonneg(a), 127.0f);
        const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
        const float sd = __fmul_rn(d, p2);  // exact
        uint32_t h[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            h[i] = h2_bits(__floats2half2_rn(__fmul_rn(sd, int_as_exact_float(q8_code(v[2 * i], id))),
                                             __fmul_rn(sd, int_as_exact_float(q8_code(v[2 * i + 1], id)))));
        }
        *reinterpret_cast<uint4 *>(out + (m * nsb + b) * QK_K + 8 * lane) = make_uint4(h[0], h[1], h[2], h[3]);
    }
}

// The same operand from canonical Q8_K blocks [M][nsb] x 292 B, for
// qmm_mul_mat_q8: the token's largest |d| first, then one warp per block, 8
// codes per lane.
__global__ void __launch_bounds__(kActThreads) import_q8_K_f16_kernel(const uint8_t *__restrict__ Xq,
                                                                      __half *__restrict__ out,
                                                                      float *__restrict__ ts, int64_t M,
                                                                      int64_t K) {
    pdl_launch_dependents();
    __shared__ float red[kActThreads / 32];
    const int64_t m = blockIdx.x, nsb = K / QK_K;
    const uint8_t *row = Xq + m * nsb * B_Q8_K;
    float a = 0.0f;
    for (int64_t b = threadIdx.x; b < nsb; b += kActThreads)
        a = fmaxf(a, fabsf(*reinterpret_cast<const float *>(row + b * B_Q8_K)));
    const int ex = prescale_exp(cta_max_nonneg(a, red));
    const float p2 = pow2f(ex);
    store_tok_scale(ts, M, ex);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t b = warp; b < nsb; b += kActThreads / 32) {
        const uint8_t *blk = row + b * B_Q8_K;
        const float sd = __fmul_rn(*reinterpret_cast<const float *>(blk), p2);
        // 292-byte blocks: 4-byte loads only
        const uint32_t cw[2] = {*reinterpret_cast<const uint32_t *>(blk + 4 + 8 * lane),
                                *reinterpret_cast<const uint32_t *>(blk + 8 + 8 * lane)};
        uint32_t h[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int q0 = (int)(int8_t)(uint8_t)(cw[i >> 1] >> (16 * (i & 1)));
            const int q1 = (int)(int8_t)(uint8_t)(cw[i >> 1] >> (16 * (i & 1) + 8));
            h[i] = h2_bits(__halves2half2(__float2half_rn(__fmul_rn(sd, (float)q0)),
                                          __float2half_rn(__fmul_rn(sd, (float)q1))));
        }
        *reinterpret_cast<uint4 *>(out + (m * nsb + b) * QK_K + 8 * lane) = make_uint4(h[0], h[1], h[2], h[3]);
    }
}

// The GEMM (programmatic dependent launch): one CTA per tile, or with more
// tiles than SMs a persistent stream-K grid and the fixup of its split tiles.
// act: the fp16 activations [M][K], read through a swizzled 2-D tensor
// map whose box is one stage (BN tokens x kActK elements). C is written through
// a 2-D tensor map (box 128 rows x 16 tokens) where its base and rows are
// 16-byte aligned, else by plain stores.
template <int F, int BN>
cudaError_t launch_stream_k_bn(Args a, const CUtensorMap &tmap_w, const CUtensorMap &tmap_d, const void *act,
                               cudaStream_t s) {
    auto fn = gemm_f16_kernel<F, BN>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(fn), FmtInfo<F>::kSmemBytes);
    if (e != cudaSuccess) return e;
    CUtensorMap tmap_a;
    if (!tc::make_tmap_2d(&tmap_a, act, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (uint64_t)a.M, (uint64_t)a.K, BN,
                          Tile<BN>::kActK,
                          Tile<BN>::kActK == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    CUtensorMap tmap_c;
    const uint32_t celem = F == kW4A16 ? 2 : 4;
    a.c_tma = ((uintptr_t)a.C % 16) == 0 && ((uint64_t)a.N * celem) % 16 == 0 &&
              tc::make_tmap_2d(&tmap_c, a.C, F == kW4A16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                               celem, (uint64_t)a.M, (uint64_t)a.N, kStageCols, kBM, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!a.c_tma) memset(&tmap_c, 0, sizeof tmap_c);
    const int64_t nsb = (a.K + kSB - 1) / kSB;
    a.mblocks = (a.M + BN - 1) / BN;
    const int64_t tiles = ((a.N + kBM - 1) / kBM) * a.mblocks;
    a.units = tiles * nsb;
    const int64_t G = stream_k_grid(tiles, a.units);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = FmtInfo<F>::kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, fn, a, tmap_w, tmap_d, tmap_a, tmap_c);
    count_launch();
    if (e != cudaSuccess || G == tiles) return e;
    return launch_stream_k_fixup(a.part, a.C, F == kW4A16, BN, a.N, a.M, a.mblocks, nsb, a.units, G, s);
}

template <int F>
cudaError_t launch_stream_k(const Args &a, const CUtensorMap &tmap_w, const CUtensorMap &tmap_d, const void *act,
                            cudaStream_t s) {
    constexpr int wt = F == kW4A16 ? QMM_TYPE_W4A16 : F == kQ40 ? QMM_TYPE_Q4_0 : F == kQ6K ? QMM_TYPE_Q6_K
                                                                                       : QMM_TYPE_Q4_K;
    return gemm_tile_cols(wt, a.M) == 256 ? launch_stream_k_bn<F, 256>(a, tmap_w, tmap_d, act, s)
                                      : launch_stream_k_bn<F, 128>(a, tmap_w, tmap_d, act, s);
}

}  // namespace

// The prefill workspace: the fp16 operand [M][K], then the per-token scales.
static size_t operand_bytes(int64_t M, int64_t K) { return align_up((size_t)M * K * 2, 256); }
static float *tok_scales(const void *ws, int64_t M, int64_t K) {
    return reinterpret_cast<float *>(static_cast<uint8_t *>(const_cast<void *>(ws)) + operand_bytes(M, K));
}
size_t prefill_operand_bytes(int64_t M, int64_t K) {
    return operand_bytes(M, K) + align_up((size_t)pad16(M) * sizeof(float), 256);
}

cudaError_t launch_import_q4_0_prefill(const void *Xq, void *ws, int64_t M, int64_t K,
                                       cudaStream_t s) {
    import_q8_0_prefill_kernel<<<(unsigned)M, kActThreads, 0, s>>>(
        static_cast<const uint8_t *>(Xq), static_cast<__half *>(ws), tok_scales(ws, M, K), M, K);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_w4a16_gemm(const void *W, const __half *S, const uint8_t *Z, const __half *lut, int64_t G,
                              const __half *A, __half *C, int64_t M, int64_t N, int64_t K,
                              float *part, cudaStream_t s) {
    Args a;
    a.S = S;
    a.Z = Z;
    a.lut = lut;
    a.C = C;
    a.M = M;
    a.N = N;
    a.K = K;
    a.ng = (int)(K / G);
    a.spg = (int)(G / kW4StepK);
    a.err = device_error_word();
    a.part = part;
    a.tok_scale = nullptr;
    const int64_t nsteps = K / kW4StepK, ntiles16 = (N + kW4Tile - 1) / kW4Tile;
    CUtensorMap tmap_w;
    // packed weights as [16-row tile][step][1 KB], in 4-byte units
    const uint64_t wdims[3] = {256, (uint64_t)nsteps, (uint64_t)ntiles16};
    const uint64_t wstrides[2] = {1024, (uint64_t)nsteps * 1024};
    const uint32_t wbox[3] = {256, kSB / kW4StepK, kBM / kW4Tile};
    if (!tc::make_tmap_3d(&tmap_w, W, CU_TENSOR_MAP_DATA_TYPE_UINT32, wdims, wstrides, wbox))
        return cudaErrorInvalidValue;
    return launch_stream_k<kW4A16>(a, tmap_w, tmap_w, A, s);
}

cudaError_t launch_quantize_q4_0_prefill(const float *X, void *ws, int64_t M, int64_t K,
                                         cudaStream_t s) {
    quantize_q4_0_prefill_kernel<<<(unsigned)M, kActThreads, 0, s>>>(X, static_cast<__half *>(ws),
                                                                    tok_scales(ws, M, K), M, K);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_gemm_q4_0(const void *Wp, int64_t N, int64_t K, const void *ws, float *part,
                             int64_t M, float *Y, cudaStream_t s) {
    Args a;
    a.S = nullptr;
    a.Z = nullptr;
    a.lut = nullptr;
    a.C = Y;
    a.M = M;
    a.N = N;
    a.K = K;
    a.ng = 0;
    a.spg = 1;
    a.err = device_error_word();
    a.part = part;
    a.tok_scale = tok_scales(ws, M, K);
    const int64_t nb = K / QK4_0, ntiles = tiles_of(N);
    const uint64_t tile_bytes = (uint64_t)nb * kQ4Tile * B_Q4_0;
    CUtensorMap tmap_w, tmap_d;
    // nibble planes as [tile][row][block][4 words], read as [tile][block][row][16 B]
    const uint64_t ndims[4] = {4, (uint64_t)kQ4Tile, (uint64_t)nb, (uint64_t)ntiles};
    const uint64_t nstrides[3] = {(uint64_t)nb * 16, 16, tile_bytes};
    const uint32_t nbox[4] = {4, (uint32_t)kQ4Tile, kQ4Blocks, kBM / kQ4Tile};
    // scale planes as [tile][block][8 fp16]
    const uint64_t ddims[3] = {(uint64_t)kQ4Tile, (uint64_t)nb, (uint64_t)ntiles};
    const uint64_t dstrides[2] = {16, tile_bytes};
    const uint32_t dbox[3] = {(uint32_t)kQ4Tile, kQ4Blocks, kBM / kQ4Tile};
    const uint8_t *dplane = static_cast<const uint8_t *>(Wp) + (size_t)nb * kQ4Tile * 16;
    if (!tc::make_tmap_4d(&tmap_w, Wp, CU_TENSOR_MAP_DATA_TYPE_UINT32, ndims, nstrides, nbox) ||
        !tc::make_tmap_3d(&tmap_d, dplane, CU_TENSOR_MAP_DATA_TYPE_UINT16, ddims, dstrides, dbox))
        return cudaErrorInvalidValue;
    return launch_stream_k<kQ40>(a, tmap_w, tmap_d, ws, s);
}

// ------------------------------------------------------------------ Q6_K prefill
cudaError_t launch_quantize_q8_K_f16(const float *X, void *ws, int64_t M, int64_t K, cudaStream_t s) {
    quantize_q8_K_f16_kernel<<<(unsigned)M, kActThreads, 0, s>>>(X, static_cast<__half *>(ws),
                                                                tok_scales(ws, M, K), M, K);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_import_q8_K_f16(const void *Xq, void *ws, int64_t M, int64_t K, cudaStream_t s) {
    import_q8_K_f16_kernel<<<(unsigned)M, kActThreads, 0, s>>>(static_cast<const uint8_t *>(Xq),
                                                              static_cast<__half *>(ws), tok_scales(ws, M, K),
                                                              M, K);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_gemm_q4_K_f16(const void *Wp, int64_t N, int64_t K, const void *ws, float *part,
                                 int64_t M, float *Y, cudaStream_t s) {
    Args a;
    a.S = nullptr;
    a.Z = nullptr;
    a.lut = nullptr;
    a.C = Y;
    a.M = M;
    a.N = N;
    a.K = K;
    a.ng = 0;
    a.spg = 1;
    a.err = device_error_word();
    a.part = part;
    a.tok_scale = tok_scales(ws, M, K);
    const int64_t nsb = K / QK_K;
    constexpr int kRec = kTileRows * B_Q4_K;  // 1152 B: one (tile, super-block)
    CUtensorMap tmap_w;
    const uint64_t wdims[3] = {kRec / 8, (uint64_t)nsb, (uint64_t)tiles_of(N)};
    const uint64_t wstrides[2] = {(uint64_t)kRec, (uint64_t)nsb * kRec};
    const uint32_t wbox[3] = {kRec / 8, 1, kBM / kTileRows};
    if (!tc::make_tmap_3d(&tmap_w, Wp, CU_TENSOR_MAP_DATA_TYPE_UINT64, wdims, wstrides, wbox))
        return cudaErrorInvalidValue;
    return launch_stream_k<kQ4K>(a, tmap_w, tmap_w, ws, s);
}

cudaError_t launch_gemm_q6_K(const void *Wp, int64_t N, int64_t K, const void *ws, float *part, int64_t M,
                             float *Y, cudaStream_t s) {
    Args a;
    a.S = nullptr;
    a.Z = nullptr;
    a.lut = nullptr;
    a.C = Y;
    a.M = M;
    a.N = N;
    a.K = K;
    a.ng = 0;
    a.spg = 1;
    a.err = device_error_word();
    a.part = part;
    a.tok_scale = tok_scales(ws, M, K);
    const int64_t nsb = K / QK_K;
    CUtensorMap tmap_w;
    // packed records as [8-row tile][super-block][1680 B], in 8-byte units
    const uint64_t wdims[3] = {kQ6Rec / 8, (uint64_t)nsb, (uint64_t)tiles_of(N)};
    const uint64_t wstrides[2] = {(uint64_t)kQ6Rec, (uint64_t)nsb * kQ6Rec};
    const uint32_t wbox[3] = {kQ6Rec / 8, 1, kBM / kTileRows};
    if (!tc::make_tmap_3d(&tmap_w, Wp, CU_TENSOR_MAP_DATA_TYPE_UINT64, wdims, wstrides, wbox))
        return cudaErrorInvalidValue;
    return launch_stream_k<kQ6K>(a, tmap_w, tmap_w, ws, s);
}

}  // namespace qmm
