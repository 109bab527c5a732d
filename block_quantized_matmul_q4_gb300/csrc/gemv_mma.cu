// gemv_mma.cu -- decode-path mul_mat (M = 1..16 tokens per launch) over packed
// Q4_K weights on the tensor cores (mma.sync m16n8k16, fp16 operands, fp32
// accumulation).
//
// What is computed is page 1's Q4_K x Q8_K dot product ("正确性: 缩放系数可以
// 提到求和号外面", "min 项与最终归约"): per super-block and (row, token)
//   isum = sum_j s_j sum_{k in sub-block j} q_k y_k,
//   msum = sum_j m_j (bs_2j + bs_2j+1),
//   y   += d_a (d isum - dmin msum).
// The integer structure is kept exactly by feeding the MMA integer-valued
// fp16 operands (page 3, "Tensor Core 数据通路": decode in registers, feed the
// MMA):
//   * A (weights, 16 rows = a pair of 8-row packed tiles) holds s_j * q_k,
//     at most 63 * 15 = 945, exact in fp16; it is made from the nibbles with
//     one lop3 (fp16 1024 + q, or 1024 + 16 q for a high nibble) and one fused
//     multiply-add by s_j (s_j / 16) that removes the bias exactly;
//   * B (activations, n8 = up to 8 tokens) holds the Q8_K codes, exact in fp16;
//   * products are exact in fp32, and so is the super-block sum while it
//     stays below 2^24 (it exceeds 2^22 only when most of the 256 products sit
//     near their bound);
//   * msum is one more m16n8k16 per super-block: A = (m_2c, m_2c+1) per row,
//     B = the sixteen 16-code sums (|bs| <= 2032, exact in fp16).
// Against the scalar dp4a GEMV, one set of weight conversions serves all the
// tokens of the launch, so the cost per weight hardly grows with M.
//
// Work split: a CTA owns a contiguous range of tile pairs. One producer warp
// streams (pair, 8 super-blocks) stages through a shared-memory ring with
// 1-D bulk copies, as in gemv.cu. Consumer warp w takes super-block w of
// every stage, so each warp only ever needs the activations of super-blocks
// w, w + 8, w + 16, ...: for small M*K it quantizes them itself from fp32 X
// into its own shared-memory area, with no CTA-wide barrier; otherwise a
// stand-alone quantizer writes the whole area once (the activation image)
// and every CTA bulk-copies it. The eight warps' partial sums of a pair are added through
// shared memory once per pair.
//
// K mapping inside one m16n8k16 step (the MMA's K order is free as long as A
// and B agree): lane (g, t) = (lane / 4, lane % 4) of the warp reads qs bytes
// 32t .. 32t + 31 of its two rows, i.e. all of sub-blocks 2t (low nibbles)
// and 2t + 1 (high nibbles). Word i of those bytes feeds steps 2i (low
// nibbles) and 2i + 1 (high nibbles); in step 2i the lane's K positions
// (2t, 2t+1) hold elements (e, e+2) and (2t+8, 2t+9) hold (e+1, e+3), with
// e = 64t + 4i (e + 32 .. for step 2i + 1).
#include "qmm_internal.cuh"

namespace qmm {
namespace {

constexpr int kMWarps = 8;                  // consumer warps
constexpr int kMConsumers = kMWarps * 32;
constexpr int kMThreads = kMConsumers + 32;  // + one producer warp
constexpr int kSbStage = 8;                  // super-blocks per stage and tile
constexpr int kMHalf = kSbStage * kTileRows * B_Q4_K;  // one tile's share: 9216 B
constexpr int kMStage = 2 * kMHalf;                    // 18432 B
constexpr int kSbCodes = 512;                // fp16 codes of one (super-block, token)
constexpr int kSbSums = 32;                  // fp16 16-code sums of one (super-block, token)

struct MmaArgs {
    MatSet ms;          // packed Q4_K weights, outputs, rows; units = tile pairs
    int64_t nsb;        // super-blocks per row
    const float *X;     // fp32 activations (fused quantizer) or nullptr
    const uint8_t *img; // activation image of this launch (when X == nullptr)
    int64_t m0;         // first token of this launch
    int mc;             // tokens in this launch (1..16)
    int stages;         // ring depth
    unsigned *err;
    uint32_t act_off, act_warp;  // per-warp activation areas: offset, bytes each
    uint32_t bs_off, d_off;      // inside one warp's area
    uint32_t red_off, bar_off;
};

__device__ __forceinline__ uint32_t lop_or(uint32_t x, uint32_t mask) {
    uint32_t d;  // (x & mask) | 0x64006400
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(x), "r"(mask), "r"(0x64006400u));
    return d;
}
__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t half2_bits(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kMConsumers) : "memory");
}

// fp16 constants (two copies each)
constexpr uint32_t kH1024 = 0x64006400u;      // 1024
constexpr uint32_t kHNeg1024 = 0xE400E400u;   // -1024
constexpr uint32_t kHSixteenth = 0x2C002C00u; // 1/16
constexpr uint32_t kHNeg64 = 0xD400D400u;     // -64

// Byte offset of the 16-byte slot (word i, lane column t) of token m inside a
// (super-block, token) code block; odd tokens flip bit 2 of the slot so that
// tokens 2p and 2p + 1 (one 8-lane phase of a 128-bit load) use both halves
// of the banks.
__device__ __forceinline__ uint32_t code_slot(int i, int t, int m) {
    return (uint32_t)(((i * 4 + t) ^ ((m & 1) << 2)) * 16);
}

// One Q8_K super-block of one token, held 8 elements per lane (lane l:
// elements 8l .. 8l+7), written to the warp's area in the MMA layout.
// h[0] = codes (8l, 8l+2), h[1] = (8l+1, 8l+3), h[2] = (8l+4, 8l+6),
// h[3] = (8l+5, 8l+7); bsum = codes 16(l/2) .. 16(l/2)+15 summed (valid on
// even lanes); d the fp32 block scale.
__device__ __forceinline__ void put_sb(uint8_t *codes, uint8_t *sums, float *dslot, int m, int lane,
                                       const uint32_t h[4], float bsum, float d) {
    const int c = lane >> 3, r = lane & 7;  // chunk (= reader lane column), 8-element run
    const int hi = r >> 2, i0 = 2 * (r & 3);
    *reinterpret_cast<uint2 *>(codes + code_slot(i0, c, m) + hi * 8) = make_uint2(h[0], h[1]);
    *reinterpret_cast<uint2 *>(codes + code_slot(i0 + 1, c, m) + hi * 8) = make_uint2(h[2], h[3]);
    if ((lane & 1) == 0) {
        // 16-code sum g = lane / 2 goes to slot 4 (g / 4) + {0, 2, 1, 3}[g % 4]
        const int g = lane >> 1, gl = g & 3;
        const int pos = 4 * (g >> 2) + ((gl & 1) << 1) + (gl >> 1);
        reinterpret_cast<__half *>(sums)[pos] = __float2half_rn(bsum);
    }
    if (lane == 0) *dslot = d;
}

// Q8_K quantization of 8 values per lane (page 1, "第一步: 激活得先变成
// Q8_K"): d = amax / 127, codes round-half-away(x / d) clamped to +-127 --
// the arithmetic of q8_K_warp -- packed into fp16 pairs (exact: integers of
// magnitude <= 127) and the 16-code sums as fp32, all without conversions.
__device__ __forceinline__ void quant_sb(const float v[8], uint32_t h[4], float &bsum, float &d) {
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
    const float amax = warp_max_nonneg(a);
    d = __fdiv_rn(amax, 127.0f);
    const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
    int q[8], s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        q[i] = q8_code(v[i], id);
        s += q[i];
    }
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    bsum = int_as_exact_float(s);
    // fp16 pairs of the codes: (1152 + q) as bits, then 1152 taken off (exact)
    auto pair = [&](int x, int y) {
        return hsub2_u(biased_half_bits(x) | (biased_half_bits(y) << 16), 0x64806480u);
    };
    h[0] = pair(q[0], q[2]);
    h[1] = pair(q[1], q[3]);
    h[2] = pair(q[4], q[6]);
    h[3] = pair(q[5], q[7]);
}

// Scale operands of one row for lane column t: field f = s_2t | m_2t << 6 |
// s_2t+1 << 12 | m_2t+1 << 18 of the packed header (bits 24..31 undefined).
struct RowScales {
    uint32_t sl, nl;  // (s_lo, s_lo), (-1024 s_lo, ...)
    uint32_t sh, nh;  // (s_hi / 16, ...), (-64 s_hi, ...)
    uint32_t mm;      // (m_lo, m_hi)
};
__device__ __forceinline__ RowScales row_scales(uint32_t f) {
    RowScales r;
    const uint32_t slo = hsub2_u(kH1024 + (f & 63u) * 0x00010001u, kH1024);
    const uint32_t shi_raw = kH1024 + ((f >> 12) & 63u) * 0x00010001u;
    r.sl = slo;
    r.nl = hmul2_u(slo, kHNeg1024);
    r.sh = hfma2_u(shi_raw, kHSixteenth, kHNeg64);  // (1024 + s) / 16 - 64 = s / 16
    r.nh = hmul2_u(r.sh, kHNeg1024);                // -1024 s / 16 = -64 s
    // m_lo sits at bits 6..11 and m_hi at 18..23 (bits 24..31 of f are not part
    // of the field): move them to the two halves
    r.mm = hsub2_u(((f >> 6) & 63u) + ((f >> 18) & 63u) * 0x00010000u + kH1024, kH1024);
    return r;
}

// A operands of steps 2i (low nibbles) and 2i + 1 (high nibbles) from word w
// of one row: e = (s q_e, s q_e+2), o = (s q_e+1, s q_e+3).
__device__ __forceinline__ void conv_word(uint32_t w, const RowScales &s, uint32_t &lo_e,
                                          uint32_t &lo_o, uint32_t &hi_e, uint32_t &hi_o) {
    const uint32_t v = w >> 8;
    lo_e = hfma2_u(lop_or(w, 0x000F000Fu), s.sl, s.nl);
    hi_e = hfma2_u(lop_or(w, 0x00F000F0u), s.sh, s.nh);
    lo_o = hfma2_u(lop_or(v, 0x000F000Fu), s.sl, s.nl);
    hi_o = hfma2_u(lop_or(v, 0x00F000F0u), s.sh, s.nh);
}

__device__ __forceinline__ uint32_t pick(const uint4 &a, const uint4 &b, int i) {
    const uint4 &v = i < 4 ? a : b;
    switch (i & 3) {
    case 0: return v.x;
    case 1: return v.y;
    case 2: return v.z;
    default: return v.w;
    }
}

// Bounded wait that, once any wait of the CTA has given up, no longer waits.
__device__ __forceinline__ void wait_or_skip(uint32_t bar, uint32_t parity, unsigned *err,
                                             volatile int *abort_flag) {
    if (*abort_flag) return;
    if (!mbar_wait(bar, parity, err)) *abort_flag = 1;
}

template <int NT>  // n8 token tiles: 1 (M <= 8) or 2 (M <= 16)
__global__ void __launch_bounds__(kMThreads, NT == 1 ? 2 : 1) gemv_mma_q4_K_kernel(const MmaArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nsb = a.nsb, K = nsb * QK_K;
    const int64_t npairs = a.ms.off[a.ms.n];
    const int64_t pb = (int64_t)blockIdx.x * npairs / gridDim.x;
    const int64_t pe = ((int64_t)blockIdx.x + 1) * npairs / gridDim.x;
    const int64_t nchunks = (nsb + kSbStage - 1) / kSbStage;
    const int64_t n_items = (pe - pb) * nchunks;
    const int S = a.stages;

    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.bar_off);
    uint64_t *empty = full + S;
    uint64_t *act_bar = empty + S;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(act_bar + 1);
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), kMWarps);
        }
        mbar_init(smem_u32(act_bar), 1);
        *abort_flag = 0;
        fence_barrier_init();
        // The next kernel in the stream may launch now: until its
        // griddepcontrol.wait it only streams weights.
        pdl_launch_dependents();
    }
    __syncthreads();

    uint8_t *act = smem + a.act_off;
    const uint32_t act_bytes = kMWarps * a.act_warp;
    if (warp == kMWarps) {  // ---------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            // the activation image is written by the preceding quantizer: copy it
            // once the first weight stages are in flight
            auto image = [&]() {
                if (!a.img) return;
                pdl_wait();
                mbar_arrive_expect_tx(smem_u32(act_bar), act_bytes);
                bulk_g2s(smem_u32(act), a.img, act_bytes, smem_u32(act_bar), policy_evict_last());
            };
            int64_t it = 0;
            bool img_done = false;
            int s = 0;
            uint32_t ph = 0;             // ring position and phase
            int64_t chunk = 0, pair = pb;  // counters instead of divisions
            for (; it < n_items; ++it) {
                if (it == S) {
                    image();
                    img_done = true;
                }
                if (*abort_flag) break;
                if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1u, a.err)) {
                    *abort_flag = 1;
                    break;
                }
                const int mi = mat_of(a.ms, pair);
                const int64_t t0 = 2 * (pair - a.ms.off[mi]);
                const int64_t sb0 = chunk * kSbStage;
                const uint32_t bytes = (uint32_t)(nsb - sb0 < kSbStage ? nsb - sb0 : kSbStage) * kTileRows * B_Q4_K;
                const bool has1 = t0 + 1 < tiles_of(a.ms.N[mi]);
                const uint8_t *W = a.ms.W[mi];
                const uint32_t dst = smem_u32(smem + (size_t)s * kMStage), bar = smem_u32(&full[s]);
                mbar_arrive_expect_tx(bar, has1 ? 2 * bytes : bytes);
                bulk_g2s(dst, W + (t0 * nsb + sb0) * (kTileRows * B_Q4_K), bytes, bar, pol);
                if (has1)
                    bulk_g2s(dst + kMHalf, W + ((t0 + 1) * nsb + sb0) * (kTileRows * B_Q4_K),
                             bytes, bar, pol);
                if (++s == S) s = 0, ph ^= 1u;
                if (++chunk == nchunks) chunk = 0, ++pair;
            }
            if (!img_done) image();
            // no copy issued by this CTA may still be landing when it exits
            for (int64_t k = it > S ? it - S : 0; k < it; ++k)
                mbar_wait(smem_u32(&full[k % S]), (uint32_t)((k / S) & 1), a.err);
            if (a.img) mbar_wait(smem_u32(act_bar), 0, a.err);
        }
        return;
    }

    // ------------------------------------------------------------ activations
    // Warp w's area: codes [j][mc][512 B], sums [j][mc][32 B], d [j][NT * 8]
    // for its super-blocks sb = 8 j + w.
    uint8_t *area = act + (size_t)warp * a.act_warp;
    uint8_t *codes = area;
    uint8_t *sums = area + a.bs_off;
    float *dsl = reinterpret_cast<float *>(area + a.d_off);
    const int mc = a.mc;
    pdl_wait();  // X / the image come from the preceding kernels; Y is written below
    if (a.X) {
        for (int64_t j = 0, sb = warp; sb < nsb; ++j, sb += kMWarps) {
            for (int m = 0; m < mc; ++m) {
                const float4 *src =
                    reinterpret_cast<const float4 *>(a.X + (a.m0 + m) * K + sb * QK_K + 8 * lane);
                const float4 v0 = __ldg(src), v1 = __ldg(src + 1);
                const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                uint32_t h[4];
                float bsum, d;
                quant_sb(v, h, bsum, d);
                put_sb(codes + (j * mc + m) * kSbCodes, sums + (j * mc + m) * kSbSums,
                       dsl + j * (NT * 8) + m, m, lane, h, bsum, d);
            }
            if (lane < NT * 8 - mc) dsl[j * (NT * 8) + mc + lane] = 0.0f;
        }
        __syncwarp();
    } else {
        wait_or_skip(smem_u32(act_bar), 0, a.err, abort_flag);
    }

    // ------------------------------------------------------------ main loop
    const int g = lane >> 2, t = lane & 3;
    const uint32_t fsh = (uint32_t)((24 * t) & 31);
    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[n][e] = 0.0f;
    float *red = reinterpret_cast<float *>(smem + a.red_off);
    int pair_no = 0;

    // B operand addresses: token m = 8 n + g, slot of (word i, column t) with
    // the odd-token swizzle: ((i ^ (m & 1)) * 4 + t) * 16 = i * 64 + (t * 16 +
    // (i even ? +64 : -64) * (m & 1))
    const int sw = (g & 1) * 64;
    const uint32_t boff_e = (uint32_t)(g * kSbCodes + t * 16 + sw);
    const uint32_t boff_o = (uint32_t)(g * kSbCodes + t * 16 - sw);
    int s = 0;
    uint32_t ph = 0;
    int64_t chunk = 0, pair = pb;
    for (int64_t it = 0; it < n_items; ++it) {
        wait_or_skip(smem_u32(&full[s]), ph, a.err, abort_flag);
        const int cnt = (int)(nsb - chunk * kSbStage < kSbStage ? nsb - chunk * kSbStage : kSbStage);
        if (warp < cnt) {
            const uint8_t *rowA = smem + (size_t)s * kMStage + (warp * kTileRows + g) * B_Q4_K;
            const uint8_t *rowB = rowA + kMHalf;
            const uint4 hA = *reinterpret_cast<const uint4 *>(rowA);
            const uint4 qA0 = *reinterpret_cast<const uint4 *>(rowA + 16 + 32 * t);
            const uint4 qA1 = *reinterpret_cast<const uint4 *>(rowA + 32 + 32 * t);
            const uint4 hB = *reinterpret_cast<const uint4 *>(rowB);
            const uint4 qB0 = *reinterpret_cast<const uint4 *>(rowB + 16 + 32 * t);
            const uint4 qB1 = *reinterpret_cast<const uint4 *>(rowB + 32 + 32 * t);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));  // the stage's bytes are in registers

            const uint32_t fA = __funnelshift_r(t >= 3 ? hA.w : (t >= 2 ? hA.z : hA.y),
                                                t >= 2 ? hA.w : hA.z, fsh);
            const uint32_t fB = __funnelshift_r(t >= 3 ? hB.w : (t >= 2 ? hB.z : hB.y),
                                                t >= 2 ? hB.w : hB.z, fsh);
            const RowScales sA = row_scales(fA), sB = row_scales(fB);

            const int64_t j = chunk;  // this warp's super-block 8 chunk + warp
            const uint8_t *cb = codes + (size_t)j * mc * kSbCodes;
            // two accumulator chains (low- and high-nibble steps), added at the end:
            // both partial sums are integers below 2^24, so the sum is exact
            float isum[NT][2][4], msum[NT][4];
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) isum[n][0][e] = isum[n][1][e] = msum[n][e] = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t aLe, aLo, aHe, aHo, bLe, bLo, bHe, bHo;
                conv_word(pick(qA0, qA1, i), sA, aLe, aLo, aHe, aHo);
                conv_word(pick(qB0, qB1, i), sB, bLe, bLo, bHe, bHo);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const int m = n * 8 + g;
                    uint4 y = make_uint4(0u, 0u, 0u, 0u);
                    if (m < mc)  // m & 1 == g & 1
                        y = *reinterpret_cast<const uint4 *>(cb + n * 8 * kSbCodes + i * 64 +
                                                             ((i & 1) ? boff_o : boff_e));
                    mma_16816(isum[n][0], aLe, bLe, aLo, bLo, y.x, y.y);  // step 2i
                    mma_16816(isum[n][1], aHe, bHe, aHo, bHo, y.z, y.w);  // step 2i + 1
                }
            }
            const float2 dA = __half22float2(*reinterpret_cast<const __half2 *>(&hA.x));
            const float2 dB = __half22float2(*reinterpret_cast<const __half2 *>(&hB.x));
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int m = n * 8 + g;
                uint2 bs = make_uint2(0u, 0u);
                if (m < mc)
                    bs = *reinterpret_cast<const uint2 *>(sums + (j * mc + m) * kSbSums + 8 * t);
                mma_16816(msum[n], sA.mm, sB.mm, sA.mm, sB.mm, bs.x, bs.y);
                const float2 da = *reinterpret_cast<const float2 *>(dsl + j * (NT * 8) + n * 8 + 2 * t);
                // C fragment: e = 0, 1 row g (tile A), columns 2t, 2t + 1; e = 2, 3 row g + 8
                float is[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) is[e] = isum[n][0][e] + isum[n][1][e];
                acc[n][0] += da.x * (dA.x * is[0] - dA.y * msum[n][0]);
                acc[n][1] += da.y * (dA.x * is[1] - dA.y * msum[n][1]);
                acc[n][2] += da.x * (dB.x * is[2] - dB.y * msum[n][2]);
                acc[n][3] += da.y * (dB.x * is[3] - dB.y * msum[n][3]);
            }
        } else {
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        }

        if (chunk == nchunks - 1) {  // pair done: add the eight warps' partial sums
            float *rb = red + (size_t)(pair_no & 1) * (kMWarps * NT * 4 * 32);
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    rb[((warp * NT + n) * 4 + e) * 32 + lane] = acc[n][e];
                    acc[n][e] = 0.0f;
                }
            consumers_sync();
            const int tid = threadIdx.x;  // one output per thread: (n, e, lane)
            if (tid < NT * 4 * 32) {
                const int n = tid >> 7, e = (tid >> 5) & 3, l = tid & 31;
                float v = 0.0f;
#pragma unroll
                for (int w = 0; w < kMWarps; ++w) v += rb[((w * NT + n) * 4 + e) * 32 + l];
                const int m = n * 8 + 2 * (l & 3) + (e & 1);
                const int mi = mat_of(a.ms, pair);
                const int64_t N = a.ms.N[mi];
                const int64_t row = (pair - a.ms.off[mi]) * 16 + (e >> 1) * 8 + (l >> 2);
                if (m < mc && row < N) a.ms.Y[mi][(a.m0 + m) * N + row] = v;
            }
            ++pair_no;
        }
        if (++s == S) s = 0, ph ^= 1u;
        if (++chunk == nchunks) chunk = 0, ++pair;
    }
}

// Per-warp activation area for mc tokens over nsb super-blocks: codes
// [J][mc][512 B], 16-code sums [J][mc][32 B], scales [J][nt * 8] fp32,
// J = ceil(nsb / 8); the CTA holds eight of them (warp w: super-blocks
// w, w + 8, ...), and so does one launch's activation image.
struct Layout {
    int nt;
    uint32_t warp_bytes, bs_off, d_off;
};
__host__ __device__ inline Layout act_layout(int64_t nsb, int mc) {
    Layout L;
    L.nt = mc <= 8 ? 1 : 2;
    const uint64_t J = (uint64_t)(nsb + kMWarps - 1) / kMWarps;
    L.bs_off = (uint32_t)(J * mc * kSbCodes);
    L.d_off = (uint32_t)(L.bs_off + J * mc * kSbSums);
    L.warp_bytes = (uint32_t)align_up(L.d_off + J * L.nt * 8 * 4, 128);
    return L;
}

// Activation quantizer for the MMA path: one warp per (token, super-block)
// writes its codes, sums and scale straight into the launch's image, in the
// layout the GEMV copies into shared memory.
__global__ void __launch_bounds__(256) quantize_mma_image_kernel(const float *X, uint8_t *img,
                                                                 int64_t M, int64_t nsb, int per) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (threadIdx.x == 0) pdl_launch_dependents();
    if (gw >= M * nsb) return;
    pdl_wait();
    const int64_t m = gw / nsb, sb = gw % nsb, K = nsb * QK_K;
    const int64_t chunk = m / per;
    const int ml = (int)(m - chunk * per);
    const int mc = (int)(M - chunk * per < per ? M - chunk * per : per);
    const Layout full = act_layout(nsb, per), L = act_layout(nsb, mc);
    uint8_t *area = img + (size_t)chunk * kMWarps * full.warp_bytes + (sb % kMWarps) * L.warp_bytes;
    const int64_t j = sb / kMWarps;
    const float4 *src = reinterpret_cast<const float4 *>(X + m * K + sb * QK_K + 8 * lane);
    const float4 v0 = __ldg(src), v1 = __ldg(src + 1);
    const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t h[4];
    float bsum, d;
    quant_sb(v, h, bsum, d);
    float *dsl = reinterpret_cast<float *>(area + L.d_off) + j * (L.nt * 8);
    put_sb(area + (j * mc + ml) * kSbCodes, area + L.bs_off + (j * mc + ml) * kSbSums, dsl + ml, ml,
           lane, h, bsum, d);
    if (ml == 0 && lane < L.nt * 8 - mc) dsl[mc + lane] = 0.0f;
}

// The same image from canonical Q8_K blocks [M][nsb] x 292 B (their codes,
// scale and stored 16-code sums), for qmm_mul_mat_q8.
__global__ void __launch_bounds__(256) import_mma_image_kernel(const uint8_t *Xq, uint8_t *img,
                                                               int64_t M, int64_t nsb, int per) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (threadIdx.x == 0) pdl_launch_dependents();
    if (gw >= M * nsb) return;
    pdl_wait();
    const int64_t m = gw / nsb, sb = gw % nsb;
    const int64_t chunk = m / per;
    const int ml = (int)(m - chunk * per);
    const int mc = (int)(M - chunk * per < per ? M - chunk * per : per);
    const Layout full = act_layout(nsb, per), L = act_layout(nsb, mc);
    uint8_t *area = img + (size_t)chunk * kMWarps * full.warp_bytes + (sb % kMWarps) * L.warp_bytes;
    const int64_t j = sb / kMWarps;
    const uint8_t *blk = Xq + gw * B_Q8_K;
    const uint32_t *qw = reinterpret_cast<const uint32_t *>(blk + 4 + 8 * lane);
    const uint32_t w[2] = {qw[0], qw[1]};
    float q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = (float)(int8_t)(w[i >> 2] >> (8 * (i & 3)));
    const uint32_t h[4] = {half2_bits(q[0], q[2]), half2_bits(q[1], q[3]), half2_bits(q[4], q[6]),
                           half2_bits(q[5], q[7])};
    const float bsum = (float)reinterpret_cast<const int16_t *>(blk + 260)[lane >> 1];
    const float d = *reinterpret_cast<const float *>(blk);
    float *dsl = reinterpret_cast<float *>(area + L.d_off) + j * (L.nt * 8);
    put_sb(area + (j * mc + ml) * kSbCodes, area + L.bs_off + (j * mc + ml) * kSbSums, dsl + ml, ml,
           lane, h, bsum, d);
    if (ml == 0 && lane < L.nt * 8 - mc) dsl[mc + lane] = 0.0f;
}

struct Plan {
    Layout L;
    int stages, ctas_per_sm;
    uint32_t act_off, red_off, bar_off, smem;
};

constexpr uint32_t kSmemMax = 227 * 1024;

// Shared-memory plan for mc tokens over nsb super-blocks:
// [ring][8 warp areas][reduction, double-buffered][barriers + abort flag].
bool make_plan(int64_t nsb, int mc, Plan *p) {
    const Layout L = act_layout(nsb, mc);
    const uint64_t red = 2ull * kMWarps * L.nt * 4 * 32 * 4;
    // Two CTAs per SM (each within half of the SM's 228 KB, less the 1 KB the
    // hardware reserves per CTA) with a ring of 4, 3 or 2 stages, else one CTA
    // with 4, 3 or 2 stages.
    static const int kTry[6][2] = {{4, 2}, {3, 2}, {2, 2}, {4, 1}, {3, 1}, {2, 1}};
    for (const auto &tr : kTry) {
        const int stages = tr[0];
        const uint64_t ring = (uint64_t)stages * kMStage;
        const uint64_t total =
            ring + (uint64_t)kMWarps * L.warp_bytes + red + (2 * stages + 1) * 8 + 8;  // + flag
        const uint64_t cap = tr[1] == 2 ? 113 * 1024 : kSmemMax;
        if (tr[1] == 2 && L.nt == 2) continue;  // its registers allow one CTA per SM
        if (total <= cap) {
            p->L = L;
            p->stages = stages;
            p->ctas_per_sm = tr[1];
            p->act_off = (uint32_t)ring;
            p->red_off = (uint32_t)(ring + (uint64_t)kMWarps * L.warp_bytes);
            p->bar_off = (uint32_t)(p->red_off + red);
            p->smem = (uint32_t)total;
            return true;
        }
    }
    return false;
}

}  // namespace

// Largest number of tokens (<= 16) one launch can hold for this K.
int gemv_mma_max_tokens(int64_t K) {
    Plan p;
    for (int mc = 16; mc >= 1; --mc)
        if (make_plan(K / QK_K, mc, &p)) return mc;
    return 0;
}

// Bytes of the activation images of all launches for M tokens.
size_t gemv_mma_image_bytes(int64_t M, int64_t K) {
    const int per = gemv_mma_max_tokens(K);
    if (per == 0) return 0;
    const int64_t nsb = K / QK_K, full = M / per, rest = M % per;
    size_t b = (size_t)full * kMWarps * act_layout(nsb, per).warp_bytes;
    if (rest) b += (size_t)kMWarps * act_layout(nsb, (int)rest).warp_bytes;
    return b;
}

cudaError_t launch_quantize_mma_image(const float *X, void *img, int64_t M, int64_t K,
                                      cudaStream_t s) {
    const int per = gemv_mma_max_tokens(K);
    if (per == 0) return cudaErrorInvalidValue;
    const int64_t nsb = K / QK_K;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((M * nsb + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, quantize_mma_image_kernel, X, static_cast<uint8_t *>(img),
                                       M, nsb, per);
    count_launch();
    return e;
}

cudaError_t launch_import_mma_image(const void *Xq, void *img, int64_t M, int64_t K, cudaStream_t s) {
    const int per = gemv_mma_max_tokens(K);
    if (per == 0) return cudaErrorInvalidValue;
    const int64_t nsb = K / QK_K;
    import_mma_image_kernel<<<(unsigned)((M * nsb + 7) / 8), 256, 0, s>>>(
        static_cast<const uint8_t *>(Xq), static_cast<uint8_t *>(img), M, nsb, per);
    count_launch();
    return cudaGetLastError();
}

// X != nullptr: the activation quantizer runs inside the kernel; otherwise the
// activations are the images written by launch_quantize_mma_image at img.
cudaError_t launch_gemv_mma_q4_K(MatSet ms, int64_t K, const float *X, const void *img, int64_t M,
                                 bool pdl, cudaStream_t s) {
    ms.off[0] = 0;
    for (int i = 0; i < ms.n; ++i) ms.off[i + 1] = ms.off[i] + (tiles_of(ms.N[i]) + 1) / 2;
    MmaArgs a;
    a.ms = ms;
    a.nsb = K / QK_K;
    a.X = X;
    a.err = device_error_word();
    const int per = gemv_mma_max_tokens(K);
    if (per == 0) return cudaErrorInvalidValue;
    const int64_t npairs = ms.off[ms.n];
    const uint8_t *im = static_cast<const uint8_t *>(img);
    for (int64_t m0 = 0; m0 < M; m0 += per) {
        Plan p;
        a.m0 = m0;
        a.mc = (int)(M - m0 < per ? M - m0 : per);
        make_plan(a.nsb, a.mc, &p);
        a.img = X ? nullptr : im;
        if (im) im += (size_t)kMWarps * p.L.warp_bytes;
        a.stages = p.stages;
        a.act_off = p.act_off;
        a.act_warp = p.L.warp_bytes;
        a.bs_off = p.L.bs_off;
        a.d_off = p.L.d_off;
        a.red_off = p.red_off;
        a.bar_off = p.bar_off;
        const void *fn = p.L.nt == 1 ? reinterpret_cast<const void *>(gemv_mma_q4_K_kernel<1>)
                                     : reinterpret_cast<const void *>(gemv_mma_q4_K_kernel<2>);
        cudaError_t e = ensure_smem_attr(fn, (int)p.smem);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)balanced_grid(npairs, (int64_t)p.ctas_per_sm * sm_count()));
        cfg.blockDim = dim3(kMThreads);
        cfg.dynamicSmemBytes = p.smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
        if (p.L.nt == 1)
            e = cudaLaunchKernelEx(&cfg, gemv_mma_q4_K_kernel<1>, a);
        else
            e = cudaLaunchKernelEx(&cfg, gemv_mma_q4_K_kernel<2>, a);
        count_launch();
        if (e != cudaSuccess) return e;
        pdl = false;
    }
    return cudaSuccess;
}

}  // namespace qmm
