// gemv_mma6.cu -- decode-path mul_mat (M = 2..16 tokens per launch) over
// packed Q6_K and Q4_0 weights on the tensor cores (mma.sync m16n8k16, fp16
// operands, fp32 accumulation), with the block arithmetic kept exact.
//
// Q6_K x Q8_K (page 1, "更低的比特: Q6_K 与 Q2_K 的取舍"): per super-block and
// (row, token)
//   S_j  = sum_{k in group j} q_k y_k       (16 groups of 16, q = u - 32),
//   isum = sum_j s_j S_j                     (s_j the signed 8-bit scales),
//   y   += d_a (d isum).
// One m16n8k16 step is one group: A holds q (|q| <= 32, exact in fp16), B the
// Q8_K codes (exact), so the step's fp32 result is S_j exactly (|S_j| <=
// 16 * 32 * 127 < 2^24), and so is s_j S_j (< 2^23 in magnitude); isum is
// their fp32 sum, exact while it stays below 2^24 in magnitude, which only
// a super-block with most of its products near their bounds reaches. (No
// float-to-integer conversions: they run on the narrow conversion pipe.)
//
// Q4_0 x Q8_0 (page 1, "最基础的两块"): per block of 32 and (row, token)
//   isum = sum_k (q_k - 8) y_k,   y += d_a (d isum).
// Two steps are one block: A holds q - 8 (exact), B the codes; the block sum
// (|isum| <= 32 * 8 * 127) is exact in fp32.
//
// Against the scalar dp4a GEMVs, one set of weight conversions serves all the
// tokens of a launch, so the cost per weight hardly grows with M.
//
// Work split (as gemv_mma.cu): a CTA owns a contiguous range of tile pairs (16
// rows). One producer warp streams (pair, 8 units of 256 elements of K)
// stages through a shared-memory ring with 1-D bulk copies; consumer warp w
// takes unit w of every stage. The activations of a launch are an image
// written by a quantizer kernel (the codes as fp16 in MMA order, the block
// scales as fp32), bulk-copied into shared memory once per CTA; warp w's area
// holds the units w, w + 8, ... The eight warps' partial sums of a pair are
// added through shared memory once per pair.
//
// K order inside one step (free, as long as A and B agree): lane (g, t) of
// the warp takes 4 consecutive elements 4t .. 4t+3 of the step's 16 (one
// 32-bit word of nibbles or 6-bit codes): K positions (2t, 2t+1) hold
// elements (4t, 4t+2), (2t+8, 2t+9) hold (4t+1, 4t+3). A Q6_K step is group
// (lane t_q of the packed record, nibble half h) = elements q6k_elem(t_q, h,
// 0..15), step index 2 t_q + h, whose scale is packed scale byte 2 t_q + h;
// Q4_0 steps 2b, 2b+1 are the low and the high nibbles (elements 0..15, 16..31)
// of block b of the unit.
#include "qmm_internal.cuh"

namespace qmm {
namespace {

constexpr int kWarps6 = 8;
constexpr int kCons6 = kWarps6 * 32;
constexpr int kThreads6 = kCons6 + 32;  // + one producer warp
constexpr int kUnits6 = 8;              // units of 256 elements per stage and tile
constexpr int kSteps6 = 16;             // m16n8k16 steps per unit
constexpr int kSlot6 = 32;              // image bytes of one (step, token): 4 lanes x 4 fp16

enum Fmt6 { kF40 = 0, kF6K = 1 };

// One tile's share of a stage. Q6_K: 8 records of 8 rows. Q4_0: nibbles [8
// rows][64 blocks][16 B] with rows 16 bytes apart more than their length (so
// that the eight rows a warp reads at once fall in different banks), then
// scales [64 blocks][8 rows] fp16.
constexpr int kRow40 = kUnits6 * 8 * 16 + 16;  // 1040
template <int F>
struct Stage6 {
    static constexpr int kNib40 = kTileRows * kRow40;
    static constexpr int kHalf = F == kF6K ? kUnits6 * kQ6Rec : kNib40 + kUnits6 * 8 * kTileRows * 2;
    static constexpr int kBytes = 2 * kHalf;
};

struct Mma6Args {
    MatSet ms;             // packed weights, outputs, rows; units = tile pairs
    int64_t nu;            // units of 256 elements per row (K / 256)
    const uint8_t *img;    // activation image of this launch
    int64_t m0;            // first token of this launch
    int mc;                // tokens in this launch (1..16)
    int stages;            // ring depth
    unsigned *err;
    uint32_t act_off, act_warp;  // per-warp activation areas: offset, bytes each
    uint32_t d_off;              // scales inside one warp's area
    uint32_t red_off, bar_off;
};

__device__ __forceinline__ uint32_t lop_mask_or(uint32_t x, uint32_t mask) {
    uint32_t d;  // (x & mask) | 0x64006400
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(x), "r"(mask), "r"(0x64006400u));
    return d;
}
__device__ __forceinline__ uint32_t h2sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t h2fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// c = A B (a fresh accumulator) or c += A B
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1, bool fresh) {
    if (fresh)
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
            "{%8, %9}, {%10, %10, %10, %10};"
            : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
    else
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
            "{%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void cons_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kCons6) : "memory"); }

// fp16 constants, two copies each
constexpr uint32_t kH1056 = 0x64206420u;     // 1024 + 32: Q6_K code u -> q = u - 32
constexpr uint32_t kH1032 = 0x64086408u;     // 1024 + 8: Q4_0 low nibble -> q - 8
constexpr uint32_t kH16th = 0x2C002C00u;     // 1/16
constexpr uint32_t kHNeg72 = 0xD480D480u;    // -(64 + 8): Q4_0 high nibble (1024 + 16 q) / 16 - 72 = q - 8

// Q6_K A operands of one row for one step: the 6-bit codes u of ql word t
// (nibble half taken by the caller) with their high bits, as (q0, q2) and
// (q1, q3).
__device__ __forceinline__ void q6_pair(uint32_t nib, uint32_t hb, int t, uint32_t &e02, uint32_t &e13) {
    const uint32_t u = q6k_u(nib, hb, t);
    e02 = h2sub(lop_mask_or(u, 0x003F003Fu), kH1056);
    e13 = h2sub(lop_mask_or(u >> 8, 0x003F003Fu), kH1056);
}
// Q4_0 A operands of one row from nibble word w: low nibbles (step 2b) and
// high nibbles (step 2b + 1), each as (e0, e2), (e1, e3), values q - 8.
__device__ __forceinline__ void q40_pairs(uint32_t w, uint32_t &l02, uint32_t &l13, uint32_t &h02,
                                          uint32_t &h13) {
    const uint32_t v = w >> 8;
    l02 = h2sub(lop_mask_or(w, 0x000F000Fu), kH1032);
    l13 = h2sub(lop_mask_or(v, 0x000F000Fu), kH1032);
    h02 = h2fma(lop_mask_or(w, 0x00F000F0u), kH16th, kHNeg72);
    h13 = h2fma(lop_mask_or(v, 0x00F000F0u), kH16th, kHNeg72);
}

// The signed byte k of x as a float, exactly, without a conversion
// instruction: 2^23 + (byte + 128) less 2^23 + 128.
__device__ __forceinline__ float sbyte_f(uint32_t x, int k) {
    const uint32_t b = ((x >> (8 * k)) & 0xFFu) ^ 0x80u;
    return __int_as_float(0x4B000000 | (int)b) - 8388736.0f;
}

__device__ __forceinline__ void wait_or_skip6(uint32_t bar, uint32_t parity, unsigned *err, volatile int *abort_flag) {
    if (*abort_flag) return;
    if (!mbar_wait(bar, parity, err)) *abort_flag = 1;
}

template <int F, int NT>  // NT n8 token tiles: 1 (M <= 8) or 2 (M <= 16)
__global__ void __launch_bounds__(kThreads6, NT == 1 ? 2 : 1) gemv_mma6_kernel(const Mma6Args a) {
    using SG = Stage6<F>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nu = a.nu;
    const int64_t npairs = a.ms.off[a.ms.n];
    const int64_t pb = (int64_t)blockIdx.x * npairs / gridDim.x;
    const int64_t pe = ((int64_t)blockIdx.x + 1) * npairs / gridDim.x;
    const int64_t nchunks = (nu + kUnits6 - 1) / kUnits6;
    const int64_t n_items = (pe - pb) * nchunks;
    const int S = a.stages;
    constexpr int nt = NT * 8;

    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.bar_off);
    uint64_t *empty = full + S;
    uint64_t *act_bar = empty + S;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(act_bar + 1);
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), kWarps6);
        }
        mbar_init(smem_u32(act_bar), 1);
        *abort_flag = 0;
        fence_barrier_init();
        // the next kernel in the stream may launch now: until its
        // griddepcontrol.wait it only streams weights
        pdl_launch_dependents();
    }
    __syncthreads();

    uint8_t *act = smem + a.act_off;
    const uint32_t act_bytes = kWarps6 * a.act_warp;
    if (warp == kWarps6) {  // ---------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            // the image is written by the preceding quantizer: copy it once
            // the first weight stages are in flight
            auto image = [&]() {
                pdl_wait();
                mbar_arrive_expect_tx(smem_u32(act_bar), act_bytes);
                bulk_g2s(smem_u32(act), a.img, act_bytes, smem_u32(act_bar), policy_evict_last());
            };
            int64_t it = 0;
            bool img_done = false;
            int s = 0;
            uint32_t ph = 0;
            int64_t chunk = 0, pair = pb;
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
                const int64_t u0 = chunk * kUnits6;
                const int cnt = (int)(nu - u0 < kUnits6 ? nu - u0 : kUnits6);
                const int ntl = t0 + 1 < tiles_of(a.ms.N[mi]) ? 2 : 1;
                const uint8_t *W = a.ms.W[mi];
                uint8_t *dst = smem + (size_t)s * SG::kBytes;
                const uint32_t bar = smem_u32(&full[s]);
                if (F == kF6K) {
                    const uint32_t bytes = (uint32_t)cnt * kQ6Rec;
                    mbar_arrive_expect_tx(bar, ntl * bytes);
                    for (int h = 0; h < ntl; ++h)
                        bulk_g2s(smem_u32(dst + h * SG::kHalf), W + ((t0 + h) * nu + u0) * kQ6Rec, bytes, bar, pol);
                } else {
                    // per tile: 8 rows of cnt * 8 blocks of nibbles, then their scales
                    const int64_t nb = nu * 8;
                    const int64_t tile_bytes = nb * kTileRows * B_Q4_0;
                    const uint32_t rb = (uint32_t)cnt * 8 * 16;
                    mbar_arrive_expect_tx(bar, ntl * (kTileRows * rb + rb));
                    for (int h = 0; h < ntl; ++h) {
                        const uint8_t *tb = W + (t0 + h) * tile_bytes;
                        uint8_t *th = dst + h * SG::kHalf;
                        for (int r = 0; r < kTileRows; ++r)
                            bulk_g2s(smem_u32(th + r * kRow40), tb + (r * nb + u0 * 8) * 16, rb, bar, pol);
                        bulk_g2s(smem_u32(th + SG::kNib40), tb + nb * kTileRows * 16 + u0 * 8 * kTileRows * 2, rb, bar,
                                 pol);
                    }
                }
                if (++s == S) s = 0, ph ^= 1u;
                if (++chunk == nchunks) chunk = 0, ++pair;
            }
            if (!img_done) image();
            // no copy issued by this CTA may still be landing when it exits
            for (int64_t k = it > S ? it - S : 0; k < it; ++k)
                mbar_wait(smem_u32(&full[k % S]), (uint32_t)((k / S) & 1), a.err);
            mbar_wait(smem_u32(act_bar), 0, a.err);
        }
        return;
    }

    // warp w's image area: codes [J][16 steps][mc tokens][32 B], then scales
    // [J][blocks per unit][nt] fp32, for its units w, w + 8, ...
    const uint8_t *codes = act + (size_t)warp * a.act_warp;
    const float *dsl = reinterpret_cast<const float *>(codes + a.d_off);
    const int mc = a.mc;
    pdl_wait();  // Y is written below; the image comes from the preceding kernel
    wait_or_skip6(smem_u32(act_bar), 0, a.err, abort_flag);

    const int g = lane >> 2, t = lane & 3;
    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[n][e] = 0.0f;
    float *red = reinterpret_cast<float *>(smem + a.red_off);
    int pair_no = 0;
    int s = 0;
    uint32_t ph = 0;
    int64_t chunk = 0, pair = pb;
    for (int64_t it = 0; it < n_items; ++it) {
        wait_or_skip6(smem_u32(&full[s]), ph, a.err, abort_flag);
        const int cnt = (int)(nu - chunk * kUnits6 < kUnits6 ? nu - chunk * kUnits6 : kUnits6);
        const uint8_t *st = smem + (size_t)s * SG::kBytes;
        if (warp < cnt) {
            const int64_t j = chunk;  // this warp's unit 8 chunk + warp
            // B operand of step q, token tile n: 8 bytes at lane (g, t)
            const uint8_t *bb = codes + (size_t)j * kSteps6 * mc * kSlot6 + g * kSlot6 + t * 8;
            if (F == kF6K) {
                const uint8_t *recA = st + warp * kQ6Rec, *recB = recA + SG::kHalf;
                const uint8_t *rowA = recA + g * kQ6Codes, *rowB = recB + g * kQ6Codes;
                const uint4 scA = *reinterpret_cast<const uint4 *>(recA + kQ6ScOff + 16 * g);
                const uint4 scB = *reinterpret_cast<const uint4 *>(recB + kQ6ScOff + 16 * g);
                const float dA = __half2float(*reinterpret_cast<const __half *>(recA + kQ6DOff + 2 * g));
                const float dB = __half2float(*reinterpret_cast<const __half *>(recB + kQ6DOff + 2 * g));
                __syncwarp();
                float isum[NT][4];
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) isum[n][e] = 0.0f;
#pragma unroll
                for (int tq = 0; tq < 8; ++tq) {
                    const uint32_t qa = *reinterpret_cast<const uint32_t *>(rowA + 16 * tq + 4 * t);
                    const uint32_t qb = *reinterpret_cast<const uint32_t *>(rowB + 16 * tq + 4 * t);
                    const uint2 ha = *reinterpret_cast<const uint2 *>(rowA + 128 + 8 * tq);
                    const uint2 hb = *reinterpret_cast<const uint2 *>(rowB + 128 + 8 * tq);
                    const uint32_t sa = tq < 2 ? scA.x : tq < 4 ? scA.y : tq < 6 ? scA.z : scA.w;
                    const uint32_t sbv = tq < 2 ? scB.x : tq < 4 ? scB.y : tq < 6 ? scB.z : scB.w;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int q = 2 * tq + h;  // step = group (tq, h); its scale is packed byte q
                        uint32_t a02, a13, b02, b13;
                        q6_pair(h ? qa >> 4 : qa, h ? ha.y : ha.x, t, a02, a13);
                        q6_pair(h ? qb >> 4 : qb, h ? hb.y : hb.x, t, b02, b13);
                        const float sA = sbyte_f(sa, q & 3), sB = sbyte_f(sbv, q & 3);
#pragma unroll
                        for (int n = 0; n < NT; ++n) {
                            uint2 y = make_uint2(0u, 0u);
                            if (n * 8 + g < mc) y = *reinterpret_cast<const uint2 *>(bb + (q * mc + n * 8) * kSlot6);
                            float c[4];
                            mma16816(c, a02, b02, a13, b13, y.x, y.y, true);
                            // C: e = 0, 1 row g (tile A), tokens 2t, 2t + 1; e = 2, 3 row g + 8
                            isum[n][0] = fmaf(sA, c[0], isum[n][0]);
                            isum[n][1] = fmaf(sA, c[1], isum[n][1]);
                            isum[n][2] = fmaf(sB, c[2], isum[n][2]);
                            isum[n][3] = fmaf(sB, c[3], isum[n][3]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&empty[s]));  // the stage is read
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const float2 da = *reinterpret_cast<const float2 *>(dsl + j * nt + n * 8 + 2 * t);
                    acc[n][0] += da.x * (dA * isum[n][0]);
                    acc[n][1] += da.y * (dA * isum[n][1]);
                    acc[n][2] += da.x * (dB * isum[n][2]);
                    acc[n][3] += da.y * (dB * isum[n][3]);
                }
            } else {
                const uint8_t *nibA = st + g * kRow40 + warp * 8 * 16 + 4 * t;
                const uint8_t *nibB = nibA + SG::kHalf;
                const __half *scA = reinterpret_cast<const __half *>(st + SG::kNib40) + warp * 8 * kTileRows + g;
                const __half *scB = reinterpret_cast<const __half *>(st + SG::kHalf + SG::kNib40) + warp * 8 * kTileRows + g;
                uint32_t wa[8], wb[8];
                float dA[8], dB[8];
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    wa[b] = *reinterpret_cast<const uint32_t *>(nibA + b * 16);
                    wb[b] = *reinterpret_cast<const uint32_t *>(nibB + b * 16);
                    dA[b] = __half2float(scA[b * kTileRows]);
                    dB[b] = __half2float(scB[b * kTileRows]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&empty[s]));  // the stage's bytes are in registers
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    uint32_t al02, al13, ah02, ah13, bl02, bl13, bh02, bh13;
                    q40_pairs(wa[b], al02, al13, ah02, ah13);
                    q40_pairs(wb[b], bl02, bl13, bh02, bh13);
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        uint2 y0 = make_uint2(0u, 0u), y1 = y0;
                        if (n * 8 + g < mc) {
                            y0 = *reinterpret_cast<const uint2 *>(bb + ((2 * b) * mc + n * 8) * kSlot6);
                            y1 = *reinterpret_cast<const uint2 *>(bb + ((2 * b + 1) * mc + n * 8) * kSlot6);
                        }
                        float c[4];
                        mma16816(c, al02, bl02, al13, bl13, y0.x, y0.y, true);
                        mma16816(c, ah02, bh02, ah13, bh13, y1.x, y1.y, false);
                        const float2 da = *reinterpret_cast<const float2 *>(dsl + (j * 8 + b) * nt + n * 8 + 2 * t);
                        acc[n][0] += da.x * (dA[b] * c[0]);
                        acc[n][1] += da.y * (dA[b] * c[1]);
                        acc[n][2] += da.x * (dB[b] * c[2]);
                        acc[n][3] += da.y * (dB[b] * c[3]);
                    }
                }
            }
        } else {
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        }

        if (chunk == nchunks - 1) {  // pair done: add the eight warps' partial sums
            float *rb = red + (size_t)(pair_no & 1) * (kWarps6 * NT * 4 * 32);
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    rb[((warp * NT + n) * 4 + e) * 32 + lane] = acc[n][e];
                    acc[n][e] = 0.0f;
                }
            cons_sync();
            const int tid = threadIdx.x;  // one output per thread: (n, e, lane)
            if (tid < NT * 4 * 32) {
                const int n = tid >> 7, e = (tid >> 5) & 3, l = tid & 31;
                float v = 0.0f;
#pragma unroll
                for (int w = 0; w < kWarps6; ++w) v += rb[((w * NT + n) * 4 + e) * 32 + l];
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

// Per-warp image area for mc tokens over nu units: codes [J][16][mc][32 B],
// scales [J][blocks per unit][nt] fp32 (nt = mc rounded up to 8 or 16, the
// padding tokens' scales zero), J = ceil(nu / 8); a launch's image is the
// eight warps' areas one after another.
struct Layout6 {
    int nt;
    uint32_t warp_bytes, d_off;
};
__host__ __device__ inline Layout6 layout6(int f, int64_t nu, int mc) {
    Layout6 L;
    L.nt = mc <= 8 ? 8 : 16;
    const uint64_t J = (uint64_t)(nu + kWarps6 - 1) / kWarps6;
    L.d_off = (uint32_t)(J * kSteps6 * mc * kSlot6);
    const int dpu = f == kF6K ? 1 : 8;
    L.warp_bytes = (uint32_t)align_up(L.d_off + J * dpu * L.nt * 4, 128);
    return L;
}

// Slot of element i (0..15) of a step inside the token's 32 bytes: lane i / 4,
// and inside the lane's 4 fp16 the order (i0, i2, i1, i3).
__device__ __forceinline__ int slot_elem(int i) { return (i >> 2) * 8 + ((i & 1) * 2 + ((i >> 1) & 1)) * 2; }

// Where token ml's code of element e of unit u goes, and its scale slot.
// Q6_K: e in 0..255 of the super-block; Q4_0: e in 0..255 of the unit, block
// e / 32.
template <int F>
__device__ __forceinline__ void image_pos(int e, int &step, int &i) {
    if (F == kF6K) {
        i = e & 15;
        const int tq = 2 * (e >> 6) + ((e >> 4) & 1), h = (e >> 5) & 1;
        step = 2 * tq + h;
    } else {
        const int b = e >> 5, k = e & 31;
        step = 2 * b + (k >> 4);
        i = k & 15;
    }
}

// A Q8 code (|q| <= 127) as fp16 without a conversion instruction.
__device__ __forceinline__ __half code_half(int q) {
    return __hsub(__ushort_as_half((unsigned short)biased_half_bits(q)), __ushort_as_half((unsigned short)0x6480));
}

// One warp per (token, unit): the unit's 256 codes (8 per lane, elements 8l
// .. 8l+7) and scales into the launch's image.
template <int F>
__device__ __forceinline__ void put_unit(uint8_t *img, int64_t nu, int mc, int ml, int64_t u, int lane,
                                         const int q[8], const float *d /* Q6_K: d[0]; Q4_0: d of block lane / 4 */) {
    const Layout6 L = layout6(F, nu, mc);
    uint8_t *area = img + (size_t)(u % kWarps6) * L.warp_bytes;
    const int64_t j = u / kWarps6;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        int step, i;
        image_pos<F>(8 * lane + k, step, i);
        *reinterpret_cast<__half *>(area + ((j * kSteps6 + step) * mc + ml) * kSlot6 + slot_elem(i)) =
            code_half(q[k]);
    }
    float *dsl = reinterpret_cast<float *>(area + L.d_off);
    if (F == kF6K) {
        if (lane == 0) dsl[j * L.nt + ml] = d[0];
        if (ml == 0 && lane >= mc && lane < L.nt) dsl[j * L.nt + lane] = 0.0f;  // padding tokens
    } else {
        if ((lane & 3) == 0) dsl[(j * 8 + (lane >> 2)) * L.nt + ml] = d[0];
        if (ml == 0)
            for (int x = lane; x < 8 * L.nt; x += 32)
                if (x % L.nt >= mc) dsl[j * 8 * L.nt + x] = 0.0f;
    }
}

// Q6_K's image of each launch of `per` tokens (the last one holds the
// rest) from fp32 X, one warp per (token, super-block): the Q8_K codes and
// scales of the planar quantizer bit for bit.
__global__ void __launch_bounds__(256) quantize_image6k_kernel(const float *X, uint8_t *img, int64_t M, int64_t nu,
                                                               int per) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (threadIdx.x == 0) pdl_launch_dependents();
    if (gw >= M * nu) return;
    pdl_wait();
    const int64_t m = gw / nu, u = gw % nu;
    const int64_t launch = m / per;
    const int ml = (int)(m - launch * per);
    const int mc = (int)(M - launch * per < per ? M - launch * per : per);
    uint8_t *base = img + (size_t)launch * kWarps6 * layout6(kF6K, nu, per).warp_bytes;
    const float4 *x = reinterpret_cast<const float4 *>(X + m * nu * 256 + u * 256 + 8 * lane);
    const float4 v0 = __ldg(x), v1 = __ldg(x + 1);
    const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t lo, hi;
    int bsum, q[8];
    float d;
    q8_K_warp(v, lo, hi, d, bsum);
#pragma unroll
    for (int k = 0; k < 8; ++k) q[k] = (int)(int8_t)(uint8_t)((k < 4 ? lo : hi) >> (8 * (k & 3)));
    put_unit<kF6K>(base, nu, mc, ml, u, lane, q, &d);
}

// Q4_0's image from fp32 X with one warp per (token, block of 32): one
// Q8_0 pass per warp (element = lane), so the quantizer's critical path is
// one block long.
__global__ void __launch_bounds__(256) quantize_image40_kernel(const float *X, uint8_t *img, int64_t M, int64_t nu,
                                                               int per) {
    const int lane = threadIdx.x & 31;
    const int64_t nb = nu * 8;
    const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (threadIdx.x == 0) pdl_launch_dependents();
    if (gw >= M * nb) return;
    pdl_wait();
    const int64_t m = gw / nb, blk = gw % nb, u = blk / 8;
    const int b = (int)(blk % 8);
    const int64_t launch = m / per;
    const int ml = (int)(m - launch * per);
    const int mc = (int)(M - launch * per < per ? M - launch * per : per);
    const Layout6 L = layout6(kF40, nu, mc);
    uint8_t *area = img + (size_t)launch * kWarps6 * layout6(kF40, nu, per).warp_bytes +
                    (size_t)(u % kWarps6) * L.warp_bytes;
    const int64_t j = u / kWarps6;
    int c, sum;
    __half dh;
    q8_0_warp(X[m * nu * 256 + blk * 32 + lane], c, dh, sum);
    const int step = 2 * b + (lane >> 4);
    *reinterpret_cast<__half *>(area + ((j * kSteps6 + step) * mc + ml) * kSlot6 + slot_elem(lane & 15)) =
        code_half(c);
    float *dsl = reinterpret_cast<float *>(area + L.d_off) + (j * 8 + b) * L.nt;
    if (lane == 0) dsl[ml] = __half2float(dh);
    if (ml == 0 && lane >= mc && lane < L.nt) dsl[lane] = 0.0f;  // padding tokens
}

// The same image from canonical blocks (qmm_mul_mat_q8): Q8_K [M][nu] x 292 B
// (Q6_K) or Q8_0 [M][8 nu] x 34 B (Q4_0).
template <int F>
__global__ void __launch_bounds__(256) import_image6_kernel(const uint8_t *Xq, uint8_t *img, int64_t M, int64_t nu,
                                                            int per) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (threadIdx.x == 0) pdl_launch_dependents();
    if (gw >= M * nu) return;
    pdl_wait();
    const int64_t m = gw / nu, u = gw % nu;
    const int64_t launch = m / per;
    const int ml = (int)(m - launch * per);
    const int mc = (int)(M - launch * per < per ? M - launch * per : per);
    uint8_t *base = img + (size_t)launch * kWarps6 * layout6(F, nu, per).warp_bytes;
    int q[8];
    float d;
    if (F == kF6K) {
        const uint8_t *blk = Xq + gw * B_Q8_K;
        const uint32_t *qw = reinterpret_cast<const uint32_t *>(blk + 4 + 8 * lane);
        const uint32_t w[2] = {qw[0], qw[1]};
#pragma unroll
        for (int k = 0; k < 8; ++k) q[k] = (int)(int8_t)(uint8_t)(w[k >> 2] >> (8 * (k & 3)));
        d = *reinterpret_cast<const float *>(blk);
    } else {
        // lane l: elements 8l .. 8l+7 = block l / 4, codes 8 (l % 4) ..
        const uint8_t *blk = Xq + (m * nu * 8 + u * 8 + (lane >> 2)) * B_Q8_0;
        const uint16_t *cw = reinterpret_cast<const uint16_t *>(blk + 2 + 8 * (lane & 3));
#pragma unroll
        for (int k = 0; k < 8; ++k) q[k] = (int)(int8_t)(uint8_t)(cw[k >> 1] >> (8 * (k & 1)));
        d = __half2float(*reinterpret_cast<const __half *>(blk));
    }
    put_unit<F>(base, nu, mc, ml, u, lane, q, &d);
}

struct Plan6 {
    Layout6 L;
    int stages, ctas_per_sm;
    uint32_t act_off, red_off, bar_off, smem;
};

// [ring][8 warp areas][reduction, double-buffered][barriers + abort flag]:
// two CTAs per SM (within 113 KB each) with a ring of 4, 3 or 2 stages, else
// one CTA with 4, 3 or 2.
bool make_plan6(int f, int64_t nu, int mc, Plan6 *p) {
    const Layout6 L = layout6(f, nu, mc);
    const int nt = L.nt / 8;
    const uint64_t stage = f == kF6K ? Stage6<kF6K>::kBytes : Stage6<kF40>::kBytes;
    const uint64_t red = 2ull * kWarps6 * nt * 4 * 32 * 4;
    static const int kTry[6][2] = {{4, 2}, {3, 2}, {2, 2}, {4, 1}, {3, 1}, {2, 1}};
    for (const auto &tr : kTry) {
        if (tr[1] == 2 && nt == 2) continue;  // its registers allow one CTA per SM
        const uint64_t ring = (uint64_t)tr[0] * stage;
        const uint64_t total = ring + (uint64_t)kWarps6 * L.warp_bytes + red + (2 * tr[0] + 1) * 8 + 8;
        if (total <= (tr[1] == 2 ? 113u * 1024 : 227u * 1024)) {
            p->L = L;
            p->stages = tr[0];
            p->ctas_per_sm = tr[1];
            p->act_off = (uint32_t)ring;
            p->red_off = (uint32_t)(ring + (uint64_t)kWarps6 * L.warp_bytes);
            p->bar_off = (uint32_t)(p->red_off + red);
            p->smem = (uint32_t)total;
            return true;
        }
    }
    return false;
}

int fmt6(qmm_type wt) { return wt == QMM_TYPE_Q6_K ? kF6K : kF40; }

}  // namespace

int gemv_mma6_max_tokens(qmm_type wt, int64_t K) {
    if (K % 256 != 0) return 0;
    Plan6 p;
    for (int mc = 16; mc >= 1; --mc)
        if (make_plan6(fmt6(wt), K / 256, mc, &p)) return mc;
    return 0;
}

size_t gemv_mma6_image_bytes(qmm_type wt, int64_t M, int64_t K) {
    const int per = gemv_mma6_max_tokens(wt, K);
    if (per == 0) return 0;
    const int64_t nu = K / 256, full = M / per, rest = M % per;
    size_t b = (size_t)full * kWarps6 * layout6(fmt6(wt), nu, per).warp_bytes;
    if (rest) b += (size_t)kWarps6 * layout6(fmt6(wt), nu, (int)rest).warp_bytes;
    return b;
}

cudaError_t launch_image6(qmm_type wt, bool import, const void *src, void *img, int64_t M, int64_t K,
                          cudaStream_t s) {
    const int per = gemv_mma6_max_tokens(wt, K);
    if (per == 0) return cudaErrorInvalidValue;
    const int64_t nu = K / 256;
    cudaLaunchConfig_t cfg = {};
    // one warp per (token, unit), or per (token, block) for Q4_0 from fp32
    const bool per_block = !import && wt == QMM_TYPE_Q4_0;
    cfg.gridDim = dim3((unsigned)((M * nu * (per_block ? 8 : 1) + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    uint8_t *out = static_cast<uint8_t *>(img);
    cudaError_t e;
    if (import)
        e = wt == QMM_TYPE_Q6_K
                ? cudaLaunchKernelEx(&cfg, import_image6_kernel<kF6K>, static_cast<const uint8_t *>(src), out, M, nu, per)
                : cudaLaunchKernelEx(&cfg, import_image6_kernel<kF40>, static_cast<const uint8_t *>(src), out, M, nu, per);
    else
        e = wt == QMM_TYPE_Q6_K
                ? cudaLaunchKernelEx(&cfg, quantize_image6k_kernel, static_cast<const float *>(src), out, M, nu, per)
                : cudaLaunchKernelEx(&cfg, quantize_image40_kernel, static_cast<const float *>(src), out, M, nu, per);
    count_launch();
    return e;
}

cudaError_t launch_gemv_mma6(qmm_type wt, MatSet ms, int64_t K, const void *img, int64_t M, bool pdl,
                             cudaStream_t s) {
    ms.off[0] = 0;
    for (int i = 0; i < ms.n; ++i) ms.off[i + 1] = ms.off[i] + (tiles_of(ms.N[i]) + 1) / 2;
    const int f = fmt6(wt);
    Mma6Args a;
    a.ms = ms;
    a.nu = K / 256;
    a.err = device_error_word();
    const int per = gemv_mma6_max_tokens(wt, K);
    if (per == 0) return cudaErrorInvalidValue;
    const int64_t npairs = ms.off[ms.n];
    const uint8_t *im = static_cast<const uint8_t *>(img);
    for (int64_t m0 = 0; m0 < M; m0 += per) {
        Plan6 p;
        a.m0 = m0;
        a.mc = (int)(M - m0 < per ? M - m0 : per);
        make_plan6(f, a.nu, a.mc, &p);
        a.img = im;
        im += (size_t)kWarps6 * p.L.warp_bytes;
        a.stages = p.stages;
        a.act_off = p.act_off;
        a.act_warp = p.L.warp_bytes;
        a.d_off = p.L.d_off;
        a.red_off = p.red_off;
        a.bar_off = p.bar_off;
        const bool two = p.L.nt == 16;
        const void *fn = f == kF6K ? (two ? reinterpret_cast<const void *>(gemv_mma6_kernel<kF6K, 2>)
                                          : reinterpret_cast<const void *>(gemv_mma6_kernel<kF6K, 1>))
                                   : (two ? reinterpret_cast<const void *>(gemv_mma6_kernel<kF40, 2>)
                                          : reinterpret_cast<const void *>(gemv_mma6_kernel<kF40, 1>));
        cudaError_t e = ensure_smem_attr(fn, (int)p.smem);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)balanced_grid(npairs, (int64_t)p.ctas_per_sm * sm_count()));
        cfg.blockDim = dim3(kThreads6);
        cfg.dynamicSmemBytes = p.smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
        if (f == kF6K)
            e = two ? cudaLaunchKernelEx(&cfg, gemv_mma6_kernel<kF6K, 2>, a) : cudaLaunchKernelEx(&cfg, gemv_mma6_kernel<kF6K, 1>, a);
        else
            e = two ? cudaLaunchKernelEx(&cfg, gemv_mma6_kernel<kF40, 2>, a) : cudaLaunchKernelEx(&cfg, gemv_mma6_kernel<kF40, 1>, a);
        count_launch();
        if (e != cudaSuccess) return e;
        pdl = false;
    }
    return cudaSuccess;
}

// The tensor-core decode path of every format: image size, image writers,
// GEMV.
size_t mma_image_bytes(qmm_type wt, int64_t M, int64_t K) {
    return wt == QMM_TYPE_Q4_K ? gemv_mma_image_bytes(M, K) : gemv_mma6_image_bytes(wt, M, K);
}
cudaError_t launch_mma_image(qmm_type wt, bool import, const void *src, void *img, int64_t M, int64_t K,
                             cudaStream_t s) {
    if (wt == QMM_TYPE_Q4_K)
        return import ? launch_import_mma_image(src, img, M, K, s)
                      : launch_quantize_mma_image(static_cast<const float *>(src), img, M, K, s);
    return launch_image6(wt, import, src, img, M, K, s);
}
cudaError_t launch_gemv_mma(qmm_type wt, MatSet ms, int64_t K, const void *img, int64_t M, bool pdl,
                            cudaStream_t s) {
    return wt == QMM_TYPE_Q4_K ? launch_gemv_mma_q4_K(ms, K, nullptr, img, M, pdl, s)
                               : launch_gemv_mma6(wt, ms, K, img, M, pdl, s);
}

}  // namespace qmm
