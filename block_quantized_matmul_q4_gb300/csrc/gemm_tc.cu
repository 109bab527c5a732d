// gemm_tc.cu -- prefill-path mul_mat (M > 16 tokens) for packed Q4_K weights
// on the 5th-generation tensor cores (tcgen05, TMEM accumulators).
//
// What is computed is the same factored form as the decode path (page 1,
// "正确性: 缩放系数可以提到求和号外面" and "min 项与最终归约"):
//   Y[m, n] = sum_sb d_a[m,sb] (d[n,sb] A_sb[n,m] - dmin[n,sb] B_sb[n,m])
//   A_sb[n,m] = sum_{k in sb} (s_j(k)[n] q[n,k]) y[m,k]   (integers)
//   B_sb[n,m] = sum_{t<16} m_{t/2}[n] bs_t[m]              (integers)
// GB300 has no kind::i8 tcgen05 MMA (ptxas rejects it for sm_103a), so the
// integer products run on kind::f16 with integer-valued fp16 operands: s_j q
// <= 63 * 15 = 945 and y in [-127, 127] are exact in fp16, their products
// exact in the fp32 accumulator; m_j <= 63 and bs_t in [-2032, 2032] likewise.
// Each super-block accumulates into its own TMEM buffers (double-buffered),
// and the epilogue warps apply the per-super-block scales in fp32 registers.
//
// CTA = 128 weight rows (MMA M) x 128 tokens (MMA N), 14 warps:
//   warp 0      producer: bulk copies of the raw Q4_K blocks of a super-block
//               (one per 8-row packed tile) and 2-D TMA tiles of the fp16 codes
//               (128B swizzle) and the fp16 bsums (32B swizzle);
//   warp 1      MMA issuer (one thread) and TMEM owner (512 columns);
//   warps 2..9  converters, two sets of four: one weight row per thread (its
//               TMEM lane), set 0 takes K-chunks 0 and 2 of a super-block,
//               set 1 chunks 1 and 3. Nibbles x s_j -> fp16 in registers,
//               stored straight into a TMEM operand ring with tcgen05.st (the
//               page-3 "decode in registers, feed the MMA" idea; the expanded
//               weights never touch shared memory). Set 0 also writes the
//               row's mins for the bsum MMA and its d, dmin;
//   warps 10..25 epilogue: tcgen05.ld both accumulators, y += d_a (d A -
//               dmin B) into 32 fp32 registers per thread, final store. The
//               per-super-block scales come from a small shared-memory ring:
//               d_a by TMA from the workspace, d and dmin from the converters
//               (who read those block headers anyway).
// All mbarrier waits are bounded; on a timeout the CTA drains its copies and
// MMAs, frees its TMEM and returns with the device error word set.
#include <mutex>

#include "tc.cuh"

namespace qmm {
namespace {

constexpr int kBM = 128;  // weight rows per CTA (MMA M)
constexpr int kBN = 128;  // tokens per CTA (MMA N)
constexpr int kBK = 64;   // K per operand chunk: one 128-byte swizzle row of fp16
constexpr int kChunksPerSB = QK_K / kBK;  // 4
constexpr int kAStages = 4, kBStages = 4, kMStages = 2, kRawStages = 2;
constexpr int kChunkBytes = kBN * kBK * 2;  // 16 KB activation tile
constexpr int kMinBytes = kBM * 16 * 2;     // 4 KB per min operand (K = 16)
constexpr int kRawBytes = (kBM / kTileRows) * kTileRows * B_Q4_K;  // 18432
constexpr int kOffB = 0;
constexpr int kOffM = kOffB + kBStages * kChunkBytes;
constexpr int kOffRaw = kOffM + kMStages * 2 * kMinBytes;
constexpr int kScBytes = kBN * 4 + 2 * kBM * 4;  // d_a[128], d[128], dmin[128]
constexpr int kOffSc = kOffRaw + kRawStages * kRawBytes;
constexpr int kOffBar = kOffSc + 2 * kScBytes;
constexpr int kNumBars = 2 * (kRawStages + kAStages + kBStages + kMStages + 2 + 2) + 2;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;  // + TMEM slot + alignment
constexpr int kConvWarps = 8, kEpiWarps = 16;
constexpr int kThreads = (2 + kConvWarps + kEpiWarps) * 32;
constexpr int kEpiCols = kBN / (kEpiWarps / 4);  // columns per epilogue thread
// TMEM columns: A accumulators (x2), the bsum accumulator, the A operand ring
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColAccA = 0, kColAccB = 2 * kBN, kColARing = 3 * kBN;
constexpr uint32_t kARingCols = kBK / 2;  // two fp16 per 32-bit column
static_assert(kColARing + kAStages * kARingCols <= kTmemCols, "TMEM budget");
static_assert(kBN == kBM, "square tiles");

struct GemmArgs {
    const uint8_t *Wp;  // packed Q4_K weights
    int64_t N, nsb, M;
    float *Y;  // [M][N]
    unsigned *err;
};

struct Bars {
    uint64_t *raw_full, *raw_empty, *a_full, *a_empty, *b_full, *b_empty, *m_full, *m_empty,
        *acc_full, *acc_empty, *sc_full, *sc_empty, *bacc_empty, *done;
};

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }
// (x & mask) | 0x64006400: two fp16 values 1024 + field
__device__ __forceinline__ uint32_t magic(uint32_t x, uint32_t mask) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(x), "r"(mask), "r"(0x64006400u));
    return d;
}

// fp16 values s * q from the nibbles of one 32-bit word of qs (bytes b0..b3;
// low nibbles are elements k0..k3 of a sub-block, high nibbles the same
// positions of the next sub-block). A nibble at bits 0-3 or 4-7 of a 16-bit
// half, or'ed into 0x6400 (1024.0, one unit in the last place), reads as
// 1024 + q or 1024 + 16 q; one fused fp16 FMA with (s, -1024 s) or
// (s / 16, -64 s) leaves q s exactly (an integer <= 945). Bytes b0, b2 sit at
// bits 0 and 16 of w, bytes b1, b3 at bits 0 and 16 of w >> 8, so the halves
// come out as the pairs (k0, k2), (k1, k3): the activation codes are stored
// with elements 1 and 2 of every group of 4 swapped to match, which leaves
// the dot product unchanged.
struct ScaleLH {
    __half2 ml, al, mh, ah;  // low nibbles: s_lo, -1024 s_lo; high: s_hi / 16, -64 s_hi
};
__device__ __forceinline__ ScaleLH make_scales(float s_lo, float s_hi) {
    ScaleLH c;
    c.ml = __float2half2_rn(s_lo);
    c.al = __float2half2_rn(-1024.0f * s_lo);
    c.mh = __float2half2_rn(s_hi * 0.0625f);
    c.ah = __float2half2_rn(-64.0f * s_hi);
    return c;
}
__device__ __forceinline__ void expand_word(uint32_t w, const ScaleLH &c, uint32_t &l02,
                                            uint32_t &l13, uint32_t &h02, uint32_t &h13) {
    const uint32_t v = w >> 8;
    l02 = h2_bits(__hfma2(bits_h2(magic(w, 0x000F000Fu)), c.ml, c.al));
    l13 = h2_bits(__hfma2(bits_h2(magic(v, 0x000F000Fu)), c.ml, c.al));
    h02 = h2_bits(__hfma2(bits_h2(magic(w, 0x00F000F0u)), c.mh, c.ah));
    h13 = h2_bits(__hfma2(bits_h2(magic(v, 0x00F000F0u)), c.mh, c.ah));
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_q4_K_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap tmap_y,
                     const __grid_constant__ CUtensorMap tmap_bs,
                     const __grid_constant__ CUtensorMap tmap_da) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base for the 128B-swizzled tiles
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t sbase = (raw_base + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw_base);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nsb = a.nsb;
    const int64_t n0 = (int64_t)blockIdx.x * kBM, m0 = (int64_t)blockIdx.y * kBN;
    const int64_t t0 = n0 / kTileRows;  // first packed tile
    const int64_t ntiles = tiles_of(a.N);
    const int nt = (int)(ntiles - t0 < kBM / kTileRows ? ntiles - t0 : kBM / kTileRows);

    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kOffBar);
    Bars B;
    B.raw_full = bar;
    B.raw_empty = B.raw_full + kRawStages;
    B.a_full = B.raw_empty + kRawStages;
    B.a_empty = B.a_full + kAStages;
    B.b_full = B.a_empty + kAStages;
    B.b_empty = B.b_full + kBStages;
    B.m_full = B.b_empty + kBStages;
    B.m_empty = B.m_full + kMStages;
    B.acc_full = B.m_empty + kMStages;
    B.acc_empty = B.acc_full + 2;
    B.sc_full = B.acc_empty + 2;
    B.sc_empty = B.sc_full + 2;
    B.bacc_empty = B.sc_empty + 2;
    B.done = B.bacc_empty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(B.done + 1);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kRawStages; ++i) {
            mbar_init(smem_u32(&B.raw_full[i]), 1);
            mbar_init(smem_u32(&B.raw_empty[i]), kConvWarps);
        }
        for (int i = 0; i < kAStages; ++i) {
            mbar_init(smem_u32(&B.a_full[i]), 4);
            mbar_init(smem_u32(&B.a_empty[i]), 1);
        }
        for (int i = 0; i < kBStages; ++i) {
            mbar_init(smem_u32(&B.b_full[i]), 1);
            mbar_init(smem_u32(&B.b_empty[i]), 1);
        }
        for (int i = 0; i < kMStages; ++i) {
            mbar_init(smem_u32(&B.m_full[i]), 1 + 4);
            mbar_init(smem_u32(&B.m_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&B.acc_full[i]), 1);
            mbar_init(smem_u32(&B.acc_empty[i]), kEpiWarps);
            mbar_init(smem_u32(&B.sc_full[i]), 1 + 4);
            mbar_init(smem_u32(&B.sc_empty[i]), kEpiWarps);
        }
        mbar_init(smem_u32(B.bacc_empty), kEpiWarps);
        mbar_init(smem_u32(B.done), 1);
        fence_barrier_init();
    }
    if (warp == 1) tc::tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tc::prefetch_tensormap(&tmap_y);
            tc::prefetch_tensormap(&tmap_bs);
            tc::prefetch_tensormap(&tmap_da);
            const uint64_t pol = policy_evict_last();  // weights and codes are reused by other CTAs
            pdl_wait();  // the codes come from the preceding quantizer kernel
            int64_t issued_raw = 0, issued_b = 0, issued_m = 0, issued_sc = 0;
            bool ok = true;
            for (int64_t sb = 0; sb < nsb && ok; ++sb) {
                const int rs = (int)(sb % kRawStages);
                ok = mbar_wait(smem_u32(&B.raw_empty[rs]), (uint32_t)(((sb / kRawStages) & 1) ^ 1), a.err);
                if (!ok) break;
                const uint32_t rbar = smem_u32(&B.raw_full[rs]);
                mbar_arrive_expect_tx(rbar, (uint32_t)nt * kTileRows * B_Q4_K);
                for (int i = 0; i < nt; ++i)
                    bulk_g2s(smem_u32(smem + kOffRaw + rs * kRawBytes + i * kTileRows * B_Q4_K),
                             a.Wp + ((t0 + i) * nsb + sb) * (kTileRows * B_Q4_K),
                             kTileRows * B_Q4_K, rbar, pol);
                ++issued_raw;
                for (int kc = 0; kc < kChunksPerSB && ok; ++kc) {
                    const int64_t it = sb * kChunksPerSB + kc;
                    const int bs = (int)(it % kBStages);
                    ok = mbar_wait(smem_u32(&B.b_empty[bs]), (uint32_t)(((it / kBStages) & 1) ^ 1), a.err);
                    if (!ok) break;
                    const uint32_t bbar = smem_u32(&B.b_full[bs]);
                    mbar_arrive_expect_tx(bbar, kBN * kBK * 2);
                    tc::tma_load_2d(smem_u32(smem + kOffB + bs * kChunkBytes), &tmap_y,
                                    (int32_t)(sb * QK_K + kc * kBK), (int32_t)m0, bbar, pol);
                    ++issued_b;
                }
                if (!ok) break;
                const int ms = (int)(sb % kMStages);
                ok = mbar_wait(smem_u32(&B.m_empty[ms]), (uint32_t)(((sb / kMStages) & 1) ^ 1), a.err);
                if (!ok) break;
                const uint32_t mbar = smem_u32(&B.m_full[ms]);
                mbar_arrive_expect_tx(mbar, kBN * 16 * 2);
                tc::tma_load_2d(smem_u32(smem + kOffM + ms * 2 * kMinBytes + kMinBytes), &tmap_bs,
                                (int32_t)(sb * 16), (int32_t)m0, mbar, pol);
                ++issued_m;
                // activation scales d_a[m0 .. m0+127] of this super-block
                const int sbuf = (int)(sb & 1);
                ok = mbar_wait(smem_u32(&B.sc_empty[sbuf]), (uint32_t)(((sb >> 1) & 1) ^ 1), a.err);
                if (!ok) break;
                const uint32_t sbar = smem_u32(&B.sc_full[sbuf]);
                mbar_arrive_expect_tx(sbar, kBN * 4);
                tc::tma_load_2d(smem_u32(smem + kOffSc + sbuf * kScBytes), &tmap_da, (int32_t)m0,
                                (int32_t)sb, sbar, pol);
                ++issued_sc;
            }
            // drain: no copy may still be landing when the CTA exits
            for (int64_t k = issued_raw > kRawStages ? issued_raw - kRawStages : 0; k < issued_raw; ++k)
                mbar_wait(smem_u32(&B.raw_full[k % kRawStages]), (uint32_t)((k / kRawStages) & 1), a.err);
            for (int64_t k = issued_b > kBStages ? issued_b - kBStages : 0; k < issued_b; ++k)
                mbar_wait(smem_u32(&B.b_full[k % kBStages]), (uint32_t)((k / kBStages) & 1), a.err);
            for (int64_t k = issued_m > kMStages ? issued_m - kMStages : 0; k < issued_m; ++k)
                mbar_wait(smem_u32(&B.m_full[k % kMStages]), (uint32_t)((k / kMStages) & 1), a.err);
            for (int64_t k = issued_sc > 2 ? issued_sc - 2 : 0; k < issued_sc; ++k)
                mbar_wait(smem_u32(&B.sc_full[k & 1]), (uint32_t)((k >> 1) & 1), a.err);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_f16_f32(kBM, kBN);
            int64_t issued = 0;
            bool ok = true;
            for (int64_t sb = 0; sb < nsb && ok; ++sb) {
                const int buf = (int)(sb & 1);
                ok = mbar_wait(smem_u32(&B.acc_empty[buf]), (uint32_t)(((sb >> 1) & 1) ^ 1), a.err);
                if (!ok) break;
                tc::fence_after_sync();
                const uint32_t dA = tmem + kColAccA + (uint32_t)(buf * kBN);
                const uint32_t dB = tmem + kColAccB;
                for (int kc = 0; kc < kChunksPerSB && ok; ++kc) {
                    const int64_t it = sb * kChunksPerSB + kc;
                    const int as = (int)(it % kAStages), bs = (int)(it % kBStages);
                    ok = mbar_wait(smem_u32(&B.a_full[as]), (uint32_t)((it / kAStages) & 1), a.err) &&
                         mbar_wait(smem_u32(&B.b_full[bs]), (uint32_t)((it / kBStages) & 1), a.err);
                    if (!ok) break;
                    tc::fence_after_sync();
                    const uint32_t acol = tmem + kColARing + (uint32_t)as * kARingCols;
                    const uint32_t bbase = smem_u32(smem + kOffB + bs * kChunkBytes);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        tc::mma_f16_ta(dA, acol + 8 * kk, tc::smem_desc(bbase + 32 * kk, 1024, 2),
                                       idesc, (kc | kk) != 0);
                    }
                    tc::commit(smem_u32(&B.a_empty[as]));
                    tc::commit(smem_u32(&B.b_empty[bs]));
                    ++issued;
                }
                if (!ok) break;
                const int ms = (int)(sb % kMStages);
                ok = mbar_wait(smem_u32(&B.m_full[ms]), (uint32_t)((sb / kMStages) & 1), a.err) &&
                     mbar_wait(smem_u32(B.bacc_empty), (uint32_t)((sb & 1) ^ 1), a.err);
                if (!ok) break;
                tc::fence_after_sync();
                const uint32_t mbase = smem_u32(smem + kOffM + ms * 2 * kMinBytes);
                tc::mma_f16(dB, tc::smem_desc(mbase, 256, 6), tc::smem_desc(mbase + kMinBytes, 256, 6),
                            idesc, false);
                tc::commit(smem_u32(&B.m_empty[ms]));
                tc::commit(smem_u32(&B.acc_full[buf]));
            }
            // no MMA may still be running when TMEM is freed
            tc::commit(smem_u32(B.done));
            mbar_wait(smem_u32(B.done), 0, a.err);
        }
    } else if (warp < 2 + kConvWarps) {
        // ------------------------------------------------------------ converters
        // warp w may only touch TMEM lanes 32 (w % 4) .. +31: those are its rows
        const int ct = 32 * (warp & 3) + lane;  // weight row within the tile
        const uint32_t lane_addr = (uint32_t)(32 * (warp & 3)) << 16;
        const int set = (warp - 2) >> 2;  // K-chunks set, set + 2
        const int ti = ct / kTileRows, r = ct % kTileRows;
        const bool valid = ti < nt;
        bool ok = true;
        for (int64_t sb = 0; sb < nsb && ok; ++sb) {
            const int rs = (int)(sb % kRawStages);
            ok = mbar_wait(smem_u32(&B.raw_full[rs]), (uint32_t)((sb / kRawStages) & 1), a.err);
            if (!ok) break;
            const uint8_t *blk = smem + kOffRaw + rs * kRawBytes + (ti * kTileRows + r) * B_Q4_K;
            const uint4 hdr = valid ? *reinterpret_cast<const uint4 *>(blk) : make_uint4(0, 0, 0, 0);
            int s[8], m[8];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t f = k4_field(hdr.y, hdr.z, hdr.w, c);
                s[2 * c] = f & 63;
                m[2 * c] = (f >> 6) & 63;
                s[2 * c + 1] = (f >> 12) & 63;
                m[2 * c + 1] = (f >> 18) & 63;
            }
            // this row's d and dmin for the epilogue (set 0)
            const int sbuf = (int)(sb & 1);
            if (set == 0) {
                ok = mbar_wait(smem_u32(&B.sc_empty[sbuf]), (uint32_t)(((sb >> 1) & 1) ^ 1), a.err);
                if (!ok) break;
                {
                    float *scd = reinterpret_cast<float *>(smem + kOffSc + sbuf * kScBytes + kBN * 4);
                    scd[ct] = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xFFFFu)));
                    scd[kBM + ct] = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&B.sc_full[sbuf]));
                // mins operand, K = 16: column t holds m_{t/2}; 32B-swizzled rows
                const int ms = (int)(sb % kMStages);
                ok = mbar_wait(smem_u32(&B.m_empty[ms]), (uint32_t)(((sb / kMStages) & 1) ^ 1), a.err);
                if (!ok) break;
                {
                    uint32_t hm[8];
    #pragma unroll
                    for (int j = 0; j < 8; ++j) hm[j] = h2_bits(__float2half2_rn((float)m[j]));
                    uint8_t *row = smem + kOffM + ms * 2 * kMinBytes + ct * 32;
                    const int sw = (ct >> 2) & 1;
                    *reinterpret_cast<uint4 *>(row + 16 * (0 ^ sw)) = make_uint4(hm[0], hm[1], hm[2], hm[3]);
                    *reinterpret_cast<uint4 *>(row + 16 * (1 ^ sw)) = make_uint4(hm[4], hm[5], hm[6], hm[7]);
                }
                tc::fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&B.m_full[ms]));
            }
            for (int kc = set; kc < kChunksPerSB && ok; kc += 2) {
                const int64_t it = sb * kChunksPerSB + kc;
                const int as = (int)(it % kAStages);
                ok = mbar_wait(smem_u32(&B.a_empty[as]), (uint32_t)(((it / kAStages) & 1) ^ 1), a.err);
                if (!ok) break;
                // 32 nibble bytes: low nibbles are k = 64kc + 0..31 (sub-block
                // 2kc), high nibbles k = 64kc + 32..63 (sub-block 2kc + 1)
                uint4 q0 = make_uint4(0, 0, 0, 0), q1 = q0;
                if (valid) {
                    q0 = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * kc);
                    q1 = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * kc);
                }
                tc::fence_after_sync();
                const ScaleLH sc = make_scales((float)s[2 * kc], (float)s[2 * kc + 1]);
                const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                // columns 0..15: k = 0..31 (low nibbles), 16..31: k = 32..63 (high),
                // column pairs in the (0, 2), (1, 3) order of every group of 4
                uint32_t lo[16], hi[16];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    expand_word(w[j], sc, lo[2 * j], lo[2 * j + 1], hi[2 * j], hi[2 * j + 1]);
                const uint32_t acol = tmem + lane_addr + kColARing + (uint32_t)as * kARingCols;
                tc::tmem_st16(acol, lo);
                tc::tmem_st16(acol + 16, hi);
                tc::tmem_st_wait();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&B.a_full[as]));
            }
            __syncwarp();
            if (lane == 0 && ok) mbar_arrive(smem_u32(&B.raw_empty[rs]));
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 2 - kConvWarps;
        const int quarter = warp & 3;  // TMEM lanes 32 * (warp % 4) ..
        const int part = ew >> 2;      // columns kEpiCols * part ..
        const int nl = quarter * 32 + lane;
        const int64_t n = n0 + nl;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        float run[kEpiCols];
#pragma unroll
        for (int j = 0; j < kEpiCols; ++j) run[j] = 0.0f;
        bool ok = true;
        for (int64_t sb = 0; sb < nsb && ok; ++sb) {
            const int buf = (int)(sb & 1);
            ok = mbar_wait(smem_u32(&B.sc_full[buf]), (uint32_t)((sb >> 1) & 1), a.err) &&
                 mbar_wait(smem_u32(&B.acc_full[buf]), (uint32_t)((sb >> 1) & 1), a.err);
            if (!ok) break;
            tc::fence_after_sync();
            const float *sc = reinterpret_cast<const float *>(smem + kOffSc + buf * kScBytes);
            const float dw = sc[kBN + nl], dmw = sc[kBN + kBM + nl];
#pragma unroll
            for (int c16 = 0; c16 < kEpiCols / 16; ++c16) {
                const uint32_t col = (uint32_t)(part * kEpiCols + c16 * 16);
                float A[16], Bv[16];
                tc::tmem_ld16(tmem + lane_addr + kColAccA + (uint32_t)(buf * kBN) + col, A);
                tc::tmem_ld16(tmem + lane_addr + kColAccB + col, Bv);
                tc::tmem_ld_wait();
#pragma unroll
                for (int j4 = 0; j4 < 4; ++j4) {
                    const float4 da = *reinterpret_cast<const float4 *>(sc + col + 4 * j4);
                    const float dv[4] = {da.x, da.y, da.z, da.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = 4 * j4 + e;
                        run[c16 * 16 + j] += dv[e] * (dw * A[j] - dmw * Bv[j]);
                    }
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(&B.acc_empty[buf]));
                mbar_arrive(smem_u32(B.bacc_empty));
                mbar_arrive(smem_u32(&B.sc_empty[buf]));
            }
        }
        if (n < a.N) {
#pragma unroll
            for (int j = 0; j < kEpiCols; ++j) {
                const int64_t m = m0 + part * kEpiCols + j;
                if (m < a.M) a.Y[m * a.N + n] = run[j];
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ prefill quantizer
// Activations fp32 -> Q8_K codes as exact fp16 [M][K] (the MMA operand),
// 16-code sums as fp16 [M][nsb * 16] and scales as fp32 [nsb][M]. Same
// arithmetic as the Q8_K quantizer (shared q8_K_warp).
__global__ void __launch_bounds__(256) quantize_q8K_prefill_kernel(const float *__restrict__ X,
                                                                   __half *__restrict__ y16,
                                                                   __half *__restrict__ bs16,
                                                                   float *__restrict__ daT,
                                                                   int64_t M, int64_t nsb) {
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t nblocks = M * nsb;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < nblocks;
         b += nwarps) {
        const int64_t m = b / nsb, sb = b % nsb;
        const float4 *src = reinterpret_cast<const float4 *>(X + b * QK_K + 8 * lane);
        const float4 v0 = src[0], v1 = src[1];
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint32_t lo, hi;
        float d;
        int bsum;
        q8_K_warp(v, lo, hi, d, bsum);
        // the MMA operand order: elements 1 and 2 of every group of 4 swapped
        uint4 o;
        uint32_t *po = &o.x;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t wsrc = i < 2 ? lo : hi;
            const int sh = 8 * (i & 1);  // pair (e0, e2), then (e1, e3)
            const int8_t c0 = (int8_t)(wsrc >> sh);
            const int8_t c1 = (int8_t)(wsrc >> (16 + sh));
            po[i] = h2_bits(__halves2half2(__int2half_rn(c0), __int2half_rn(c1)));
        }
        *reinterpret_cast<uint4 *>(y16 + b * QK_K + 8 * lane) = o;
        if ((lane & 1) == 0) bs16[b * 16 + (lane >> 1)] = __int2half_rn(bsum);
        if (lane == 0) daT[sb * ((M + 3) & ~(int64_t)3) + m] = d;
    }
}

}  // namespace

namespace tc {
bool make_tmap_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype,
                  uint32_t elem_bytes, uint64_t rows, uint64_t cols, uint32_t box_rows,
                  uint32_t box_cols, CUtensorMapSwizzle swizzle) {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    std::call_once(once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!encode) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * elem_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return encode(map, dtype, 2, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}
}  // namespace tc

// Prefill workspace: fp16 codes [M][K], fp16 bsums [M][nsb*16], fp32 scales
// [nsb][M]; 256-byte aligned sections.
size_t prefill_bytes(int64_t M, int64_t K, PrefillWs *p, uint8_t *base) {
    const int64_t nsb = K / QK_K;
    size_t off = 0;
    const size_t o_y = off;
    off = align_up(off + (size_t)M * K * 2, 256);
    const size_t o_bs = off;
    off = align_up(off + (size_t)M * nsb * 16 * 2, 256);
    const size_t o_d = off;
    off = align_up(off + (size_t)((M + 3) & ~(int64_t)3) * nsb * 4, 256);
    if (p) {
        p->y16 = reinterpret_cast<__half *>(base + o_y);
        p->bs16 = reinterpret_cast<__half *>(base + o_bs);
        p->daT = reinterpret_cast<float *>(base + o_d);
    }
    return off;
}

cudaError_t launch_quantize_prefill(const float *X, PrefillWs p, int64_t M, int64_t K,
                                    cudaStream_t s) {
    const int64_t nblocks = M * (K / QK_K);
    int64_t grid = (nblocks + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 16;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    quantize_q8K_prefill_kernel<<<(int)grid, 256, 0, s>>>(X, p.y16, p.bs16, p.daT, M, K / QK_K);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_gemm_q4_K(const void *Wp, int64_t N, int64_t K, PrefillWs p, int64_t M,
                             float *Y, cudaStream_t s) {
    const int64_t nsb = K / QK_K;
    CUtensorMap tmap_y, tmap_bs, tmap_da;
    const uint64_t Mpad = (uint64_t)((M + 3) & ~(int64_t)3);
    if (!tc::make_tmap_2d(&tmap_y, p.y16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (uint64_t)M,
                          (uint64_t)K, kBN, kBK, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !tc::make_tmap_2d(&tmap_bs, p.bs16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (uint64_t)M,
                          (uint64_t)nsb * 16, kBN, 16, CU_TENSOR_MAP_SWIZZLE_32B) ||
        !tc::make_tmap_2d(&tmap_da, p.daT, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)nsb, Mpad,
                          1, kBN, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(gemm_q4_K_kernel), kSmemBytes);
    if (e != cudaSuccess) return e;
    GemmArgs a;
    a.Wp = static_cast<const uint8_t *>(Wp);
    a.N = N;
    a.nsb = nsb;
    a.M = M;
    a.Y = Y;
    a.err = device_error_word();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((N + kBM - 1) / kBM), (unsigned)((M + kBN - 1) / kBN));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gemm_q4_K_kernel, a, tmap_y, tmap_bs, tmap_da);
    count_launch();
    return e;
}

}  // namespace qmm
