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
// CTA = 128 weight rows (MMA M) x 128 tokens (MMA N), 27 warps:
//   warp 0      producer: per super-block one 3-D TMA copy of the raw Q4_K
//               blocks (16 packed 8-row tiles) and one activation stage: four
//               2-D TMA tiles of fp16 codes (128B swizzle) plus the fp16 bsums
//               (32B swizzle), all on one barrier;
//   warp 1      MMA issuer (one thread) and TMEM owner (512 columns);
//   warp 2      MMA waiter: all the issuer's barrier waits, handed over per
//               group of MMAs through a named barrier;
//   warps 3..10 converters, two sets of four: one weight row per thread (its
//               TMEM lane), set 0 takes K-chunks 0 and 2 of a super-block,
//               set 1 chunks 1 and 3. Nibbles x s_j -> fp16 in registers,
//               stored straight into a TMEM operand ring with tcgen05.st (the
//               page-3 "decode in registers, feed the MMA" idea; the expanded
//               weights never touch shared memory). Set 0 also writes the
//               row's mins, the A operand of the bsum MMA;
//   warps 11..26 epilogue: tcgen05.ld both accumulators, y += d_a (d A -
//               dmin B) in packed fp32 pairs, 32 columns per thread, final
//               store. d, dmin (block header) and d_a (workspace) are read
//               from global memory one super-block ahead.
// Every wait costs a shared-memory round trip, so the pipeline is built to
// need few of them per super-block: one barrier per activation stage, one
// per pair of A chunks. All mbarrier waits are bounded; on a timeout the
// CTA drains its copies and MMAs, frees its TMEM and returns with the
// device error word set.
#include <mutex>

#include "tc.cuh"

namespace qmm {
namespace {

constexpr int kBM = 128;  // weight rows per CTA (MMA M)
constexpr int kBN = 128;  // tokens per CTA (MMA N)
constexpr int kBK = 64;   // K per operand chunk: one 128-byte swizzle row of fp16
constexpr int kChunksPerSB = QK_K / kBK;  // 4
constexpr int kGroups = 2;                // A handed over in pairs of chunks
constexpr int kActStages = 2, kRawStages = 4, kMinStages = 2;
constexpr int kChunkBytes = kBN * kBK * 2;  // 16 KB activation tile
constexpr int kBsBytes = kBN * 16 * 2;      // 4 KB bsum tile (K = 16)
constexpr int kActBytes = kChunksPerSB * kChunkBytes + kBsBytes;  // one super-block
constexpr int kMinBytes = kBM * 16 * 2;     // 4 KB mins operand (K = 16)
constexpr int kRawBytes = (kBM / kTileRows) * kTileRows * B_Q4_K;  // 18432
constexpr int kConvWarps = 8, kEpiWarps = 16;
constexpr int kThreads = (3 + kConvWarps + kEpiWarps) * 32;
constexpr int kEpiCols = kBN / (kEpiWarps / 4);  // columns per epilogue thread
constexpr int kOffAct = 0;
constexpr int kOffMin = kOffAct + kActStages * kActBytes;
constexpr int kOffRaw = kOffMin + kMinStages * kMinBytes;
constexpr int kOffDa = kOffRaw + kRawStages * kRawBytes;  // per epilogue warp: its 32 d_a
constexpr int kOffBar = kOffDa + kEpiWarps * kEpiCols * 4;
constexpr int kNumBars = 2 * (kRawStages + kActStages + kGroups + 2) + 2;  // + bacc_empty, done
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;  // + TMEM slot + alignment
static_assert(kActBytes % 1024 == 0 && kOffMin % 1024 == 0, "128B-swizzle tiles need 1 KB alignment");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
// TMEM columns: A accumulators (x2), the bsum accumulator, the A operand ring
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColAccA = 0, kColAccB = 2 * kBN, kColARing = 3 * kBN;
constexpr uint32_t kARingCols = kBK / 2;  // two fp16 per 32-bit column
static_assert(kColARing + kChunksPerSB * kARingCols <= kTmemCols, "TMEM budget");
static_assert(kBN == kBM, "square tiles");

struct GemmArgs {
    const uint8_t *Wp;  // packed Q4_K weights
    const float *daT;   // activation scales [nsb][Mpad]
    int64_t N, nsb, M;
    float *Y;  // [M][N]
    unsigned *err;
    // stream-K: tile t = (row block t / mblocks, token block t % mblocks);
    // unit u = t * nsb + super-block; CTA c takes units [c U / G, (c+1) U / G)
    int64_t mblocks, units;
    float *part;  // split tiles: [CTA][slot 0: first tile, 1: last tile][128 cols][128 rows]
};

struct Bars {
    uint64_t *raw_full, *raw_empty, *act_full, *act_empty, *a_full, *a_empty, *acc_full,
        *acc_empty, *bacc_empty, *done;
};

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }
// Packed fp32 pairs (sm_100 family f32x2 arithmetic): half the FP
// instructions of the per-super-block epilogue.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint32_t ldg_nc_u32(const void *p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ float ldg_nc_f32(const float *p) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}
// Named barrier 1: the MMA waiter and issuer warps (64 threads).
__device__ __forceinline__ void handoff_sync() { asm volatile("bar.sync 1, 64;" ::: "memory"); }
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
    gemm_q4_K_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap tmap_w,
                     const __grid_constant__ CUtensorMap tmap_y,
                     const __grid_constant__ CUtensorMap tmap_bs) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base for the 128B-swizzled tiles
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t sbase = (raw_base + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw_base);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nsb = a.nsb;
    const int64_t ntiles = tiles_of(a.N);
    // this CTA's units (stream-K): a contiguous range of (tile, super-block)
    const int64_t u0 = (int64_t)blockIdx.x * a.units / gridDim.x;
    const int64_t u1 = ((int64_t)blockIdx.x + 1) * a.units / gridDim.x;
    const int64_t nunits = u1 - u0;

    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kOffBar);
    Bars B;
    B.raw_full = bar;
    B.raw_empty = B.raw_full + kRawStages;
    B.act_full = B.raw_empty + kRawStages;
    B.act_empty = B.act_full + kActStages;
    B.a_full = B.act_empty + kActStages;
    B.a_empty = B.a_full + kGroups;
    B.acc_full = B.a_empty + kGroups;
    B.acc_empty = B.acc_full + 2;
    B.bacc_empty = B.acc_empty + 2;
    B.done = B.bacc_empty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(B.done + 1);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kRawStages; ++i) {
            mbar_init(smem_u32(&B.raw_full[i]), 1);
            mbar_init(smem_u32(&B.raw_empty[i]), kConvWarps);
        }
        for (int i = 0; i < kActStages; ++i) {
            mbar_init(smem_u32(&B.act_full[i]), 1);
            mbar_init(smem_u32(&B.act_empty[i]), 1);
        }
        for (int i = 0; i < kGroups; ++i) {
            mbar_init(smem_u32(&B.a_full[i]), kConvWarps);  // both sets, one chunk each
            mbar_init(smem_u32(&B.a_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&B.acc_full[i]), 1);
            mbar_init(smem_u32(&B.acc_empty[i]), kEpiWarps);
        }
        mbar_init(smem_u32(B.bacc_empty), kEpiWarps);
        mbar_init(smem_u32(B.done), 1);
        fence_barrier_init();
    }
    __syncwarp();  // warps meet converged at every CTA barrier below
    if (warp == 1) tc::tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tc::prefetch_tensormap(&tmap_w);
            tc::prefetch_tensormap(&tmap_y);
            tc::prefetch_tensormap(&tmap_bs);
            const uint64_t pol = policy_evict_last();  // weights and codes are reused by other CTAs
            pdl_wait();  // the codes come from the preceding quantizer kernel
            int64_t issued_raw = 0, issued_act = 0;
            bool ok = true;
            for (int64_t i = 0; i < nunits && ok; ++i) {
                const int64_t u = u0 + i, tile = u / nsb, sb = u - tile * nsb;
                const int64_t t0 = (tile / a.mblocks) * (kBM / kTileRows);  // first packed tile
                const int64_t m0 = (tile % a.mblocks) * kBN;
                const int rs = (int)(i % kRawStages);
                ok = mbar_wait(smem_u32(&B.raw_empty[rs]), (uint32_t)(((i / kRawStages) & 1) ^ 1), a.err);
                if (!ok) break;
                // tiles past the last one read as zeros (and are never stored)
                const uint32_t rbar = smem_u32(&B.raw_full[rs]);
                mbar_arrive_expect_tx(rbar, kRawBytes);
                tc::tma_load_3d(smem_u32(smem + kOffRaw + rs * kRawBytes), &tmap_w, 0, (int32_t)sb,
                                (int32_t)t0, rbar, pol);
                ++issued_raw;
                const int st = (int)(i % kActStages);
                ok = mbar_wait(smem_u32(&B.act_empty[st]), (uint32_t)(((i / kActStages) & 1) ^ 1), a.err);
                if (!ok) break;
                const uint32_t abar = smem_u32(&B.act_full[st]);
                uint8_t *stage = smem + kOffAct + st * kActBytes;
                mbar_arrive_expect_tx(abar, kActBytes);
                for (int kc = 0; kc < kChunksPerSB; ++kc)
                    tc::tma_load_2d(smem_u32(stage + kc * kChunkBytes), &tmap_y,
                                    (int32_t)(sb * QK_K + kc * kBK), (int32_t)m0, abar, pol);
                tc::tma_load_2d(smem_u32(stage + kChunksPerSB * kChunkBytes), &tmap_bs,
                                (int32_t)(sb * 16), (int32_t)m0, abar, pol);
                ++issued_act;
            }
            // drain: no copy may still be landing when the CTA exits
            for (int64_t k = issued_raw > kRawStages ? issued_raw - kRawStages : 0; k < issued_raw; ++k)
                mbar_wait(smem_u32(&B.raw_full[k % kRawStages]), (uint32_t)((k / kRawStages) & 1), a.err);
            for (int64_t k = issued_act > kActStages ? issued_act - kActStages : 0; k < issued_act; ++k)
                mbar_wait(smem_u32(&B.act_full[k % kActStages]), (uint32_t)((k / kActStages) & 1), a.err);
        }
        __syncwarp();  // lanes 1..31 wait here for the producer lane
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Never touches an mbarrier on the way: a shared-memory access by the
        // issuing thread waits for its MMAs in flight, which would drain the
        // tensor pipe at every chunk. The waiter warp does the waiting and
        // hands over each group through a named barrier. Both warps pass it
        // the same number of times whatever happens, so neither can hang; after
        // a timeout the MMAs run on stale operands and the error word reports it.
        constexpr uint32_t idesc = tc::idesc_f16_f32(kBM, kBN);
        const uint64_t bdesc0 = tc::smem_desc(smem_u32(smem + kOffAct), 1024, 2);
        for (int64_t i = 0; i < nunits; ++i) {
            const int buf = (int)(i & 1), st = (int)(i % kActStages);
            const uint32_t dA = tmem + kColAccA + (uint32_t)(buf * kBN);
#pragma unroll 1
            for (int g = 0; g < kGroups; ++g) {
                handoff_sync();
                if (lane == 0) {
                    tc::fence_after_sync();
#pragma unroll
                    for (int h = 0; h < kChunksPerSB / kGroups; ++h) {
                        const int kc = g * (kChunksPerSB / kGroups) + h;
                        const uint32_t acol = tmem + kColARing + (uint32_t)kc * kARingCols;
                        // K step of 16 fp16 = 32 bytes = 2 in the descriptor's address field
                        const uint64_t bdesc = bdesc0 + (uint64_t)((st * kActBytes + kc * kChunkBytes) >> 4);
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            tc::mma_f16_ta(dA, acol + 8 * kk, bdesc + 2 * kk, idesc, (kc | kk) != 0);
                    }
                    tc::commit(smem_u32(&B.a_empty[g]));
                }
                __syncwarp();
            }
            handoff_sync();
            if (lane == 0) {
                tc::fence_after_sync();
                const uint32_t mins = smem_u32(smem + kOffMin + (int)(i % kMinStages) * kMinBytes);
                const uint32_t bsum = smem_u32(smem + kOffAct + st * kActBytes + kChunksPerSB * kChunkBytes);
                tc::mma_f16(tmem + kColAccB, tc::smem_desc(mins, 256, 6), tc::smem_desc(bsum, 256, 6),
                            idesc, false);
                tc::commit(smem_u32(&B.act_empty[st]));
                tc::commit(smem_u32(&B.acc_full[buf]));
            }
            __syncwarp();
        }
        if (lane == 0) {
            // no MMA may still be running when TMEM is freed
            tc::commit(smem_u32(B.done));
            mbar_wait(smem_u32(B.done), 0, a.err);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------------ MMA waiter
        // Waits for the operands (and free accumulators) of each group, then
        // meets the issuer at the named barrier. After a timeout it stops
        // waiting but keeps meeting the issuer.
        bool ok = true;
        for (int64_t i = 0; i < nunits; ++i) {
            const int buf = (int)(i & 1), st = (int)(i % kActStages);
            const uint32_t par = (uint32_t)(i & 1);
            if (lane == 0 && ok)
                ok = mbar_wait(smem_u32(&B.acc_empty[buf]), (uint32_t)(((i >> 1) & 1) ^ 1), a.err) &&
                     mbar_wait(smem_u32(&B.act_full[st]), (uint32_t)((i / kActStages) & 1), a.err);
#pragma unroll 1
            for (int g = 0; g < kGroups; ++g) {
                if (lane == 0 && ok) ok = mbar_wait(smem_u32(&B.a_full[g]), par, a.err);
                __syncwarp();
                handoff_sync();
            }
            if (lane == 0 && ok) ok = mbar_wait(smem_u32(B.bacc_empty), par ^ 1, a.err);
            __syncwarp();
            handoff_sync();
        }
    } else if (warp < 3 + kConvWarps) {
        // ------------------------------------------------------------ converters
        // warp w may only touch TMEM lanes 32 (w % 4) .. +31: those are its rows
        const int ct = 32 * (warp & 3) + lane;  // weight row within the tile
        const uint32_t lane_addr = (uint32_t)(32 * (warp & 3)) << 16;
        const int set = (warp - 3) >> 2;  // chunk `set` of each group
        const int ti = ct / kTileRows, r = ct % kTileRows;
        bool ok = true;
        int i = 0;  // units done: the pipeline position
        // the CTA's units as pieces of tiles; per piece, its super-blocks
        for (int64_t u = u0; u < u1 && ok;) {
            const int64_t tile = u / nsb;
            const int sb_begin = (int)(u - tile * nsb);
            const int sb_end = (int)(nsb < sb_begin + (u1 - u) ? nsb : sb_begin + (u1 - u));
            const bool valid = (tile / a.mblocks) * (kBM / kTileRows) + ti < ntiles;
            u += sb_end - sb_begin;
        for (int sb = sb_begin; sb < sb_end && ok; ++sb, ++i) {
            const int rs = (int)(i % kRawStages);
            const uint32_t par = (uint32_t)(i & 1);
            ok = mbar_wait_warp(smem_u32(&B.raw_full[rs]), (uint32_t)((i / kRawStages) & 1), a.err);
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
#pragma unroll 1
            for (int g = 0; g < kGroups && ok; ++g) {
                const int kc = g * (kChunksPerSB / kGroups) + set;
                // the slots of group g are free once the MMAs of group g of the
                // previous super-block are done -- and with them every MMA
                // issued before, including the bsum MMA two super-blocks back
                // that read the mins slot reused below
                ok = mbar_wait_warp(smem_u32(&B.a_empty[g]), par ^ 1, a.err);
                if (!ok) break;
                if (g == 0 && set == 0) {
                    // mins operand, K = 16: column t holds m_{t/2}; 32B-swizzled rows
                    uint32_t hm[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) hm[j] = h2_bits(__float2half2_rn((float)m[j]));
                    uint8_t *row = smem + kOffMin + (int)(i % kMinStages) * kMinBytes + ct * 32;
                    const int sw = (ct >> 2) & 1;
                    *reinterpret_cast<uint4 *>(row + 16 * (0 ^ sw)) = make_uint4(hm[0], hm[1], hm[2], hm[3]);
                    *reinterpret_cast<uint4 *>(row + 16 * (1 ^ sw)) = make_uint4(hm[4], hm[5], hm[6], hm[7]);
                    tc::fence_proxy_async();
                }
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
                const uint32_t acol = tmem + lane_addr + kColARing + (uint32_t)kc * kARingCols;
                tc::tmem_st16(acol, lo);
                tc::tmem_st16(acol + 16, hi);
                tc::tmem_st_wait();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&B.a_full[g]));
            }
            __syncwarp();
            if (lane == 0 && ok) mbar_arrive(smem_u32(&B.raw_empty[rs]));
        }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 3 - kConvWarps;
        const int quarter = warp & 3;  // TMEM lanes 32 * (warp % 4) ..
        const int cpart = ew >> 2;     // columns kEpiCols * cpart ..
        const int nl = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        float *da_stage = reinterpret_cast<float *>(smem + kOffDa) + ew * kEpiCols;
        const int64_t Mpad = (a.M + 3) & ~(int64_t)3;
        pdl_wait();  // d_a comes from the preceding quantizer kernel
        bool ok = true;
        int i = 0;  // units done: the pipeline position
        // the CTA's units as pieces of tiles: a whole tile goes to Y, a part
        // of one to this CTA's partial slot for the fixup kernel
        for (int64_t u = u0; u < u1;) {
            const int64_t tile = u / nsb;
            const int sb_begin = (int)(u - tile * nsb);
            const int sb_end = (int)(nsb < sb_begin + (u1 - u) ? nsb : sb_begin + (u1 - u));
            u += sb_end - sb_begin;
            const int64_t n = (tile / a.mblocks) * kBM + nl;
            const int64_t mb0 = (tile % a.mblocks) * kBN + cpart * kEpiCols;
            // this row's block headers (d, dmin as two fp16) and this warp's 32
            // activation scales, read one super-block ahead
            const bool row_ok = n < a.N;
            const uint8_t *hdr_ptr = a.Wp + ((n / kTileRows) * nsb * kTileRows + (n % kTileRows)) * B_Q4_K;
            const int64_t mcol = mb0 + lane;
            uint32_t hdr_next = row_ok ? ldg_nc_u32(hdr_ptr + sb_begin * (kTileRows * B_Q4_K)) : 0u;
            float da_next = mcol < Mpad ? ldg_nc_f32(a.daT + sb_begin * Mpad + mcol) : 0.0f;
            uint64_t run[kEpiCols / 2];  // column pairs
#pragma unroll
            for (int j = 0; j < kEpiCols / 2; ++j) run[j] = 0;  // (+0.0f, +0.0f)
            for (int sb = sb_begin; sb < sb_end && ok; ++sb, ++i) {
                const int buf = i & 1;
                const uint32_t hdr = hdr_next;
                const float da = da_next;
                if (sb + 1 < sb_end) {
                    if (row_ok) hdr_next = ldg_nc_u32(hdr_ptr + (sb + 1) * (kTileRows * B_Q4_K));
                    if (mcol < Mpad) da_next = ldg_nc_f32(a.daT + (sb + 1) * Mpad + mcol);
                }
                da_stage[lane] = da;
                __syncwarp();
                ok = mbar_wait_warp(smem_u32(&B.acc_full[buf]), (uint32_t)((i >> 1) & 1), a.err);
                if (!ok) break;
                tc::fence_after_sync();
                const float dw = __half2float(__ushort_as_half((unsigned short)(hdr & 0xFFFFu)));
                const float dmw = __half2float(__ushort_as_half((unsigned short)(hdr >> 16)));
                const uint64_t dw2 = pk2(dw, dw), ndmw2 = pk2(-dmw, -dmw);
#pragma unroll
                for (int c8 = 0; c8 < kEpiCols / 8; ++c8) {
                    const uint32_t col = (uint32_t)(cpart * kEpiCols + c8 * 8);
                    float A[8], Bv[8];
                    tc::tmem_ld8(tmem + lane_addr + kColAccA + (uint32_t)(buf * kBN) + col, A);
                    tc::tmem_ld8(tmem + lane_addr + kColAccB + col, Bv);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j4 = 0; j4 < 2; ++j4) {
                        const float4 dav = *reinterpret_cast<const float4 *>(da_stage + c8 * 8 + 4 * j4);
                        const uint64_t dv[2] = {pk2(dav.x, dav.y), pk2(dav.z, dav.w)};
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int j = 4 * j4 + 2 * e;
                            // run += d_a (d A - dmin B), two columns at a time
                            const uint64_t t = fma2(pk2(A[j], A[j + 1]), dw2,
                                                    mul2(pk2(Bv[j], Bv[j + 1]), ndmw2));
                            run[(c8 * 8 + j) / 2] = fma2(dv[e], t, run[(c8 * 8 + j) / 2]);
                        }
                    }
                }
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(smem_u32(&B.acc_empty[buf]));
                    mbar_arrive(smem_u32(B.bacc_empty));
                }
            }
            if (sb_begin == 0 && sb_end == nsb) {
                if (row_ok && ok) {
#pragma unroll
                    for (int j = 0; j < kEpiCols; j += 2) {
                        float lo, hi;
                        upk2(run[j / 2], lo, hi);
                        const int64_t m = mb0 + j;
                        if (m < a.M) a.Y[m * a.N + n] = lo;
                        if (m + 1 < a.M) a.Y[(m + 1) * a.N + n] = hi;
                    }
                }
            } else if (ok) {
                // a part of a split tile: to this CTA's slot (column-major:
                // column j of this row at j * kBM) for the fixup kernel
                float *mine = a.part + sk_slot(blockIdx.x, tile, a.units, gridDim.x, nsb) +
                              (int64_t)(cpart * kEpiCols) * kBM + nl;
#pragma unroll
                for (int j = 0; j < kEpiCols; j += 2) {
                    float lo, hi;
                    upk2(run[j / 2], lo, hi);
                    mine[j * kBM] = lo;
                    mine[(j + 1) * kBM] = hi;
                }
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

// The same layout from canonical Q8_K blocks [M][nsb] x 292 B (codes, scale
// and stored 16-code sums), for qmm_mul_mat_q8.
__global__ void __launch_bounds__(256) import_q8K_prefill_kernel(const uint8_t *__restrict__ Xq,
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
        const uint8_t *blk = Xq + b * B_Q8_K;
        const uint32_t *qw = reinterpret_cast<const uint32_t *>(blk + 4 + 8 * lane);
        const uint32_t lo = qw[0], hi = qw[1];
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
        if (lane < 16)
            bs16[b * 16 + lane] = __int2half_rn(reinterpret_cast<const int16_t *>(blk + 260)[lane]);
        if (lane == 0) daT[sb * ((M + 3) & ~(int64_t)3) + m] = *reinterpret_cast<const float *>(blk);
    }
}

}  // namespace

namespace tc {
namespace {
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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
    return encode;
}
}  // namespace

bool make_tmap_3d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype,
                  const uint64_t dims[3], const uint64_t strides[2], const uint32_t box[3],
                  CUtensorMapSwizzle swizzle) {
    const auto encode = encoder();
    if (!encode) return false;
    const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
    const cuuint64_t st[2] = {strides[0], strides[1]};
    const cuuint32_t bx[3] = {box[0], box[1], box[2]};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode(map, dtype, 3, const_cast<void *>(base), d, st, bx, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

bool make_tmap_4d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype,
                  const uint64_t dims[4], const uint64_t strides[3], const uint32_t box[4]) {
    const auto encode = encoder();
    if (!encode) return false;
    const cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
    const cuuint64_t st[3] = {strides[0], strides[1], strides[2]};
    const cuuint32_t bx[4] = {box[0], box[1], box[2], box[3]};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return encode(map, dtype, 4, const_cast<void *>(base), d, st, bx, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

bool make_tmap_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype,
                  uint32_t elem_bytes, uint64_t rows, uint64_t cols, uint32_t box_rows,
                  uint32_t box_cols, CUtensorMapSwizzle swizzle) {
    const auto encode = encoder();
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

cudaError_t launch_import_prefill(const void *Xq, PrefillWs p, int64_t M, int64_t K,
                                  cudaStream_t s) {
    const int64_t nblocks = M * (K / QK_K);
    int64_t grid = (nblocks + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 16;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    import_q8K_prefill_kernel<<<(int)grid, 256, 0, s>>>(static_cast<const uint8_t *>(Xq), p.y16,
                                                        p.bs16, p.daT, M, K / QK_K);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_gemm_q4_K(const void *Wp, int64_t N, int64_t K, PrefillWs p, float *part, int64_t M,
                             float *Y, cudaStream_t s) {
    const int64_t nsb = K / QK_K;
    GemmArgs a;
    a.Wp = static_cast<const uint8_t *>(Wp);
    a.daT = p.daT;
    a.N = N;
    a.nsb = nsb;
    a.M = M;
    a.Y = Y;
    a.err = device_error_word();
    CUtensorMap tmap_w, tmap_y, tmap_bs;
    // packed weights as [tile][super-block][8 rows x 144 bytes], in 8-byte units
    const uint64_t wdims[3] = {kTileRows * B_Q4_K / 8, (uint64_t)nsb, (uint64_t)tiles_of(N)};
    const uint64_t wstrides[2] = {kTileRows * B_Q4_K, (uint64_t)nsb * kTileRows * B_Q4_K};
    const uint32_t wbox[3] = {kTileRows * B_Q4_K / 8, 1, kBM / kTileRows};
    if (!tc::make_tmap_3d(&tmap_w, Wp, CU_TENSOR_MAP_DATA_TYPE_UINT64, wdims, wstrides, wbox) ||
        !tc::make_tmap_2d(&tmap_y, p.y16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (uint64_t)M,
                          (uint64_t)K, kBN, kBK, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !tc::make_tmap_2d(&tmap_bs, p.bs16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (uint64_t)M,
                          (uint64_t)nsb * 16, kBN, 16, CU_TENSOR_MAP_SWIZZLE_32B))
        return cudaErrorInvalidValue;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(gemm_q4_K_kernel), kSmemBytes);
    if (e != cudaSuccess) return e;
    // one CTA per tile, or with more tiles than SMs stream-K over (tile,
    // super-block) units with one persistent CTA per SM
    const int64_t nblocks = (N + kBM - 1) / kBM;
    a.mblocks = (M + kBN - 1) / kBN;
    const int64_t tiles = nblocks * a.mblocks;
    a.units = tiles * nsb;
    a.part = part;
    const int64_t G = stream_k_grid(tiles);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gemm_q4_K_kernel, a, tmap_w, tmap_y, tmap_bs);
    count_launch();
    if (e != cudaSuccess || G == tiles) return e;
    return launch_stream_k_fixup(part, Y, false, N, M, a.mblocks, nsb, a.units, G, s);
}

}  // namespace qmm
