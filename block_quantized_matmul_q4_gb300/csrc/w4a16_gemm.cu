// w4a16_gemm.cu -- W4A16 for M > 16 tokens on the 5th-generation tensor
// cores (page 3, "BitBLAS 完全拆解": decode the low-bit weight on the way
// into the tensor-core operand, "边解码边计算").
//   C[m, n] = sum_k A[m, k] * w[n, k],  w = fp16(s[n, g] * (q[n, k] - z[n, g]))
// The weight is rounded once to fp16 (relative error <= 2^-11; q - z and s
// are exact), multiplied with the fp16 activations on kind::f16 with fp32
// accumulation over all of K, and the result rounded to fp16.
//
// CTA = 128 weight rows (MMA M) x 128 tokens (MMA N), 15 warps:
//   warp 0      producer: per 256 elements of K one 3-D TMA copy of the 8
//               packed 16-row tiles (2 steps each, 16 KB) and one activation
//               stage of four 2-D TMA tiles of A (128B swizzle, 64 KB);
//   warp 1      MMA issuer (one thread) and TMEM owner;
//   warp 2      MMA waiter: the issuer's barrier waits, handed over per pair
//               of K chunks through a named barrier (a shared-memory access
//               by the issuing thread would drain the tensor pipe);
//   warps 3..10 converters, two sets of four: one weight row per thread
//               (its TMEM lane); nibbles -> q - z -> x s in fp16 registers,
//               stored into a TMEM operand ring with tcgen05.st;
//   warps 11..14 epilogue: one tcgen05.ld pass over the accumulator at the
//               end, fp16 stores.
// All mbarrier waits are bounded; on a timeout the CTA drains its copies and
// MMAs, frees its TMEM and returns with the device error word set.
#include "tc.cuh"

namespace qmm {
namespace {

constexpr int kBM = 128, kBN = 128, kBK = 64;  // rows, tokens, K per chunk
constexpr int kSB = 256;                       // K per pipeline round
constexpr int kChunks = kSB / kBK;             // 4
constexpr int kGroups = 2;                     // A handed over in pairs of chunks
constexpr int kStepK = 128;                    // packed step: 16 rows x 16 words per tile
constexpr int kTileRows16 = 16;
constexpr int kWStages = 3, kActStages = 2;
constexpr int kWBytes = (kBM / kTileRows16) * (kSB / kStepK) * 1024;  // 16 KB
constexpr int kChunkBytes = kBN * kBK * 2;                           // 16 KB
constexpr int kActBytes = kChunks * kChunkBytes;                     // 64 KB
constexpr int kConvWarps = 8, kEpiWarps = 4;
constexpr int kThreads = (3 + kConvWarps + kEpiWarps) * 32;
constexpr int kOffAct = 0;
constexpr int kOffW = kOffAct + kActStages * kActBytes;
constexpr int kOffBar = kOffW + kWStages * kWBytes;
constexpr int kNumBars = 2 * (kWStages + kActStages + kGroups) + 2;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColAcc = 0, kColARing = kBN;
constexpr uint32_t kARingCols = kBK / 2;
static_assert(kColARing + kChunks * kARingCols <= kTmemCols, "TMEM budget");

struct Args {
    const __half *S;   // [N][ng]
    const uint8_t *Z;  // [N][ng]
    __half *C;         // [M][N]
    int64_t M, N, K;
    int ng, spg;  // groups per row, 128-element steps per group
    unsigned *err;
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
__device__ __forceinline__ void handoff_sync() { asm volatile("bar.sync 1, 64;" ::: "memory"); }

// fp16 s (q - z) for the 8 codes of one packed word, as pairs (k0, k1),
// (k2, k3), (k4, k5), (k6, k7): q - z exactly (1024 + q minus 1024 + z, or
// the x16 form through one FMA), then one rounding for the product with s.
__device__ __forceinline__ void weight_word(uint32_t w, uint32_t zz, uint32_t zh, uint32_t ss,
                                           uint32_t (&p)[4]) {
    constexpr uint32_t kSixteenth = 0x2C002C00u;  // fp16 1/16 twice
    const uint32_t v = w >> 8;
    p[0] = hmul2_u(hsub2_u(lop_or(w, 0x000F000Fu), zz), ss);
    p[1] = hmul2_u(hfma2_u(lop_or(w, 0x00F000F0u), kSixteenth, zh), ss);
    p[2] = hmul2_u(hsub2_u(lop_or(v, 0x000F000Fu), zz), ss);
    p[3] = hmul2_u(hfma2_u(lop_or(v, 0x00F000F0u), kSixteenth, zh), ss);
}

__global__ void __launch_bounds__(kThreads, 1)
    w4a16_gemm_kernel(const Args a, const __grid_constant__ CUtensorMap tmap_w,
                      const __grid_constant__ CUtensorMap tmap_a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t sbase = (raw_base + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw_base);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n0 = (int64_t)blockIdx.x * kBM, m0 = (int64_t)blockIdx.y * kBN;
    const int64_t nsteps = a.K / kStepK;
    const int64_t nsb = (a.K + kSB - 1) / kSB;

    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *w_full = bar, *w_empty = w_full + kWStages;
    uint64_t *act_full = w_empty + kWStages, *act_empty = act_full + kActStages;
    uint64_t *a_full = act_empty + kActStages, *a_empty = a_full + kGroups;
    uint64_t *acc_full = a_empty + kGroups, *done = acc_full + 1;
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
        for (int i = 0; i < kGroups; ++i) {
            mbar_init(smem_u32(&a_full[i]), kConvWarps);  // both sets, one chunk each
            mbar_init(smem_u32(&a_empty[i]), 1);
        }
        mbar_init(smem_u32(acc_full), 1);
        mbar_init(smem_u32(done), 1);
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
            tc::prefetch_tensormap(&tmap_w);
            tc::prefetch_tensormap(&tmap_a);
            const uint64_t pol = policy_evict_last();  // weights and A are reused by other CTAs
            pdl_wait();  // A may come from the preceding kernel
            int64_t issued_w = 0, issued_a = 0;
            bool ok = true;
            for (int64_t sb = 0; sb < nsb && ok; ++sb) {
                const int ws = (int)(sb % kWStages);
                ok = mbar_wait(smem_u32(&w_empty[ws]), (uint32_t)(((sb / kWStages) & 1) ^ 1), a.err);
                if (!ok) break;
                // 8 tiles x 2 steps; tiles past the last and steps past K read as zeros
                const uint32_t wbar = smem_u32(&w_full[ws]);
                mbar_arrive_expect_tx(wbar, kWBytes);
                tc::tma_load_3d(smem_u32(smem + kOffW + ws * kWBytes), &tmap_w, 0, (int32_t)(2 * sb),
                                (int32_t)(n0 / kTileRows16), wbar, pol);
                ++issued_w;
                const int st = (int)(sb % kActStages);
                ok = mbar_wait(smem_u32(&act_empty[st]), (uint32_t)(((sb / kActStages) & 1) ^ 1), a.err);
                if (!ok) break;
                const uint32_t abar = smem_u32(&act_full[st]);
                mbar_arrive_expect_tx(abar, kActBytes);
                for (int c = 0; c < kChunks; ++c)
                    tc::tma_load_2d(smem_u32(smem + kOffAct + st * kActBytes + c * kChunkBytes), &tmap_a,
                                    (int32_t)(sb * kSB + c * kBK), (int32_t)m0, abar, pol);
                ++issued_a;
            }
            for (int64_t k = issued_w > kWStages ? issued_w - kWStages : 0; k < issued_w; ++k)
                mbar_wait(smem_u32(&w_full[k % kWStages]), (uint32_t)((k / kWStages) & 1), a.err);
            for (int64_t k = issued_a > kActStages ? issued_a - kActStages : 0; k < issued_a; ++k)
                mbar_wait(smem_u32(&act_full[k % kActStages]), (uint32_t)((k / kActStages) & 1), a.err);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Meets the waiter at the named barrier the same number of times
        // whatever happens; after a timeout the MMAs run on stale operands and
        // the error word reports it.
        constexpr uint32_t idesc = tc::idesc_f16_f32(kBM, kBN);
        const uint64_t bdesc0 = tc::smem_desc(smem_u32(smem + kOffAct), 1024, 2);
        for (int64_t sb = 0; sb < nsb; ++sb) {
            const int st = (int)(sb % kActStages);
#pragma unroll 1
            for (int g = 0; g < kGroups; ++g) {
                handoff_sync();
                if (lane == 0) {
                    tc::fence_after_sync();
#pragma unroll
                    for (int h = 0; h < kChunks / kGroups; ++h) {
                        const int c = g * (kChunks / kGroups) + h;
                        const uint32_t acol = tmem + kColARing + (uint32_t)c * kARingCols;
                        // K step of 16 fp16 = 32 bytes = 2 in the descriptor's address field
                        const uint64_t bdesc = bdesc0 + (uint64_t)((st * kActBytes + c * kChunkBytes) >> 4);
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            tc::mma_f16_ta(tmem + kColAcc, acol + 8 * kk, bdesc + 2 * kk, idesc,
                                           (sb | c | kk) != 0);
                    }
                    tc::commit(smem_u32(&a_empty[g]));
                    if (g == kGroups - 1) tc::commit(smem_u32(&act_empty[st]));
                }
                __syncwarp();
            }
        }
        if (lane == 0) {
            tc::commit(smem_u32(acc_full));
            tc::commit(smem_u32(done));
            mbar_wait(smem_u32(done), 0, a.err);  // no MMA may run when TMEM is freed
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------------ MMA waiter
        bool ok = true;
        for (int64_t sb = 0; sb < nsb; ++sb) {
            const int st = (int)(sb % kActStages);
            const uint32_t par = (uint32_t)(sb & 1);
            if (lane == 0 && ok)
                ok = mbar_wait(smem_u32(&act_full[st]), (uint32_t)((sb / kActStages) & 1), a.err);
#pragma unroll 1
            for (int g = 0; g < kGroups; ++g) {
                if (lane == 0 && ok) ok = mbar_wait(smem_u32(&a_full[g]), par, a.err);
                __syncwarp();
                handoff_sync();
            }
        }
    } else if (warp < 3 + kConvWarps) {
        // ------------------------------------------------------------ converters
        const int ct = 32 * (warp & 3) + lane;  // weight row within the CTA = TMEM lane
        const uint32_t lane_addr = (uint32_t)(32 * (warp & 3)) << 16;
        const int set = (warp - 3) >> 2;  // chunk `set` of each group
        const int64_t n = n0 + ct;
        const int64_t nc = n < a.N ? n : a.N - 1;  // rows past N: zero codes, clamped scales
        const __half *s_row = a.S + nc * a.ng;
        const uint8_t *z_row = a.Z + nc * a.ng;
        bool ok = true;
        for (int64_t sb = 0; sb < nsb && ok; ++sb) {
            const int ws = (int)(sb % kWStages);
            const uint32_t par = (uint32_t)(sb & 1);
            ok = mbar_wait(smem_u32(&w_full[ws]), (uint32_t)((sb / kWStages) & 1), a.err);
            if (!ok) break;
            const uint8_t *wst = smem + kOffW + ws * kWBytes;
#pragma unroll 1
            for (int g = 0; g < kGroups && ok; ++g) {
                const int c = g * (kChunks / kGroups) + set;  // chunk of this sb
                const int sl = c >> 1;                        // step within the stage
                int64_t step = 2 * sb + sl;
                if (step >= nsteps) step = nsteps - 1;  // past K: activations are zero there
                const int grp = a.spg == 1 ? (int)step : (int)step / a.spg;
                const uint32_t zv = z_row[grp];
                const uint32_t sv = (uint32_t)__half_as_ushort(s_row[grp]);
                const uint32_t zz = 0x64006400u + zv * 0x00010001u;  // fp16 1024 + z twice
                const uint32_t zh = 0xD400D400u + zv * 0x00100010u;  // fp16 -(64 + z) twice
                const uint32_t ss = sv | (sv << 16);
                ok = mbar_wait(smem_u32(&a_empty[g]), par ^ 1, a.err);
                if (!ok) break;
                // row ct's 16 words of step sl: tile ct / 16, row ct % 16; this
                // chunk is half (c & 1) of them
                const uint8_t *src = wst + ((ct >> 4) * (kSB / kStepK) + sl) * 1024 + (ct & 15) * 64 +
                                     (c & 1) * 32;
                const uint4 w0 = *reinterpret_cast<const uint4 *>(src);
                const uint4 w1 = *reinterpret_cast<const uint4 *>(src + 16);
                const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                tc::fence_after_sync();
                // columns 0..31: elements 64c + 2i, 64c + 2i + 1 in column i
                uint32_t lo[16], hi[16];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t p[4];
                    weight_word(wv[i], zz, zh, ss, p);
                    lo[4 * i] = p[0], lo[4 * i + 1] = p[1], lo[4 * i + 2] = p[2], lo[4 * i + 3] = p[3];
                    weight_word(wv[i + 4], zz, zh, ss, p);
                    hi[4 * i] = p[0], hi[4 * i + 1] = p[1], hi[4 * i + 2] = p[2], hi[4 * i + 3] = p[3];
                }
                const uint32_t acol = tmem + lane_addr + kColARing + (uint32_t)c * kARingCols;
                tc::tmem_st16(acol, lo);
                tc::tmem_st16(acol + 16, hi);
                tc::tmem_st_wait();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&a_full[g]));
            }
            __syncwarp();
            if (lane == 0 && ok) mbar_arrive(smem_u32(&w_empty[ws]));
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;  // TMEM lanes 32 * (warp % 4) ..
        const int64_t n = n0 + quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const bool ok = mbar_wait(smem_u32(acc_full), 0, a.err);
        tc::fence_after_sync();
        if (ok) {
#pragma unroll 1
            for (int c16 = 0; c16 < kBN / 16; ++c16) {
                float v[16];
                tc::tmem_ld16(tmem + lane_addr + kColAcc + (uint32_t)(c16 * 16), v);
                tc::tmem_ld_wait();
                if (n < a.N) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int64_t m = m0 + c16 * 16 + i;
                        if (m < a.M) a.C[m * a.N + n] = __float2half_rn(v[i]);
                    }
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

}  // namespace

cudaError_t launch_w4a16_gemm(const void *W, const __half *S, const uint8_t *Z, int64_t G,
                              const __half *A, __half *C, int64_t M, int64_t N, int64_t K,
                              cudaStream_t s) {
    Args a;
    a.S = S;
    a.Z = Z;
    a.C = C;
    a.M = M;
    a.N = N;
    a.K = K;
    a.ng = (int)(K / G);
    a.spg = (int)(G / kStepK);
    a.err = device_error_word();
    const int64_t nsteps = K / kStepK, ntiles16 = (N + kTileRows16 - 1) / kTileRows16;
    CUtensorMap tmap_w, tmap_a;
    // packed weights as [16-row tile][step][1 KB], in 4-byte units
    const uint64_t wdims[3] = {256, (uint64_t)nsteps, (uint64_t)ntiles16};
    const uint64_t wstrides[2] = {1024, (uint64_t)nsteps * 1024};
    const uint32_t wbox[3] = {256, kSB / kStepK, kBM / kTileRows16};
    if (!tc::make_tmap_3d(&tmap_w, W, CU_TENSOR_MAP_DATA_TYPE_UINT32, wdims, wstrides, wbox) ||
        !tc::make_tmap_2d(&tmap_a, A, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (uint64_t)M, (uint64_t)K,
                          kBN, kBK, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(w4a16_gemm_kernel), kSmemBytes);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((N + kBM - 1) / kBM), (unsigned)((M + kBN - 1) / kBN));
    w4a16_gemm_kernel<<<grid, kThreads, kSmemBytes, s>>>(a, tmap_w, tmap_a);
    count_launch();
    return cudaGetLastError();
}

}  // namespace qmm
