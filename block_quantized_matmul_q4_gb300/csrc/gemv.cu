// gemv.cu -- decode-path mul_mat (M = 1..16 tokens per launch) over packed
// Q4_0 / Q4_K weights and planar Q8_0 / Q8_K activations.
//
// Page 1 sets what is computed ("正确性: 缩放系数可以提到求和号外面", the
// generic vec_dot in "通用实现" and the min term in "min 项与最终归约"):
//   Q4_K: per super-block, S_j = sum q y (unsigned nibbles x int8),
//         isum = sum_j s_j S_j, msum = sum_j m_j (bs_2j + bs_2j+1),
//         y += d_a (d isum - dmin msum)
//   Q4_0: per block, isum = sum (q - 8) y = sum q y - 8 sum y,
//         y += d_w d_a isum
// and why decode is bound by the weight bytes ("先把账算清楚": every token
// reads every weight once). The GB300 design:
//   * one producer warp streams each CTA's contiguous tiles of packed weights
//     through a 4-stage shared-memory ring with 1-D bulk async copies
//     (cp.async.bulk + mbarrier transaction counts, L2 evict-first), so the
//     HBM stream is a few large copies per CTA, never gated by the ALU;
//   * eight consumer warps unpack nibbles and the 6-bit scales in registers
//     and take the integer dot products with dp4a against the activations
//     (read through the read-only path; they are small and L1/L2-resident);
//   * programmatic dependent launch: the producer starts streaming weights
//     while the activation quantizer still runs; consumers wait for it with
//     griddepcontrol.wait before touching the activations.
// Every mbarrier wait is bounded; a timeout sets the device error word and
// the CTA leaves after draining its own copies in flight.
#include "qmm_internal.cuh"

namespace qmm {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 4;
constexpr int kStageBytes = 18432;
constexpr int kQ4KChunk = 16;   // super-blocks per stage: 16 * 8 rows * 144 B = 18432
constexpr int kQ40Chunk = 128;  // blocks per stage: 128 * 8 rows * 18 B = 18432
constexpr int kBarBytes = 2 * kStages * 8;
constexpr int kMaxMT = 16;
constexpr int kSmemBytes = kStages * kStageBytes + kBarBytes;
static_assert(kQ4KChunk * kTileRows * B_Q4_K == kStageBytes, "stage size");
static_assert(kQ40Chunk * kTileRows * B_Q4_0 == kStageBytes, "stage size");

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ void my_tiles(int64_t ntiles, int64_t &tb, int64_t &te) {
    tb = (int64_t)blockIdx.x * ntiles / gridDim.x;
    te = ((int64_t)blockIdx.x + 1) * ntiles / gridDim.x;
}

__device__ __forceinline__ void init_barriers(uint64_t *full, uint64_t *empty) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), kConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();
}

// Producer: for items 0 .. n_items-1, wait for the stage to be free, then
// issue its copies (copy(item, dst, bar, policy) posts expect_tx + copies).
template <class Copy>
__device__ __forceinline__ void producer_loop(int64_t n_items, uint8_t *ring, uint64_t *full,
                                              uint64_t *empty, unsigned *err, Copy copy) {
    const uint64_t pol = policy_evict_first();
    int64_t it = 0;
    for (; it < n_items; ++it) {
        const int s = (int)(it % kStages);
        const uint32_t ph = (uint32_t)((it / kStages) & 1);
        if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1u, err)) break;
        copy(it, smem_u32(ring + s * kStageBytes), smem_u32(&full[s]), pol);
    }
    // never leave while an issued copy may still be landing in shared memory
    for (int64_t k = it > kStages ? it - kStages : 0; k < it; ++k)
        mbar_wait(smem_u32(&full[k % kStages]), (uint32_t)((k / kStages) & 1), err);
}

__device__ __forceinline__ void consumer_release(uint64_t *empty, int s, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Scales and mins of sub-blocks j0 = 2 c and j1 = 2 c + 1 from the 12 packed
// bytes (page 1, "6-bit 参数是怎么塞进 12 字节的"): j < 4 keeps them in the low
// 6 bits of bytes j and j + 4; j >= 4 splits them into the nibbles of byte
// j + 4 and the top 2 bits of bytes j - 4 (scale) and j (min).
__device__ __forceinline__ void scale_min_pair(const uint4 &hdr, int c, int &s0, int &m0,
                                               int &s1, int &m1) {
    const int sh = 8 * ((2 * c) & 3);
    const uint32_t y = hdr.y >> sh, z = hdr.z >> sh, w = hdr.w >> sh;
    const int ls0 = y & 63, lm0 = z & 63, ls1 = (y >> 8) & 63, lm1 = (z >> 8) & 63;
    const int hs0 = (w & 15) | (((y >> 6) & 3) << 4);
    const int hm0 = ((w >> 4) & 15) | (((z >> 6) & 3) << 4);
    const int hs1 = ((w >> 8) & 15) | (((y >> 14) & 3) << 4);
    const int hm1 = ((w >> 12) & 15) | (((z >> 14) & 3) << 4);
    const bool hi = c >= 2;
    s0 = hi ? hs0 : ls0;
    m0 = hi ? hm0 : lm0;
    s1 = hi ? hs1 : ls1;
    m1 = hi ? hm1 : lm1;
}

// ------------------------------------------------------------------ Q4_K
// Stage = one tile (8 rows) x up to 16 super-blocks. Warp w owns row w of the
// tile; lane (g, t) = (lane / 8, lane % 8) owns super-blocks g, g+4, ... of
// the stage and, within each, qs bytes 16t .. 16t+15: chunk c = t / 2 half
// h = t % 2, i.e. 16 elements of sub-block 2c (low nibbles) and 16 of 2c+1
// (high nibbles).
template <int MT>
__global__ void __launch_bounds__(kThreads, 2)
    gemv_q4_K_kernel(const uint8_t *__restrict__ Wp, int64_t N, int64_t nsb, Planar x, int64_t M,
                     int64_t m0, float *__restrict__ Y, unsigned *err) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
    uint64_t *empty = full + kStages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int64_t tb, te;
    my_tiles(tiles_of(N), tb, te);
    const int64_t nchunks = (nsb + kQ4KChunk - 1) / kQ4KChunk;
    const int64_t n_items = (te - tb) * nchunks;
    init_barriers(full, empty);

    if (warp == kConsumerWarps) {
        if (lane == 0) {
            producer_loop(n_items, smem, full, empty, err,
                          [&](int64_t it, uint32_t dst, uint32_t bar, uint64_t pol) {
                              const int64_t tile = tb + it / nchunks;
                              const int64_t sb0 = (it % nchunks) * kQ4KChunk;
                              const int cnt = (int)min64(kQ4KChunk, nsb - sb0);
                              const uint32_t bytes = (uint32_t)cnt * kTileRows * B_Q4_K;
                              mbar_arrive_expect_tx(bar, bytes);
                              bulk_g2s(dst, Wp + (tile * nsb + sb0) * (kTileRows * B_Q4_K), bytes,
                                       bar, pol);
                          });
        }
        return;
    }

    pdl_wait();  // the activations come from the preceding quantizer kernel
    const int g = lane >> 3, t = lane & 7, c = t >> 1, h = t & 1;
    const int mcount = (int)min64(MT, M - m0);
    const int64_t K = nsb * QK_K;
    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.0f;

    for (int64_t it = 0; it < n_items; ++it) {
        const int s = (int)(it % kStages);
        if (!mbar_wait(smem_u32(&full[s]), (uint32_t)((it / kStages) & 1), err)) break;
        const int64_t tile = tb + it / nchunks;
        const int64_t chunk = it % nchunks;
        const int64_t sb0 = chunk * kQ4KChunk;
        const int cnt = (int)min64(kQ4KChunk, nsb - sb0);
        const uint32_t base = smem_u32(smem + s * kStageBytes);
        for (int sl = g; sl < cnt; sl += 4) {
            const uint32_t blk = base + (uint32_t)(sl * kTileRows + warp) * B_Q4_K;
            const uint4 hdr = lds128(blk);           // d, dmin, scales[12]
            const uint4 q = lds128(blk + 16 + 16 * t);
            int sc0, mn0, sc1, mn1;
            scale_min_pair(hdr, c, sc0, mn0, sc1, mn1);
            const float dw = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xFFFFu)));
            const float dmw = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
            const int l0 = q.x & 0x0F0F0F0F, l1 = q.y & 0x0F0F0F0F;
            const int l2 = q.z & 0x0F0F0F0F, l3 = q.w & 0x0F0F0F0F;
            const int h0 = (q.x >> 4) & 0x0F0F0F0F, h1 = (q.y >> 4) & 0x0F0F0F0F;
            const int h2 = (q.z >> 4) & 0x0F0F0F0F, h3 = (q.w >> 4) & 0x0F0F0F0F;
            const int64_t sbg = sb0 + sl;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m < mcount) {
                    const int64_t row = m0 + m;
                    const int8_t *yp = x.qs + row * K + sbg * QK_K + 64 * c + 16 * h;
                    const uint4 y0 = ldg_nc128(yp);       // sub-block 2c
                    const uint4 y1 = ldg_nc128(yp + 32);  // sub-block 2c + 1
                    int S0 = __dp4a(l0, (int)y0.x, 0);
                    S0 = __dp4a(l1, (int)y0.y, S0);
                    S0 = __dp4a(l2, (int)y0.z, S0);
                    S0 = __dp4a(l3, (int)y0.w, S0);
                    int S1 = __dp4a(h0, (int)y1.x, 0);
                    S1 = __dp4a(h1, (int)y1.y, S1);
                    S1 = __dp4a(h2, (int)y1.z, S1);
                    S1 = __dp4a(h3, (int)y1.w, S1);
                    // this lane's 16 codes of sub-block j are bsums[2j + h]
                    const int16_t *bs = x.sums + (row * nsb + sbg) * 16 + 4 * c + h;
                    const int isum = sc0 * S0 + sc1 * S1;
                    const int msum = mn0 * (int)__ldg(bs) + mn1 * (int)__ldg(bs + 2);
                    const float da = __ldg(x.d + row * nsb + sbg);
                    acc[m] += da * (dw * (float)isum - dmw * (float)msum);
                }
            }
        }
        consumer_release(empty, s, lane);
        if (chunk == nchunks - 1) {
            const int64_t n = tile * kTileRows + warp;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float v = warp_sum(acc[m]);
                if (lane == 0 && m < mcount && n < N) Y[(m0 + m) * N + n] = v;
                acc[m] = 0.0f;
            }
        }
    }
}

// ------------------------------------------------------------------ Q4_0
// Stage = one tile (8 rows) x up to 128 blocks. Shared layout: nibble rows
// [8][128][16 B] at offset 0 (one bulk copy per row segment) and the fp16
// scales [cnt][8] at offset kDOff (one copy). Warp w owns row w; lane l takes
// blocks l, l + 32, ... so each 8-lane phase of a 128-bit load reads 128
// contiguous bytes.
template <int MT>
__global__ void __launch_bounds__(kThreads, 2)
    gemv_q4_0_kernel(const uint8_t *__restrict__ Wp, int64_t N, int64_t nb, Planar x, int64_t M,
                     int64_t m0, float *__restrict__ Y, unsigned *err) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
    uint64_t *empty = full + kStages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int64_t tb, te;
    my_tiles(tiles_of(N), tb, te);
    const int64_t nchunks = (nb + kQ40Chunk - 1) / kQ40Chunk;
    const int64_t n_items = (te - tb) * nchunks;
    const int64_t tile_bytes = nb * kTileRows * B_Q4_0;
    constexpr uint32_t kRowBytes = kQ40Chunk * 16;
    constexpr uint32_t kDOff = kTileRows * kRowBytes;
    init_barriers(full, empty);

    if (warp == kConsumerWarps) {
        if (lane == 0) {
            producer_loop(n_items, smem, full, empty, err,
                          [&](int64_t it, uint32_t dst, uint32_t bar, uint64_t pol) {
                              const int64_t tile = tb + it / nchunks;
                              const int64_t b0 = (it % nchunks) * kQ40Chunk;
                              const uint32_t cnt = (uint32_t)min64(kQ40Chunk, nb - b0);
                              const uint8_t *tbase = Wp + tile * tile_bytes;
                              mbar_arrive_expect_tx(bar, cnt * kTileRows * B_Q4_0);
                              for (int r = 0; r < kTileRows; ++r)
                                  bulk_g2s(dst + r * kRowBytes, tbase + (r * nb + b0) * 16, cnt * 16,
                                           bar, pol);
                              bulk_g2s(dst + kDOff, tbase + nb * kTileRows * 16 + b0 * kTileRows * 2,
                                       cnt * kTileRows * 2, bar, pol);
                          });
        }
        return;
    }

    pdl_wait();
    const int mcount = (int)min64(MT, M - m0);
    const int64_t K = nb * QK4_0;
    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.0f;

    for (int64_t it = 0; it < n_items; ++it) {
        const int s = (int)(it % kStages);
        if (!mbar_wait(smem_u32(&full[s]), (uint32_t)((it / kStages) & 1), err)) break;
        const int64_t tile = tb + it / nchunks;
        const int64_t chunk = it % nchunks;
        const int64_t b0 = chunk * kQ40Chunk;
        const int cnt = (int)min64(kQ40Chunk, nb - b0);
        const uint32_t base = smem_u32(smem + s * kStageBytes);
        for (int bl = lane; bl < cnt; bl += 32) {
            const uint4 q = lds128(base + warp * kRowBytes + (uint32_t)bl * 16);
            unsigned short dbits;
            asm volatile("ld.shared.u16 %0, [%1];"
                         : "=h"(dbits)
                         : "r"(base + kDOff + (uint32_t)(bl * kTileRows + warp) * 2));
            const float dw = __half2float(__ushort_as_half(dbits));
            const int l0 = q.x & 0x0F0F0F0F, l1 = q.y & 0x0F0F0F0F;
            const int l2 = q.z & 0x0F0F0F0F, l3 = q.w & 0x0F0F0F0F;
            const int h0 = (q.x >> 4) & 0x0F0F0F0F, h1 = (q.y >> 4) & 0x0F0F0F0F;
            const int h2 = (q.z >> 4) & 0x0F0F0F0F, h3 = (q.w >> 4) & 0x0F0F0F0F;
            const int64_t bg = b0 + bl;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m < mcount) {
                    const int64_t row = m0 + m;
                    const int8_t *yp = x.qs + row * K + bg * QK4_0;
                    const uint4 y0 = ldg_nc128(yp);       // elements 0..15
                    const uint4 y1 = ldg_nc128(yp + 16);  // elements 16..31
                    int sq = __dp4a(l0, (int)y0.x, 0);
                    sq = __dp4a(l1, (int)y0.y, sq);
                    sq = __dp4a(l2, (int)y0.z, sq);
                    sq = __dp4a(l3, (int)y0.w, sq);
                    sq = __dp4a(h0, (int)y1.x, sq);
                    sq = __dp4a(h1, (int)y1.y, sq);
                    sq = __dp4a(h2, (int)y1.z, sq);
                    sq = __dp4a(h3, (int)y1.w, sq);
                    // sum (q - 8) y = sum q y - 8 sum y, with sum y from the quantizer
                    const int isum = sq - 8 * (int)__ldg(x.sums + row * nb + bg);
                    const float da = __ldg(x.d + row * nb + bg);
                    acc[m] += (dw * da) * (float)isum;
                }
            }
        }
        consumer_release(empty, s, lane);
        if (chunk == nchunks - 1) {
            const int64_t n = tile * kTileRows + warp;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float v = warp_sum(acc[m]);
                if (lane == 0 && m < mcount && n < N) Y[(m0 + m) * N + n] = v;
                acc[m] = 0.0f;
            }
        }
    }
}

template <class Kern>
cudaError_t launch_one(Kern kern, int smem, int64_t ntiles, bool pdl, cudaStream_t s,
                       const uint8_t *Wp, int64_t N, int64_t nblk, Planar x, int64_t M,
                       int64_t m0, float *Y) {
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    const int64_t cap = 2LL * sm_count();
    const int grid = (int)(ntiles < cap ? ntiles : cap);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    unsigned *err = device_error_word();
    e = cudaLaunchKernelEx(&cfg, kern, Wp, N, nblk, x, M, m0, Y, err);
    count_launch();
    return e;
}

template <int MT>
cudaError_t launch_mt(qmm_type wt, const uint8_t *Wp, int64_t N, int64_t K, Planar x, int64_t M,
                      int64_t m0, float *Y, bool pdl, cudaStream_t s) {
    const int64_t ntiles = tiles_of(N);
    if (wt == QMM_TYPE_Q4_K)
        return launch_one(gemv_q4_K_kernel<MT>, kSmemBytes, ntiles, pdl, s, Wp, N, K / QK_K, x, M,
                          m0, Y);
    return launch_one(gemv_q4_0_kernel<MT>, kSmemBytes, ntiles, pdl, s, Wp, N, K / QK4_0, x, M,
                      m0, Y);
}

}  // namespace

cudaError_t launch_gemv(qmm_type wt, const void *Wp, int64_t N, int64_t K, Planar x, int64_t M,
                        float *Y, bool pdl, cudaStream_t s) {
    const uint8_t *w = static_cast<const uint8_t *>(Wp);
    for (int64_t m0 = 0; m0 < M; m0 += kMaxMT) {
        const int64_t mt = M - m0 < kMaxMT ? M - m0 : kMaxMT;
        cudaError_t e;
        if (mt == 1)
            e = launch_mt<1>(wt, w, N, K, x, M, m0, Y, pdl, s);
        else if (mt == 2)
            e = launch_mt<2>(wt, w, N, K, x, M, m0, Y, pdl, s);
        else if (mt <= 4)
            e = launch_mt<4>(wt, w, N, K, x, M, m0, Y, pdl, s);
        else if (mt <= 8)
            e = launch_mt<8>(wt, w, N, K, x, M, m0, Y, pdl, s);
        else
            e = launch_mt<16>(wt, w, N, K, x, M, m0, Y, pdl, s);
        if (e != cudaSuccess) return e;
        pdl = false;  // only the first launch follows the quantizer directly
    }
    return cudaSuccess;
}

}  // namespace qmm
