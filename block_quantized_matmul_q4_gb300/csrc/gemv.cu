// gemv.cu -- decode-path mul_mat (M = 1..16 tokens per launch) over packed
// Q4_0 / Q4_K weights and Q8_0 / Q8_K activations.
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
//   * the activations live in shared memory for the whole kernel, filled one
//     of three ways (Mode): quantized from fp32 by the consumer warps in the
//     prologue (the activation quantizer fused into the GEMV, for small M*K),
//     bulk-copied from a workspace written by the stand-alone quantizer
//     (after griddepcontrol.wait, so the weight stream starts first), or --
//     when they do not fit -- read from global memory in place;
//   * eight consumer warps, one weight row each, unpack nibbles and the 6-bit
//     scales in registers and take the integer dot products with dp4a; each
//     lane owns four super-blocks per stage, unrolled for independent loads.
// Every mbarrier wait is bounded; a timeout sets the device error word and
// the CTA leaves after draining its own copies in flight.
#include "qmm_internal.cuh"

namespace qmm {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;
constexpr int kStages = 4;
constexpr int kStageBytes = 18432;
constexpr int kRingBytes = kStages * kStageBytes;
constexpr int kQ4KChunk = 8;    // super-blocks per stage and tile: 2 tiles * 8 * 8 * 144 B = 18432
constexpr int kHalfStage = kQ4KChunk * kTileRows * B_Q4_K;  // one tile's share of a stage
constexpr int kQ40Chunk = 128;  // blocks per stage: 128 * 8 rows * 18 B = 18432
constexpr int kBarBytes = (2 * kStages + 1) * 8;  // full[4], empty[4], act
constexpr int kMaxMT = 16;
constexpr int kActMax = 36 * 1024;        // shared memory for staged activations
constexpr int64_t kFuseMaxElems = 8192;  // fused quantizer up to M*K fp32 elements
static_assert(2 * kHalfStage == kStageBytes, "stage size");
static_assert(kQ40Chunk * kTileRows * B_Q4_0 == kStageBytes, "stage size");
static_assert(kBarBytes == 72, "barrier area must hold 2 * kStages + 1 mbarriers");

enum Mode { kDirect = 0, kStaged = 1, kFused = 2 };

struct GemvArgs {
    MatSet ms;          // packed weights, outputs and rows of each matrix
    int64_t nblk;       // blocks per row (nsb for Q4_K, nb for Q4_0)
    Planar x;           // planar activations (kDirect, kStaged)
    const float *X;     // fp32 activations (kFused)
    int64_t M, m0;      // all tokens, first token of this launch
    unsigned *err;
    uint32_t act_bs, act_d, act_bytes;  // shared activation layout (offsets, total)
};

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ uint32_t align16(uint64_t x) {
    return (uint32_t)((x + 15) & ~15ull);
}

__device__ __forceinline__ void my_tiles(int64_t ntiles, int64_t &tb, int64_t &te) {
    tb = (int64_t)blockIdx.x * ntiles / gridDim.x;
    te = ((int64_t)blockIdx.x + 1) * ntiles / gridDim.x;
}

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <class T>
__device__ __forceinline__ T ld(const T *p, bool global) {
    return global ? __ldg(p) : *p;
}
__device__ __forceinline__ uint4 ld4(const void *p, bool global) {
    return global ? __ldg(reinterpret_cast<const uint4 *>(p)) : *reinterpret_cast<const uint4 *>(p);
}

// ------------------------------------------------------------------ pipeline
struct Ring {
    uint8_t *smem;
    uint64_t *full, *empty, *act;
};

__device__ __forceinline__ Ring ring_init(uint8_t *smem, uint32_t act_bytes) {
    Ring r;
    r.smem = smem;
    r.full = reinterpret_cast<uint64_t *>(smem + kRingBytes + act_bytes);
    r.empty = r.full + kStages;
    r.act = r.empty + kStages;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&r.full[s]), 1);
            mbar_init(smem_u32(&r.empty[s]), kConsumerWarps);
        }
        mbar_init(smem_u32(r.act), 1);
        fence_barrier_init();
        // The next kernel in the stream may launch now: it only streams
        // weights until its griddepcontrol.wait, which waits for this grid.
        pdl_launch_dependents();
    }
    __syncthreads();
    return r;
}

// Producer: issue stage copies for items 0 .. n_items-1 (copy(item, dst, bar,
// policy) posts expect_tx and the copies). The first kStages items need no
// wait; `after_prefill` runs once they are in flight (it brings in the
// activations, which depend on the previous kernel). Before returning, waits
// (bounded) until no issued copy can still be landing in shared memory.
template <class Copy, class After>
__device__ __forceinline__ void producer_loop(const Ring &r, int64_t n_items, unsigned *err,
                                              Copy copy, After after_prefill) {
    const uint64_t pol = policy_evict_first();
    int64_t it = 0;
    bool after_done = false;
    for (; it < n_items; ++it) {
        const int s = (int)(it % kStages);
        if (it == kStages) {
            after_prefill();
            after_done = true;
        }
        if (!mbar_wait(smem_u32(&r.empty[s]), (uint32_t)(((it / kStages) & 1) ^ 1), err)) break;
        copy(it, smem_u32(r.smem + s * kStageBytes), smem_u32(&r.full[s]), pol);
    }
    if (!after_done) after_prefill();
    for (int64_t k = it > kStages ? it - kStages : 0; k < it; ++k)
        mbar_wait(smem_u32(&r.full[k % kStages]), (uint32_t)((k / kStages) & 1), err);
}

// Copies this launch's token rows of the planar workspace into shared memory.
__device__ __forceinline__ void stage_activations(const Ring &r, const GemvArgs &a, int mc,
                                                  int64_t K, int groups) {
    pdl_wait();  // the workspace is written by the preceding quantizer kernel
    const uint64_t pol = policy_evict_last();
    const uint32_t bar = smem_u32(r.act);
    const uint32_t base = smem_u32(r.smem + kRingBytes);
    const uint32_t qs_bytes = (uint32_t)(mc * K);
    const uint32_t bs_bytes = align16((uint64_t)mc * a.nblk * groups * 2);
    const uint32_t d_bytes = align16((uint64_t)mc * a.nblk * 4);
    mbar_arrive_expect_tx(bar, qs_bytes + bs_bytes + d_bytes);
    bulk_g2s(base, a.x.qs + a.m0 * K, qs_bytes, bar, pol);
    bulk_g2s(base + a.act_bs, a.x.sums + a.m0 * a.nblk * groups, bs_bytes, bar, pol);
    bulk_g2s(base + a.act_d, a.x.d + a.m0 * a.nblk, d_bytes, bar, pol);
}

// ------------------------------------------------------------------ Q4_K
// Stage = a pair of tiles (rows 16p .. 16p+15) x up to 8 super-blocks: tile
// 2p's blocks [sb][8 rows][144 B] at offset 0, tile 2p+1's at kHalfStage (one
// bulk copy each). Warp w owns row w of both tiles, so every activation value
// it loads serves two weight rows. Lane (g, t) = (lane / 8, lane % 8) owns
// super-blocks g and g + 4 of the stage and, within each, qs bytes 16t ..
// 16t+15: chunk c = t / 2, half h = t % 2, i.e. 16 elements of sub-block 2c
// (low nibbles) and 16 of sub-block 2c+1 (high nibbles). The planar
// activation layout puts exactly those 2 x 16 codes at bytes 16t and
// 128 + 16t of the super-block and the two matching 16-code sums in word t;
// the packed header puts the lane's two scales and mins in 24-bit field c.

// dp4a with an unsigned first operand: bytes of a are 0..255.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

struct KLane {
    bool c_ge2, c_ge3;  // which header words hold field c
    uint32_t fsh;       // bit offset of field c within them
};

// One (row, super-block) share of this lane: d_a (d isum - dmin msum) over
// its 16 + 16 elements (page 1, "正确性" and "min 项与最终归约").
__device__ __forceinline__ float q4k_dot(const uint4 &hdr, const uint4 &q, const uint4 &y0,
                                         const uint4 &y1, int bw, float da, const KLane &L) {
    const uint32_t f =
        __funnelshift_r(L.c_ge3 ? hdr.w : (L.c_ge2 ? hdr.z : hdr.y), L.c_ge2 ? hdr.w : hdr.z, L.fsh);
    const int sc0 = f & 63, mn0 = (f >> 6) & 63;
    const int sc1 = (f >> 12) & 63, mn1 = (f >> 18) & 63;
    const float dw = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xFFFFu)));
    const float dmw = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
    // low nibbles as bytes; high nibbles left in place, giving 16 x their sum
    int s0 = dp4a_us(q.x & 0x0F0F0F0Fu, y0.x, 0);
    int s0b = dp4a_us(q.y & 0x0F0F0F0Fu, y0.y, 0);
    s0 = dp4a_us(q.z & 0x0F0F0F0Fu, y0.z, s0);
    s0b = dp4a_us(q.w & 0x0F0F0F0Fu, y0.w, s0b);
    int s1 = dp4a_us(q.x & 0xF0F0F0F0u, y1.x, 0);
    int s1b = dp4a_us(q.y & 0xF0F0F0F0u, y1.y, 0);
    s1 = dp4a_us(q.z & 0xF0F0F0F0u, y1.z, s1);
    s1b = dp4a_us(q.w & 0xF0F0F0F0u, y1.w, s1b);
    const int isum = sc0 * (s0 + s0b) + sc1 * ((s1 + s1b) >> 4);
    const int msum = mn0 * (int)(int16_t)(bw & 0xFFFF) + mn1 * (bw >> 16);
    // |isum| <= 2 * 63 * 16 * 15 * 127 and msum <= 2 * 63 * 2032: exact
    // conversions without the conversion pipe
    return da * (dw * int_as_exact_float(isum) - dmw * int_as_exact_float(msum));
}

// The Q8_K quantizer fused into the GEMV prologue (K-quant weights): the
// launch's mc token rows of X into the planar layout in shared memory at aw.
// Super-blocks b = warp + 8 j of all the tokens' rows (b = row * nsb + sb, X
// rows contiguous, so b * QK_K is the element offset): up to kQBatch per
// warp with all their loads issued before any reduction.
__device__ __forceinline__ void fused_q8K(const GemvArgs &a, int mc, int64_t nsb, int64_t K, int warp,
                                          int lane, uint8_t *aw) {
    constexpr int kQBatch = 4;
    const int nq = (int)(mc * nsb);  // at most 16 x 4096 blocks
    for (int b0 = warp; b0 < nq; b0 += kQBatch * kConsumerWarps) {
        float4 v[kQBatch][2];
#pragma unroll
        for (int j = 0; j < kQBatch; ++j) {
            const int b = b0 + j * kConsumerWarps;
            if (b < nq) {
                const float4 *src = reinterpret_cast<const float4 *>(a.X + a.m0 * K + (int64_t)b * QK_K) +
                                    2 * lane;
                v[j][0] = __ldg(src);
                v[j][1] = __ldg(src + 1);
            }
        }
#pragma unroll
        for (int j = 0; j < kQBatch; ++j) {
            const int b = b0 + j * kConsumerWarps;
            if (b < nq) {
                const float x[8] = {v[j][0].x, v[j][0].y, v[j][0].z, v[j][0].w,
                                    v[j][1].x, v[j][1].y, v[j][1].z, v[j][1].w};
                uint32_t lo, hi;
                float d;
                int bsum;
                q8_K_warp(x, lo, hi, d, bsum);
                *reinterpret_cast<uint2 *>(aw + (int64_t)b * QK_K + q8K_code_offset(lane)) = make_uint2(lo, hi);
                if ((lane & 1) == 0)
                    *reinterpret_cast<int16_t *>(aw + a.act_bs + b * 32 + q8K_bsum_offset(lane >> 1)) =
                        (int16_t)bsum;
                if (lane == 0) reinterpret_cast<float *>(aw + a.act_d)[b] = d;
            }
        }
    }
}

template <int MT, int kMode>
__global__ void __launch_bounds__(kThreads, 2) gemv_q4_K_kernel(const GemvArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nsb = a.nblk, K = nsb * QK_K;
    const int mc = (int)min64(MT, a.M - a.m0);
    int64_t pb, pe;
    my_tiles(a.ms.off[a.ms.n], pb, pe);  // this CTA's tile pairs (over all matrices)
    const int64_t nchunks = (nsb + kQ4KChunk - 1) / kQ4KChunk;
    const int64_t n_items = (pe - pb) * nchunks;
    const Ring r = ring_init(smem, kMode == kDirect ? 0 : a.act_bytes);

    if (warp == kConsumerWarps) {
        if (lane == 0) {
            producer_loop(
                r, n_items, a.err,
                [&, chunk = (int64_t)0, p = pb](int64_t, uint32_t dst, uint32_t bar,
                                                 uint64_t pol) mutable {
                    // items in order: (pair, chunk) counted, not divided out
                    const int mi = mat_of(a.ms, p);
                    const int64_t t0 = 2 * (p - a.ms.off[mi]);
                    const int64_t sb0 = chunk * kQ4KChunk;
                    if (++chunk == nchunks) chunk = 0, ++p;
                    const uint32_t bytes =
                        (uint32_t)min64(kQ4KChunk, nsb - sb0) * kTileRows * B_Q4_K;
                    const bool has1 = t0 + 1 < tiles_of(a.ms.N[mi]);
                    const uint8_t *W = a.ms.W[mi];
                    mbar_arrive_expect_tx(bar, has1 ? 2 * bytes : bytes);
                    bulk_g2s(dst, W + (t0 * nsb + sb0) * (kTileRows * B_Q4_K), bytes, bar, pol);
                    if (has1)
                        bulk_g2s(dst + kHalfStage, W + ((t0 + 1) * nsb + sb0) * (kTileRows * B_Q4_K),
                                 bytes, bar, pol);
                },
                [&]() {
                    if (kMode == kStaged) stage_activations(r, a, mc, K, 16);
                });
            if (kMode == kStaged) mbar_wait(smem_u32(r.act), 0, a.err);
        }
        return;
    }

    // ---- activations: where this launch's token rows are read from
    const uint8_t *act = smem + kRingBytes;
    const bool gl = kMode == kDirect;
    const int8_t *xqs = gl ? a.x.qs + a.m0 * K : reinterpret_cast<const int8_t *>(act);
    const int32_t *xbs = gl ? reinterpret_cast<const int32_t *>(a.x.sums) + a.m0 * nsb * 8
                            : reinterpret_cast<const int32_t *>(act + a.act_bs);
    const float *xd = gl ? a.x.d + a.m0 * nsb : reinterpret_cast<const float *>(act + a.act_d);
    if (kMode == kFused) {
        pdl_wait();
        fused_q8K(a, mc, nsb, K, warp, lane, smem + kRingBytes);
        consumer_sync();
    } else if (kMode == kStaged) {
        if (!mbar_wait(smem_u32(r.act), 0, a.err)) return;
    } else {
        pdl_wait();
    }

    const int g = lane >> 3, t = lane & 7, c = t >> 1;
    const KLane L{c >= 2, c >= 3, (uint32_t)((24 * c) & 31)};
    float acc0[MT], acc1[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc0[m] = acc1[m] = 0.0f;

    int64_t chunk = 0, p = pb;  // the item's K chunk and tile pair, counted
    for (int64_t it = 0; it < n_items; ++it) {
        const int s = (int)(it % kStages);
        if (!mbar_wait(smem_u32(&r.full[s]), (uint32_t)((it / kStages) & 1), a.err)) break;
        const int64_t sb0 = chunk * kQ4KChunk;
        const int cnt = (int)min64(kQ4KChunk, nsb - sb0);
        const uint8_t *stage = smem + s * kStageBytes;
        // super-block sl of the stage: both rows of this warp, all tokens
        auto body = [&](int sl) {
            const uint8_t *ba = stage + (sl * kTileRows + warp) * B_Q4_K;
            const uint4 ha = *reinterpret_cast<const uint4 *>(ba);
            const uint4 qa = *reinterpret_cast<const uint4 *>(ba + 16 + 16 * t);
            const uint4 hb = *reinterpret_cast<const uint4 *>(ba + kHalfStage);
            const uint4 qb = *reinterpret_cast<const uint4 *>(ba + kHalfStage + 16 + 16 * t);
            const int64_t sbg = sb0 + sl;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m < mc) {
                    const int8_t *yp = xqs + m * K + sbg * QK_K;
                    const uint4 y0 = ld4(yp + 16 * t, gl);        // sub-block 2c
                    const uint4 y1 = ld4(yp + 128 + 16 * t, gl);  // sub-block 2c + 1
                    const int bw = ld(xbs + (m * nsb + sbg) * 8 + t, gl);
                    const float da = ld(xd + m * nsb + sbg, gl);
                    acc0[m] += q4k_dot(ha, qa, y0, y1, bw, da, L);
                    acc1[m] += q4k_dot(hb, qb, y0, y1, bw, da, L);
                }
            }
        };
        if (cnt == kQ4KChunk) {
            body(g);
            body(g + 4);
        } else {
            if (g < cnt) body(g);
            if (g + 4 < cnt) body(g + 4);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&r.empty[s]));
        if (chunk == nchunks - 1) {
            const int mi = mat_of(a.ms, p);
            const int64_t N = a.ms.N[mi];
            float *Y = a.ms.Y[mi];
            const int64_t n0 = 2 * (p - a.ms.off[mi]) * kTileRows + warp, n1 = n0 + kTileRows;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float v0 = warp_sum(acc0[m]);
                const float v1 = warp_sum(acc1[m]);
                if (lane == 0 && m < mc) {
                    if (n0 < N) Y[(a.m0 + m) * N + n0] = v0;
                    if (n1 < N) Y[(a.m0 + m) * N + n1] = v1;
                }
                acc0[m] = acc1[m] = 0.0f;
            }
        }
        if (++chunk == nchunks) chunk = 0, ++p;
    }
}

// ------------------------------------------------------------------ Q6_K
// Page 1, "更低的比特: Q6_K 与 Q2_K 的取舍": w = d s_j q, q = u - 32 in
// -32..31, 16 groups of 16, no min term. Per super-block and lane t:
//   S_g = sum_i q_i y_i = sum_i u_i y_i - 32 bs_g   (bs_g the group's code sum)
//   isum = s_lo S_lo + s_hi S_hi,   y += d_a (d isum)
// Stage = a pair of tiles x up to 4 super-blocks (records of kQ6Rec bytes:
// tile 2p's at offset 0, tile 2p+1's at kQ6Half). Warp w owns row w of both
// tiles; lane (g, t) takes super-block g of the stage and ql bytes 16t ..
// 16t+15, whose elements are exactly the planar activation bytes 16t.. and
// 128 + 16t.. of the super-block and whose two groups' code sums are word t.
constexpr int kQ6KChunk = 4;
constexpr int kQ6Half = kQ6KChunk * kQ6Rec;  // 6720
static_assert(2 * kQ6Half <= kStageBytes, "stage size");

__device__ __forceinline__ float q6k_dot(const uint4 &q, const uint2 &h, uint32_t sc, float dw,
                                         const uint4 &y0, const uint4 &y1, int bw, float da) {
    int s0 = dp4a_us(q6k_u(q.x, h.x, 0), y0.x, 0);
    int s0b = dp4a_us(q6k_u(q.y, h.x, 1), y0.y, 0);
    s0 = dp4a_us(q6k_u(q.z, h.x, 2), y0.z, s0);
    s0b = dp4a_us(q6k_u(q.w, h.x, 3), y0.w, s0b);
    int s1 = dp4a_us(q6k_u(q.x >> 4, h.y, 0), y1.x, 0);
    int s1b = dp4a_us(q6k_u(q.y >> 4, h.y, 1), y1.y, 0);
    s1 = dp4a_us(q6k_u(q.z >> 4, h.y, 2), y1.z, s1);
    s1b = dp4a_us(q6k_u(q.w >> 4, h.y, 3), y1.w, s1b);
    const int S0 = s0 + s0b - 32 * (int)(int16_t)(bw & 0xFFFF);
    const int S1 = s1 + s1b - 32 * (bw >> 16);
    const int isum = (int)(int8_t)(sc & 0xFF) * S0 + (int)(int8_t)(sc >> 8) * S1;
    return da * (dw * (float)isum);
}

template <int MT, int kMode>
__global__ void __launch_bounds__(kThreads, 2) gemv_q6_K_kernel(const GemvArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nsb = a.nblk, K = nsb * QK_K;
    const int mc = (int)min64(MT, a.M - a.m0);
    int64_t pb, pe;
    my_tiles(a.ms.off[a.ms.n], pb, pe);  // this CTA's tile pairs (over all matrices)
    const int64_t nchunks = (nsb + kQ6KChunk - 1) / kQ6KChunk;
    const int64_t n_items = (pe - pb) * nchunks;
    const Ring r = ring_init(smem, kMode == kDirect ? 0 : a.act_bytes);

    if (warp == kConsumerWarps) {
        if (lane == 0) {
            producer_loop(
                r, n_items, a.err,
                [&, chunk = (int64_t)0, p = pb](int64_t, uint32_t dst, uint32_t bar,
                                                 uint64_t pol) mutable {
                    const int mi = mat_of(a.ms, p);
                    const int64_t t0 = 2 * (p - a.ms.off[mi]);
                    const int64_t sb0 = chunk * kQ6KChunk;
                    if (++chunk == nchunks) chunk = 0, ++p;
                    const uint32_t bytes = (uint32_t)min64(kQ6KChunk, nsb - sb0) * kQ6Rec;
                    const bool has1 = t0 + 1 < tiles_of(a.ms.N[mi]);
                    const uint8_t *W = a.ms.W[mi];
                    mbar_arrive_expect_tx(bar, has1 ? 2 * bytes : bytes);
                    bulk_g2s(dst, W + (t0 * nsb + sb0) * kQ6Rec, bytes, bar, pol);
                    if (has1)
                        bulk_g2s(dst + kQ6Half, W + ((t0 + 1) * nsb + sb0) * kQ6Rec, bytes, bar, pol);
                },
                [&]() {
                    if (kMode == kStaged) stage_activations(r, a, mc, K, 16);
                });
            if (kMode == kStaged) mbar_wait(smem_u32(r.act), 0, a.err);
        }
        return;
    }

    const uint8_t *act = smem + kRingBytes;
    const bool gl = kMode == kDirect;
    const int8_t *xqs = gl ? a.x.qs + a.m0 * K : reinterpret_cast<const int8_t *>(act);
    const int32_t *xbs = gl ? reinterpret_cast<const int32_t *>(a.x.sums) + a.m0 * nsb * 8
                            : reinterpret_cast<const int32_t *>(act + a.act_bs);
    const float *xd = gl ? a.x.d + a.m0 * nsb : reinterpret_cast<const float *>(act + a.act_d);
    if (kMode == kFused) {
        pdl_wait();
        fused_q8K(a, mc, nsb, K, warp, lane, smem + kRingBytes);
        consumer_sync();
    } else if (kMode == kStaged) {
        if (!mbar_wait(smem_u32(r.act), 0, a.err)) return;
    } else {
        pdl_wait();
    }

    const int g = lane >> 3, t = lane & 7;
    float acc0[MT], acc1[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc0[m] = acc1[m] = 0.0f;

    int64_t chunk = 0, p = pb;  // the item's K chunk and tile pair, counted
    for (int64_t it = 0; it < n_items; ++it) {
        const int s = (int)(it % kStages);
        if (!mbar_wait(smem_u32(&r.full[s]), (uint32_t)((it / kStages) & 1), a.err)) break;
        const int64_t sb0 = chunk * kQ6KChunk;
        const int cnt = (int)min64(kQ6KChunk, nsb - sb0);
        if (g < cnt) {
            const uint8_t *ra = smem + s * kStageBytes + g * kQ6Rec;
            const uint8_t *rb = ra + kQ6Half;
            const uint4 qa = *reinterpret_cast<const uint4 *>(ra + warp * kQ6Codes + 16 * t);
            const uint2 ha = *reinterpret_cast<const uint2 *>(ra + warp * kQ6Codes + 128 + 8 * t);
            const uint32_t sca = *reinterpret_cast<const uint16_t *>(ra + kQ6ScOff + 16 * warp + 2 * t);
            const float dwa = __half2float(*reinterpret_cast<const __half *>(ra + kQ6DOff + 2 * warp));
            const uint4 qb = *reinterpret_cast<const uint4 *>(rb + warp * kQ6Codes + 16 * t);
            const uint2 hb = *reinterpret_cast<const uint2 *>(rb + warp * kQ6Codes + 128 + 8 * t);
            const uint32_t scb = *reinterpret_cast<const uint16_t *>(rb + kQ6ScOff + 16 * warp + 2 * t);
            const float dwb = __half2float(*reinterpret_cast<const __half *>(rb + kQ6DOff + 2 * warp));
            const int64_t sbg = sb0 + g;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m < mc) {
                    const int8_t *yp = xqs + m * K + sbg * QK_K;
                    const uint4 y0 = ld4(yp + 16 * t, gl);        // group 4c + h
                    const uint4 y1 = ld4(yp + 128 + 16 * t, gl);  // group 4c + 2 + h
                    const int bw = ld(xbs + (m * nsb + sbg) * 8 + t, gl);
                    const float da = ld(xd + m * nsb + sbg, gl);
                    acc0[m] += q6k_dot(qa, ha, sca, dwa, y0, y1, bw, da);
                    acc1[m] += q6k_dot(qb, hb, scb, dwb, y0, y1, bw, da);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&r.empty[s]));
        if (chunk == nchunks - 1) {
            const int mi = mat_of(a.ms, p);
            const int64_t N = a.ms.N[mi];
            float *Y = a.ms.Y[mi];
            const int64_t n0 = 2 * (p - a.ms.off[mi]) * kTileRows + warp, n1 = n0 + kTileRows;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float v0 = warp_sum(acc0[m]);
                const float v1 = warp_sum(acc1[m]);
                if (lane == 0 && m < mc) {
                    if (n0 < N) Y[(a.m0 + m) * N + n0] = v0;
                    if (n1 < N) Y[(a.m0 + m) * N + n1] = v1;
                }
                acc0[m] = acc1[m] = 0.0f;
            }
        }
        if (++chunk == nchunks) chunk = 0, ++p;
    }
}

// ------------------------------------------------------------------ Q4_0
// Stage = one tile (8 rows) x up to 128 blocks. Shared layout: nibble rows
// [8][128][16 B] at offset 0 (one bulk copy per row segment) and the fp16
// scales [cnt][8] at offset kDOff (one copy). Warp w owns row w; lane l takes
// blocks l, l + 32, l + 64, l + 96, so each 8-lane phase of a 128-bit load
// reads 128 contiguous bytes.
template <int MT, int kMode>
__global__ void __launch_bounds__(kThreads, 2) gemv_q4_0_kernel(const GemvArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nb = a.nblk, K = nb * QK4_0;
    const int mc = (int)min64(MT, a.M - a.m0);
    int64_t tb, te;
    my_tiles(a.ms.off[a.ms.n], tb, te);  // this CTA's tiles (over all matrices)
    const int64_t nchunks = (nb + kQ40Chunk - 1) / kQ40Chunk;
    const int64_t n_items = (te - tb) * nchunks;
    const int64_t tile_bytes = nb * kTileRows * B_Q4_0;
    constexpr uint32_t kRowBytes = kQ40Chunk * 16;
    constexpr uint32_t kDOff = kTileRows * kRowBytes;
    const Ring r = ring_init(smem, kMode == kDirect ? 0 : a.act_bytes);

    if (warp == kConsumerWarps) {
        if (lane == 0) {
            producer_loop(
                r, n_items, a.err,
                [&, chunk = (int64_t)0, tile = tb](int64_t, uint32_t dst, uint32_t bar,
                                                    uint64_t pol) mutable {
                    const int mi = mat_of(a.ms, tile);
                    const int64_t b0 = chunk * kQ40Chunk;
                    const uint32_t cnt = (uint32_t)min64(kQ40Chunk, nb - b0);
                    const uint8_t *tbase = a.ms.W[mi] + (tile - a.ms.off[mi]) * tile_bytes;
                    mbar_arrive_expect_tx(bar, cnt * kTileRows * B_Q4_0);
                    for (int rr = 0; rr < kTileRows; ++rr)
                        bulk_g2s(dst + rr * kRowBytes, tbase + (rr * nb + b0) * 16, cnt * 16, bar,
                                 pol);
                    bulk_g2s(dst + kDOff, tbase + nb * kTileRows * 16 + b0 * kTileRows * 2,
                             cnt * kTileRows * 2, bar, pol);
                    if (++chunk == nchunks) chunk = 0, ++tile;
                },
                [&]() {
                    if (kMode == kStaged) stage_activations(r, a, mc, K, 1);
                });
            if (kMode == kStaged) mbar_wait(smem_u32(r.act), 0, a.err);
        }
        return;
    }

    const uint8_t *act = smem + kRingBytes;
    const bool gl = kMode == kDirect;
    const int8_t *xqs = gl ? a.x.qs + a.m0 * K : reinterpret_cast<const int8_t *>(act);
    const int16_t *xsum =
        gl ? a.x.sums + a.m0 * nb : reinterpret_cast<const int16_t *>(act + a.act_bs);
    const float *xd = gl ? a.x.d + a.m0 * nb : reinterpret_cast<const float *>(act + a.act_d);
    if (kMode == kFused) {
        pdl_wait();
        uint8_t *aw = smem + kRingBytes;
        // groups of eight blocks, four lanes per block (b * QK4_0 is the
        // element offset over all the tokens' rows): group g0 + 8 j of warp
        // g0, up to kQBatch per warp with their loads issued first; lanes
        // past the last block take zeros and store nothing
        constexpr int kQBatch = 2;
        const int nq = (int)(mc * nb);
        const int bl = lane >> 2, part = lane & 3;
        for (int g0 = warp * 8; g0 < nq; g0 += kQBatch * kConsumerWarps * 8) {
            float4 v[kQBatch][2];
#pragma unroll
            for (int j = 0; j < kQBatch; ++j) {
                const int b = g0 + j * kConsumerWarps * 8 + bl;
                v[j][0] = v[j][1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (b < nq) {
                    const float4 *src =
                        reinterpret_cast<const float4 *>(a.X + a.m0 * K + (int64_t)b * QK4_0 + 8 * part);
                    v[j][0] = __ldg(src);
                    v[j][1] = __ldg(src + 1);
                }
            }
#pragma unroll
            for (int j = 0; j < kQBatch; ++j) {
                const int gb = g0 + j * kConsumerWarps * 8;
                if (gb < nq) {  // warp-uniform: the shuffles need every lane
                    const int b = gb + bl;
                    const float x[8] = {v[j][0].x, v[j][0].y, v[j][0].z, v[j][0].w,
                                        v[j][1].x, v[j][1].y, v[j][1].z, v[j][1].w};
                    uint32_t lo, hi;
                    int sum;
                    __half dh;
                    q8_0_quad(x, lo, hi, dh, sum);
                    if (b < nq) {
                        *reinterpret_cast<uint2 *>(aw + (int64_t)b * QK4_0 + 8 * part) = make_uint2(lo, hi);
                        if (part == 0) {
                            reinterpret_cast<int16_t *>(aw + a.act_bs)[b] = (int16_t)sum;
                            reinterpret_cast<float *>(aw + a.act_d)[b] = __half2float(dh);
                        }
                    }
                }
            }
        }
        consumer_sync();
    } else if (kMode == kStaged) {
        if (!mbar_wait(smem_u32(r.act), 0, a.err)) return;
    } else {
        pdl_wait();
    }

    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.0f;

    int64_t chunk = 0, tile = tb;  // the item's K chunk and tile, counted
    for (int64_t it = 0; it < n_items; ++it) {
        const int s = (int)(it % kStages);
        if (!mbar_wait(smem_u32(&r.full[s]), (uint32_t)((it / kStages) & 1), a.err)) break;
        const int64_t b0 = chunk * kQ40Chunk;
        const int cnt = (int)min64(kQ40Chunk, nb - b0);
        const uint8_t *stage = smem + s * kStageBytes;
#pragma unroll
        for (int i = 0; i < kQ40Chunk / 32; ++i) {
            const int bl = lane + 32 * i;
            if (bl < cnt) {
                const uint4 q = *reinterpret_cast<const uint4 *>(stage + warp * kRowBytes + bl * 16);
                const unsigned short dbits = *reinterpret_cast<const unsigned short *>(
                    stage + kDOff + (bl * kTileRows + warp) * 2);
                const float dw = __half2float(__ushort_as_half(dbits));
                const uint32_t l0 = q.x & 0x0F0F0F0Fu, l1 = q.y & 0x0F0F0F0Fu;
                const uint32_t l2 = q.z & 0x0F0F0F0Fu, l3 = q.w & 0x0F0F0F0Fu;
                const uint32_t h0 = q.x & 0xF0F0F0F0u, h1 = q.y & 0xF0F0F0F0u;
                const uint32_t h2 = q.z & 0xF0F0F0F0u, h3 = q.w & 0xF0F0F0F0u;
                const int64_t bg = b0 + bl;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (m < mc) {
                        const int8_t *yp = xqs + m * K + bg * QK4_0;
                        const uint4 y0 = ld4(yp, gl);       // elements 0..15
                        const uint4 y1 = ld4(yp + 16, gl);  // elements 16..31
                        int sl = dp4a_us(l0, y0.x, 0);
                        sl = dp4a_us(l1, y0.y, sl);
                        sl = dp4a_us(l2, y0.z, sl);
                        sl = dp4a_us(l3, y0.w, sl);
                        int sh16 = dp4a_us(h0, y1.x, 0);  // 16 x the high-nibble sum
                        sh16 = dp4a_us(h1, y1.y, sh16);
                        sh16 = dp4a_us(h2, y1.z, sh16);
                        sh16 = dp4a_us(h3, y1.w, sh16);
                        // sum (q - 8) y = sum q y - 8 sum y, sum y from the quantizer
                        const int isum =
                            sl + (sh16 >> 4) - 8 * (int)ld(xsum + m * nb + bg, gl);
                        const float da = ld(xd + m * nb + bg, gl);
                        acc[m] += (dw * da) * (float)isum;
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&r.empty[s]));
        if (chunk == nchunks - 1) {
            const int mi = mat_of(a.ms, tile);
            const int64_t N = a.ms.N[mi];
            const int64_t n = (tile - a.ms.off[mi]) * kTileRows + warp;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float v = warp_sum(acc[m]);
                if (lane == 0 && m < mc && n < N) a.ms.Y[mi][(a.m0 + m) * N + n] = v;
                acc[m] = 0.0f;
            }
        }
        if (++chunk == nchunks) chunk = 0, ++tile;
    }
}

// ------------------------------------------------------------------ launch
template <int MT, int kMode>
cudaError_t launch_kernel(qmm_type wt, const GemvArgs &a, bool pdl, cudaStream_t s) {
    const void *fn = wt == QMM_TYPE_Q4_K   ? reinterpret_cast<const void *>(gemv_q4_K_kernel<MT, kMode>)
                     : wt == QMM_TYPE_Q6_K ? reinterpret_cast<const void *>(gemv_q6_K_kernel<MT, kMode>)
                                           : reinterpret_cast<const void *>(gemv_q4_0_kernel<MT, kMode>);
    const int smem = kRingBytes + (kMode == kDirect ? 0 : (int)a.act_bytes) + kBarBytes;
    cudaError_t e = ensure_smem_attr(fn, smem);
    if (e != cudaSuccess) return e;
    // K-quant CTAs work on pairs of tiles, Q4_0 CTAs on single tiles
    const int64_t units = a.ms.off[a.ms.n];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)balanced_grid(units, 2LL * sm_count()));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (wt == QMM_TYPE_Q4_K)
        e = cudaLaunchKernelEx(&cfg, gemv_q4_K_kernel<MT, kMode>, a);
    else if (wt == QMM_TYPE_Q6_K)
        e = cudaLaunchKernelEx(&cfg, gemv_q6_K_kernel<MT, kMode>, a);
    else
        e = cudaLaunchKernelEx(&cfg, gemv_q4_0_kernel<MT, kMode>, a);
    count_launch();
    return e;
}

template <int MT>
cudaError_t launch_mode(qmm_type wt, int mode, const GemvArgs &a, bool pdl, cudaStream_t s) {
    if (mode == kFused) return launch_kernel<MT, kFused>(wt, a, pdl, s);
    if (mode == kStaged) return launch_kernel<MT, kStaged>(wt, a, pdl, s);
    return launch_kernel<MT, kDirect>(wt, a, pdl, s);
}

uint32_t act_layout(qmm_type wt, int64_t mt, int64_t K, uint32_t *bs_off, uint32_t *d_off) {
    const int qk = wt == QMM_TYPE_Q4_0 ? QK4_0 : QK_K;
    const int groups = wt == QMM_TYPE_Q4_0 ? 1 : 16;
    const uint32_t bs = align16((uint64_t)mt * K);
    const uint32_t d = bs + align16((uint64_t)mt * (K / qk) * groups * 2);
    if (bs_off) *bs_off = bs;
    if (d_off) *d_off = d;
    return d + align16((uint64_t)mt * (K / qk) * 4);
}

}  // namespace

bool gemv_use_mma(qmm_type wt, int64_t M, int64_t K) {
    if (M < kMmaMinM) return false;
    if (wt == QMM_TYPE_Q4_K) return gemv_mma_max_tokens(K) >= 1;
    // Q6_K at two tokens small enough for the fused quantizer: the one-kernel
    // dp4a GEMV beats the quantizer kernel plus the tensor-core GEMV (4096^2:
    // 5.5 against 7.4 us); from three tokens the tensor cores win
    if (wt == QMM_TYPE_Q6_K && M == 2 && M * K <= kFuseMaxElems) return false;
    return (wt == QMM_TYPE_Q6_K || wt == QMM_TYPE_Q4_0) && gemv_mma6_max_tokens(wt, K) >= 1;
}

bool gemv_can_fuse(qmm_type wt, int64_t M, int64_t K) {
    // only the Q4_K tensor-core GEMV has its quantizer inside
    if (gemv_use_mma(wt, M, K)) return wt == QMM_TYPE_Q4_K && M * K <= kMmaFuseElems;
    const int64_t mt = min64(M, kMaxMT);
    return act_layout(wt, mt, K, nullptr, nullptr) <= (uint32_t)kActMax && mt * K <= kFuseMaxElems;
}

MatSet single_mat(const void *Wp, int64_t N, float *Y) {
    MatSet ms = {};
    ms.n = 1;
    ms.W[0] = static_cast<const uint8_t *>(Wp);
    ms.N[0] = N;
    ms.Y[0] = Y;
    return ms;
}

// X != nullptr runs the quantizer fused into the GEMV prologue (X is the fp32
// activation; the caller checked gemv_can_fuse); otherwise the activations
// come from the planar workspace x written by launch_quantize_q8.
cudaError_t launch_gemv(qmm_type wt, MatSet ms, int64_t K, Planar x, const float *X, int64_t M,
                        bool pdl, cudaStream_t s) {
    if (X && gemv_use_mma(wt, M, K)) return launch_gemv_mma_q4_K(ms, K, X, nullptr, M, pdl, s);
    // work units: tile pairs (K-quant CTAs work on two 8-row tiles) or tiles
    const bool pairs = wt != QMM_TYPE_Q4_0;
    ms.off[0] = 0;
    for (int i = 0; i < ms.n; ++i)
        ms.off[i + 1] = ms.off[i] + (pairs ? (tiles_of(ms.N[i]) + 1) / 2 : tiles_of(ms.N[i]));
    GemvArgs a;
    a.ms = ms;
    a.nblk = K / (pairs ? QK_K : QK4_0);
    a.x = x;
    a.X = X;
    a.M = M;
    a.err = device_error_word();
    for (int64_t m0 = 0; m0 < M; m0 += kMaxMT) {
        const int64_t mt = min64(M - m0, kMaxMT);
        a.m0 = m0;
        a.act_bytes = act_layout(wt, mt, K, &a.act_bs, &a.act_d);
        int mode = kDirect;
        if (X)
            mode = kFused;
        else if (a.act_bytes <= (uint32_t)kActMax)
            mode = kStaged;
        cudaError_t e;
        if (mt == 1)
            e = launch_mode<1>(wt, mode, a, pdl, s);
        else if (mt == 2)
            e = launch_mode<2>(wt, mode, a, pdl, s);
        else if (mt <= 4)
            e = launch_mode<4>(wt, mode, a, pdl, s);
        else if (mt <= 8)
            e = launch_mode<8>(wt, mode, a, pdl, s);
        else
            e = launch_mode<16>(wt, mode, a, pdl, s);
        if (e != cudaSuccess) return e;
        pdl = false;  // only the first launch follows the quantizer directly
    }
    return cudaSuccess;
}

cudaError_t launch_gemv(qmm_type wt, const void *Wp, int64_t N, int64_t K, Planar x,
                        const float *X, int64_t M, float *Y, bool pdl, cudaStream_t s) {
    return launch_gemv(wt, single_mat(Wp, N, Y), K, x, X, M, pdl, s);
}

}  // namespace qmm
