// qmm_internal.cuh -- device helpers and private layouts shared by the
// libqmm translation units (never by the CPU oracle).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qmm.h"

namespace qmm {

// ------------------------------------------------------------------ formats
constexpr int QK4_0 = 32;   // elements per Q4_0 / Q8_0 block
constexpr int QK_K = 256;   // elements per Q4_K / Q8_K super-block
constexpr int B_Q4_0 = 18;  // canonical bytes per block (page 1 block layouts)
constexpr int B_Q8_0 = 34;
constexpr int B_Q4_K = 144;
constexpr int B_Q8_K = 292;
constexpr int B_Q6_K = 210;  // ql[128] qh[64] int8 scales[16] fp16 d

// Packed weight layout: rows grouped in tiles of kTileRows. Within a tile,
// the blocks of one K position are adjacent, so a (tile, K-range) is one
// contiguous byte range that a single bulk copy moves:
//   Q4_K: tile t = [nsb][kTileRows][144 B]   (canonical block bytes, except
//         the 12 scale bytes, see k4_header_to_packed)
//   Q4_0: tile t = [kTileRows][nb][16 B nibbles] then [nb][kTileRows] fp16 d
//         (a (tile, K-range) is then 8 row segments plus one scale segment)
//   Q6_K: tile t = [nsb] records of kQ6Rec = 8 x 210 B:
//         [8 rows][192 B codes] [8 rows][16 B scales] [8 rows] fp16 d.
//         Codes of a row: the canonical ql (bytes 16t.. serve GEMV lane t),
//         then per lane t two words of high bits (q6k_* below); the scales
//         re-ordered so lane t's two are bytes 2t, 2t + 1.
constexpr int kTileRows = 8;
constexpr int kQ6Codes = 192;                            // ql 128 B + qh 64 B per row
constexpr int kQ6ScOff = kTileRows * kQ6Codes;           // 1536
constexpr int kQ6DOff = kQ6ScOff + kTileRows * 16;       // 1664
constexpr int kQ6Rec = kQ6DOff + kTileRows * 2;          // 1680 = 8 x 210
static_assert(kQ6Rec == kTileRows * B_Q6_K && kQ6Rec % 16 == 0, "Q6_K record");

// Q6_K lane geometry, shared by the repack and the GEMV. Lane t (0..7) of a
// row reads ql bytes 16t + i (i < 16): with c = t / 2, h = t % 2, the low
// nibbles are elements 64c + 16h + i (group 4c + h) and the high nibbles
// elements 64c + 32 + 16h + i (group 4c + 2 + h) -- the Q8_K planar order.
// Its high-bit word for either set holds element i's 2 bits at bit
// 8 (i % 4) + 2 (i / 4), so (word >> 2w) & 0x03030303 lines them up with
// the 4 code bytes of ql word w.
__host__ __device__ inline int q6k_elem(int t, int hi, int i) {
    return 64 * (t >> 1) + 32 * hi + 16 * (t & 1) + i;
}
__host__ __device__ inline int q6k_hbit_pos(int i) { return 8 * (i & 3) + 2 * (i >> 2); }
// The stored 6-bit codes u (0..63) of ql word w of a lane (its 4 bytes' low
// nibbles, or the high nibbles after a shift by 4) as 4 bytes.
__host__ __device__ inline uint32_t q6k_u(uint32_t nib, uint32_t hbits, int w) {
    return (nib & 0x0F0F0F0Fu) | (((hbits >> (2 * w)) & 0x03030303u) << 4);
}

__host__ __device__ inline int64_t tiles_of(int64_t N) { return (N + kTileRows - 1) / kTileRows; }

// Private quantized-activation layout ("planar"), written by the quantizer
// for the mul_mat kernels:
//   qs   : int8  [M][K]          codes, rows 16-byte aligned (K % 32 == 0).
//                                Q8_0: natural order. Q8_K: each super-block's
//                                256 codes permuted for the GEMV lanes (see
//                                q8K_code_offset): bytes 16t..16t+15 hold
//                                elements 64c + 16h + 0..15 and bytes
//                                128 + 16t .. hold 64c + 32 + 16h + 0..15,
//                                with c = t / 2, h = t % 2 (t = 0..7).
//   d    : float [M][K/QK]       block scales (Q8_0: the fp16 scale widened)
//   sums : int16 [M][K/QK][G]    Q8_K: G = 16 sums of 16 codes (bsums),
//                                stored as 8 words, word t = bs[4c + h] in
//                                the low and bs[4c + 2 + h] in the high half;
//                                Q8_0: G = 1, the sum of the block's 32 codes
struct Planar {
    int8_t *qs;
    float *d;
    int16_t *sums;
};

// Weight matrices that share K and the activations X of one decode launch
// (a layer's q/k/v or gate/up projections): Y_i = X W_i^T. Their work units
// (tile pairs for Q4_K, tiles for Q4_0) are numbered one after another:
// matrix i owns units off[i] .. off[i+1]-1.
constexpr int kMaxMats = 8;
struct MatSet {
    int n;
    const uint8_t *W[kMaxMats];
    float *Y[kMaxMats];
    int64_t N[kMaxMats];
    int64_t off[kMaxMats + 1];
};
__host__ __device__ __forceinline__ int mat_of(const MatSet &s, int64_t unit) {
    int i = 0;
    while (i + 1 < s.n && unit >= s.off[i + 1]) ++i;
    return i;
}

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Tokens per call from which mul_mat runs the tensor-core GEMM; below, every
// format has a tensor-core GEMV from 2 tokens on (4096 x 4096, measured: the
// Q4_0 / Q6_K GEMVs take 10.8 / 11.0 us at 12 tokens and 11.7 / 12.2 at 16,
// the split-K GEMM 18.9 / 21.6 and 16.8 / 18.2).
constexpr int64_t kGemmMinM = 17;

// Workspace carve-up for M rows of K activations with block size qk.
__host__ __device__ inline size_t planar_bytes(int64_t M, int64_t K, int qk, Planar *p,
                                               uint8_t *base) {
    const int64_t nb = K / qk;
    const int g = qk == QK_K ? 16 : 1;
    size_t off = 0;
    size_t o_qs = off;
    off = align_up(off + (size_t)M * K, 256);
    size_t o_d = off;
    off = align_up(off + (size_t)M * nb * sizeof(float), 256);
    size_t o_s = off;
    off = align_up(off + (size_t)M * nb * g * sizeof(int16_t), 256);
    off += 256;  // slack: bulk copies round their sizes up to 16 bytes
    if (p) {
        p->qs = (int8_t *)(base + o_qs);
        p->d = (float *)(base + o_d);
        p->sums = (int16_t *)(base + o_s);
    }
    return off;
}

// Q4_K block header (first 16 bytes: fp16 d, fp16 dmin, 12 bytes of scales).
// Canonical scale bytes follow the page's 6-bit packing ("6-bit 参数是怎么塞进
// 12 字节的"). The packed layout keeps the same 96 bits of information in an
// order one GEMV lane can read in a few operations: four 24-bit fields, field
// c at bit 24c of the little-endian 96-bit value, each
//   s_{2c} | m_{2c} << 6 | s_{2c+1} << 12 | m_{2c+1} << 18.
__host__ __device__ inline void k4_scales_canonical(const uint4 &h, int s[8], int m[8]) {
    uint8_t q[12];
    for (int i = 0; i < 4; ++i) {
        q[i] = (uint8_t)(h.y >> (8 * i));
        q[4 + i] = (uint8_t)(h.z >> (8 * i));
        q[8 + i] = (uint8_t)(h.w >> (8 * i));
    }
    for (int j = 0; j < 8; ++j) {
        if (j < 4) {
            s[j] = q[j] & 63;
            m[j] = q[j + 4] & 63;
        } else {
            s[j] = (q[j + 4] & 0x0F) | ((q[j - 4] >> 6) << 4);
            m[j] = (q[j + 4] >> 4) | ((q[j] >> 6) << 4);
        }
    }
}

__host__ __device__ inline uint4 k4_header_to_packed(const uint4 &h) {
    int s[8], m[8];
    k4_scales_canonical(h, s, m);
    uint64_t lo = 0;
    uint32_t hi = 0;
    for (int c = 0; c < 4; ++c) {
        const uint64_t f = (uint64_t)(s[2 * c] | (m[2 * c] << 6) | (s[2 * c + 1] << 12) |
                                      (m[2 * c + 1] << 18));
        if (c < 2) {
            lo |= f << (24 * c);
        } else if (c == 2) {
            lo |= f << 48;
            hi |= (uint32_t)(f >> 16);
        } else {
            hi |= (uint32_t)(f << 8);
        }
    }
    return make_uint4(h.x, (uint32_t)lo, (uint32_t)(lo >> 32), hi);
}

// Field c (24 bits) of a packed header; w1..w3 are its scale words.
__host__ __device__ __forceinline__ uint32_t k4_field(uint32_t w1, uint32_t w2, uint32_t w3, int c) {
    const uint64_t v = c < 2 ? ((uint64_t)w2 << 32 | w1) : ((uint64_t)w3 << 32 | w2);
    const int sh = c < 2 ? 24 * c : 24 * c - 32;
    return (uint32_t)(v >> sh) & 0xFFFFFFu;
}

__host__ __device__ inline uint4 k4_header_to_canonical(const uint4 &h) {
    uint8_t q[12] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
    for (int c = 0; c < 4; ++c) {
        const uint32_t f = k4_field(h.y, h.z, h.w, c);
        const int sv[2] = {(int)(f & 63), (int)((f >> 12) & 63)};
        const int mv[2] = {(int)((f >> 6) & 63), (int)((f >> 18) & 63)};
        for (int e = 0; e < 2; ++e) {
            const int j = 2 * c + e;
            if (j < 4) {
                q[j] |= (uint8_t)sv[e];
                q[j + 4] |= (uint8_t)mv[e];
            } else {
                q[j + 4] = (uint8_t)((sv[e] & 15) | ((mv[e] & 15) << 4));
                q[j - 4] |= (uint8_t)((sv[e] >> 4) << 6);
                q[j] |= (uint8_t)((mv[e] >> 4) << 6);
            }
        }
    }
    uint4 o;
    o.x = h.x;
    o.y = q[0] | (q[1] << 8) | (q[2] << 16) | ((uint32_t)q[3] << 24);
    o.z = q[4] | (q[5] << 8) | (q[6] << 16) | ((uint32_t)q[7] << 24);
    o.w = q[8] | (q[9] << 8) | (q[10] << 16) | ((uint32_t)q[11] << 24);
    return o;
}

// ------------------------------------------------------------------ errors
// Device error word bits (read and cleared by qmm_check_device_error).
constexpr unsigned kDevErrTimeout = 1u;

// A bounded wait gives up after this many SM clock cycles (about 2 s).
constexpr long long kWaitTimeoutCycles = 4000000000LL;

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete. Returns
// false (and records a timeout in *err) if it has not after the bound.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, unsigned *err,
                                              long long limit_cycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit_cycles) {
            atomicOr(err, kDevErrTimeout);
            return false;
        }
    }
    return true;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned *err) {
    return mbar_wait_for(bar, parity, err, kWaitTimeoutCycles);
}
// The same wait by every lane of a warp, with one answer for the whole warp:
// warps that go on to warp-collective tcgen05 loads or stores must agree.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, unsigned *err) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, err));
}

// 1-D bulk async copy global -> shared, completing on an mbarrier.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue / wait for the previous kernel's memory to be visible.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint4 ldg_nc128(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Round half away from zero in fp32 without contraction: sign(v) floor(|v| + 0.5).
__device__ __forceinline__ float round_half_away(float v) {
    return v < 0.0f ? -floorf(__fadd_rn(-v, 0.5f)) : floorf(__fadd_rn(v, 0.5f));
}

__device__ __forceinline__ int clampi(int v, int lo, int hi) { return min(max(v, lo), hi); }

// floor(a + 0.5) for 0 <= a < 2^22 without a float-to-integer conversion
// (those run on the narrow conversion pipe): a + 0.5 rounded to nearest, then
// 2^23 added with rounding toward zero leaves the integer part in the low
// mantissa bits. The same value as round_half_away's floor for such a.
__device__ __forceinline__ int floor_half_up(float a) {
    return __float_as_int(__fadd_rz(__fadd_rn(a, 0.5f), 8388608.0f)) - 0x4B000000;
}

// n with the sign of p (the sign bit as a mask; n = 0 gives 0 for p = -0).
__device__ __forceinline__ int with_sign_of(int n, float p) {
    const int s = __float_as_int(p) >> 31;
    return (n ^ s) - s;
}

// (int)round_half_away(p) for |p| < 2^22.
__device__ __forceinline__ int round_half_away_int(float p) {
    return with_sign_of(floor_half_up(fabsf(p)), p);
}

// An integer |v| < 2^22 as fp32 without a conversion: 1.5 * 2^23 + v has v
// in its low mantissa bits; subtracting 1.5 * 2^23 is exact.
__device__ __forceinline__ float int_as_exact_float(int v) {
    return __int_as_float(0x4B400000 + v) - 12582912.0f;
}

// An integer |v| < 2^10 as fp16 bits without a conversion: 1152 + v lies in
// [1024, 2048), where fp16 holds every integer, so its bits are 0x6480 + v.
// Subtracting 1152 (0x6480) in fp16 afterwards is exact.
__device__ __forceinline__ uint32_t biased_half_bits(int v) { return (uint32_t)(0x6480 + v); }

// ------------------------------------------------------------------ stream-K
// The tensor-core GEMMs run a grid of G CTAs over units u = tile * nsb +
// k-round (U units), CTA c taking [c U / G, (c+1) U / G). With at most as
// many tiles as SMs, G = tiles: one whole tile per CTA. With more, G = the
// SM count and a tile may span several CTAs: each CTA that holds only part of
// it writes that piece to its partial slot (slot 0 when the tile is the
// CTA's first, 1 when its last), and the fixup kernel (streamk.cu) adds the
// pieces in CTA order and writes the tile. A tile is 128 weight rows by
// gemm_tile_cols(wt, M) tokens: 256 above 128 tokens (every decoded weight
// then serves 256 tokens), else 128; Q4_0, whose weights decode in a few fp16
// instructions, measured faster at 128 whatever M.
constexpr int kSkTile = 128;   // tile rows
constexpr int kSkRound = 256;  // K elements per unit
constexpr int kSkColsMax = 256;
__host__ __device__ inline int gemm_tile_cols(int wt, int64_t M) {
    return wt != QMM_TYPE_Q4_0 && M > 128 ? 256 : 128;
}

// The CTA whose range holds unit u.
__host__ __device__ __forceinline__ int64_t sk_cta_of(int64_t u, int64_t U, int64_t G) {
    return ((u + 1) * G - 1) / U;
}
// Float offset of CTA c's slot for `tile` in the partial area
// [G][2][cols][128 rows] (a column's 128 rows contiguous), cols the tile's.
__host__ __device__ __forceinline__ int64_t sk_slot(int64_t c, int64_t tile, int64_t U, int64_t G,
                                                    int64_t nsb, int cols) {
    return (c * 2 + ((c * U / G) / nsb == tile ? 0 : 1)) * (int64_t)(kSkTile * cols);
}

// ------------------------------------------------------------------ activation quantization
// Shared by the stand-alone quantizer kernels and the quantizer fused into the
// GEMV prologue, so both produce identical codes. Page 1 ("最基础的两块",
// "更低的比特"): symmetric int8 per block, d = amax / 127, q = round-half-away
// of x * (1/d) clamped to +-127, in IEEE fp32 with explicit rounding.

__device__ __forceinline__ float warp_max_nonneg(float v) {
    // v >= +0 (no -0, no NaN): the IEEE bit patterns order like the values
    return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
}

// clamp(round_half_away(x id), -127, 127); min(|p|, 255) keeps floor_half_up
// in range. Equal to the conversion form for every non-NaN p.
__device__ __forceinline__ int q8_code(float x, float id) {
    const float p = __fmul_rn(x, id);
    return with_sign_of(min(floor_half_up(fminf(fabsf(p), 255.0f)), 127), p);
}

// Q8_0 block held one element per lane: code, scale (fp32 value of the fp16
// scale that is stored), and the block's code sum (all lanes).
__device__ __forceinline__ void q8_0_warp(float x, int &q, __half &dh, int &sum) {
    const float amax = warp_max_nonneg(fabsf(x));
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
    q = q8_code(x, id);
    dh = __float2half_rn(d);
    sum = __reduce_add_sync(0xffffffffu, q);
}

// Q8_0 block held 8 elements per lane by four consecutive lanes (lane l:
// elements 8 (l % 4) .. 8 (l % 4) + 7 of the warp's block l / 4), so a warp
// quantizes eight blocks at once: the arithmetic of q8_0_warp, the codes
// packed little-endian in (lo, hi), the block's code sum on all four lanes.
__device__ __forceinline__ void q8_0_quad(const float v[8], uint32_t &lo, uint32_t &hi, __half &dh,
                                          int &sum) {
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    const float amax = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
    int q[8], s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        q[i] = q8_code(v[i], id);
        s += q[i];
    }
    lo = __byte_perm(__byte_perm(q[0], q[1], 0x0040), __byte_perm(q[2], q[3], 0x0040), 0x5410);
    hi = __byte_perm(__byte_perm(q[4], q[5], 0x0040), __byte_perm(q[6], q[7], 0x0040), 0x5410);
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    sum = s + __shfl_xor_sync(0xffffffffu, s, 2);
    dh = __float2half_rn(d);
}

// Q8_K super-block held 8 elements per lane (lane l: elements 8l .. 8l+7):
// the lane's codes packed little-endian in (lo, hi), the fp32 scale d, and
// the sum of codes 16 (l/2) .. 16 (l/2) + 15 (valid on every lane).
__device__ __forceinline__ void q8_K_warp(const float v[8], uint32_t &lo, uint32_t &hi, float &d,
                                          int &bsum) {
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
    const float amax = warp_max_nonneg(a);
    d = __fdiv_rn(amax, 127.0f);
    const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
    // |x| <= amax, so |x * id| <= 127 (1 + 2^-23)^3 < 127.5: the clamp to
    // +-127 of q8_code never acts here and is left out
    int q[8], s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        q[i] = round_half_away_int(__fmul_rn(v[i], id));
        s += q[i];
    }
    // low bytes of q[0..3] and q[4..7], little-endian
    lo = __byte_perm(__byte_perm(q[0], q[1], 0x0040), __byte_perm(q[2], q[3], 0x0040), 0x5410);
    hi = __byte_perm(__byte_perm(q[4], q[5], 0x0040), __byte_perm(q[6], q[7], 0x0040), 0x5410);
    bsum = s + __shfl_xor_sync(0xffffffffu, s, 1);
}

// Byte offset, inside the planar layout's 256-byte super-block, of the 8 codes
// lane l computed (elements 8l .. 8l+7).
__host__ __device__ __forceinline__ int q8K_code_offset(int lane) {
    const int c = lane >> 3, j = lane & 7;
    const int part = j >> 2, rr = (j & 3) * 8;
    return part * 128 + 16 * (2 * c + (rr >> 4)) + (rr & 15);
}

// Byte offset, inside the planar layout's 32-byte bsum group, of bsum b.
__host__ __device__ __forceinline__ int q8K_bsum_offset(int b) {
    const int c = b >> 2, w = b & 3;
    return 4 * (2 * c + (w & 1)) + 2 * (w >> 1);
}

}  // namespace qmm

// ------------------------------------------------------------------ host side
namespace qmm {
struct Launch;
// Defined in api.cu.
unsigned *device_error_word();           // device pointer for the current device
// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (kernel, device)
cudaError_t ensure_smem_attr(const void *kernel, int bytes);
int sm_count();                          // SMs of the current device
void count_launch(unsigned n = 1);       // bump the launch counter
qmm_status set_error(qmm_status s, const char *fmt, ...);

// Kernel launchers (each .cu file); all return cudaSuccess or the launch error.
// Grid for `units` equal work items on at most `cap` CTAs that each take a
// contiguous range: the fewest items per CTA the cap allows, then the fewest
// CTAs with that many, so that no CTA has more items than another by more
// than one and the grid is not padded with CTAs that hold fewer. (A memory-
// bound kernel finishes when its busiest CTA does.)
inline int64_t balanced_grid(int64_t units, int64_t cap) {
    if (units <= 0) return 1;
    const int64_t per = (units + cap - 1) / cap;
    return (units + per - 1) / per;
}

cudaError_t launch_quantize_q8(qmm_type vt, bool planar, const float *X, void *out, Planar p,
                               int64_t M, int64_t K, cudaStream_t s);
cudaError_t launch_quantize_weights(qmm_type wt, const float *W, void *Wq, int64_t N, int64_t K,
                                    cudaStream_t s);
// Canonical Q8 blocks (qmm_mul_mat_q8) into each private activation layout:
// planar (scalar GEMV), image (tensor-core GEMV), the fp16 prefill operands.
cudaError_t launch_import_q8_planar(qmm_type vt, const void *Xq, Planar p, int64_t M, int64_t K,
                                    cudaStream_t s);
cudaError_t launch_import_mma_image(const void *Xq, void *img, int64_t M, int64_t K, cudaStream_t s);
cudaError_t launch_import_q4_0_prefill(const void *Xq, void *ws, int64_t M, int64_t K,
                                       cudaStream_t s);
cudaError_t launch_repack(qmm_type wt, bool inverse, const void *src, void *dst, int64_t N,
                          int64_t K, cudaStream_t s);
// X != nullptr: fused quantizer (requires gemv_can_fuse(wt, M, K)). The
// MatSet form runs all its matrices in one launch (n, W, Y, N filled by the
// caller; off is computed here).
cudaError_t launch_gemv(qmm_type wt, MatSet ms, int64_t K, Planar x, const float *X, int64_t M,
                        bool pdl, cudaStream_t s);
cudaError_t launch_gemv(qmm_type wt, const void *Wp, int64_t N, int64_t K, Planar x,
                        const float *X, int64_t M, float *Y, bool pdl, cudaStream_t s);
MatSet single_mat(const void *Wp, int64_t N, float *Y);
bool gemv_can_fuse(qmm_type wt, int64_t M, int64_t K);
// Tensor-core decode GEMV for Q4_K (gemv_mma.cu): used from kMmaMinM tokens
// on while one token's activations fit its shared memory
// (gemv_mma_max_tokens(K) >= 1). Up to kMmaFuseElems activation elements per
// call it quantizes inside the kernel; beyond, launch_quantize_mma_image
// writes the activation images (gemv_mma_image_bytes) into the workspace.
constexpr int64_t kMmaMinM = 2;
constexpr int64_t kMmaFuseElems = 8192;
int gemv_mma_max_tokens(int64_t K);
bool gemv_use_mma(qmm_type wt, int64_t M, int64_t K);
size_t gemv_mma_image_bytes(int64_t M, int64_t K);
cudaError_t launch_quantize_mma_image(const float *X, void *img, int64_t M, int64_t K,
                                      cudaStream_t s);
cudaError_t launch_gemv_mma_q4_K(MatSet ms, int64_t K, const float *X, const void *img, int64_t M,
                                 bool pdl, cudaStream_t s);
// Tensor-core decode GEMV for Q6_K and Q4_0 (gemv_mma6.cu), from kMmaMinM
// tokens on where K is a multiple of 256 and one token's activations fit its
// shared memory; its activations are always an image written ahead of it.
int gemv_mma6_max_tokens(qmm_type wt, int64_t K);
size_t gemv_mma6_image_bytes(qmm_type wt, int64_t M, int64_t K);
cudaError_t launch_image6(qmm_type wt, bool import, const void *src, void *img, int64_t M, int64_t K,
                          cudaStream_t s);
cudaError_t launch_gemv_mma6(qmm_type wt, MatSet ms, int64_t K, const void *img, int64_t M, bool pdl,
                             cudaStream_t s);
// The tensor-core decode path of any format (gemv_use_mma): the image bytes
// for M tokens; the image from fp32 X (import = false) or from canonical Q8
// blocks (import = true); the GEMV over the image.
size_t mma_image_bytes(qmm_type wt, int64_t M, int64_t K);
cudaError_t launch_mma_image(qmm_type wt, bool import, const void *src, void *img, int64_t M, int64_t K,
                             cudaStream_t s);
cudaError_t launch_gemv_mma(qmm_type wt, MatSet ms, int64_t K, const void *img, int64_t M, bool pdl,
                            cudaStream_t s);
// W4A16: nibble interleave of the packed layout (or its inverse), the decode
// kernel (M <= 16) and the tensor-core GEMM (M > 16).
cudaError_t launch_w4a16_repack(bool inverse, const void *src, void *dst, int64_t N, int64_t K,
                                cudaStream_t s);
// Prefill workspace (every weight type): the activations as fp16(2^e d_a y)
// [M][K] (Q8 codes y, block scale d_a, a power of two 2^e per token), then
// 2^-e per token, fp32, padded with 1.0 to a multiple of 16 tokens.
size_t prefill_operand_bytes(int64_t M, int64_t K);
// Q4_K and Q6_K prefill: the operand from Q8_K codes in natural order, from
// fp32 X or from canonical Q8_K blocks, then the fp16-operand GEMM.
cudaError_t launch_quantize_q8_K_f16(const float *X, void *ws, int64_t M, int64_t K, cudaStream_t s);
cudaError_t launch_import_q8_K_f16(const void *Xq, void *ws, int64_t M, int64_t K, cudaStream_t s);
cudaError_t launch_gemm_q6_K(const void *Wp, int64_t N, int64_t K, const void *ws, float *part, int64_t M,
                             float *Y, cudaStream_t s);
cudaError_t launch_gemm_q4_K_f16(const void *Wp, int64_t N, int64_t K, const void *ws, float *part,
                                 int64_t M, float *Y, cudaStream_t s);
// lut == nullptr: W-hat = s (q - z); otherwise W-hat = s LUT(q) (Z unused).
cudaError_t launch_w4a16_decode(const void *W, const __half *S, const uint8_t *Z, const __half *lut,
                                int64_t G, const __half *A, __half *C, int64_t M, int64_t N, int64_t K,
                                cudaStream_t s);
cudaError_t launch_w4a16_gemm(const void *W, const __half *S, const uint8_t *Z, const __half *lut,
                              int64_t G, const __half *A, __half *C, int64_t M, int64_t N, int64_t K,
                              float *part, cudaStream_t s);
cudaError_t launch_w4a16_unpack_zeros(const uint32_t *zp, uint8_t *z, int64_t N, int64_t ng,
                                      cudaStream_t s);
// Q4_0 prefill (M > 8): the operand from Q8_0 codes, each 32-block permuted
// for the converter, then the fp16-operand tensor-core GEMM.
cudaError_t launch_quantize_q4_0_prefill(const float *X, void *ws, int64_t M, int64_t K,
                                         cudaStream_t s);
cudaError_t launch_gemm_q4_0(const void *Wp, int64_t N, int64_t K, const void *ws, float *part,
                             int64_t M, float *Y, cudaStream_t s);
cudaError_t launch_debug_block_sums(qmm_type wt, const void *Wp, int64_t N, int64_t K,
                                    const void *Xq, int64_t M, int32_t *out, cudaStream_t s);
cudaError_t launch_debug_wait_timeout(int64_t limit_cycles, cudaStream_t s);
// Tensor-core throughput microbenchmark `which` (qmm_peak_kind); *ops = the
// multiply-add operations (2 per MAC) the launch performs.
cudaError_t launch_debug_peak(int which, int64_t iters, cudaStream_t s, double *ops);
// Stream-K GEMMs (streamk.cu): CTAs for `tiles` tiles of `units` units (the
// SM count above it, one per tile from half of it, else split K over up to
// the SM count); bytes of the partial area (enough for either tile width);
// the fixup that adds the split tiles' pieces into C (fp32, or fp16 when
// half_out), launched only when G != tiles.
int64_t stream_k_grid(int64_t tiles, int64_t units);
size_t stream_k_part_bytes();
// Whether an N x M output of depth K (128 x gemm_tile_cols(wt, M) tiles,
// 256-element units) of weight type wt runs split tiles, i.e. needs the
// partial area.
bool stream_k_splits(int wt, int64_t N, int64_t M, int64_t K);
cudaError_t launch_stream_k_fixup(const float *part, void *C, bool half_out, int cols, int64_t N, int64_t M,
                                  int64_t mblocks, int64_t nsb, int64_t units, int64_t G,
                                  cudaStream_t s);
}  // namespace qmm
