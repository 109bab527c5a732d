// w4a16.cu -- the W4A16 group-asymmetric path of page 3 ("BitBLAS 完全拆解",
// "从数学表达式到真实存储" and "位级打包"):
//   C[m, n] = sum_k A[m, k] * s[n, g] * (q[n, k] - z[n, g]),  g = k / G,
// with A and C fp16, q 4-bit codes (8 per uint32 word, element 8c + i in
// bits 4i of word c), s fp16 and z uint8 per (row, group).
//
// Layout (qmm_repack_weights, QMM_TYPE_W4A16): the same words, with the
// nibbles of each word interleaved -- even elements in the low 16 bits,
// odd ones in the high 16 bits (slots 0..7 hold elements 0,2,4,6,1,3,5,7).
// One lop3 then turns a word into fp16 pairs (k, k+1) laid out exactly as
// the tensor-core operands want them (page 3, "Ladder": lay the bits out
// offline for the decoder), so neither kernel permutes the activations.
//
// Decode (M <= 16): mma.sync m16n8k16, weights as the A operand (16 rows per
// warp), tokens as B (8 per MMA). q - z is exact in fp16 (1024 + q minus
// 1024 + z, or the x16 form through one fp16 FMA), the products are exact in
// the fp32 accumulator, and each 128-element step of a group is scaled by s
// in fp32. Weight and activation words stream from global memory with
// one step of register prefetch; eight warps split K, then reduce.
#include "qmm_internal.cuh"

namespace qmm {
namespace {

constexpr int kStepK = 128;  // elements per warp step (16 words per row)
constexpr int kDecodeWarps = 8;
constexpr int kDecodeThreads = kDecodeWarps * 32;
constexpr int kRowsPerCta = 16;

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
    const uint32_t a = 0x6400u | z;  // fp16 1024 + z (z <= 15)
    const __half h = __float2half_rn(-64.0f - (float)z);
    const uint32_t b = (uint32_t)__half_as_ushort(h);
    return Zero2{a | (a << 16), b | (b << 16)};
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

__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

struct DecodeArgs {
    const uint32_t *W;  // packed [N][K/8]
    const __half *S;    // [N][K/G]
    const uint8_t *Z;   // [N][K/G]
    const __half *A;    // [M][K]
    __half *C;          // [M][N]
    int64_t M, N, K, G;
};

// One step's operands for one thread: its 4 words of rows r0 and r1, the
// scale and zero of each row for the step's group, and its 32 activation
// elements of tokens t/4 (+8 for the second N tile).
template <int NT>
struct StepRegs {
    uint4 w0, w1;
    __half s0, s1;
    uint8_t z0, z1;
    uint4 x[NT][4];
};

template <int NT>
__device__ __forceinline__ void load_step(const DecodeArgs &a, int64_t st, int64_t r0, int64_t r1,
                                          int j, int tok, StepRegs<NT> &R) {
    const int64_t kw = a.K / 8, ng = a.K / a.G;
    const int64_t g = st * kStepK / a.G;
    const int64_t word = st * (kStepK / 8) + 4 * j;
    R.w0 = r0 < a.N ? ldg_nc128(a.W + r0 * kw + word) : make_uint4(0, 0, 0, 0);
    R.w1 = r1 < a.N ? ldg_nc128(a.W + r1 * kw + word) : make_uint4(0, 0, 0, 0);
    R.s0 = r0 < a.N ? a.S[r0 * ng + g] : __float2half_rn(0.0f);
    R.s1 = r1 < a.N ? a.S[r1 * ng + g] : __float2half_rn(0.0f);
    R.z0 = r0 < a.N ? a.Z[r0 * ng + g] : 0;
    R.z1 = r1 < a.N ? a.Z[r1 * ng + g] : 0;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int64_t m = nt * 8 + tok;
        const __half *xp = a.A + m * a.K + st * kStepK + 32 * j;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            R.x[nt][q] = m < a.M ? ldg_nc128(xp + 8 * q) : make_uint4(0, 0, 0, 0);
    }
}

template <int NT>
__global__ void __launch_bounds__(kDecodeThreads, 2) w4a16_decode_kernel(const DecodeArgs a) {
    __shared__ float red[kDecodeWarps][NT][4][32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = lane & 3, tok = lane >> 2;
    const int64_t n0 = (int64_t)blockIdx.x * kRowsPerCta;
    const int64_t r0 = n0 + tok, r1 = n0 + tok + 8;
    const int64_t nsteps = a.K / kStepK;
    float tot[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) tot[nt][i] = 0.0f;

    StepRegs<NT> cur, nxt;
    int64_t st = warp;
    if (st < nsteps) load_step<NT>(a, st, r0, r1, j, tok, cur);
    for (; st < nsteps; st += kDecodeWarps) {
        if (st + kDecodeWarps < nsteps) load_step<NT>(a, st + kDecodeWarps, r0, r1, j, tok, nxt);
        const Zero2 z0 = make_zero2(cur.z0), z1 = make_zero2(cur.z1);
        const uint32_t w0[4] = {cur.w0.x, cur.w0.y, cur.w0.z, cur.w0.w};
        const uint32_t w1[4] = {cur.w1.x, cur.w1.y, cur.w1.z, cur.w1.w};
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
            // (q - z) pairs of row r0 (u*) and row r1 (v*) for this word
            uint32_t u01, u23, u45, u67, v01, v23, v45, v67;
            dequant_word(w0[wi], z0, u01, u23, u45, u67);
            dequant_word(w1[wi], z1, v01, v23, v45, v67);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint32_t xs[4] = {cur.x[nt][wi].x, cur.x[nt][wi].y, cur.x[nt][wi].z,
                                        cur.x[nt][wi].w};
                // MMA 2wi takes elements 8wi + 0..3 of each thread's 32 as the
                // fragment columns 2j, 2j+1, 2j+8, 2j+9; MMA 2wi + 1 elements
                // 8wi + 4..7. A (rows r0, r1) and B (token t/4) agree, so the
                // sum over the step is unchanged.
                mma_16816(acc[nt], u01, v01, u23, v23, xs[0], xs[1]);
                mma_16816(acc[nt], u45, v45, u67, v67, xs[2], xs[3]);
            }
        }
        const float s0 = __half2float(cur.s0), s1 = __half2float(cur.s1);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            tot[nt][0] = fmaf(s0, acc[nt][0], tot[nt][0]);
            tot[nt][1] = fmaf(s0, acc[nt][1], tot[nt][1]);
            tot[nt][2] = fmaf(s1, acc[nt][2], tot[nt][2]);
            tot[nt][3] = fmaf(s1, acc[nt][3], tot[nt][3]);
        }
        cur = nxt;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) red[warp][nt][i][lane] = tot[nt][i];
    __syncthreads();
    if (warp < NT) {
        const int nt = warp;
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < kDecodeWarps; ++w) sum += red[w][nt][i][lane];
            v[i] = sum;
        }
        // c0, c1: row t/4, tokens 2j, 2j+1; c2, c3: row t/4 + 8, same tokens
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t n = (i < 2) ? r0 : r1;
            const int64_t m = nt * 8 + 2 * j + (i & 1);
            if (n < a.N && m < a.M) a.C[m * a.N + n] = __float2half_rn(v[i]);
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
__global__ void w4a16_repack_kernel(const uint32_t *__restrict__ src, uint32_t *__restrict__ dst,
                                    int64_t nwords, bool inverse) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nwords;
         i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = inverse ? unpack_word(src[i]) : pack_word(src[i]);
}

}  // namespace

cudaError_t launch_w4a16_repack(bool inverse, const void *src, void *dst, int64_t N, int64_t K,
                                cudaStream_t s) {
    const int64_t nwords = N * (K / 8);
    int64_t grid = (nwords + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    w4a16_repack_kernel<<<(int)grid, 256, 0, s>>>(static_cast<const uint32_t *>(src),
                                                  static_cast<uint32_t *>(dst), nwords, inverse);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_w4a16_decode(const void *W, const __half *S, const uint8_t *Z, int64_t G,
                                const __half *A, __half *C, int64_t M, int64_t N, int64_t K,
                                cudaStream_t s) {
    DecodeArgs a;
    a.W = static_cast<const uint32_t *>(W);
    a.S = S;
    a.Z = Z;
    a.A = A;
    a.C = C;
    a.M = M;
    a.N = N;
    a.K = K;
    a.G = G;
    const unsigned grid = (unsigned)((N + kRowsPerCta - 1) / kRowsPerCta);
    if (M <= 8)
        w4a16_decode_kernel<1><<<grid, kDecodeThreads, 0, s>>>(a);
    else
        w4a16_decode_kernel<2><<<grid, kDecodeThreads, 0, s>>>(a);
    count_launch();
    return cudaGetLastError();
}

}  // namespace qmm
