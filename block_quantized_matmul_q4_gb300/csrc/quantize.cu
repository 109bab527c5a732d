// quantize.cu -- block quantizers on the GPU.
//
//  * Activations fp32 -> Q8_0 / Q8_K (page 1, "最基础的两块: Q4_0 与 Q8_0",
//    "更低的比特" for block_q8_K and its bsums, mul_mat step 1 "激活得先变成
//    Q8_K"): symmetric int8 per block, d = amax / 127, q = round-half-away of
//    x * (1/d), clamp to +-127. Output either in the canonical block bytes or
//    in the private planar layout the mul_mat kernels read.
//  * Weights fp32 -> Q4_0 / Q4_K (page 1 Q4_0 and K-quant sections, the
//    6-bit packing section and the nibble packing loop in "正确性").
//
// Every step that decides an integer code is done in IEEE fp32 with explicit
// round-to-nearest intrinsics (no contraction), in the order the formulas
// state, so the codes are bit-identical to any other IEEE fp32 evaluation of
// the same formulas.
#include "qmm_internal.cuh"

namespace qmm {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float group_min(float v, int width) {
    for (int o = 1; o < width; o <<= 1) v = fminf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}
__device__ __forceinline__ float group_max(float v, int width) {
    for (int o = 1; o < width; o <<= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

// ---------------------------------------------------------------- Q8_0
// One warp per 32-element block; lane i holds element i.
template <bool kPlanar>
__global__ void __launch_bounds__(256) quantize_q8_0_kernel(const float *__restrict__ X,
                                                            uint8_t *__restrict__ out, Planar p,
                                                            int64_t nblocks) {
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < nblocks;
         b += nwarps) {
        const float x = X[b * 32 + lane];
        int q, s;
        __half dh;
        q8_0_warp(x, q, dh, s);
        if (kPlanar) {
            p.qs[b * 32 + lane] = (int8_t)q;
            if (lane == 0) {
                p.d[b] = __half2float(dh);
                p.sums[b] = (int16_t)s;
            }
        } else {
            uint8_t *blk = out + b * B_Q8_0;
            blk[2 + lane] = (uint8_t)(int8_t)q;
            if (lane == 0) *reinterpret_cast<__half *>(blk) = dh;
        }
    }
}

// ---------------------------------------------------------------- Q8_K
// One warp per 256-element block; lane l holds elements 8l .. 8l+7.
template <bool kPlanar>
__global__ void __launch_bounds__(256) quantize_q8_K_kernel(const float *__restrict__ X,
                                                            uint8_t *__restrict__ out, Planar p,
                                                            int64_t nblocks) {
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < nblocks;
         b += nwarps) {
        const float4 *src = reinterpret_cast<const float4 *>(X + b * 256 + 8 * lane);
        const float4 v0 = src[0], v1 = src[1];
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint32_t lo, hi;
        float d;
        int s;
        q8_K_warp(v, lo, hi, d, s);
        if (kPlanar) {
            // lane-permuted private layout (see Planar)
            *reinterpret_cast<uint2 *>(p.qs + b * 256 + q8K_code_offset(lane)) = make_uint2(lo, hi);
            if ((lane & 1) == 0)
                *reinterpret_cast<int16_t *>(reinterpret_cast<uint8_t *>(p.sums + b * 16) +
                                             q8K_bsum_offset(lane >> 1)) = (int16_t)s;
            if (lane == 0) p.d[b] = d;
        } else {
            uint8_t *blk = out + b * B_Q8_K;
            uint32_t *qw = reinterpret_cast<uint32_t *>(blk + 4 + 8 * lane);
            qw[0] = lo;
            qw[1] = hi;
            if ((lane & 1) == 0) reinterpret_cast<int16_t *>(blk + 260)[lane >> 1] = (int16_t)s;
            if (lane == 0) *reinterpret_cast<float *>(blk) = d;
        }
    }
}

// ---------------------------------------------------------------- canonical Q8 -> planar
// qmm_mul_mat_q8: the caller's canonical blocks (their codes, scales and, for
// Q8_K, the stored 16-code sums) rewritten into the planar layout.
__global__ void __launch_bounds__(256) import_q8_0_planar_kernel(const uint8_t *__restrict__ Xq,
                                                                 Planar p, int64_t nblocks) {
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < nblocks;
         b += nwarps) {
        const uint8_t *blk = Xq + b * B_Q8_0;
        const int q = (int8_t)blk[2 + lane];
        const int s = __reduce_add_sync(kFull, q);
        p.qs[b * 32 + lane] = (int8_t)q;
        if (lane == 0) {
            p.d[b] = __half2float(*reinterpret_cast<const __half *>(blk));
            p.sums[b] = (int16_t)s;
        }
    }
}

__global__ void __launch_bounds__(256) import_q8_K_planar_kernel(const uint8_t *__restrict__ Xq,
                                                                 Planar p, int64_t nblocks) {
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < nblocks;
         b += nwarps) {
        const uint8_t *blk = Xq + b * B_Q8_K;
        const uint32_t *qw = reinterpret_cast<const uint32_t *>(blk + 4 + 8 * lane);
        *reinterpret_cast<uint2 *>(p.qs + b * 256 + q8K_code_offset(lane)) = make_uint2(qw[0], qw[1]);
        if (lane < 16)
            *reinterpret_cast<int16_t *>(reinterpret_cast<uint8_t *>(p.sums + b * 16) +
                                         q8K_bsum_offset(lane)) =
                reinterpret_cast<const int16_t *>(blk + 260)[lane];
        if (lane == 0) p.d[b] = *reinterpret_cast<const float *>(blk);
    }
}

// ---------------------------------------------------------------- Q4_0 weights
// One warp per block. d = -x_max / 8, x_max the signed value of largest
// magnitude (first index on ties); q = clamp(floor(x * (1/d) + 8.5), 0, 15).
__global__ void __launch_bounds__(256) quantize_q4_0_kernel(const float *__restrict__ W,
                                                            uint8_t *__restrict__ out,
                                                            int64_t nblocks) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < nblocks;
         b += nwarps) {
        const float x = W[b * 32 + lane];
        const uint32_t a = __float_as_uint(fabsf(x));
        const uint32_t amax = __reduce_max_sync(kFull, a);
        const int first = __ffs(__ballot_sync(kFull, a == amax)) - 1;
        float vmax = __shfl_sync(kFull, x, first);
        if (amax == 0u) vmax = 0.0f;  // a block of zeros keeps x_max = +0
        const float d = __fdiv_rn(vmax, -8.0f);
        const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
        const int q = clampi((int)floorf(__fadd_rn(__fmul_rn(x, id), 8.5f)), 0, 15);
        const int qhi = __shfl_down_sync(kFull, q, 16);
        uint8_t *blk = out + b * B_Q4_0;
        if (lane < 16) blk[2 + lane] = (uint8_t)(q | (qhi << 4));
        if (lane == 0) *reinterpret_cast<__half *>(blk) = __float2half_rn(d);
    }
}

// ---------------------------------------------------------------- Q4_K weights
// One warp per super-block; lane l holds sub-block j = l / 4, elements
// 8 (l % 4) .. +7 of it. Reading of the unprinted scale search: per sub-block
// lo = min(0, min x), hi = max x, sc = (hi - lo)/15, mn = -lo; d = max sc / 63,
// dmin = max mn / 63; s_j, m_j rounded to 6 bits; codes from the stored fp16
// d, dmin.
__global__ void __launch_bounds__(256) quantize_q4_K_kernel(const float *__restrict__ W,
                                                            uint8_t *__restrict__ out,
                                                            int64_t nblocks) {
    const int lane = threadIdx.x & 31;
    const int j = lane >> 2, part = lane & 3;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < nblocks;
         b += nwarps) {
        const float4 *src = reinterpret_cast<const float4 *>(W + b * 256 + 32 * j + 8 * part);
        const float4 v0 = src[0], v1 = src[1];
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        float lo = 0.0f, hi = v[0];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            lo = fminf(lo, v[i]);
            hi = fmaxf(hi, v[i]);
        }
        lo = group_min(lo, 4);
        hi = group_max(hi, 4);
        const float sc = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
        const float mn = -lo;
        const float max_sc = warp_max_nonneg(sc > 0.0f ? sc : 0.0f);
        const float max_mn = warp_max_nonneg(mn > 0.0f ? mn : 0.0f);
        const float d = __fdiv_rn(max_sc, 63.0f);
        const float dmin = __fdiv_rn(max_mn, 63.0f);
        const int s = d > 0.0f ? clampi((int)round_half_away(__fdiv_rn(sc, d)), 0, 63) : 0;
        const int m = dmin > 0.0f ? clampi((int)round_half_away(__fdiv_rn(mn, dmin)), 0, 63) : 0;
        const __half d16 = __float2half_rn(d);
        const __half dmin16 = __float2half_rn(dmin);
        const float D = __fmul_rn(__half2float(d16), (float)s);
        const float Mo = __fmul_rn(__half2float(dmin16), (float)m);
        uint32_t qlo = 0, qhi = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int q = 0;
            if (D != 0.0f) q = clampi((int)round_half_away(__fdiv_rn(__fadd_rn(v[i], Mo), D)), 0, 15);
            if (i < 4)
                qlo |= (uint32_t)q << (8 * i);
            else
                qhi |= (uint32_t)q << (8 * (i - 4));
        }
        // sub-block 2c holds the low nibbles and 2c+1 the high nibbles of
        // bytes 32c .. 32c+31: lane 8c+p pairs with lane 8c+4+p.
        const uint32_t olo = __shfl_down_sync(kFull, qlo, 4);
        const uint32_t ohi = __shfl_down_sync(kFull, qhi, 4);
        uint8_t *blk = out + b * B_Q4_K;
        if ((j & 1) == 0) {
            const int c = j >> 1;
            *reinterpret_cast<uint2 *>(blk + 16 + 32 * c + 8 * part) =
                make_uint2(qlo | (olo << 4), qhi | (ohi << 4));
        }
        // 6-bit scales and mins into 12 bytes (page 1, "6-bit 参数")
        uint32_t sm = (uint32_t)s | ((uint32_t)m << 8);
        uint32_t all[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) all[jj] = __shfl_sync(kFull, sm, 4 * jj);
        if (lane == 0) {
            uint8_t sc12[12] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const uint32_t sj = all[jj] & 63, mj = (all[jj] >> 8) & 63;
                if (jj < 4) {
                    sc12[jj] |= (uint8_t)sj;
                    sc12[jj + 4] |= (uint8_t)mj;
                } else {
                    sc12[jj + 4] = (uint8_t)((sj & 15) | ((mj & 15) << 4));
                    sc12[jj - 4] |= (uint8_t)((sj >> 4) << 6);
                    sc12[jj] |= (uint8_t)((mj >> 4) << 6);
                }
            }
            uint4 hdr;
            hdr.x = (uint32_t)__half_as_ushort(d16) | ((uint32_t)__half_as_ushort(dmin16) << 16);
            hdr.y = sc12[0] | (sc12[1] << 8) | (sc12[2] << 16) | ((uint32_t)sc12[3] << 24);
            hdr.z = sc12[4] | (sc12[5] << 8) | (sc12[6] << 16) | ((uint32_t)sc12[7] << 24);
            hdr.w = sc12[8] | (sc12[9] << 8) | (sc12[10] << 16) | ((uint32_t)sc12[11] << 24);
            *reinterpret_cast<uint4 *>(blk) = hdr;
        }
    }
}

// ---------------------------------------------------------------- Q6_K weights
// One warp per super-block; lane l holds elements 8l .. 8l+7, half of group
// l / 2. Reading of the unprinted scale search (page 1 gives the format):
// sc_j = -x_max,j / 32 with x_max,j the signed value of largest magnitude in
// group j (the first on ties), d = max |sc_j| / 127, s_j = round(sc_j / d)
// clamped to int8 +-127, codes q = clamp(round(x / (d16 s_j)), -32, 31) from
// the stored fp16 d, stored as u = q + 32. Canonical bit order: ql[32c + l] =
// low(u[64c + l]) | low(u[64c + 32 + l]) << 4, qh[32h + l] = sum_i
// high2(u[128h + 32i + l]) << 2i (the pairing of Q4_K's nibbles, fields 32
// elements apart).
__global__ void __launch_bounds__(256) quantize_q6_K_kernel(const float *__restrict__ W,
                                                            uint8_t *__restrict__ out,
                                                            int64_t nblocks) {
    __shared__ __align__(16) uint8_t us_all[8][256];
    const int lane = threadIdx.x & 31;
    uint8_t *us = us_all[threadIdx.x >> 5];
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < nblocks;
         b += nwarps) {
        const float4 *src = reinterpret_cast<const float4 *>(W + b * 256 + 8 * lane);
        const float4 v0 = src[0], v1 = src[1];
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        float amax = 0.0f, vmax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float a = fabsf(v[i]);
            if (a > amax) {
                amax = a;
                vmax = v[i];
            }
        }
        // the group's first half (even lane) wins ties, as in a scan from 0
        const float amax_o = __shfl_xor_sync(kFull, amax, 1);
        const float vmax_o = __shfl_xor_sync(kFull, vmax, 1);
        const bool first = (lane & 1) == 0;
        const float a0 = first ? amax : amax_o, a1 = first ? amax_o : amax;
        const float x0 = first ? vmax : vmax_o, x1 = first ? vmax_o : vmax;
        const float vg = a1 > a0 ? x1 : x0;
        const float sc = __fdiv_rn(vg, -32.0f);
        const float max_sc = warp_max_nonneg(fabsf(sc));
        const float d = __fdiv_rn(max_sc, 127.0f);
        const __half d16 = __float2half_rn(d);
        const int s = d > 0.0f ? clampi((int)round_half_away(__fdiv_rn(sc, d)), -127, 127) : 0;
        const float D = __fmul_rn(__half2float(d16), (float)s);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int q = 0;
            if (D != 0.0f) q = clampi((int)round_half_away(__fdiv_rn(v[i], D)), -32, 31);
            const uint32_t u = (uint32_t)(q + 32);
            if (i < 4)
                lo |= u << (8 * i);
            else
                hi |= u << (8 * (i - 4));
        }
        *reinterpret_cast<uint2 *>(us + 8 * lane) = make_uint2(lo, hi);
        __syncwarp();
        uint8_t *blk = out + b * B_Q6_K;
        uint32_t ql = 0;  // ql bytes 4 lane .. 4 lane + 3
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int idx = 4 * lane + k, c = idx >> 5, l = idx & 31;
            ql |= (uint32_t)((us[64 * c + l] & 15) | ((us[64 * c + 32 + l] & 15) << 4)) << (8 * k);
        }
        uint32_t qh = 0;  // qh bytes 2 lane, 2 lane + 1
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int idx = 2 * lane + k, h = idx >> 5, l = idx & 31;
            uint32_t byte = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) byte |= (uint32_t)(us[128 * h + 32 * i + l] >> 4) << (2 * i);
            qh |= byte << (8 * k);
        }
        // 210-byte blocks: 2-byte stores only
        reinterpret_cast<uint16_t *>(blk)[2 * lane] = (uint16_t)ql;
        reinterpret_cast<uint16_t *>(blk)[2 * lane + 1] = (uint16_t)(ql >> 16);
        reinterpret_cast<uint16_t *>(blk + 128)[lane] = (uint16_t)qh;
        if (first) blk[192 + (lane >> 1)] = (uint8_t)(int8_t)s;
        if (lane == 0) *reinterpret_cast<uint16_t *>(blk + 208) = __half_as_ushort(d16);
        __syncwarp();  // us is rewritten by the next super-block
    }
}

int grid_for(int64_t nwarp_items) {
    const int64_t ctas = (nwarp_items + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 16;
    return (int)(ctas < cap ? (ctas > 0 ? ctas : 1) : cap);
}

}  // namespace

cudaError_t launch_quantize_q8(qmm_type vt, bool planar, const float *X, void *out, Planar p,
                               int64_t M, int64_t K, cudaStream_t s) {
    const int64_t nblocks = M * (K / (vt == QMM_TYPE_Q8_0 ? QK4_0 : QK_K));
    const int grid = grid_for(nblocks);
    uint8_t *o = static_cast<uint8_t *>(out);
    if (vt == QMM_TYPE_Q8_0) {
        if (planar)
            quantize_q8_0_kernel<true><<<grid, 256, 0, s>>>(X, o, p, nblocks);
        else
            quantize_q8_0_kernel<false><<<grid, 256, 0, s>>>(X, o, p, nblocks);
    } else {
        if (planar)
            quantize_q8_K_kernel<true><<<grid, 256, 0, s>>>(X, o, p, nblocks);
        else
            quantize_q8_K_kernel<false><<<grid, 256, 0, s>>>(X, o, p, nblocks);
    }
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_import_q8_planar(qmm_type vt, const void *Xq, Planar p, int64_t M, int64_t K,
                                    cudaStream_t s) {
    const int64_t nblocks = M * (K / (vt == QMM_TYPE_Q8_0 ? QK4_0 : QK_K));
    const uint8_t *x = static_cast<const uint8_t *>(Xq);
    if (vt == QMM_TYPE_Q8_0)
        import_q8_0_planar_kernel<<<grid_for(nblocks), 256, 0, s>>>(x, p, nblocks);
    else
        import_q8_K_planar_kernel<<<grid_for(nblocks), 256, 0, s>>>(x, p, nblocks);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_quantize_weights(qmm_type wt, const float *W, void *Wq, int64_t N, int64_t K,
                                    cudaStream_t s) {
    uint8_t *o = static_cast<uint8_t *>(Wq);
    if (wt == QMM_TYPE_Q4_0) {
        const int64_t nblocks = N * (K / QK4_0);
        quantize_q4_0_kernel<<<grid_for(nblocks), 256, 0, s>>>(W, o, nblocks);
    } else if (wt == QMM_TYPE_Q6_K) {
        const int64_t nblocks = N * (K / QK_K);
        quantize_q6_K_kernel<<<grid_for(nblocks), 256, 0, s>>>(W, o, nblocks);
    } else {
        const int64_t nblocks = N * (K / QK_K);
        quantize_q4_K_kernel<<<grid_for(nblocks), 256, 0, s>>>(W, o, nblocks);
    }
    count_launch();
    return cudaGetLastError();
}

}  // namespace qmm
