// repack.cu -- canonical weight blocks <-> the private GPU layout.
//
// The layout change is done once at load time (page 3, "Ladder Permutation":
// a permutation applied offline pays off when R * dT > T_P, and turns
// run-time address shuffles into contiguous reads; page 4 on GGML_CPU_REPACK).
// It is a pure byte permutation:
//   Q4_K: canonical [N][nsb][144 B] -> tiles of 8 rows, [T][nsb][8][144 B].
//         One (tile, super-block range) is then one contiguous byte range.
//         The 12 scale bytes are re-ordered into four 24-bit lane fields
//         (k4_header_to_packed), the same 96 bits in another order.
//   Q4_0: canonical [N][nb][18 B]   -> per tile [8][nb][16 B nibbles] followed
//         by [nb][8] fp16 scales, so the nibbles are 16-byte aligned (the
//         18-byte block defeats 128-bit loads).
//   Q6_K: canonical [N][nsb][210 B] -> records of 8 rows per (tile,
//         super-block), [T][nsb][1680 B] (qmm_internal.cuh): ql unchanged,
//         the high bits and the scales re-ordered for the GEMV lanes.
// Padding rows (N not a multiple of 8) are zero blocks: d = 0 contributes 0.
#include "qmm_internal.cuh"

namespace qmm {
namespace {

// Q4_K: one thread per 16-byte chunk of the packed buffer (or of the
// canonical buffer for the inverse).
template <bool kInverse>
__global__ void repack_q4_K_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                   int64_t N, int64_t nsb) {
    const int64_t Npad = tiles_of(N) * kTileRows;
    const int64_t total = Npad * nsb * 9;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t pblk = i / 9;  // packed block index
        const int chunk = (int)(i % 9);
        const int64_t tile = pblk / (nsb * kTileRows);
        const int64_t rem = pblk % (nsb * kTileRows);
        const int64_t sb = rem / kTileRows;
        const int64_t n = tile * kTileRows + rem % kTileRows;
        const int64_t cblk = n * nsb + sb;  // canonical block index
        if (!kInverse) {
            uint4 v = n < N ? src[cblk * 9 + chunk] : make_uint4(0, 0, 0, 0);
            if (chunk == 0) v = k4_header_to_packed(v);
            dst[i] = v;
        } else if (n < N) {
            uint4 v = src[i];
            if (chunk == 0) v = k4_header_to_canonical(v);
            dst[cblk * 9 + chunk] = v;
        }
    }
}

// Q4_0: one thread per (row, block).
template <bool kInverse>
__global__ void repack_q4_0_kernel(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst,
                                   int64_t N, int64_t nb) {
    const int64_t Npad = tiles_of(N) * kTileRows;
    const int64_t total = Npad * nb;
    const int64_t tile_bytes = nb * kTileRows * B_Q4_0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / nb, b = i % nb;
        const int64_t tile = n / kTileRows;
        const int r = (int)(n % kTileRows);
        uint8_t *packed_base = kInverse ? nullptr : dst + tile * tile_bytes;
        const uint8_t *packed_src = kInverse ? src + tile * tile_bytes : nullptr;
        const int64_t qs_off = (r * nb + b) * 16;
        const int64_t d_off = nb * kTileRows * 16 + (b * kTileRows + r) * 2;
        if (!kInverse) {
            uint16_t h[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
            if (n < N) {
                const uint16_t *c = reinterpret_cast<const uint16_t *>(src + (n * nb + b) * B_Q4_0);
#pragma unroll
                for (int k = 0; k < 9; ++k) h[k] = c[k];
            }
            uint4 q;
            q.x = h[1] | ((uint32_t)h[2] << 16);
            q.y = h[3] | ((uint32_t)h[4] << 16);
            q.z = h[5] | ((uint32_t)h[6] << 16);
            q.w = h[7] | ((uint32_t)h[8] << 16);
            *reinterpret_cast<uint4 *>(packed_base + qs_off) = q;
            *reinterpret_cast<uint16_t *>(packed_base + d_off) = h[0];
        } else if (n < N) {
            const uint4 q = *reinterpret_cast<const uint4 *>(packed_src + qs_off);
            const uint16_t d = *reinterpret_cast<const uint16_t *>(packed_src + d_off);
            uint16_t *c = reinterpret_cast<uint16_t *>(dst + (n * nb + b) * B_Q4_0);
            c[0] = d;
            c[1] = (uint16_t)q.x;
            c[2] = (uint16_t)(q.x >> 16);
            c[3] = (uint16_t)q.y;
            c[4] = (uint16_t)(q.y >> 16);
            c[5] = (uint16_t)q.z;
            c[6] = (uint16_t)(q.z >> 16);
            c[7] = (uint16_t)q.w;
            c[8] = (uint16_t)(q.w >> 16);
        }
    }
}

// Canonical Q6_K high bits of element e (page 1's qh[64], in the order the
// oracle states: qh[32 (e / 128) + e % 32] bits 2 ((e % 128) / 32)).
__device__ __forceinline__ int q6k_qh_byte(int e) { return 32 * (e >> 7) + (e & 31); }
__device__ __forceinline__ int q6k_qh_shift(int e) { return 2 * ((e & 127) >> 5); }

// Q6_K: one thread per (row, super-block).
template <bool kInverse>
__global__ void repack_q6_K_kernel(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst,
                                   int64_t N, int64_t nsb) {
    const int64_t Npad = tiles_of(N) * kTileRows;
    const int64_t total = Npad * nsb;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / nsb, sb = i % nsb;
        const int r = (int)(n % kTileRows);
        const int64_t rec_off = ((n / kTileRows) * nsb + sb) * kQ6Rec;
        if (!kInverse) {
            uint8_t *rec = dst + rec_off;
            uint8_t ql[128], qh[64], sc[16];
            uint16_t d = 0;
            if (n < N) {
                const uint8_t *c = src + (n * nsb + sb) * B_Q6_K;
                for (int k = 0; k < 128; ++k) ql[k] = c[k];
                for (int k = 0; k < 64; ++k) qh[k] = c[128 + k];
                for (int k = 0; k < 16; ++k) sc[k] = c[192 + k];
                d = *reinterpret_cast<const uint16_t *>(c + 208);
            } else {
                for (int k = 0; k < 128; ++k) ql[k] = 0;
                for (int k = 0; k < 64; ++k) qh[k] = 0;
                for (int k = 0; k < 16; ++k) sc[k] = 0;
            }
            uint8_t *row = rec + r * kQ6Codes;
            for (int k = 0; k < 8; ++k) {
                uint4 v;
                v.x = ql[16 * k] | (ql[16 * k + 1] << 8) | (ql[16 * k + 2] << 16) | ((uint32_t)ql[16 * k + 3] << 24);
                v.y = ql[16 * k + 4] | (ql[16 * k + 5] << 8) | (ql[16 * k + 6] << 16) | ((uint32_t)ql[16 * k + 7] << 24);
                v.z = ql[16 * k + 8] | (ql[16 * k + 9] << 8) | (ql[16 * k + 10] << 16) | ((uint32_t)ql[16 * k + 11] << 24);
                v.w = ql[16 * k + 12] | (ql[16 * k + 13] << 8) | (ql[16 * k + 14] << 16) | ((uint32_t)ql[16 * k + 15] << 24);
                *reinterpret_cast<uint4 *>(row + 16 * k) = v;
            }
            for (int t = 0; t < 8; ++t) {
                uint32_t h[2] = {0, 0};
                for (int hi = 0; hi < 2; ++hi)
                    for (int k = 0; k < 16; ++k) {
                        const int e = q6k_elem(t, hi, k);
                        h[hi] |= (uint32_t)((qh[q6k_qh_byte(e)] >> q6k_qh_shift(e)) & 3) << q6k_hbit_pos(k);
                    }
                *reinterpret_cast<uint2 *>(row + 128 + 8 * t) = make_uint2(h[0], h[1]);
            }
            uint8_t ps[16];
            for (int t = 0; t < 8; ++t) {
                ps[2 * t] = sc[q6k_elem(t, 0, 0) / 16];
                ps[2 * t + 1] = sc[q6k_elem(t, 1, 0) / 16];
            }
            uint4 v;
            v.x = ps[0] | (ps[1] << 8) | (ps[2] << 16) | ((uint32_t)ps[3] << 24);
            v.y = ps[4] | (ps[5] << 8) | (ps[6] << 16) | ((uint32_t)ps[7] << 24);
            v.z = ps[8] | (ps[9] << 8) | (ps[10] << 16) | ((uint32_t)ps[11] << 24);
            v.w = ps[12] | (ps[13] << 8) | (ps[14] << 16) | ((uint32_t)ps[15] << 24);
            *reinterpret_cast<uint4 *>(rec + kQ6ScOff + 16 * r) = v;
            *reinterpret_cast<uint16_t *>(rec + kQ6DOff + 2 * r) = d;
        } else if (n < N) {
            const uint8_t *rec = src + rec_off;
            const uint8_t *row = rec + r * kQ6Codes;
            uint8_t *c = dst + (n * nsb + sb) * B_Q6_K;
            for (int k = 0; k < 128; ++k) c[k] = row[k];
            uint8_t qh[64];
            for (int k = 0; k < 64; ++k) qh[k] = 0;
            for (int t = 0; t < 8; ++t) {
                const uint2 hw = *reinterpret_cast<const uint2 *>(row + 128 + 8 * t);
                const uint32_t h[2] = {hw.x, hw.y};
                for (int hi = 0; hi < 2; ++hi)
                    for (int k = 0; k < 16; ++k) {
                        const int e = q6k_elem(t, hi, k);
                        qh[q6k_qh_byte(e)] |= (uint8_t)(((h[hi] >> q6k_hbit_pos(k)) & 3) << q6k_qh_shift(e));
                    }
            }
            for (int k = 0; k < 64; ++k) c[128 + k] = qh[k];
            const uint8_t *ps = rec + kQ6ScOff + 16 * r;
            for (int t = 0; t < 8; ++t) {
                c[192 + q6k_elem(t, 0, 0) / 16] = ps[2 * t];
                c[192 + q6k_elem(t, 1, 0) / 16] = ps[2 * t + 1];
            }
            *reinterpret_cast<uint16_t *>(c + 208) = *reinterpret_cast<const uint16_t *>(rec + kQ6DOff + 2 * r);
        }
    }
}

int grid_1d(int64_t n, int threads) {
    const int64_t ctas = (n + threads - 1) / threads;
    const int64_t cap = (int64_t)sm_count() * 32;
    return (int)(ctas < 1 ? 1 : (ctas < cap ? ctas : cap));
}

}  // namespace

cudaError_t launch_repack(qmm_type wt, bool inverse, const void *src, void *dst, int64_t N,
                          int64_t K, cudaStream_t s) {
    const int64_t Npad = tiles_of(N) * kTileRows;
    if (wt == QMM_TYPE_Q4_K) {
        const int64_t nsb = K / QK_K;
        const int grid = grid_1d(Npad * nsb * 9, 256);
        if (inverse)
            repack_q4_K_kernel<true><<<grid, 256, 0, s>>>((const uint4 *)src, (uint4 *)dst, N, nsb);
        else
            repack_q4_K_kernel<false><<<grid, 256, 0, s>>>((const uint4 *)src, (uint4 *)dst, N, nsb);
    } else if (wt == QMM_TYPE_Q6_K) {
        const int64_t nsb = K / QK_K;
        const int grid = grid_1d(Npad * nsb, 128);
        if (inverse)
            repack_q6_K_kernel<true><<<grid, 128, 0, s>>>((const uint8_t *)src, (uint8_t *)dst, N, nsb);
        else
            repack_q6_K_kernel<false><<<grid, 128, 0, s>>>((const uint8_t *)src, (uint8_t *)dst, N, nsb);
    } else {
        const int64_t nb = K / QK4_0;
        const int grid = grid_1d(Npad * nb, 256);
        if (inverse)
            repack_q4_0_kernel<true><<<grid, 256, 0, s>>>((const uint8_t *)src, (uint8_t *)dst, N, nb);
        else
            repack_q4_0_kernel<false><<<grid, 256, 0, s>>>((const uint8_t *)src, (uint8_t *)dst, N, nb);
    }
    count_launch();
    return cudaGetLastError();
}

}  // namespace qmm
