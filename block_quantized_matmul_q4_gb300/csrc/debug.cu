// debug.cu -- per-block integer sums of the factored form, for bit-exact
// checks of the packed layout and the block arithmetic (page 1, "正确性:
// 缩放系数可以提到求和号外面" and "通用实现"). Slow on purpose: one thread per
// (token, row, block), reading packed weights and canonical Q8 blocks.
#include "qmm_internal.cuh"

namespace qmm {
namespace {

__global__ void block_sums_q4_0_kernel(const uint8_t *__restrict__ Wp, int64_t N, int64_t nb,
                                       const uint8_t *__restrict__ Xq, int64_t M,
                                       int32_t *__restrict__ out) {
    const int64_t total = M * N * nb;
    const int64_t tile_bytes = nb * kTileRows * B_Q4_0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = i % nb, n = (i / nb) % N, m = i / (nb * N);
        const uint8_t *qs = Wp + (n / kTileRows) * tile_bytes + ((n % kTileRows) * nb + b) * 16;
        const int8_t *y = reinterpret_cast<const int8_t *>(Xq + (m * nb + b) * B_Q8_0 + 2);
        int32_t s = 0;
        for (int l = 0; l < 16; ++l) {
            s += ((qs[l] & 0x0F) - 8) * y[l];
            s += ((qs[l] >> 4) - 8) * y[l + 16];
        }
        out[i] = s;
    }
}

__global__ void block_sums_q4_K_kernel(const uint8_t *__restrict__ Wp, int64_t N, int64_t nsb,
                                       const uint8_t *__restrict__ Xq, int64_t M,
                                       int32_t *__restrict__ out) {
    const int64_t total = M * N * nsb;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t sb = i % nsb, n = (i / nsb) % N, m = i / (nsb * N);
        const uint8_t *blk =
            Wp + (((n / kTileRows) * nsb + sb) * kTileRows + n % kTileRows) * B_Q4_K;
        int sj[8], mj[8];
        k4_scales_canonical(k4_header_to_canonical(*reinterpret_cast<const uint4 *>(blk)), sj, mj);
        const uint8_t *qs = blk + 16;
        const uint8_t *yb = Xq + (m * nsb + sb) * B_Q8_K;
        const int8_t *y = reinterpret_cast<const int8_t *>(yb + 4);
        const int16_t *bs = reinterpret_cast<const int16_t *>(yb + 260);
        int32_t S[8];
        for (int c = 0; c < 4; ++c) {
            int32_t lo = 0, hi = 0;
            for (int l = 0; l < 32; ++l) {
                lo += (qs[32 * c + l] & 0x0F) * y[64 * c + l];
                hi += (qs[32 * c + l] >> 4) * y[64 * c + 32 + l];
            }
            S[2 * c] = lo;
            S[2 * c + 1] = hi;
        }
        int32_t isum = 0, msum = 0;
        for (int j = 0; j < 8; ++j) {
            isum += sj[j] * S[j];
            msum += mj[j] * (bs[2 * j] + bs[2 * j + 1]);
        }
        int32_t *o = out + i * 10;
        for (int j = 0; j < 8; ++j) o[j] = S[j];
        o[8] = isum;
        o[9] = msum;
    }
}

// Q6_K: each element decoded from the packed record through the lane
// geometry the GEMV uses (ql bytes 16t.., high-bit words, scale bytes 2t,
// 2t + 1), summed per group of 16 in natural element order.
__global__ void block_sums_q6_K_kernel(const uint8_t *__restrict__ Wp, int64_t N, int64_t nsb,
                                       const uint8_t *__restrict__ Xq, int64_t M,
                                       int32_t *__restrict__ out) {
    const int64_t total = M * N * nsb;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t sb = i % nsb, n = (i / nsb) % N, m = i / (nsb * N);
        const uint8_t *rec = Wp + ((n / kTileRows) * nsb + sb) * kQ6Rec;
        const int r = (int)(n % kTileRows);
        const uint8_t *row = rec + r * kQ6Codes;
        const int8_t *ps = reinterpret_cast<const int8_t *>(rec + kQ6ScOff + 16 * r);
        const int8_t *y = reinterpret_cast<const int8_t *>(Xq + (m * nsb + sb) * B_Q8_K + 4);
        int32_t S[16], isum = 0;
        for (int j = 0; j < 16; ++j) S[j] = 0;
        int sj[16];
        for (int t = 0; t < 8; ++t) {
            for (int hi = 0; hi < 2; ++hi) {
                const uint32_t hw = reinterpret_cast<const uint32_t *>(row + 128 + 8 * t)[hi];
                sj[q6k_elem(t, hi, 0) / 16] = ps[2 * t + hi];
                for (int k = 0; k < 16; ++k) {
                    const int e = q6k_elem(t, hi, k);
                    const int nib = hi ? (row[16 * t + k] >> 4) : (row[16 * t + k] & 15);
                    const int u = nib | (int)(((hw >> q6k_hbit_pos(k)) & 3) << 4);
                    S[e / 16] += (u - 32) * y[e];
                }
            }
        }
        int32_t *o = out + i * 17;
        for (int j = 0; j < 16; ++j) {
            o[j] = S[j];
            isum += sj[j] * S[j];
        }
        o[16] = isum;
    }
}

}  // namespace

cudaError_t launch_debug_block_sums(qmm_type wt, const void *Wp, int64_t N, int64_t K,
                                    const void *Xq, int64_t M, int32_t *out, cudaStream_t s) {
    const int64_t nblk = K / (wt == QMM_TYPE_Q4_0 ? QK4_0 : QK_K);
    const int64_t total = M * N * nblk;
    int64_t grid = (total + 255) / 256;
    if (grid > (int64_t)sm_count() * 32) grid = (int64_t)sm_count() * 32;
    if (grid < 1) grid = 1;
    if (wt == QMM_TYPE_Q4_0)
        block_sums_q4_0_kernel<<<(int)grid, 256, 0, s>>>((const uint8_t *)Wp, N, nblk,
                                                         (const uint8_t *)Xq, M, out);
    else if (wt == QMM_TYPE_Q6_K)
        block_sums_q6_K_kernel<<<(int)grid, 256, 0, s>>>((const uint8_t *)Wp, N, nblk,
                                                         (const uint8_t *)Xq, M, out);
    else
        block_sums_q4_K_kernel<<<(int)grid, 256, 0, s>>>((const uint8_t *)Wp, N, nblk,
                                                         (const uint8_t *)Xq, M, out);
    count_launch();
    return cudaGetLastError();
}

// A bounded wait that is made to run out: one CTA waits on an mbarrier that
// nothing completes, with the same helper as every pipeline wait of the
// library and a short limit, so the failure path (error word set, kernel
// returns, context usable) can be checked without any fault.
namespace {
__global__ void wait_timeout_kernel(unsigned *err, long long limit_cycles) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_barrier_init();
    }
    __syncthreads();
    mbar_wait_for(smem_u32(&bar), 0, err, limit_cycles);
}
}  // namespace

cudaError_t launch_debug_wait_timeout(int64_t limit_cycles, cudaStream_t s) {
    wait_timeout_kernel<<<1, 32, 0, s>>>(device_error_word(), (long long)limit_cycles);
    count_launch();
    return cudaGetLastError();
}

}  // namespace qmm
