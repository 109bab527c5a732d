// peaks.cu -- tensor-core throughput microbenchmarks, the denominators the
// prefill GEMMs are measured against (page 3, "性能判断: 带宽、解码和 Tensor
// Core 谁是瓶颈": a kernel is judged against the peak of the unit it uses).
//   QMM_PEAK_MMA_S8     legacy warp-level mma.sync m16n8k32 s8 x s8 -> s32
//                       (the int8 tensor path sm_103a offers: tcgen05 has no
//                       kind::i8 there)
//   QMM_PEAK_MMA_F16    legacy mma.sync m16n8k16 f16 x f16 -> f32
//   QMM_PEAK_TC_SS_128  tcgen05.mma kind::f16, M = 128, N = 128, K = 16, both
//                       operands in shared memory, fp32 accumulator in TMEM
//   QMM_PEAK_TC_TS_128  the same with A in TMEM (the prefill GEMMs' form)
//   QMM_PEAK_TC_SS_256  M = 128, N = 256, operands in shared memory
//   QMM_PEAK_TC_TS_256  M = 128, N = 256, A in TMEM
// Operands are nonzero pseudo-random values; every result is folded into a
// comparison whose (practically never taken) branch writes a device word, so
// that nothing is dead code. The caller times the launch with CUDA events;
// ops = 2 M N K per MMA times the MMAs issued.
#include "tc.cuh"

namespace qmm {
namespace {

constexpr int kSyncThreads = 256;  // 8 warps per CTA
constexpr int kChains = 8;         // independent accumulators per warp

__device__ __forceinline__ uint32_t mix(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7feb352du;
    x ^= x >> 15;
    return x;
}

__global__ void __launch_bounds__(kSyncThreads) peak_mma_s8_kernel(int64_t iters, unsigned *sink) {
    const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t a[4], b[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = mix(t * 8 + i) & 0x3F3F3F3Fu;
#pragma unroll
    for (int i = 0; i < 2; ++i) b[i] = mix(t * 8 + 4 + i) & 0x3F3F3F3Fu;
    int c[kChains][4] = {};
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int ch = 0; ch < kChains; ++ch)
            asm volatile(
                "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                "{%8, %9}, {%0, %1, %2, %3};"
                : "+r"(c[ch][0]), "+r"(c[ch][1]), "+r"(c[ch][2]), "+r"(c[ch][3])
                : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
    }
    int acc = 0;
#pragma unroll
    for (int ch = 0; ch < kChains; ++ch) acc ^= c[ch][0] ^ c[ch][1] ^ c[ch][2] ^ c[ch][3];
    if (acc == 0x12345678) atomicAdd(sink, 1u);
}

__global__ void __launch_bounds__(kSyncThreads) peak_mma_f16_kernel(int64_t iters, unsigned *sink) {
    const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t a[4], b[2];
    // fp16 values in [1, 2): exponent 15, random mantissa
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = (mix(t * 8 + i) & 0x03FF03FFu) | 0x3C003C00u;
#pragma unroll
    for (int i = 0; i < 2; ++i) b[i] = (mix(t * 8 + 4 + i) & 0x03FF03FFu) | 0x3C003C00u;
    float c[kChains][4] = {};
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int ch = 0; ch < kChains; ++ch)
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                "{%8, %9}, {%0, %1, %2, %3};"
                : "+f"(c[ch][0]), "+f"(c[ch][1]), "+f"(c[ch][2]), "+f"(c[ch][3])
                : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
    }
    float acc = 0.0f;
#pragma unroll
    for (int ch = 0; ch < kChains; ++ch) acc += c[ch][0] + c[ch][1] + c[ch][2] + c[ch][3];
    if (acc == 1.2345f) atomicAdd(sink, 1u);
}

// tcgen05: one CTA per SM, 128 threads. Shared memory: A tile [128 rows][64
// K] and B tile [N rows][64 K], fp16, 128-byte swizzled K-major rows (the
// layout the prefill GEMM's TMA writes). One thread issues `iters` rounds of
// 4 MMAs (K = 64) into one accumulator, then commits; all four warps read a
// few accumulator columns back.
template <int N, bool kTmemA>
__global__ void __launch_bounds__(128, 1) peak_tc_kernel(int64_t iters, unsigned *sink, unsigned *err) {
    constexpr int kM = 128, kK = 64;
    constexpr int kABytes = kM * kK * 2, kBBytes = N * kK * 2;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kABytes + kBBytes);
    uint32_t *slot = reinterpret_cast<uint32_t *>(bar + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // operands: fp16 in [1, 2) (any bit pattern of the swizzled tile is a valid element)
    uint32_t *words = reinterpret_cast<uint32_t *>(smem);
    for (int i = threadIdx.x; i < (kABytes + kBBytes) / 4; i += 128)
        words[i] = (mix(i * 131 + blockIdx.x) & 0x03FF03FFu) | 0x3C003C00u;
    tc::fence_proxy_async();
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(bar), 1);
        fence_barrier_init();
    }
    __syncwarp();
    if (warp == 0) tc::tmem_alloc(smem_u32(slot), 512);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *slot;
    constexpr uint32_t kColA = 256;  // A operand columns (TMEM-A form): 4 K steps x 8 columns
    if (kTmemA) {
        uint32_t r[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = (mix(threadIdx.x * 16 + i) & 0x03FF03FFu) | 0x3C003C00u;
        const uint32_t lane_addr = (uint32_t)(32 * warp) << 16;
        tc::tmem_st16(tmem + lane_addr + kColA, r);
        tc::tmem_st16(tmem + lane_addr + kColA + 16, r);
        tc::tmem_st_wait();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (threadIdx.x == 0) {
        constexpr uint32_t idesc = tc::idesc_f16_f32(kM, N);
        const uint64_t adesc = tc::smem_desc(base, 1024, 2);
        const uint64_t bdesc = tc::smem_desc(base + kABytes, 1024, 2);
        for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
            for (int kk = 0; kk < kK / 16; ++kk) {
                // K step of 16 fp16 = 32 bytes = 2 in the descriptors' address field
                if (kTmemA)
                    tc::mma_f16_ta(tmem, tmem + kColA + 8 * kk, bdesc + 2 * kk, idesc, (it | kk) != 0);
                else
                    tc::mma_f16(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (it | kk) != 0);
            }
        }
        tc::commit(smem_u32(bar));
    }
    __syncwarp();
    const bool ok = mbar_wait_warp(smem_u32(bar), 0, err);
    tc::fence_after_sync();
    if (ok) {
        float v[16];
        tc::tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16), v);
        tc::tmem_ld_wait();
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) s += v[i];
        if (s == 1.2345f) atomicAdd(sink, 1u);
    }
    (void)lane;
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

template <int N, bool kTmemA>
cudaError_t launch_tc(int64_t iters, unsigned *sink, cudaStream_t s, double *ops) {
    // at least 116 KB so that one CTA (and one 512-column TMEM allocation)
    // sits on each SM
    constexpr int kNeed = 128 * 64 * 2 + N * 64 * 2 + 1024 + 64;
    constexpr int kSmem = kNeed > 116 * 1024 ? kNeed : 116 * 1024;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(peak_tc_kernel<N, kTmemA>), kSmem);
    if (e != cudaSuccess) return e;
    const int grid = sm_count();
    peak_tc_kernel<N, kTmemA><<<grid, 128, kSmem, s>>>(iters, sink, device_error_word());
    count_launch();
    *ops = 2.0 * 128 * N * 64 * (double)iters * grid;
    return cudaGetLastError();
}

__device__ unsigned g_peak_sink;  // written only if a result hits a sentinel value

}  // namespace

cudaError_t launch_debug_peak(int which, int64_t iters, cudaStream_t s, double *ops) {
    unsigned *sink = nullptr;
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(&sink), g_peak_sink);
    if (e != cudaSuccess) return e;
    const int sms = sm_count();
    switch (which) {
    case QMM_PEAK_MMA_S8:
    case QMM_PEAK_MMA_F16: {
        const int grid = sms * 4;  // 32 warps per SM
        if (which == QMM_PEAK_MMA_S8)
            peak_mma_s8_kernel<<<grid, kSyncThreads, 0, s>>>(iters, sink);
        else
            peak_mma_f16_kernel<<<grid, kSyncThreads, 0, s>>>(iters, sink);
        count_launch();
        const double per = which == QMM_PEAK_MMA_S8 ? 2.0 * 16 * 8 * 32 : 2.0 * 16 * 8 * 16;
        *ops = per * kChains * (double)iters * (kSyncThreads / 32) * grid;
        return cudaGetLastError();
    }
    case QMM_PEAK_TC_SS_128: return launch_tc<128, false>(iters, sink, s, ops);
    case QMM_PEAK_TC_TS_128: return launch_tc<128, true>(iters, sink, s, ops);
    case QMM_PEAK_TC_SS_256: return launch_tc<256, false>(iters, sink, s, ops);
    case QMM_PEAK_TC_TS_256: return launch_tc<256, true>(iters, sink, s, ops);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
