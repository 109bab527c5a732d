// static_scratch.cu -- qmm_mul_mat_static: the quantize-then-GEMV path with
// its activation workspace in a fixed device array instead of memory the
// library or the caller allocates.
//
// Who needs it: callers that may not allocate device memory once they are
// running -- a serving loop whose allocator is frozen after start-up, a
// runtime that hands this library no allocator of its own, or code that must
// never block on cudaMalloc/cudaFree in a latency-critical step. They still
// own and pass X, the weights and Y; only the scratch moves into the library.
#include <mutex>

#include "qmm_internal.cuh"

namespace qmm {

// The scratch: quantized activations in the planar layout. Every GPU that
// loads this library reserves it until the process exits.
constexpr size_t kStaticScratchBytes = 4u << 20;  // 4 MiB
__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_static_mutex;
uint8_t *g_static_ptr[kMaxDevices] = {nullptr};

bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }

// Device address of the scratch for the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device with that device current.
qmm_status scratch_address(uint8_t **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_error(QMM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return set_error(QMM_ERR_UNSUPPORTED, "device %d", dev);
    std::lock_guard<std::mutex> lk(g_static_mutex);
    if (!g_static_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || !p)
            return set_error(QMM_ERR_CUDA, "cudaGetSymbolAddress(static scratch): %s",
                             cudaGetErrorString(e));
        g_static_ptr[dev] = static_cast<uint8_t *>(p);
    }
    *out = g_static_ptr[dev];
    return QMM_OK;
}
}  // namespace
}  // namespace qmm

using namespace qmm;

extern "C" qmm_status qmm_mul_mat_static(qmm_type wt, const void *W_packed, int64_t N, int64_t K,
                                         const float *X, int64_t M, float *Y,
                                         qmm_stream_t stream) {
    if (wt != QMM_TYPE_Q4_0 && wt != QMM_TYPE_Q4_K && wt != QMM_TYPE_Q6_K)
        return set_error(QMM_ERR_ARG, "weight type must be Q4_0, Q4_K or Q6_K (got %d)", (int)wt);
    const int qk = wt == QMM_TYPE_Q4_0 ? QK4_0 : QK_K;
    if (N < 0 || M < 0 || K <= 0 || K % qk != 0 || K > ((int64_t)1 << 30) || N > ((int64_t)1 << 31))
        return set_error(QMM_ERR_ARG, "bad sizes N=%lld K=%lld M=%lld (K must be a multiple of %d)",
                         (long long)N, (long long)K, (long long)M, qk);
    if (M == 0 || N == 0) return set_error(QMM_OK, "");
    if (!W_packed || !X || !Y) return set_error(QMM_ERR_ARG, "null pointer argument");
    if (!aligned16(W_packed) || !aligned16(X) || ((uintptr_t)Y & 3))
        return set_error(QMM_ERR_ARG, "W_packed and X must be 16-byte aligned, Y 4-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    if (gemv_can_fuse(wt, M, K)) {  // one kernel, no scratch
        Planar none{nullptr, nullptr, nullptr};
        cudaError_t e = launch_gemv(wt, W_packed, N, K, none, X, M, Y, /*pdl=*/true, s);
        if (e != cudaSuccess)
            return set_error(QMM_ERR_CUDA, "mul_mat kernel launch: %s", cudaGetErrorString(e));
        return set_error(QMM_OK, "");
    }
    const bool mma = gemv_use_mma(wt, M, K);
    const size_t need = mma ? mma_image_bytes(wt, M, K) : planar_bytes(M, K, qk, nullptr, nullptr);
    if (need > kStaticScratchBytes)
        return set_error(QMM_ERR_WORKSPACE,
                         "qmm_mul_mat_static: M=%lld x K=%lld needs %zu bytes of scratch, more than "
                         "its fixed %zu; use qmm_mul_mat_ws with a caller workspace",
                         (long long)M, (long long)K, need, kStaticScratchBytes);
    uint8_t *scratch = nullptr;
    qmm_status st = scratch_address(&scratch);
    if (st != QMM_OK) return st;
    // Nothing in the scratch has to start at zero: the quantizer writes every
    // byte the GEMV reads.
    if (mma) {
        cudaError_t e = launch_mma_image(wt, false, X, scratch, M, K, s);
        if (e == cudaSuccess) e = launch_gemv_mma(wt, single_mat(W_packed, N, Y), K, scratch, M, true, s);
        if (e != cudaSuccess)
            return set_error(QMM_ERR_CUDA, "mul_mat launch: %s", cudaGetErrorString(e));
        return set_error(QMM_OK, "");
    }
    Planar p;
    planar_bytes(M, K, qk, &p, scratch);
    const qmm_type at = wt == QMM_TYPE_Q4_0 ? QMM_TYPE_Q8_0 : QMM_TYPE_Q8_K;
    cudaError_t e = launch_quantize_q8(at, true, X, nullptr, p, M, K, s);
    if (e != cudaSuccess)
        return set_error(QMM_ERR_CUDA, "activation quantizer launch: %s", cudaGetErrorString(e));
    e = launch_gemv(wt, W_packed, N, K, p, nullptr, M, Y, /*pdl=*/true, s);
    if (e != cudaSuccess)
        return set_error(QMM_ERR_CUDA, "mul_mat kernel launch: %s", cudaGetErrorString(e));
    return set_error(QMM_OK, "");
}
