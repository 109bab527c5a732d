// api.cu -- the extern "C" entry points declared in include/qmm.h: argument
// validation, workspace handling, dispatch to the kernel launchers, status
// and error reporting.
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <mutex>
#include <map>
#include <utility>

#include "qmm_internal.cuh"

namespace qmm {

// Device error word: bit kDevErrTimeout is set by a kernel that gave up a
// bounded wait. Read and cleared by qmm_check_device_error.
__device__ unsigned g_device_error = 0;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned *g_err_ptr[kMaxDevices] = {nullptr};
int g_sms[kMaxDevices] = {0};
bool g_pool_ready[kMaxDevices] = {false};
std::map<std::pair<const void *, int>, int> g_smem_set;  // (kernel, device) -> bytes
std::atomic<uint64_t> g_launches{0};
thread_local char g_msg[512] = "";

int current_device() {
    int d = 0;
    cudaGetDevice(&d);
    return d < 0 ? 0 : (d >= kMaxDevices ? kMaxDevices - 1 : d);
}
}  // namespace

unsigned *device_error_word() {
    const int d = current_device();
    std::lock_guard<std::mutex> lk(g_mutex);
    if (!g_err_ptr[d]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) == cudaSuccess) g_err_ptr[d] = (unsigned *)p;
    }
    return g_err_ptr[d];
}

int sm_count() {
    const int d = current_device();
    std::lock_guard<std::mutex> lk(g_mutex);
    if (!g_sms[d]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
        g_sms[d] = n > 0 ? n : 1;
    }
    return g_sms[d];
}

cudaError_t ensure_smem_attr(const void *kernel, int bytes) {
    const int d = current_device();
    std::lock_guard<std::mutex> lk(g_mutex);
    auto it = g_smem_set.find({kernel, d});
    if (it != g_smem_set.end() && it->second >= bytes) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) g_smem_set[{kernel, d}] = bytes;
    return e;
}

void count_launch(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

qmm_status set_error(qmm_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return s;
}

namespace {

bool is_weight(qmm_type t) { return t == QMM_TYPE_Q4_0 || t == QMM_TYPE_Q4_K || t == QMM_TYPE_Q6_K; }
bool is_act(qmm_type t) { return t == QMM_TYPE_Q8_0 || t == QMM_TYPE_Q8_K; }
int elems(qmm_type t) { return (t == QMM_TYPE_Q4_0 || t == QMM_TYPE_Q8_0) ? QK4_0 : QK_K; }
qmm_type act_of(qmm_type wt) { return wt == QMM_TYPE_Q4_0 ? QMM_TYPE_Q8_0 : QMM_TYPE_Q8_K; }
bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

qmm_status ok() {
    g_msg[0] = 0;
    return QMM_OK;
}

qmm_status cuda_status(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return ok();
    return set_error(QMM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define QMM_CHECK_ARG(cond, ...)                            \
    do {                                                    \
        if (!(cond)) return set_error(QMM_ERR_ARG, __VA_ARGS__); \
    } while (0)

qmm_status check_weight_args(qmm_type wt, int64_t N, int64_t K) {
    QMM_CHECK_ARG(is_weight(wt), "weight type must be Q4_0, Q4_K or Q6_K (got %d)", (int)wt);
    QMM_CHECK_ARG(N >= 0 && K > 0, "sizes must satisfy N >= 0, K > 0 (N=%lld K=%lld)",
                  (long long)N, (long long)K);
    QMM_CHECK_ARG(K % elems(wt) == 0, "K=%lld is not a multiple of the block size %d",
                  (long long)K, elems(wt));
    QMM_CHECK_ARG(K <= (int64_t)1 << 30 && N <= (int64_t)1 << 31, "sizes too large");
    return QMM_OK;
}

// Default mem pool: keep freed workspace instead of returning it to the
// driver at every synchronization. Skipped while `s` is being captured (a
// pool attribute change would end the capture; allocations in a graph come
// from the graph's own memory anyway) and done by the next call outside one.
void prepare_pool(cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return;
    const int d = current_device();
    std::lock_guard<std::mutex> lk(g_mutex);
    if (g_pool_ready[d]) return;
    cudaMemPool_t pool;
    if (cudaDeviceGetDefaultMemPool(&pool, d) == cudaSuccess) {
        uint64_t thr = UINT64_MAX;
        cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &thr);
    }
    g_pool_ready[d] = true;
}

// More than 16 tokens run the fp16-operand tensor-core GEMM on fp16(2^e d_a y)
// activations with a power of two 2^e per token (Q4_0: 32-blocks, permuted
// for its converter; Q4_K and Q6_K: Q8_K codes in natural order); fewer the
// decode GEMVs: from 2 tokens the mma.sync kernels and their activation
// images, otherwise the scalar GEMV and the planar layout. A decode batch
// whose activation image does not fit one CTA's shared memory (large K) takes
// several tensor-core GEMV launches, each reading all the weights again; from
// three such launches (two for Q4_0 and Q6_K) the GEMM, which reads them
// once, is faster (Q4_K 8192 x 28672, 16 tokens: 255 -> 81 us; Q6_K 8192^2,
// 12 tokens: 44 -> 32 us; at two Q4_K launches the GEMV is as fast or faster).
bool use_gemm(qmm_type wt, int64_t M, int64_t K) {
    if (M >= kGemmMinM) return true;
    const int per = wt == QMM_TYPE_Q4_K ? gemv_mma_max_tokens(K) : gemv_mma6_max_tokens(wt, K);
    if (!gemv_use_mma(wt, M, K) || M <= per) return false;
    return (M + per - 1) / per >= (wt == QMM_TYPE_Q4_K ? 3 : 2);
}

// Prefill workspaces: the quantized activations with their per-token scales
// (read-only in the GEMM), then the stream-K partial area that calls owning
// the workspace use.
size_t prefill_act_bytes(qmm_type wt, int64_t M, int64_t K) {
    (void)wt;
    return prefill_operand_bytes(M, K);  // the same layout for every weight type
}

size_t ws_bytes_for(qmm_type wt, int64_t M, int64_t K) {
    if (!use_gemm(wt, M, K) && gemv_use_mma(wt, M, K)) return mma_image_bytes(wt, M, K);
    if (!use_gemm(wt, M, K)) return planar_bytes(M, K, elems(wt), nullptr, nullptr);
    return prefill_act_bytes(wt, M, K) + stream_k_part_bytes();
}

float *ws_part(qmm_type wt, int64_t M, int64_t K, void *ws) {
    return reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + prefill_act_bytes(wt, M, K));
}

qmm_status carve(qmm_type wt, int64_t M, int64_t K, const void *ws, size_t ws_bytes, Planar *p) {
    const size_t need = planar_bytes(M, K, elems(wt), p, (uint8_t *)ws);
    if (ws_bytes < need)
        return set_error(QMM_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", ws_bytes, need);
    return QMM_OK;
}

qmm_status quantize_acts_impl(qmm_type wt, const float *X, int64_t M, int64_t K, void *ws,
                              size_t ws_bytes, cudaStream_t s) {
    if (use_gemm(wt, M, K)) {
        const size_t need = ws_bytes_for(wt, M, K);
        if (ws_bytes < need)
            return set_error(QMM_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", ws_bytes, need);
        if (wt == QMM_TYPE_Q4_0)
            return cuda_status(launch_quantize_q4_0_prefill(X, ws, M, K, s), "prefill quantizer launch");
        return cuda_status(launch_quantize_q8_K_f16(X, ws, M, K, s), "prefill quantizer launch");
    }
    if (gemv_use_mma(wt, M, K)) {
        const size_t need = ws_bytes_for(wt, M, K);
        if (ws_bytes < need)
            return set_error(QMM_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", ws_bytes, need);
        return cuda_status(launch_mma_image(wt, false, X, ws, M, K, s), "activation quantizer launch");
    }
    Planar p;
    qmm_status st = carve(wt, M, K, ws, ws_bytes, &p);
    if (st != QMM_OK) return st;
    return cuda_status(launch_quantize_q8(act_of(wt), true, X, nullptr, p, M, K, s),
                       "activation quantizer launch");
}

// part: for the prefill GEMMs, stream_k_part_bytes() of device memory that
// no other work uses until this call's work on `s` is done.
qmm_status prepared_impl(qmm_type wt, const void *Wp, int64_t N, int64_t K, const void *ws,
                         size_t ws_bytes, int64_t M, float *Y, float *part, cudaStream_t s) {
    if (use_gemm(wt, M, K)) {
        const size_t need = prefill_act_bytes(wt, M, K);
        if (ws_bytes < need)
            return set_error(QMM_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", ws_bytes, need);
        if (wt == QMM_TYPE_Q4_0)
            return cuda_status(launch_gemm_q4_0(Wp, N, K, ws, part, M, Y, s), "prefill GEMM launch");
        if (wt == QMM_TYPE_Q6_K)
            return cuda_status(launch_gemm_q6_K(Wp, N, K, ws, part, M, Y, s), "prefill GEMM launch");
        return cuda_status(launch_gemm_q4_K_f16(Wp, N, K, ws, part, M, Y, s), "prefill GEMM launch");
    }
    if (gemv_use_mma(wt, M, K)) {
        const size_t need = ws_bytes_for(wt, M, K);
        if (ws_bytes < need)
            return set_error(QMM_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", ws_bytes, need);
        return cuda_status(launch_gemv_mma(wt, single_mat(Wp, N, Y), K, ws, M, /*pdl=*/true, s),
                           "mul_mat kernel launch");
    }
    Planar p;
    qmm_status st = carve(wt, M, K, ws, ws_bytes, &p);
    if (st != QMM_OK) return st;
    return cuda_status(launch_gemv(wt, Wp, N, K, p, nullptr, M, Y, /*pdl=*/true, s),
                       "mul_mat kernel launch");
}

// Decode with small M*K quantizes the activations inside the GEMV (one
// launch); otherwise the quantizer runs first into the workspace.
qmm_status mul_mat_impl(qmm_type wt, const void *Wp, int64_t N, int64_t K, const float *X,
                        int64_t M, float *Y, void *ws, size_t ws_bytes, cudaStream_t s) {
    if (gemv_can_fuse(wt, M, K)) {
        Planar none{nullptr, nullptr, nullptr};
        return cuda_status(launch_gemv(wt, Wp, N, K, none, X, M, Y, /*pdl=*/true, s),
                           "mul_mat kernel launch");
    }
    qmm_status st = quantize_acts_impl(wt, X, M, K, ws, ws_bytes, s);
    if (st != QMM_OK) return st;
    return prepared_impl(wt, Wp, N, K, ws, ws_bytes, M, Y, use_gemm(wt, M, K) ? ws_part(wt, M, K, ws) : nullptr,
                         s);
}

// A stream-K partial area of its own for a call whose workspace is shared
// read-only (or that has none): allocated on the stream, freed after `run`.
template <class F>
qmm_status with_own_part(cudaStream_t s, F run) {
    prepare_pool(s);
    void *mem = nullptr;
    const size_t need = stream_k_part_bytes();
    cudaError_t e = cudaMallocAsync(&mem, need, s);
    if (e != cudaSuccess || !mem) {
        cudaGetLastError();
        return set_error(QMM_ERR_NOMEM, "cudaMallocAsync(%zu): %s", need, cudaGetErrorString(e));
    }
    qmm_status st = run(static_cast<float *>(mem));
    cudaError_t ef = cudaFreeAsync(mem, s);
    if (st == QMM_OK && ef != cudaSuccess) return cuda_status(ef, "cudaFreeAsync");
    return st;
}

qmm_status check_mul_mat_args(qmm_type wt, const void *Wp, int64_t N, int64_t K, const float *X,
                              int64_t M, float *Y) {
    qmm_status st = check_weight_args(wt, N, K);
    if (st != QMM_OK) return st;
    QMM_CHECK_ARG(M >= 0, "M must be >= 0 (got %lld)", (long long)M);
    if (M == 0 || N == 0) return QMM_OK;
    QMM_CHECK_ARG(Wp && X && Y, "null pointer argument");
    QMM_CHECK_ARG(aligned(Wp, 16) && aligned(X, 16) && aligned(Y, 4),
                  "W_packed and X must be 16-byte aligned, Y 4-byte aligned");
    return QMM_OK;
}

}  // namespace
}  // namespace qmm

using namespace qmm;

extern "C" {

size_t qmm_block_bytes(qmm_type t) {
    switch (t) {
    case QMM_TYPE_Q4_0: return B_Q4_0;
    case QMM_TYPE_Q4_K: return B_Q4_K;
    case QMM_TYPE_Q8_0: return B_Q8_0;
    case QMM_TYPE_Q8_K: return B_Q8_K;
    case QMM_TYPE_W4A16: return 4;
    case QMM_TYPE_Q6_K: return B_Q6_K;
    default: return 0;
    }
}

int qmm_block_elems(qmm_type t) {
    if (t == QMM_TYPE_W4A16) return 8;
    return (is_weight(t) || is_act(t)) ? elems(t) : 0;
}

size_t qmm_packed_bytes(qmm_type wt, int64_t N, int64_t K) {
    if (wt == QMM_TYPE_W4A16)
        return (N > 0 && K > 0 && K % 128 == 0 && K <= ((int64_t)1 << 30) && N <= ((int64_t)1 << 31))
                   ? (size_t)((N + 15) / 16 * 16) * (size_t)(K / 2)
                   : 0;
    if (!is_weight(wt) || N <= 0 || K <= 0 || K % elems(wt)) return 0;
    return (size_t)tiles_of(N) * kTileRows * (size_t)(K / elems(wt)) * qmm_block_bytes(wt);
}

size_t qmm_workspace_bytes(qmm_type wt, int64_t M, int64_t K) {
    if (!is_weight(wt) || M < 0 || K <= 0 || K % elems(wt)) return 0;
    return ws_bytes_for(wt, M, K);
}

qmm_status qmm_quantize_row_q8(qmm_type vt, const float *X, void *Xq, int64_t M, int64_t K,
                               qmm_stream_t stream) {
    QMM_CHECK_ARG(is_act(vt), "activation type must be Q8_0 or Q8_K (got %d)", (int)vt);
    QMM_CHECK_ARG(M >= 0 && K > 0 && K % elems(vt) == 0,
                  "need M >= 0, K > 0, K %% %d == 0 (M=%lld K=%lld)", elems(vt), (long long)M,
                  (long long)K);
    if (M == 0) return ok();
    QMM_CHECK_ARG(X && Xq, "null pointer argument");
    QMM_CHECK_ARG(aligned(X, 16), "X must be 16-byte aligned");
    QMM_CHECK_ARG(aligned(Xq, vt == QMM_TYPE_Q8_K ? 4 : 2), "Xq misaligned");
    Planar none{nullptr, nullptr, nullptr};
    return cuda_status(launch_quantize_q8(vt, false, X, Xq, none, M, K, (cudaStream_t)stream),
                       "quantizer launch");
}

qmm_status qmm_quantize_weights(qmm_type wt, const float *W, void *Wq, int64_t N, int64_t K,
                                qmm_stream_t stream) {
    qmm_status st = check_weight_args(wt, N, K);
    if (st != QMM_OK) return st;
    if (N == 0) return ok();
    QMM_CHECK_ARG(W && Wq, "null pointer argument");
    QMM_CHECK_ARG(aligned(W, 16), "W must be 16-byte aligned");
    QMM_CHECK_ARG(aligned(Wq, wt == QMM_TYPE_Q4_K ? 16 : 2), "Wq misaligned");
    return cuda_status(launch_quantize_weights(wt, W, Wq, N, K, (cudaStream_t)stream),
                       "weight quantizer launch");
}

static qmm_status repack_common(qmm_type wt, const void *src, void *dst, int64_t N, int64_t K,
                                bool inverse, qmm_stream_t stream) {
    if (wt == QMM_TYPE_W4A16) {
        QMM_CHECK_ARG(N > 0 && K > 0 && K % 128 == 0, "W4A16 needs N > 0, K > 0, K %% 128 == 0 "
                      "(N=%lld K=%lld)", (long long)N, (long long)K);
        QMM_CHECK_ARG(qmm_packed_bytes(wt, N, K) > 0, "sizes too large");
        QMM_CHECK_ARG(src && dst, "null pointer argument");
        QMM_CHECK_ARG(aligned(src, 16) && aligned(dst, 16), "W4A16 buffers must be 16-byte aligned");
        const uintptr_t a = (uintptr_t)src, b = (uintptr_t)dst;
        const size_t pb = qmm_packed_bytes(wt, N, K), cb = (size_t)N * (size_t)(K / 2);
        const size_t sb = inverse ? pb : cb, db = inverse ? cb : pb;
        QMM_CHECK_ARG(a + sb <= b || b + db <= a, "source and destination overlap");
        return cuda_status(launch_w4a16_repack(inverse, src, dst, N, K, (cudaStream_t)stream),
                           "repack launch");
    }
    qmm_status st = check_weight_args(wt, N, K);
    if (st != QMM_OK) return st;
    QMM_CHECK_ARG(N > 0, "N must be > 0");
    QMM_CHECK_ARG(src && dst, "null pointer argument");
    const void *canon = inverse ? dst : src;
    const void *packed = inverse ? src : dst;
    QMM_CHECK_ARG(aligned(packed, 16), "packed weights must be 16-byte aligned");
    QMM_CHECK_ARG(aligned(canon, wt == QMM_TYPE_Q4_K ? 16 : 2), "canonical weights misaligned");
    // canonical blocks span N rows, packed ones are padded to whole tiles
    const uintptr_t a = (uintptr_t)src, b = (uintptr_t)dst;
    const size_t pb = qmm_packed_bytes(wt, N, K);
    const size_t cb = (size_t)N * (size_t)(K / qmm_block_elems(wt)) * qmm_block_bytes(wt);
    const size_t sb = inverse ? pb : cb, db = inverse ? cb : pb;
    QMM_CHECK_ARG(a + sb <= b || b + db <= a, "source and destination overlap");
    return cuda_status(launch_repack(wt, inverse, src, dst, N, K, (cudaStream_t)stream),
                       "repack launch");
}

qmm_status qmm_repack_weights(qmm_type wt, const void *W_canon, void *W_packed, int64_t N,
                              int64_t K, qmm_stream_t stream) {
    return repack_common(wt, W_canon, W_packed, N, K, false, stream);
}

qmm_status qmm_unrepack_weights(qmm_type wt, const void *W_packed, void *W_canon, int64_t N,
                                int64_t K, qmm_stream_t stream) {
    return repack_common(wt, W_packed, W_canon, N, K, true, stream);
}

qmm_status qmm_mul_mat_ws(qmm_type wt, const void *W_packed, int64_t N, int64_t K, const float *X,
                          int64_t M, float *Y, void *workspace, size_t ws_bytes,
                          qmm_stream_t stream) {
    qmm_status st = check_mul_mat_args(wt, W_packed, N, K, X, M, Y);
    if (st != QMM_OK) return st;
    if (M == 0 || N == 0) return ok();
    QMM_CHECK_ARG(workspace && aligned(workspace, 16), "workspace must be non-null, 16-byte aligned");
    const size_t need = qmm_workspace_bytes(wt, M, K);
    if (ws_bytes < need)
        return set_error(QMM_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", ws_bytes, need);
    return mul_mat_impl(wt, W_packed, N, K, X, M, Y, workspace, ws_bytes, (cudaStream_t)stream);
}

// X of qmm_mul_mat_host from mapped host memory into device_buf: one pass,
// 16 bytes per thread (X_host and the buffer are 16-byte aligned, M K is a
// multiple of 32). It follows the previous kernel in the stream, which may
// still read the buffer, and lets the GEMV after it launch early.
__global__ void __launch_bounds__(256) pull_x_kernel(const float4 *__restrict__ src, float4 *__restrict__ dst,
                                                     int64_t n4) {
    if (threadIdx.x == 0) pdl_launch_dependents();
    pdl_wait();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

// Whether a host pointer from cudaHostAlloc / cudaHostRegister is usable on
// the current device as it is (cached per device).
static bool host_pointers_usable() {
    static int cached[64] = {};  // 0 unknown, 1 yes, 2 no
    const int d = current_device();
    if (d < 0 || d >= 64) return false;
    if (!cached[d]) {
        int uva = 0, reg = 0;
        cudaDeviceGetAttribute(&uva, cudaDevAttrUnifiedAddressing, d);
        cudaDeviceGetAttribute(&reg, cudaDevAttrCanUseHostPointerForRegisteredMem, d);
        cudaGetLastError();
        cached[d] = uva && reg ? 1 : 2;
    }
    return cached[d] == 1;
}

// Device buffer of qmm_mul_mat_host: X, then Y, then the workspace.
static size_t host_x_bytes(int64_t M, int64_t K) { return (size_t)align_up((uint64_t)M * K * 4, 16); }
static size_t host_y_bytes(int64_t M, int64_t N) { return (size_t)align_up((uint64_t)M * N * 4, 16); }

size_t qmm_host_call_bytes(qmm_type wt, int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || (M > 0 && qmm_workspace_bytes(wt, M, K) == 0)) return 0;
    if (M == 0 || N == 0) return 16;
    return host_x_bytes(M, K) + host_y_bytes(M, N) + qmm_workspace_bytes(wt, M, K);
}

qmm_status qmm_mul_mat_host(qmm_type wt, const void *W_packed, int64_t N, int64_t K, const float *X_host,
                            int64_t M, float *Y_host, void *device_buf, size_t buf_bytes, unsigned flags,
                            qmm_stream_t stream) {
    qmm_status st = check_weight_args(wt, N, K);
    if (st != QMM_OK) return st;
    QMM_CHECK_ARG(M >= 0, "M must be >= 0 (got %lld)", (long long)M);
    if (M == 0 || N == 0) return ok();
    QMM_CHECK_ARG(W_packed && X_host && Y_host && device_buf, "null pointer argument");
    QMM_CHECK_ARG(aligned(W_packed, 16) && aligned(device_buf, 16),
                  "W_packed and device_buf must be 16-byte aligned");
    const size_t need = qmm_host_call_bytes(wt, M, N, K);
    if (buf_bytes < need)
        return set_error(QMM_ERR_WORKSPACE, "device buffer of %zu bytes < %zu needed", buf_bytes, need);
    cudaStream_t s = (cudaStream_t)stream;
    uint8_t *base = static_cast<uint8_t *>(device_buf);
    float *Xd = reinterpret_cast<float *>(base);
    float *Yd = reinterpret_cast<float *>(base + host_x_bytes(M, K));
    void *ws = base + host_x_bytes(M, K) + host_y_bytes(M, N);
    const size_t ws_bytes = buf_bytes - host_x_bytes(M, K) - host_y_bytes(M, N);
    QMM_CHECK_ARG((flags & ~QMM_HOST_MAPPED) == 0, "unknown flags 0x%x", flags);
    if (flags & QMM_HOST_MAPPED) {
        if (!host_pointers_usable())
            return set_error(QMM_ERR_UNSUPPORTED, "this device cannot use host pointers directly");
        QMM_CHECK_ARG(aligned(X_host, 16) && aligned(Y_host, 4), "X_host must be 16-byte aligned, Y_host 4-byte");
        const int64_t n4 = M * K / 4;
        cudaLaunchConfig_t cfg = {};
        const int64_t blocks = (n4 + 255) / 256;
        cfg.gridDim = dim3((unsigned)(blocks < 64 ? blocks : 64));
        cfg.blockDim = dim3(256);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, pull_x_kernel, reinterpret_cast<const float4 *>(X_host),
                                           reinterpret_cast<float4 *>(Xd), n4);
        count_launch();
        if (e != cudaSuccess) return cuda_status(e, "X pull launch");
        return mul_mat_impl(wt, W_packed, N, K, Xd, M, Y_host, ws, ws_bytes, s);
    }
    // X goes in by one asynchronous copy (the kernels read it many times,
    // from L2); Y, written once, goes straight to the caller's memory when
    // that is page-locked and mapped into the device's address space (what
    // cudaHostAlloc and cudaHostRegister give on this system), which saves
    // the copy call back -- else by a copy from device_buf.
    cudaPointerAttributes ay = {};
    const bool y_mapped = cudaPointerGetAttributes(&ay, Y_host) == cudaSuccess && ay.type == cudaMemoryTypeHost &&
                          ay.devicePointer && aligned(ay.devicePointer, 4);
    cudaGetLastError();  // a failed query is not an error of this call
    cudaError_t e = cudaMemcpyAsync(Xd, X_host, (size_t)M * K * 4, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_status(e, "X host-to-device copy");
    if (y_mapped) return mul_mat_impl(wt, W_packed, N, K, Xd, M, static_cast<float *>(ay.devicePointer), ws, ws_bytes, s);
    st = mul_mat_impl(wt, W_packed, N, K, Xd, M, Yd, ws, ws_bytes, s);
    if (st != QMM_OK) return st;
    e = cudaMemcpyAsync(Y_host, Yd, (size_t)M * N * 4, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_status(e, "Y device-to-host copy");
    return ok();
}

qmm_status qmm_quantize_activations(qmm_type wt, const float *X, int64_t M, int64_t K,
                                    void *workspace, size_t ws_bytes, qmm_stream_t stream) {
    qmm_status st = check_weight_args(wt, 1, K);
    if (st != QMM_OK) return st;
    QMM_CHECK_ARG(M >= 0, "M must be >= 0 (got %lld)", (long long)M);
    if (M == 0) return ok();
    QMM_CHECK_ARG(X && workspace, "null pointer argument");
    QMM_CHECK_ARG(aligned(X, 16) && aligned(workspace, 16),
                  "X and workspace must be 16-byte aligned");
    return quantize_acts_impl(wt, X, M, K, workspace, ws_bytes, (cudaStream_t)stream);
}

qmm_status qmm_mul_mat_prepared(qmm_type wt, const void *W_packed, int64_t N, int64_t K,
                                const void *workspace, size_t ws_bytes, int64_t M, float *Y,
                                qmm_stream_t stream) {
    qmm_status st = check_weight_args(wt, N, K);
    if (st != QMM_OK) return st;
    QMM_CHECK_ARG(M >= 0, "M must be >= 0 (got %lld)", (long long)M);
    if (M == 0 || N == 0) return ok();
    QMM_CHECK_ARG(W_packed && workspace && Y, "null pointer argument");
    QMM_CHECK_ARG(aligned(W_packed, 16) && aligned(workspace, 16) && aligned(Y, 4),
                  "W_packed and workspace must be 16-byte aligned, Y 4-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    if (!use_gemm(wt, M, K) || !stream_k_splits(wt, N, M, K))  // nothing to allocate
        return prepared_impl(wt, W_packed, N, K, workspace, ws_bytes, M, Y, nullptr, s);
    if (ws_bytes < prefill_act_bytes(wt, M, K))  // before allocating anything
        return set_error(QMM_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", ws_bytes,
                         prefill_act_bytes(wt, M, K));
    return with_own_part(s, [&](float *part) {
        return prepared_impl(wt, W_packed, N, K, workspace, ws_bytes, M, Y, part, s);
    });
}

qmm_status qmm_mul_mat(qmm_type wt, const void *W_packed, int64_t N, int64_t K, const float *X,
                       int64_t M, float *Y, qmm_stream_t stream) {
    qmm_status st = check_mul_mat_args(wt, W_packed, N, K, X, M, Y);
    if (st != QMM_OK) return st;
    if (M == 0 || N == 0) return ok();
    cudaStream_t s = (cudaStream_t)stream;
    if (gemv_can_fuse(wt, M, K))  // one kernel, no workspace to allocate
        return mul_mat_impl(wt, W_packed, N, K, X, M, Y, nullptr, 0, s);
    prepare_pool(s);
    const size_t need = qmm_workspace_bytes(wt, M, K);
    void *ws = nullptr;
    cudaError_t e = cudaMallocAsync(&ws, need, s);
    if (e != cudaSuccess || !ws) {
        cudaGetLastError();
        return set_error(QMM_ERR_NOMEM, "cudaMallocAsync(%zu): %s", need, cudaGetErrorString(e));
    }
    st = mul_mat_impl(wt, W_packed, N, K, X, M, Y, ws, need, s);
    cudaError_t ef = cudaFreeAsync(ws, s);
    if (st == QMM_OK && ef != cudaSuccess) return cuda_status(ef, "cudaFreeAsync");
    return st;
}

qmm_status qmm_mul_mat_q8(qmm_type wt, const void *W_packed, int64_t N, int64_t K, const void *Xq,
                          int64_t M, float *Y, qmm_stream_t stream) {
    qmm_status st = check_weight_args(wt, N, K);
    if (st != QMM_OK) return st;
    QMM_CHECK_ARG(M >= 0, "M must be >= 0 (got %lld)", (long long)M);
    if (M == 0 || N == 0) return ok();
    QMM_CHECK_ARG(W_packed && Xq && Y, "null pointer argument");
    QMM_CHECK_ARG(aligned(W_packed, 16) && aligned(Y, 4), "W_packed must be 16-byte aligned, Y 4-byte");
    QMM_CHECK_ARG(aligned(Xq, act_of(wt) == QMM_TYPE_Q8_K ? 4 : 2),
                  "Xq must be aligned like its blocks (Q8_K: 4 bytes, Q8_0: 2 bytes)");
    cudaStream_t s = (cudaStream_t)stream;
    prepare_pool(s);
    const size_t need = qmm_workspace_bytes(wt, M, K);
    void *ws = nullptr;
    cudaError_t e = cudaMallocAsync(&ws, need, s);
    if (e != cudaSuccess || !ws) {
        cudaGetLastError();
        return set_error(QMM_ERR_NOMEM, "cudaMallocAsync(%zu): %s", need, cudaGetErrorString(e));
    }
    // the caller's blocks, rewritten into the layout the kernel for (wt, M, K) reads
    if (use_gemm(wt, M, K)) {
        if (wt == QMM_TYPE_Q4_0) {
            e = launch_import_q4_0_prefill(Xq, ws, M, K, s);
        } else {
            e = launch_import_q8_K_f16(Xq, ws, M, K, s);
        }
    } else if (gemv_use_mma(wt, M, K)) {
        e = launch_mma_image(wt, true, Xq, ws, M, K, s);
    } else {
        Planar p;
        planar_bytes(M, K, elems(wt), &p, (uint8_t *)ws);
        e = launch_import_q8_planar(act_of(wt), Xq, p, M, K, s);
    }
    st = cuda_status(e, "activation import launch");
    if (st == QMM_OK)
        st = prepared_impl(wt, W_packed, N, K, ws, need, M, Y, use_gemm(wt, M, K) ? ws_part(wt, M, K, ws) : nullptr, s);
    cudaError_t ef = cudaFreeAsync(ws, s);
    if (st == QMM_OK && ef != cudaSuccess) return cuda_status(ef, "cudaFreeAsync");
    return st;
}

qmm_status qmm_mul_mat_multi(qmm_type wt, int n, const void *const *W_packed, const int64_t *N,
                             int64_t K, const float *X, int64_t M, float *const *Y,
                             qmm_stream_t stream) {
    QMM_CHECK_ARG(n >= 1 && n <= kMaxMats, "n must be 1..%d (got %d)", kMaxMats, n);
    QMM_CHECK_ARG(W_packed && N && Y, "null array argument");
    MatSet ms = {};
    for (int i = 0; i < n; ++i) {
        qmm_status st = check_mul_mat_args(wt, W_packed[i], N[i], K, X, M, Y[i]);
        if (st != QMM_OK) return st;
        if (N[i] == 0) continue;
        ms.W[ms.n] = static_cast<const uint8_t *>(W_packed[i]);
        ms.N[ms.n] = N[i];
        ms.Y[ms.n] = Y[i];
        ++ms.n;
    }
    if (M == 0 || ms.n == 0) return ok();
    cudaStream_t s = (cudaStream_t)stream;
    if (!use_gemm(wt, M, K) && gemv_can_fuse(wt, M, K)) {  // one kernel, no workspace
        Planar none{nullptr, nullptr, nullptr};
        return cuda_status(launch_gemv(wt, ms, K, none, X, M, /*pdl=*/true, s), "mul_mat kernel launch");
    }
    prepare_pool(s);
    const size_t need = qmm_workspace_bytes(wt, M, K);
    void *ws = nullptr;
    cudaError_t e = cudaMallocAsync(&ws, need, s);
    if (e != cudaSuccess || !ws) {
        cudaGetLastError();
        return set_error(QMM_ERR_NOMEM, "cudaMallocAsync(%zu): %s", need, cudaGetErrorString(e));
    }
    // one quantization of X serves every matrix; the GEMMs take the
    // stream-K partial area in turn, in stream order
    qmm_status st = quantize_acts_impl(wt, X, M, K, ws, need, s);
    if (st == QMM_OK) {
        if (use_gemm(wt, M, K)) {
            for (int i = 0; i < ms.n && st == QMM_OK; ++i)
                st = prepared_impl(wt, ms.W[i], ms.N[i], K, ws, need, M, ms.Y[i], ws_part(wt, M, K, ws), s);
        } else if (gemv_use_mma(wt, M, K)) {
            st = cuda_status(launch_gemv_mma(wt, ms, K, ws, M, /*pdl=*/true, s),
                             "mul_mat kernel launch");
        } else {
            Planar p;
            st = carve(wt, M, K, ws, need, &p);
            if (st == QMM_OK)
                st = cuda_status(launch_gemv(wt, ms, K, p, nullptr, M, /*pdl=*/true, s),
                                 "mul_mat kernel launch");
        }
    }
    cudaError_t ef = cudaFreeAsync(ws, s);
    if (st == QMM_OK && ef != cudaSuccess) return cuda_status(ef, "cudaFreeAsync");
    return st;
}

qmm_status qmm_w4a16_unpack_zeros(const uint32_t *zeros_packed, uint8_t *zeros, int64_t N,
                                  int64_t ngroups, qmm_stream_t stream) {
    QMM_CHECK_ARG(N >= 0 && ngroups >= 1, "need N >= 0 and ngroups >= 1 (N=%lld ngroups=%lld)",
                  (long long)N, (long long)ngroups);
    QMM_CHECK_ARG(N <= ((int64_t)1 << 31) && ngroups <= ((int64_t)1 << 30), "sizes too large");
    if (N == 0) return ok();
    QMM_CHECK_ARG(zeros_packed && zeros, "null pointer argument");
    return cuda_status(launch_w4a16_unpack_zeros(zeros_packed, zeros, N, ngroups, (cudaStream_t)stream),
                       "W4A16 zero unpack launch");
}

qmm_status qmm_debug_block_sums(qmm_type wt, const void *W_packed, int64_t N, int64_t K,
                                const void *Xq, int64_t M, int32_t *out, qmm_stream_t stream) {
    qmm_status st = check_weight_args(wt, N, K);
    if (st != QMM_OK) return st;
    QMM_CHECK_ARG(M >= 0, "M must be >= 0");
    if (M == 0 || N == 0) return ok();
    QMM_CHECK_ARG(W_packed && Xq && out, "null pointer argument");
    QMM_CHECK_ARG(aligned(W_packed, 16) && aligned(out, 4), "misaligned pointer");
    QMM_CHECK_ARG(aligned(Xq, act_of(wt) == QMM_TYPE_Q8_K ? 4 : 2), "Xq misaligned");
    return cuda_status(
        launch_debug_block_sums(wt, W_packed, N, K, Xq, M, out, (cudaStream_t)stream),
        "debug kernel launch");
}

qmm_status qmm_debug_wait_timeout(int64_t limit_cycles, qmm_stream_t stream) {
    QMM_CHECK_ARG(limit_cycles > 0 && limit_cycles <= 20000000000LL,
                  "limit_cycles must be in (0, 2e10] (got %lld)", (long long)limit_cycles);
    return cuda_status(launch_debug_wait_timeout(limit_cycles, (cudaStream_t)stream),
                       "debug kernel launch");
}

qmm_status qmm_debug_peak(int which, int64_t iters, double *ops, qmm_stream_t stream) {
    QMM_CHECK_ARG(which >= QMM_PEAK_MMA_S8 && which <= QMM_PEAK_TC_TS_256, "unknown peak kind %d", which);
    QMM_CHECK_ARG(iters >= 1 && iters <= 1000000, "iters must be in [1, 1e6] (got %lld)", (long long)iters);
    QMM_CHECK_ARG(ops != nullptr, "null pointer argument");
    return cuda_status(launch_debug_peak(which, iters, (cudaStream_t)stream, ops), "peak kernel launch");
}

const char *qmm_status_string(qmm_status s) {
    switch (s) {
    case QMM_OK: return "QMM_OK";
    case QMM_ERR_ARG: return "QMM_ERR_ARG";
    case QMM_ERR_UNSUPPORTED: return "QMM_ERR_UNSUPPORTED";
    case QMM_ERR_CUDA: return "QMM_ERR_CUDA";
    case QMM_ERR_TIMEOUT: return "QMM_ERR_TIMEOUT";
    case QMM_ERR_NOMEM: return "QMM_ERR_NOMEM";
    case QMM_ERR_WORKSPACE: return "QMM_ERR_WORKSPACE";
    default: return "QMM_ERR_UNKNOWN";
    }
}

const char *qmm_last_error(void) { return g_msg; }

qmm_status qmm_check_device_error(qmm_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_status(e, "stream synchronize");
    unsigned *w = device_error_word();
    if (!w) return set_error(QMM_ERR_CUDA, "device error word unavailable");
    unsigned v = 0;
    e = cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_status(e, "read device error word");
    if (v) {
        const unsigned zero = 0;
        cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    }
    if (v & kDevErrTimeout)
        return set_error(QMM_ERR_TIMEOUT, "a kernel gave up a bounded device-side wait");
    return ok();
}

uint64_t qmm_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

// Both W4A16 forms: zeros != nullptr, W-hat = s (q - z); lut != nullptr,
// W-hat = s LUT(q).
static qmm_status w4a16_impl(const char *fn, const void *W_packed, const uint16_t *scales,
                             const uint8_t *zeros, const uint16_t *lut, int64_t G, const uint16_t *A,
                             uint16_t *C, int64_t M, int64_t N, int64_t K, qmm_stream_t stream) {
    QMM_CHECK_ARG(M >= 0 && N >= 0 && K > 0 && G > 0,
                  "%s: sizes must satisfy M, N >= 0, K, G > 0 (M=%lld N=%lld K=%lld G=%lld)", fn,
                  (long long)M, (long long)N, (long long)K, (long long)G);
    QMM_CHECK_ARG(K % G == 0 && G % 8 == 0, "%s: need K %% G == 0 and G %% 8 == 0 (K=%lld G=%lld)",
                  fn, (long long)K, (long long)G);
    QMM_CHECK_ARG(K <= ((int64_t)1 << 30) && N <= ((int64_t)1 << 31) && M <= ((int64_t)1 << 31),
                  "%s: sizes too large", fn);
    if (G % 128 != 0)
        return set_error(QMM_ERR_UNSUPPORTED, "%s: group size %lld: this build needs G %% 128 == 0", fn,
                         (long long)G);
    if (M == 0 || N == 0) return ok();
    QMM_CHECK_ARG(W_packed && scales && (zeros || lut) && A && C, "%s: null pointer argument", fn);
    QMM_CHECK_ARG(aligned(W_packed, 16) && aligned(A, 16) && aligned(scales, 16) &&
                      (lut ? aligned(lut, 2) : aligned(zeros, 16)),
                  "%s: W_packed, scales, zeros and A must be 16-byte aligned, lut 2-byte", fn);
    QMM_CHECK_ARG(aligned(C, 2), "%s: C must be 2-byte aligned", fn);
    if (K / G > 256)
        return set_error(QMM_ERR_UNSUPPORTED, "%s: %lld groups per row: this build stages "
                         "at most 256 (K / G)", fn, (long long)(K / G));
    cudaStream_t s = (cudaStream_t)stream;
    const __half *S = reinterpret_cast<const __half *>(scales);
    const __half *L = reinterpret_cast<const __half *>(lut);
    const __half *Ah = reinterpret_cast<const __half *>(A);
    __half *Ch = reinterpret_cast<__half *>(C);
    // up to 16 tokens: the decode kernel (HBM-bound); more: the tensor-core
    // GEMM, whose split tiles go through a stream-ordered partial area
    if (M <= 16)
        return cuda_status(launch_w4a16_decode(W_packed, S, zeros, L, G, Ah, Ch, M, N, K, s),
                           "W4A16 kernel launch");
    if (!stream_k_splits(QMM_TYPE_W4A16, N, M, K))  // one CTA per tile: no partial area
        return cuda_status(launch_w4a16_gemm(W_packed, S, zeros, L, G, Ah, Ch, M, N, K, nullptr, s),
                           "W4A16 kernel launch");
    return with_own_part(s, [&](float *part) {
        return cuda_status(launch_w4a16_gemm(W_packed, S, zeros, L, G, Ah, Ch, M, N, K, part, s),
                           "W4A16 kernel launch");
    });
}

qmm_status qmm_w4a16(const void *W_packed, const uint16_t *scales, const uint8_t *zeros, int64_t G,
                     const uint16_t *A, uint16_t *C, int64_t M, int64_t N, int64_t K,
                     qmm_stream_t stream) {
    if (M > 0 && N > 0 && !zeros) return set_error(QMM_ERR_ARG, "qmm_w4a16: null pointer argument");
    return w4a16_impl("qmm_w4a16", W_packed, scales, zeros, nullptr, G, A, C, M, N, K, stream);
}

qmm_status qmm_w4a16_lut(const void *W_packed, const uint16_t *scales, const uint16_t *lut, int64_t G,
                         const uint16_t *A, uint16_t *C, int64_t M, int64_t N, int64_t K,
                         qmm_stream_t stream) {
    if (M > 0 && N > 0 && !lut) return set_error(QMM_ERR_ARG, "qmm_w4a16_lut: null pointer argument");
    return w4a16_impl("qmm_w4a16_lut", W_packed, scales, nullptr, lut, G, A, C, M, N, K, stream);
}

}  // extern "C"
