/*
 * qmm.h -- C ABI of libqmm, block-quantized matrix multiplication on GB300
 * (sm_103a).
 *
 * The library computes a linear layer y = W x whose weights are stored in
 * ggml's 4-bit block formats, with the activations quantized on the fly to
 * 8-bit blocks and the product taken as an integer block dot product with
 * fp32 accumulation, as described on the page
 *   "llama.cpp 源码完全拆解(十三): ggml-cpu 的一次 mul_mat"
 * (sections on the Q4_0/Q8_0 and K-quant block layouts, the 6-bit scale
 * packing, the scale-factoring identity and the mul_mat steps), plus the
 * W4A16 group-asymmetric form of
 *   "BitBLAS 完全拆解: 低比特权重如何在 Tensor Core 上边解码边计算"
 * (sections "从数学表达式到真实存储" and "位级打包").
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers unless the argument says "host".
 *   - W is [N, K]: N output rows of K/QK blocks each (QK = 32 for Q4_0 and
 *     Q8_0, 256 for Q4_K, Q6_K and Q8_K). X is fp32 [M, K] row-major. Y is fp32
 *     [M, N] row-major: Y[m * N + n] = sum_k W[n, k] X[m, k].
 *   - "Canonical" blocks are the packed little-endian structs the page prints
 *     (no padding): block_q4_0 {fp16 d; u8 qs[16]} 18 B; block_q8_0 {fp16 d;
 *     i8 qs[32]} 34 B; block_q4_K {fp16 d; fp16 dmin; u8 scales[12];
 *     u8 qs[128]} 144 B; block_q8_K {f32 d; i8 qs[256]; i16 bsums[16]} 292 B;
 *     block_q6_K {u8 ql[128]; u8 qh[64]; i8 scales[16]; fp16 d} 210 B
 *     (field order as the page lists them; bit order in qmm_quantize_weights).
 *     A row of K elements is K/QK consecutive blocks; rows are consecutive.
 *     This is the interchange format. "Packed" weights are this library's
 *     private GPU layout, made from canonical blocks by qmm_repack_weights.
 *   - The caller owns every buffer; the library never frees caller memory.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream);
 *     no call synchronizes the host except qmm_check_device_error.
 *   - The mul_mat and W4A16 kernels launch with programmatic dependent launch:
 *     they may start while the preceding kernel on the stream is finishing
 *     and stream their weights (packed weights, W4A16 scales, zeros and code
 *     table) at once; they read the activations and write the outputs only
 *     after that kernel has completed. Weights are load-time data: the kernel
 *     immediately preceding a call must not write them (a repack or weight
 *     quantizer of this library never lets the next kernel start early).
 *   - Device buffers must be 16-byte aligned, except canonical Q4_0/Q8_0/Q6_K
 *     buffers (18/34/210-byte blocks), which need 2-byte alignment.
 *   - Errors: arguments are validated before anything is enqueued; on any
 *     error nothing is launched and a qmm_status other than QMM_OK is
 *     returned (qmm_last_error() gives a one-line reason). Kernels never trap:
 *     a device-side wait that exceeds its bound records QMM_ERR_TIMEOUT in a
 *     device error word, read and cleared by qmm_check_device_error.
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-compatible with cudaStream_t / CUstream. */
typedef struct CUstream_st *qmm_stream_t;

typedef enum {
    QMM_TYPE_Q4_0 = 0, /* weights: 32 x 4-bit, fp16 d;       w = d (q - 8)            */
    QMM_TYPE_Q4_K = 1, /* weights: 256 x 4-bit, 8 sub-blocks; w = d s_j q - dmin m_j  */
    QMM_TYPE_Q8_0 = 2, /* activations: 32 x int8, fp16 d;     a = d q                  */
    QMM_TYPE_Q8_K = 3, /* activations: 256 x int8, fp32 d, 16 sums of 16 codes        */
    QMM_TYPE_W4A16 = 4, /* weights: 4-bit codes q, 8 per uint32 word; per row and group
                          of G elements an fp16 scale s and a uint8 zero z:
                          w = s (q - z). Used by qmm_w4a16 only.               */
    QMM_TYPE_Q6_K = 5   /* weights: 256 x 6-bit (ql[128] low 4 bits, qh[64] high 2),
                          16 int8 scales, fp16 d; w = d s_j q, q in -32..31, no
                          min (page 1, "更低的比特: Q6_K 与 Q2_K 的取舍"); 210 B.
                          Activations Q8_K.                                    */
} qmm_type;

typedef enum {
    QMM_OK = 0,
    QMM_ERR_ARG = 1,         /* null pointer, bad size, misaligned pointer, bad type */
    QMM_ERR_UNSUPPORTED = 2, /* valid request this build does not implement          */
    QMM_ERR_CUDA = 3,        /* a CUDA runtime call failed                           */
    QMM_ERR_TIMEOUT = 4,     /* a device-side wait exceeded its bound                */
    QMM_ERR_NOMEM = 5,       /* the library could not allocate its workspace         */
    QMM_ERR_WORKSPACE = 6    /* caller workspace smaller than qmm_workspace_bytes    */
} qmm_status;

/* ---------------------------------------------------------------- sizes */

/* Bytes of one canonical block: 18, 144, 34, 292, 210 (Q6_K), and 4 for
 * W4A16 (one uint32 word of 8 codes); 0 for an invalid type.
 * (Block layouts: page 1, "最基础的两块: Q4_0 与 Q8_0", "K-quant", "更低的比特";
 * W4A16: page 3, "位级打包".) */
size_t qmm_block_bytes(qmm_type t);

/* Elements per block: 32, 256, or 8 for W4A16; 0 for an invalid type. */
int qmm_block_elems(qmm_type t);

/* Bytes of the packed (repacked) weight buffer for an [N, K] weight of type
 * Q4_0, Q4_K, Q6_K or W4A16; 0 if the type or sizes are invalid. Q4_0, Q4_K
 * and Q6_K rows are padded to a multiple of 8 with zero blocks, W4A16 rows to a multiple
 * of 16 (K % 128 == 0): ceil(N / 16) * 16 * K / 2 bytes. */
size_t qmm_packed_bytes(qmm_type wt, int64_t N, int64_t K);

/* Bytes of the workspace qmm_mul_mat_ws needs for M activation rows of
 * length K against weights of type wt (Q4_0, Q4_K or Q6_K); 0 if invalid.
 * When the call runs the tensor-core GEMM (above 16 tokens, or a decode
 * batch with a K too large for the tensor-core GEMV's single launch, see
 * qmm_mul_mat) it ends with a partial area of about 20 MB: with more output tiles
 * than SMs the GEMM gives each SM an equal share of the
 * (tile, K-step) work (stream-K), with fewer than half as many it splits K
 * over the SMs, and the parts of tiles that several CTAs computed meet
 * there before a second kernel adds them. */
size_t qmm_workspace_bytes(qmm_type wt, int64_t M, int64_t K);

/* ---------------------------------------------------------------- quantizers */

/* Quantize fp32 activations X [M, K] into canonical blocks Xq of type vt
 * (Q8_0 or Q8_K), M rows of K/QK blocks (page 1, "最基础的两块" for Q8_0 and
 * "更低的比特" for Q8_K with its bsums; the mul_mat step "激活得先变成 Q8_K").
 * Per block: amax = max |x|, d = amax / 127, q = round-half-away(x / d)
 * clamped to [-127, 127] (computed as x * (1/d) in fp32); Q8_0 stores d as
 * fp16, Q8_K as fp32 plus bsums[t] = sum of codes 16t..16t+15. An all-zero
 * block gives d = 0 and q = 0. Bit-identical to the CPU oracle.
 * Errors: QMM_ERR_ARG if vt is not Q8_0/Q8_K, M < 0, K <= 0 or K % QK != 0,
 * or a pointer is null while M > 0. M == 0 is a no-op. */
qmm_status qmm_quantize_row_q8(qmm_type vt, const float *X, void *Xq, int64_t M, int64_t K,
                               qmm_stream_t stream);

/* Quantize fp32 weights W [N, K] into canonical blocks Wq of type wt (Q4_0,
 * Q4_K or Q6_K) -- the offline quantizer's job, done on the GPU.
 * Q4_0 (page 1, "最基础的两块"): d = -x_max / 8 where x_max is the signed
 * value of largest magnitude (the first on ties); q = clamp(floor(x * (1/d)
 * + 8.5), 0, 15); d stored as fp16; byte l holds element l (low nibble) and
 * element l + 16 (high nibble).
 * Q4_K (page 1, "K-quant", "6-bit 参数", nibble packing in "正确性"): per
 * sub-block j of 32: lo = min(0, min x), hi = max x, sc_j = (hi - lo) / 15,
 * mn_j = -lo; d = max sc_j / 63, dmin = max mn_j / 63 (fp16);
 * s_j = clamp(round(sc_j / d), 0, 63), m_j = clamp(round(mn_j / dmin), 0, 63);
 * q = clamp(round((x + dmin16 m_j) / (d16 s_j)), 0, 15) with the stored fp16
 * d16, dmin16; scales packed in 12 bytes, qs[32c + l] = q[64c + l] |
 * q[64c + 32 + l] << 4. The pages print the format but not the scale search;
 * this single-pass min/max search is this library's reading.
 * Q6_K (page 1, "更低的比特"): per group j of 16: sc_j = -x_max,j / 32 (x_max,j
 * the signed value of largest magnitude, the first on ties); d = max |sc_j|
 * / 127 (fp16); s_j = clamp(round(sc_j / d), -127, 127) (int8); q =
 * clamp(round(x / (d16 s_j)), -32, 31), stored u = q + 32 with
 * ql[32c + l] = (u[64c + l] & 15) | (u[64c + 32 + l] & 15) << 4 and
 * qh[32h + l] = sum_i (u[128h + 32i + l] >> 4) << 2i. The scale search and
 * the bit order are this library's readings (the page gives the fields).
 * Bit-identical to the CPU oracle. Errors as qmm_quantize_row_q8. */
qmm_status qmm_quantize_weights(qmm_type wt, const float *W, void *Wq, int64_t N, int64_t K,
                                qmm_stream_t stream);

/* ---------------------------------------------------------------- layout */

/* Repack canonical weight blocks W_canon ([N] rows of K/QK blocks) into the
 * private GPU layout W_packed (qmm_packed_bytes bytes), once at load time
 * (page 3, "Ladder Permutation": permute offline so run-time reads are
 * contiguous; page 4 on GGML_CPU_REPACK). A pure byte permutation: rows are
 * grouped in tiles of 8 and, within a tile, blocks of the same K position are
 * adjacent; Q4_0 blocks are split into a 16-byte nibble plane and an fp16
 * scale plane; Q6_K blocks of a tile and super-block form one 1680-byte
 * record (8 x 192 bytes of codes, the high bits regrouped per 16-byte ql
 * slice; 8 x 16 scale bytes, regrouped likewise; 8 fp16 d). W_packed must
 * not overlap W_canon.
 * Errors: QMM_ERR_ARG for a non-weight type, N <= 0, K <= 0, K % QK != 0,
 * null or misaligned pointers. */
qmm_status qmm_repack_weights(qmm_type wt, const void *W_canon, void *W_packed, int64_t N,
                              int64_t K, qmm_stream_t stream);

/* W4A16 (wt = QMM_TYPE_W4A16): W_canon is qweight [N][K/8] uint32, element
 * k = 8c + i of a row in bits 4i..4i+3 of word c (page 3, "位级打包"). The
 * packed layout groups rows in tiles of 16 (zero rows pad the last one) and
 * stores a tile as consecutive 1 KB pieces, one per 128 elements of K (its
 * 16 rows x 16 words), and interleaves the nibbles of every word, even
 * elements in the low 16 bits and odd ones in the high 16 bits (nibble
 * slots 0..7 hold elements 0, 2, 4, 6, 1, 3, 5, 7), so that one mask turns
 * a word into fp16 pairs (k, k + 1) (page 3, "Ladder": the weight is laid
 * out once for the decoder). Needs K % 128 == 0; both buffers 16-byte
 * aligned; the packed buffer has qmm_packed_bytes bytes. */

/* Inverse of qmm_repack_weights (a test and debugging aid). */
qmm_status qmm_unrepack_weights(qmm_type wt, const void *W_packed, void *W_canon, int64_t N,
                                int64_t K, qmm_stream_t stream);

/* ---------------------------------------------------------------- mul_mat */

/* Y [M, N] = W [N, K] . X [M, K]^T, the whole method (page 1, mul_mat steps
 * 1-3 and "正确性: 缩放系数可以提到求和号外面"): the activations are
 * quantized once per call to Q8_0 (for Q4_0 weights) or Q8_K (for Q4_K and
 * Q6_K) in the same stream, then every output is
 *   Q4_0: sum_b fp16(d_w) fp16(d_a) sum_{i<32} (q_i - 8) y_i
 *   Q4_K: sum_sb d_a (d * sum_j s_j sum_i q_i y_i - dmin * sum_j m_j sum_i y_i)
 *   Q6_K: sum_sb d_a d sum_j s_j sum_i q_i y_i  (16 groups j of 16, no min)
 * Decode (up to 16 tokens): the GEMV kernels take integer block sums with
 * fp32 accumulation across blocks (dp4a for one token, and for two Q6_K
 * tokens of at most 8192 elements in all; otherwise from 2 tokens mma.sync
 * on integer-valued fp16 operands, each block's integer sum exact). When
 * M*K is small (Q4_0, Q6_K: at most 8192 elements on the dp4a GEMV; Q4_K:
 * 16-token groups of at most 8192 elements) the activation quantizer runs
 * inside the GEMV kernel (no workspace). The tensor-core GEMV holds all of
 * a launch's activations in shared memory, so a large K caps its tokens
 * per launch; a decode batch that would take three or more launches (two
 * for Q4_0 and Q6_K), each reading the weights again, runs the GEMM below.
 * Above 16 tokens (prefill), and for those batches, the tensor-core GEMM
 * multiplies fp16 operands with fp32 accumulation: each weight is its exact
 * value rounded once to fp16 (Q4_0 d (q - 8); Q4_K d s_j q - dmin m_j,
 * formed in fp32 first; Q6_K d s_j q) and each activation is 2^e d_a y
 * rounded once to fp16, y the same Q8 codes and 2^e a power of two per
 * token that puts the token's largest block scale 2^e d_a in [2^7, 2^8)
 * (taken off again, exactly, before Y is written: any magnitude of X works,
 * including values past fp16's 65504). Each product is then within
 * 2^-10 (1 + 2^-11) of the factored form's, plus, only for weights below
 * fp16's normal range (|w| < 2^-14), 2^-25 |a| from the weight's subnormal
 * rounding; the prefill weights must satisfy |w| <= 65504 (any weight that
 * came from fp16 storage does). Otherwise the quantized activations go to
 * a workspace that the library allocates stream-ordered (cudaMallocAsync)
 * and frees after the call, in the same stream.
 * W_packed comes from qmm_repack_weights.
 * Errors: QMM_ERR_ARG (type, sizes, null/misaligned pointers),
 * QMM_ERR_NOMEM (workspace allocation failed), QMM_ERR_CUDA (launch failed).
 * M == 0 or N == 0 is a no-op. */
qmm_status qmm_mul_mat(qmm_type wt, const void *W_packed, int64_t N, int64_t K, const float *X,
                       int64_t M, float *Y, qmm_stream_t stream);

/* qmm_mul_mat on activations that are already quantized: Xq holds M rows of
 * canonical blocks as qmm_quantize_row_q8 writes them -- Q8_0 [M][K/32] x 34 B
 * for Q4_0 weights, Q8_K [M][K/256] x 292 B for Q4_K and Q6_K (page 1: vec_dot takes
 * the weight row and the Q8 activation row; for Q8_K the stored 16-code sums
 * are used for the min term as they are). The blocks are rewritten into the
 * private layout of the kernel that runs (in a workspace allocated like
 * qmm_mul_mat's) and the result is that of qmm_mul_mat on any X that
 * quantizes to Xq. Xq: device, aligned like its blocks (Q8_K 4 bytes, Q8_0
 * 2 bytes); other arguments and errors as qmm_mul_mat. */
qmm_status qmm_mul_mat_q8(qmm_type wt, const void *W_packed, int64_t N, int64_t K, const void *Xq,
                          int64_t M, float *Y, qmm_stream_t stream);

/* Several weight matrices that read the same activations (a layer's q, k and
 * v projections, or gate and up): Y_i [M, N_i] = W_i [N_i, K] . X [M, K]^T for
 * i < n, 1 <= n <= 8. X is quantized once for all of them (page 1, "为什么
 * 每个任务都要重新量化激活": re-quantizing one input per projection is
 * repeated work), and up to 16 tokens run as ONE decode launch whose work is
 * the rows of all the matrices, so the small ones no longer pay a launch and
 * a tail each. Results equal n qmm_mul_mat calls (same codes, same sums).
 * W_packed, N and Y are HOST arrays of n entries (device pointers to packed
 * weights / outputs, row counts); K, X, M, stream and the errors are those of
 * qmm_mul_mat, checked for every i. Matrices with N_i == 0 are skipped.
 * Where qmm_mul_mat would run the tensor-core GEMM, it runs once per matrix
 * on the shared quantized activations. */
qmm_status qmm_mul_mat_multi(qmm_type wt, int n, const void *const *W_packed, const int64_t *N,
                             int64_t K, const float *X, int64_t M, float *const *Y,
                             qmm_stream_t stream);

/* qmm_mul_mat with a caller-provided workspace of at least
 * qmm_workspace_bytes(wt, M, K) bytes (QMM_ERR_WORKSPACE otherwise). The
 * workspace is in use until the call's work on `stream` has finished. */
qmm_status qmm_mul_mat_ws(qmm_type wt, const void *W_packed, int64_t N, int64_t K, const float *X,
                          int64_t M, float *Y, void *workspace, size_t ws_bytes,
                          qmm_stream_t stream);

/* qmm_mul_mat on HOST activations and outputs, for a caller whose X starts
 * and whose Y ends in host memory (the same y = W x over block formats,
 * page 1, "通用实现"): in stream order, X_host [M, K] fp32 is copied to the
 * device, the product runs exactly as qmm_mul_mat_ws (same kernels, same
 * bits), and Y [M, N] fp32 is copied back to Y_host; one call, so the host
 * pays one library call per product instead of three.
 *   device_buf: caller-owned device memory of at least
 *     qmm_host_call_bytes(wt, M, N, K) bytes, 16-byte aligned; it holds X,
 *     Y and the workspace, and is in use until the call's work on `stream`
 *     has finished.
 *   X_host, Y_host: host memory. X is copied into device_buf by
 *     cudaMemcpyAsync (the kernels read it many times). Y, written once, is
 *     stored by the kernels straight into Y_host when that is page-locked
 *     memory mapped into the device's address space (cudaHostAlloc,
 *     cudaHostRegister), saving the copy back; else it is copied from
 *     device_buf. Page-locked memory lets the copies run asynchronously;
 *     with pageable memory the runtime stages them and the call may block.
 *     Y_host holds the result only once the stream has reached the end of
 *     the call.
 * Errors: those of qmm_mul_mat_ws; QMM_ERR_WORKSPACE when buf_bytes is too
 * small; QMM_ERR_CUDA when a copy cannot be enqueued.

 *   flags: 0, or QMM_HOST_MAPPED: the caller states that X_host and Y_host
 *     are page-locked memory the device can address by the same pointers
 *     (cudaHostAlloc under unified addressing, or cudaHostRegister where
 *     the device attribute cudaDevAttrCanUseHostPointerForRegisteredMem is
 *     1; QMM_ERR_UNSUPPORTED if the device has neither). Then no copy call
 *     and no pointer query is made: a small kernel pulls X into device_buf
 *     and the kernels store Y into Y_host. Passing the flag for any other
 *     memory is undefined behaviour. */
#define QMM_HOST_MAPPED 1u
size_t qmm_host_call_bytes(qmm_type wt, int64_t M, int64_t N, int64_t K);
qmm_status qmm_mul_mat_host(qmm_type wt, const void *W_packed, int64_t N, int64_t K, const float *X_host,
                            int64_t M, float *Y_host, void *device_buf, size_t buf_bytes, unsigned flags,
                            qmm_stream_t stream);

/* The two halves of qmm_mul_mat_ws, for callers that reuse one quantized
 * activation across several weight matrices (page 1, "为什么每个任务都要重新
 * 量化激活": a mul_mat quantizes its activations once; projections sharing an
 * input need not each re-quantize it).
 * qmm_quantize_activations: quantize X [M, K] for weights of type wt into
 *   `workspace` (qmm_workspace_bytes(wt, M, K) bytes, 16-byte aligned), in
 *   a private layout chosen by (wt, M, K) for the kernel that will read it:
 *   int8 codes with fp32 block scales and int16 code sums for the scalar
 *   decode GEMV; the fp16 codes, fp16 16-code sums and fp32 scales of the
 *   tensor-core kernels (Q4_K decode from 2 tokens, and prefill). The codes
 *   and scales are those of qmm_quantize_row_q8.
 * qmm_mul_mat_prepared: Y [M, N] from packed weights and a workspace filled
 *   by qmm_quantize_activations with the same wt, M and K (the contents are
 *   not checked). The workspace is read-only here, so several calls may
 *   share it; when the GEMM splits tiles (more 128 x 128 output tiles than
 *   SMs, or fewer than half as many), the call therefore takes its partial area
 *   (about 20 MB) from the device's default memory pool,
 *   stream-ordered, and frees it after the call on the same stream.
 *   Errors as qmm_mul_mat_ws, plus QMM_ERR_NOMEM for that area. */
qmm_status qmm_quantize_activations(qmm_type wt, const float *X, int64_t M, int64_t K,
                                    void *workspace, size_t ws_bytes, qmm_stream_t stream);
qmm_status qmm_mul_mat_prepared(qmm_type wt, const void *W_packed, int64_t N, int64_t K,
                                const void *workspace, size_t ws_bytes, int64_t M, float *Y,
                                qmm_stream_t stream);

/* qmm_mul_mat for callers that cannot allocate device memory. The pages have
 * no counterpart: this is a deployment variant of the same computation.
 * Some callers may not allocate once they are running: a serving loop whose
 * allocator is frozen after start-up, a host runtime that gives this library
 * no allocator to draw from, or a latency-critical step that must never block
 * in cudaMalloc/cudaFree. This call allocates nothing: the quantized
 * activations go to a fixed 4 MiB device array inside libqmm (reserved on
 * every GPU that loads the library, until the process exits), then a decode
 * GEMV runs on them (the one qmm_mul_mat runs for up to 16 tokens of a
 * small K). It never switches to the prefill GEMM (whose
 * operands and stream-K area would not fit): it runs the GEMV in launches of
 * up to 16 tokens, each of which reads the weights again. The caller still
 * owns and passes X, W_packed and Y (same layouts, alignment and errors as
 * qmm_mul_mat).
 *   - Limit: the activations of the whole call must fit the 4 MiB. From 2
 *     tokens on they are the tensor-core GEMV's images (about 2.0 to 2.2
 *     bytes per element of X: M*K up to about 1.9 million); one token is
 *     stored as Q8 codes with their scales and sums (about 1.14 to 1.19
 *     bytes per element: K up to about 3.5 million). Calls small enough for
 *     the decode kernel's fused quantizer use no scratch at all.
 *     Larger requests return QMM_ERR_WORKSPACE and launch nothing.
 *   - The first call on a device looks up the array's device address (once,
 *     with that device current); make that first call before any stream
 *     capture. The address is kept for the life of the process: after
 *     cudaDeviceReset on that device, do not call this again.
 *   - All calls share the one array and it keeps the last call's contents;
 *     nothing in it needs to start at zero. Calls whose GPU work overlaps
 *     (different streams, or graphs replayed concurrently) race on it: order
 *     them on one stream or use qmm_mul_mat_ws with separate workspaces. */
qmm_status qmm_mul_mat_static(qmm_type wt, const void *W_packed, int64_t N, int64_t K,
                              const float *X, int64_t M, float *Y, qmm_stream_t stream);

/* ---------------------------------------------------------------- W4A16 */

/* W4A16 group-asymmetric linear layer (page 3, "从数学表达式到真实存储"):
 *   C[m, n] = sum_k A[m, k] * s[n, k/G] * (q[n, k] - z[n, k/G])
 * W_packed: [N, K] codes from qmm_repack_weights(QMM_TYPE_W4A16, ...);
 * scales: fp16 bit patterns [N][K/G]; zeros: uint8 [N][K/G] (0..15);
 * A: fp16 [M, K] row-major; C: fp16 [M, N] row-major (written).
 * Arithmetic: q - z is exact in fp16 and every product A (q - z) exact in
 * fp32. M <= 16 (decode, mma.sync): fp32 sums over each 128-element step,
 * times s in fp32. M > 16 (tensor-core GEMM): the weight s (q - z) is
 * rounded once to fp16 (relative error <= 2^-11) and multiplied on the
 * tensor cores with fp32 accumulation. C is the fp32 sum rounded to fp16.
 * Needs G % 128 == 0 and K % G == 0 (QMM_ERR_UNSUPPORTED for other G that
 * divide K) and K / G <= 256 (QMM_ERR_UNSUPPORTED above); W_packed,
 * scales, zeros and A 16-byte aligned, C 2-byte aligned.
 * M > 16 with more 128 x 128 output tiles than SMs runs over a persistent
 * grid (stream-K), with fewer than half as many it splits K over the SMs;
 * tiles split across CTAs are added up, in a fixed order,
 * through a partial area of about 20 MB that such a call allocates and
 * frees stream-ordered on `stream` (the device's default memory pool).
 * Errors: QMM_ERR_ARG for sizes (M, N >= 0, K > 0, G > 0, K % G == 0) or
 * null/misaligned pointers; QMM_ERR_NOMEM if the partial area cannot be
 * allocated. M == 0 or N == 0 is a no-op. */
qmm_status qmm_w4a16(const void *W_packed, const uint16_t *scales, const uint8_t *zeros, int64_t G,
                     const uint16_t *A, uint16_t *C, int64_t M, int64_t N, int64_t K,
                     qmm_stream_t stream);

/* W4A16 with non-uniform 4-bit codes (page 3, "从数学表达式到真实存储": for
 * NF4-like formats q indexes a code table, W-hat = s LUT(q), one more table
 * lookup after the bit extraction, no zero point):
 *   C[m, n] = sum_k A[m, k] * s[n, k/G] * LUT[q[n, k]]
 * lut: device pointer to the 16 table values as fp16 bit patterns (2-byte
 * aligned), read by every launch like the weights and scales (it must be
 * written before the call is issued on `stream`). Weights, scales, A and C
 * as qmm_w4a16; the same packed codes serve both forms.
 * Arithmetic: table values are exact fp16, so every product A LUT(q) is
 * exact in fp32. M <= 16: fp32 sums over each 128-element step, times s in
 * fp32. M > 16: s LUT(q) rounded once to fp16, tensor cores, fp32
 * accumulation. C is the fp32 sum rounded to fp16.
 * Errors, sizes and the partial area as qmm_w4a16. */
qmm_status qmm_w4a16_lut(const void *W_packed, const uint16_t *scales, const uint16_t *lut, int64_t G,
                         const uint16_t *A, uint16_t *C, int64_t M, int64_t N, int64_t K,
                         qmm_stream_t stream);

/* W4A16 zero points stored 4-bit packed (page 3, "从数学表达式到真实存储": a
 * zero point packed in low bits needs one more bit extraction), unpacked
 * once at load time into the uint8 [N][ngroups] array qmm_w4a16 reads.
 * zeros_packed: [N][ceil(ngroups / 8)] uint32, row-major; group g of row n
 * at bits 4 (g mod 8) .. 4 (g mod 8) + 3 of word g / 8 (the nibble order of
 * the codes, page 3, "位级打包"); unused high nibbles of a row's last word
 * are ignored. zeros: [N][ngroups] uint8 (written, values 0..15). Device
 * pointers; both owned by the caller; the call only enqueues on `stream`.
 * Errors: QMM_ERR_ARG for N < 0, ngroups < 1 or null pointers (N == 0 is
 * a no-op). */
qmm_status qmm_w4a16_unpack_zeros(const uint32_t *zeros_packed, uint8_t *zeros, int64_t N,
                                  int64_t ngroups, qmm_stream_t stream);

/* Per-block integer sums of the factored form, for bit-exact checking
 * (page 1, "正确性" and "通用实现"). Xq holds canonical activation blocks
 * (Q8_0 for Q4_0 weights, Q8_K for Q4_K and Q6_K), M rows.
 *   Q4_0: out[(m * N + n) * (K/32) + b] = sum_{i<32} (q_i - 8) y_i
 *   Q4_K: out[((m * N + n) * (K/256) + sb) * 10 + t] with t = 0..7 the
 *         sub-block sums S_j = sum_i q_i y_i, t = 8 the scaled sum
 *         sum_j s_j S_j and t = 9 the min sum sum_j m_j (bs_2j + bs_2j+1).
 *   Q6_K: out[((m * N + n) * (K/256) + sb) * 17 + t] with t = 0..15 the
 *         group sums S_j = sum_i q_i y_i (q in -32..31), t = 16 sum_j s_j S_j.
 * Errors as qmm_mul_mat. */
qmm_status qmm_debug_block_sums(qmm_type wt, const void *W_packed, int64_t N, int64_t K,
                                const void *Xq, int64_t M, int32_t *out, qmm_stream_t stream);

/* Failure-detection check without a fault: launches one CTA that waits, with
 * the same bounded-wait helper as every pipeline wait of this library but a
 * limit of limit_cycles SM clocks (0 < limit_cycles <= 2e10), on an mbarrier
 * that nothing completes. The wait gives up, records QMM_ERR_TIMEOUT in the
 * device error word and the kernel returns; the next qmm_check_device_error
 * on the stream reports it (and clears it). The CUDA context stays usable.
 * Returns QMM_ERR_ARG for a bad limit, QMM_ERR_CUDA if the launch failed. */
qmm_status qmm_debug_wait_timeout(int64_t limit_cycles, qmm_stream_t stream);

/* ---------------------------------------------------------------- status */

/* Tensor-core throughput microbenchmarks: the peaks the prefill GEMMs are
 * measured against (page 3, "性能判断: 带宽、解码和 Tensor Core 谁是瓶颈":
 * judge a kernel against the unit it runs on). One launch on `stream` that
 * runs `iters` rounds of back-to-back MMAs on nonzero operands over the
 * whole GPU; *ops (host pointer) receives the operations it performs
 * (2 per multiply-add), for the caller to divide by the launch's event time.
 *   QMM_PEAK_MMA_S8     mma.sync m16n8k32 s8 x s8 -> s32 (the int8 tensor path
 *                       of sm_103a: tcgen05 has no kind::i8 there), 32 warps
 *                       per SM, 8 independent accumulators per warp
 *   QMM_PEAK_MMA_F16    mma.sync m16n8k16 f16 x f16 -> f32, the same way
 *   QMM_PEAK_TC_SS_128  tcgen05.mma kind::f16 M = 128, N = 128, K = 16, both
 *                       operands in shared memory, one CTA per SM
 *   QMM_PEAK_TC_TS_128  the same with A in TMEM (the prefill GEMMs' form)
 *   QMM_PEAK_TC_SS_256, QMM_PEAK_TC_TS_256   the same with N = 256
 * iters: 1 .. 10^6 (a round is 8 MMAs per warp for mma.sync, 4 (K = 64) for
 * tcgen05); keep a launch well under a second. Errors: QMM_ERR_ARG for a bad
 * kind or count, QMM_ERR_CUDA if the launch failed. */
typedef enum {
    QMM_PEAK_MMA_S8 = 0,
    QMM_PEAK_MMA_F16 = 1,
    QMM_PEAK_TC_SS_128 = 2,
    QMM_PEAK_TC_TS_128 = 3,
    QMM_PEAK_TC_SS_256 = 4,
    QMM_PEAK_TC_TS_256 = 5
} qmm_peak_kind;
qmm_status qmm_debug_peak(int which, int64_t iters, double *ops, qmm_stream_t stream);

/* Static string naming a status code. */
const char *qmm_status_string(qmm_status s);

/* Host: one-line description of the last error returned on this thread. */
const char *qmm_last_error(void);

/* Synchronize `stream`, then read and clear the device error word of the
 * current device. Returns QMM_ERR_TIMEOUT if a kernel gave up a bounded
 * wait since the last check, QMM_ERR_CUDA if the stream reported an error,
 * QMM_OK otherwise. */
qmm_status qmm_check_device_error(qmm_stream_t stream);

/* Number of kernels this library has launched on this process (all devices).
 * A monotone counter for accounting in benchmarks and tests. */
uint64_t qmm_kernel_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* QMM_H */
