/*
 * oracle.h -- plain CPU reference ("oracle") for the block-quantized matmul.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may include, link,
 * load or call this code: only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it. It shares no code, header, table or helper with
 * the CUDA library.
 *
 * Sources (page title, section):
 *   [P1] "llama.cpp 源码完全拆解(十三): ggml-cpu 的一次 mul_mat"
 *        sections "最基础的两块: Q4_0 与 Q8_0", "K-quant: 为什么需要超级块",
 *        "6-bit 参数是怎么塞进 12 字节的", "更低的比特: Q6_K 与 Q2_K 的取舍",
 *        "正确性: 缩放系数可以提到求和号外面", "通用实现", "手算一个子块".
 *   [P3] "BitBLAS 完全拆解: 低比特权重如何在 Tensor Core 上边解码边计算"
 *        sections "从数学表达式到真实存储" (W-hat = s(q - z), g = floor(k/G))
 *        and "位级打包" (u = sum (q_i & 15) << 4i).
 *
 * Every routine is written in the order the pages state the computation; no
 * blocking, fusion or reordering beyond that. Floating point follows the
 * precision the pages fix: fp16 block scales (ggml_half), fp32 quantization
 * arithmetic and fp32 accumulation for the vec_dot, plus fp64 variants used
 * as the "exact" reference. Built with -ffp-contract=off so that no multiply
 * and add are fused.
 *
 * Parity pins: every function here is pinned by tests/test_oracle.py against
 * facts the pages print or mathematics fixes. None is "parity unpinned"
 * except the Q4_K and Q6_K scale searches, whose pages describe only the
 * format; the readings used here are pinned by their reconstruction bounds
 * and invariants, but not against any other implementation's blocks. The
 * Q6_K bit order within ql and qh is a reading too (the pages give the field
 * sizes only), pinned by a hand-derived golden block.
 */
#ifndef QMM_ORACLE_H
#define QMM_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_Q4_0 = 0, ORC_Q4_K = 1, ORC_Q8_0 = 2, ORC_Q8_K = 3, ORC_Q6_K = 5 };

/* Bytes per block: 18 (Q4_0), 144 (Q4_K), 34 (Q8_0), 292 (Q8_K), 210 (Q6_K);
 * 0 otherwise. */
size_t orc_block_bytes(int type);
/* Elements per block: 32 or 256. */
int orc_block_elems(int type);

/* IEEE binary16 conversions, round-to-nearest-even, subnormals kept. */
uint16_t orc_fp32_to_fp16(float f);
uint16_t orc_fp64_to_fp16(double f);
float orc_fp16_to_fp32(uint16_t h);

/* Q4_K 6-bit scale/min packing into 12 bytes ([P1] "6-bit 参数..."). */
void orc_get_scale_min_k4(int j, const uint8_t *scales, uint8_t *s, uint8_t *m);
void orc_set_scale_min_k4(int j, uint8_t *scales, uint8_t s, uint8_t m);

/* Row quantizers: k must be a multiple of the block size. */
void orc_quantize_row_q4_0(const float *x, void *blocks, int64_t k);
void orc_quantize_row_q4_K(const float *x, void *blocks, int64_t k);
void orc_quantize_row_q8_0(const float *x, void *blocks, int64_t k);
void orc_quantize_row_q8_K(const float *x, void *blocks, int64_t k);
void orc_quantize_row_q6_K(const float *x, void *blocks, int64_t k);
/* Quantize rows [r0, r1) of a row-major [rows, k] fp32 matrix. */
void orc_quantize_rows(int type, const float *x, void *blocks, int64_t rows, int64_t k,
                       int nthreads);

/* Dequantizers (debug/brute-force tools; not the method's hot path). */
void orc_dequantize_row(int type, const void *blocks, float *y, int64_t k);
void orc_dequantize_row_f64(int type, const void *blocks, double *y, int64_t k);

/* vec_dot of one weight row with one activation row, fp32 accumulation. */
float orc_vec_dot_q4_0_q8_0(int64_t k, const void *w, const void *a);
float orc_vec_dot_q4_K_q8_K(int64_t k, const void *w, const void *a);
float orc_vec_dot_q6_K_q8_K(int64_t k, const void *w, const void *a);
/* Same factored form, accumulated in fp64. */
double orc_vec_dot_f64(int wtype, int64_t k, const void *w, const void *a);

/* Per-block integer sums of the factored form.
 * Q4_0 x Q8_0: isum[b] = sum_i (q_i - 8) * y_i, b < k/32.
 * Q4_K x Q8_K: S[sb*8 + j] = sum_i q_i * y_i over sub-block j,
 *              isum[sb] = sum_j s_j S_j, msum[sb] = sum_j m_j (bs_2j + bs_2j+1). */
void orc_block_sums_q4_0(int64_t k, const void *w, const void *a, int32_t *isum);
void orc_block_sums_q4_K(int64_t k, const void *w, const void *a, int32_t *S, int32_t *isum,
                         int32_t *msum);
/* Q6_K x Q8_K: S[sb*16 + j] = sum_i q_i * y_i over group j (q signed, -32..31),
 *              isum[sb] = sum_j s_j S_j (no min term). */
void orc_block_sums_q6_K(int64_t k, const void *w, const void *a, int32_t *S, int32_t *isum);

/*
 * mul_mat over already-quantized activations.
 *   W   : [N] rows of k/QK weight blocks (canonical byte layout)
 *   Xq  : [M] rows of activation blocks (Q8_0 for Q4_0 weights, Q8_K for Q4_K
 *         and Q6_K)
 *   rows: optional list of nrows weight-row indices (NULL = all N rows)
 * Outputs, [M][nrows] row-major:
 *   Y32 : fp32 vec_dot (factored integer form, fp32 accumulation)
 *   Y64 : fp64 brute force, dequantize both operands then dot
 *   den : fp64 sum_k |w_k a_k|, the normalisation of the error bound
 * Any output pointer may be NULL.
 */
void orc_mul_mat_q8(int wtype, const void *W, int64_t N, int64_t K, const void *Xq, int64_t M,
                    const int64_t *rows, int64_t nrows, float *Y32, double *Y64, double *den,
                    int nthreads);

/* W4A16 group-asymmetric path ([P3]). q is [N][K] uint8 in 0..15,
 * qweight is [N][K/8] uint32 with k = 8c + i in bits 4i..4i+3 of word c. */
void orc_w4a16_pack(const uint8_t *q, uint32_t *qweight, int64_t N, int64_t K);
void orc_w4a16_unpack(const uint32_t *qweight, uint8_t *q, int64_t N, int64_t K);
/* Zero points packed 8 per word like the codes: [N][ceil(ng/8)] -> [N][ng]. */
void orc_w4a16_unpack_zeros(const uint32_t *zp, uint8_t *z, int64_t N, int64_t ng);
/* C[m,n] = sum_k A[m,k] * s[n,g] * (q[n,k] - z[n,g]), g = k / G.
 * scales, A hold fp16 bit patterns; zeros is uint8 [N][K/G].
 * Outputs [M][nrows]: C16 (fp16 bits of the fp64 sum), C64, den (any may be NULL). */
void orc_w4a16_matmul(const uint32_t *qweight, const uint16_t *scales, const uint8_t *zeros,
                      int64_t G, const uint16_t *A, int64_t M, int64_t N, int64_t K,
                      const int64_t *rows, int64_t nrows, uint16_t *C16, double *C64, double *den,
                      int nthreads);
/* C[m,n] = sum_k A[m,k] * s[n,g] * LUT[q[n,k]] (NF4-like code table, no zero
 * point); lut holds 16 fp16 bit patterns. Outputs as orc_w4a16_matmul. */
void orc_w4a16_lut_matmul(const uint32_t *qweight, const uint16_t *scales, const uint16_t *lut,
                          int64_t G, const uint16_t *A, int64_t M, int64_t N, int64_t K,
                          const int64_t *rows, int64_t nrows, uint16_t *C16, double *C64,
                          double *den, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
