/*
 * oracle.c -- plain, slow, obviously-correct CPU reference for the
 * block-quantized matmul (Q4_0 / Q4_K weights x Q8_0 / Q8_K activations,
 * and the W4A16 group-asymmetric form).
 *
 * TEST INFRASTRUCTURE ONLY: the product path never includes or calls this.
 * See oracle.h for the page/section citations. Compile with
 *   gcc -std=c11 -O2 -ffp-contract=off -fopenmp -shared -fPIC
 * No intrinsics, no inline assembly, no reliance on the signedness of char.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Block layouts, exactly as [P1] prints them (ggml_half is stored as the    */
/* uint16 bit pattern of an IEEE binary16).                                  */
/* ------------------------------------------------------------------------ */
typedef struct {
    uint16_t d;      /* delta */
    uint8_t qs[16];  /* 32 nibbles */
} orc_block_q4_0;

typedef struct {
    uint16_t d;     /* fp16 scale */
    int8_t qs[32];  /* int8 codes */
} orc_block_q8_0;

typedef struct {
    uint16_t d;          /* super-block scale */
    uint16_t dmin;       /* super-block scale of the mins */
    uint8_t scales[12];  /* 8 scales + 8 mins, 6 bits each */
    uint8_t qs[128];     /* 256 nibbles */
} orc_block_q4_K;

typedef struct {
    float d;            /* fp32 scale */
    int8_t qs[256];     /* int8 codes */
    int16_t bsums[16];  /* sums of 16 consecutive codes */
} orc_block_q8_K;

typedef struct {
    uint8_t ql[128];    /* low 4 bits of the 256 6-bit codes */
    uint8_t qh[64];     /* high 2 bits */
    int8_t scales[16];  /* one int8 scale per 16 elements */
    uint16_t d;         /* super-block scale */
} orc_block_q6_K;

/* Sizes the pages state: 2+16 = 18 B, 2+32 = 34 B, 2+2+12+128 = 144 B,
 * 4+256+32 = 292 B, 128+64+16+2 = 210 B. */
_Static_assert(sizeof(orc_block_q4_0) == 18, "block_q4_0 must be 18 bytes");
_Static_assert(sizeof(orc_block_q8_0) == 34, "block_q8_0 must be 34 bytes");
_Static_assert(sizeof(orc_block_q4_K) == 144, "block_q4_K must be 144 bytes");
_Static_assert(sizeof(orc_block_q8_K) == 292, "block_q8_K must be 292 bytes");
_Static_assert(sizeof(orc_block_q6_K) == 210, "block_q6_K must be 210 bytes");

size_t orc_block_bytes(int type) {
    switch (type) {
    case ORC_Q4_0: return sizeof(orc_block_q4_0);
    case ORC_Q4_K: return sizeof(orc_block_q4_K);
    case ORC_Q8_0: return sizeof(orc_block_q8_0);
    case ORC_Q8_K: return sizeof(orc_block_q8_K);
    case ORC_Q6_K: return sizeof(orc_block_q6_K);
    default: return 0;
    }
}

int orc_block_elems(int type) {
    switch (type) {
    case ORC_Q4_0:
    case ORC_Q8_0: return 32;
    case ORC_Q4_K:
    case ORC_Q8_K:
    case ORC_Q6_K: return 256;
    default: return 0;
    }
}

/* ------------------------------------------------------------------------ */
/* IEEE binary16 <-> binary32/64, written from the IEEE 754 encoding.        */
/* ------------------------------------------------------------------------ */

/* Round the non-negative real value man * 2^exp2 (man < 2^63) to binary16 and
 * return the magnitude bits. Round to nearest, ties to even; overflow -> Inf. */
static uint16_t round_to_half_bits(uint64_t man, int exp2) {
    if (man == 0) return 0;
    /* normalise so that the leading one sits at bit 62 */
    int lead = 63;
    while (!((man >> lead) & 1)) --lead;
    /* value = 1.f * 2^(exp2 + lead) */
    int e = exp2 + lead;      /* unbiased exponent of the value */
    int target_lsb;           /* exponent of the unit in the last place kept */
    if (e >= -14) {
        target_lsb = e - 10;  /* normal: 10 fraction bits */
    } else {
        target_lsb = -24;     /* subnormal: fixed unit 2^-24 */
    }
    int shift = target_lsb - exp2;  /* bits to drop from man */
    uint64_t q;
    if (shift <= 0) {
        q = man << (-shift);
    } else if (shift >= 64) {
        q = 0;
        /* all bits dropped: value < 2^-25 when shift >= 64 here -> rounds to 0 */
        return 0;
    } else {
        q = man >> shift;
        uint64_t rem = man & ((((uint64_t)1) << shift) - 1);
        uint64_t half = ((uint64_t)1) << (shift - 1);
        if (rem > half || (rem == half && (q & 1))) q += 1;
    }
    /* q counts units of 2^target_lsb */
    if (target_lsb == -24) {
        /* subnormal range; q may have rounded up to 0x400 = smallest normal */
        return (uint16_t)q;
    }
    /* normal: q in [2^10, 2^11]; 2^11 means carry into the exponent */
    int be = e + 15;
    if (q >= 2048) {
        q >>= 1;
        be += 1;
    }
    if (be >= 31) return 0x7C00;
    return (uint16_t)(((uint32_t)be << 10) | ((uint32_t)q & 0x3FF));
}

uint16_t orc_fp32_to_fp16(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000);
    uint32_t exp = (x >> 23) & 0xFF;
    uint32_t frac = x & 0x7FFFFF;
    if (exp == 0xFF) return (uint16_t)(sign | (frac ? 0x7E00 : 0x7C00));
    if (exp == 0) {
        if (frac == 0) return sign;
        return (uint16_t)(sign | round_to_half_bits(frac, -149));
    }
    return (uint16_t)(sign | round_to_half_bits(frac | 0x800000u, (int)exp - 150));
}

uint16_t orc_fp64_to_fp16(double f) {
    uint64_t x;
    memcpy(&x, &f, 8);
    uint16_t sign = (uint16_t)((x >> 48) & 0x8000);
    uint32_t exp = (uint32_t)((x >> 52) & 0x7FF);
    uint64_t frac = x & 0xFFFFFFFFFFFFFull;
    if (exp == 0x7FF) return (uint16_t)(sign | (frac ? 0x7E00 : 0x7C00));
    if (exp == 0) {
        if (frac == 0) return sign;
        return (uint16_t)(sign | round_to_half_bits(frac, -1074));
    }
    return (uint16_t)(sign | round_to_half_bits(frac | 0x10000000000000ull, (int)exp - 1075));
}

float orc_fp16_to_fp32(uint16_t h) {
    uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
    uint32_t exp = ((uint32_t)h >> 10) & 0x1F;
    uint32_t frac = (uint32_t)h & 0x3FF;
    uint32_t bits;
    if (exp == 0) {
        /* zero or subnormal: frac * 2^-24, exact in binary32 */
        float v = (float)frac * 5.9604644775390625e-8f;
        return sign ? -v : v;
    } else if (exp == 31) {
        bits = sign | 0x7F800000u | (frac << 13);
    } else {
        bits = sign | ((exp - 15 + 127) << 23) | (frac << 13);
    }
    float out;
    memcpy(&out, &bits, 4);
    return out;
}

/* ------------------------------------------------------------------------ */
/* Rounding helpers (readings of the pages' "round").                        */
/* ------------------------------------------------------------------------ */

/* Round half away from zero, in fp32: sign(v) * floor(|v| + 0.5). */
static float rha(float v) {
    if (v < 0.0f) return -floorf(-v + 0.5f);
    return floorf(v + 0.5f);
}

static int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* ------------------------------------------------------------------------ */
/* Q4_K scale/min packing ([P1] "6-bit 参数是怎么塞进 12 字节的").            */
/* Sub-blocks 0..3: scale in the low 6 bits of scales[j], min in the low 6   */
/* bits of scales[j+4]. Sub-blocks 4..7: the low 4 bits of scale and min go  */
/* into the low and high nibble of scales[j+4]; their top 2 bits go into the */
/* top 2 bits of scales[j-4] (scale) and scales[j] (min).                    */
/* ------------------------------------------------------------------------ */
void orc_get_scale_min_k4(int j, const uint8_t *q, uint8_t *s, uint8_t *m) {
    if (j < 4) {
        *s = (uint8_t)(q[j] & 63);
        *m = (uint8_t)(q[j + 4] & 63);
    } else {
        *s = (uint8_t)((q[j + 4] & 0x0F) | ((q[j - 4] >> 6) << 4));
        *m = (uint8_t)((q[j + 4] >> 4) | ((q[j] >> 6) << 4));
    }
}

void orc_set_scale_min_k4(int j, uint8_t *q, uint8_t s, uint8_t m) {
    s &= 63;
    m &= 63;
    if (j < 4) {
        q[j] = (uint8_t)((q[j] & 0xC0) | s);
        q[j + 4] = (uint8_t)((q[j + 4] & 0xC0) | m);
    } else {
        q[j + 4] = (uint8_t)((s & 0x0F) | ((m & 0x0F) << 4));
        q[j - 4] = (uint8_t)((q[j - 4] & 0x3F) | ((s >> 4) << 6));
        q[j] = (uint8_t)((q[j] & 0x3F) | ((m >> 4) << 6));
    }
}

/* ------------------------------------------------------------------------ */
/* Quantizers.                                                               */
/* ------------------------------------------------------------------------ */

/* Q4_0 ([P1] "最基础的两块"): d = -x_max / 8 with x_max the signed value of
 * largest magnitude (first one wins on ties); q = clamp(round(x/d) + 8, 0, 15)
 * computed as floor(x * (1/d) + 8.5); stored d is fp16. Nibble order: the low
 * nibble of qs[l] is element l, the high nibble element l + 16. */
void orc_quantize_row_q4_0(const float *x, void *blocks, int64_t k) {
    orc_block_q4_0 *y = (orc_block_q4_0 *)blocks;
    const int64_t nb = k / 32;
    for (int64_t b = 0; b < nb; ++b) {
        const float *xb = x + b * 32;
        float amax = 0.0f, vmax = 0.0f;
        for (int i = 0; i < 32; ++i) {
            float a = fabsf(xb[i]);
            if (a > amax) {
                amax = a;
                vmax = xb[i];
            }
        }
        const float d = vmax / -8.0f;
        const float id = d != 0.0f ? 1.0f / d : 0.0f;
        y[b].d = orc_fp32_to_fp16(d);
        for (int l = 0; l < 16; ++l) {
            float v0 = xb[l] * id;
            float v1 = xb[l + 16] * id;
            int q0 = clampi((int)floorf(v0 + 8.5f), 0, 15);
            int q1 = clampi((int)floorf(v1 + 8.5f), 0, 15);
            y[b].qs[l] = (uint8_t)(q0 | (q1 << 4));
        }
    }
}

/* Q8_0 ([P1] "最基础的两块"): symmetric int8 per 32, d = amax / 127 stored as
 * fp16, q = round-half-away(x / d) clamped to [-127, 127]. */
void orc_quantize_row_q8_0(const float *x, void *blocks, int64_t k) {
    orc_block_q8_0 *y = (orc_block_q8_0 *)blocks;
    const int64_t nb = k / 32;
    for (int64_t b = 0; b < nb; ++b) {
        const float *xb = x + b * 32;
        float amax = 0.0f;
        for (int i = 0; i < 32; ++i) {
            float a = fabsf(xb[i]);
            if (a > amax) amax = a;
        }
        const float d = amax / 127.0f;
        const float id = d != 0.0f ? 1.0f / d : 0.0f;
        y[b].d = orc_fp32_to_fp16(d);
        for (int i = 0; i < 32; ++i) {
            y[b].qs[i] = (int8_t)clampi((int)rha(xb[i] * id), -127, 127);
        }
    }
}

/* Q8_K ([P1] "更低的比特"): int8 per 256 with an fp32 d, plus bsums[t] = the
 * sum of codes 16t .. 16t+15 ([P1] "正确性" on why the sums are kept). */
void orc_quantize_row_q8_K(const float *x, void *blocks, int64_t k) {
    orc_block_q8_K *y = (orc_block_q8_K *)blocks;
    const int64_t nb = k / 256;
    for (int64_t b = 0; b < nb; ++b) {
        const float *xb = x + b * 256;
        float amax = 0.0f;
        for (int i = 0; i < 256; ++i) {
            float a = fabsf(xb[i]);
            if (a > amax) amax = a;
        }
        const float d = amax / 127.0f;
        const float id = d != 0.0f ? 1.0f / d : 0.0f;
        y[b].d = d;
        for (int i = 0; i < 256; ++i) {
            y[b].qs[i] = (int8_t)clampi((int)rha(xb[i] * id), -127, 127);
        }
        for (int t = 0; t < 16; ++t) {
            int s = 0;
            for (int i = 0; i < 16; ++i) s += y[b].qs[16 * t + i];
            y[b].bsums[t] = (int16_t)s;
        }
    }
}

/* Q4_K ([P1] "K-quant", "6-bit 参数", "正确性"): w = d * s_j * q - dmin * m_j.
 * The pages give the format and the packing, not the scale search; the
 * reading used is a single pass per sub-block j of 32 values:
 *   lo_j = min(0, min x), hi_j = max x, sc_j = (hi_j - lo_j) / 15, mn_j = -lo_j
 *   d = max_j sc_j / 63, dmin = max_j mn_j / 63 (stored as fp16)
 *   s_j = clamp(round(sc_j / d), 0, 63), m_j = clamp(round(mn_j / dmin), 0, 63)
 *   q   = clamp(round((x + dmin16 * m_j) / (d16 * s_j)), 0, 15)
 * using the stored (fp16) d and dmin for the codes. Nibble order per 64
 * elements: qs[32c + l] = q[64c + l] | q[64c + 32 + l] << 4. */
void orc_quantize_row_q4_K(const float *x, void *blocks, int64_t k) {
    orc_block_q4_K *y = (orc_block_q4_K *)blocks;
    const int64_t nb = k / 256;
    for (int64_t b = 0; b < nb; ++b) {
        const float *xb = x + b * 256;
        float sc[8], mn[8];
        float max_sc = 0.0f, max_mn = 0.0f;
        for (int j = 0; j < 8; ++j) {
            float lo = 0.0f, hi = xb[32 * j];
            for (int i = 0; i < 32; ++i) {
                float v = xb[32 * j + i];
                if (v < lo) lo = v;
                if (v > hi) hi = v;
            }
            sc[j] = (hi - lo) / 15.0f;
            mn[j] = -lo;
            if (sc[j] > max_sc) max_sc = sc[j];
            if (mn[j] > max_mn) max_mn = mn[j];
        }
        const float d = max_sc / 63.0f;
        const float dmin = max_mn / 63.0f;
        y[b].d = orc_fp32_to_fp16(d);
        y[b].dmin = orc_fp32_to_fp16(dmin);
        memset(y[b].scales, 0, sizeof(y[b].scales));
        int s[8], m[8];
        for (int j = 0; j < 8; ++j) {
            s[j] = d > 0.0f ? clampi((int)rha(sc[j] / d), 0, 63) : 0;
            m[j] = dmin > 0.0f ? clampi((int)rha(mn[j] / dmin), 0, 63) : 0;
            orc_set_scale_min_k4(j, y[b].scales, (uint8_t)s[j], (uint8_t)m[j]);
        }
        const float d16 = orc_fp16_to_fp32(y[b].d);
        const float dmin16 = orc_fp16_to_fp32(y[b].dmin);
        uint8_t q[256];
        for (int j = 0; j < 8; ++j) {
            const float D = d16 * (float)s[j];
            const float Mo = dmin16 * (float)m[j];
            for (int i = 0; i < 32; ++i) {
                int qi = 0;
                if (D != 0.0f) qi = clampi((int)rha((xb[32 * j + i] + Mo) / D), 0, 15);
                q[32 * j + i] = (uint8_t)qi;
            }
        }
        for (int c = 0; c < 4; ++c) {
            for (int l = 0; l < 32; ++l) {
                y[b].qs[32 * c + l] = (uint8_t)(q[64 * c + l] | (q[64 * c + 32 + l] << 4));
            }
        }
    }
}

/* Q6_K ([P1] "更低的比特: Q6_K 与 Q2_K 的取舍"): w = d * s_j * q with q in
 * -32..31, 16 groups j of 16 elements, int8 s_j, fp16 d, no min. The pages
 * give the format, not the scale search; the reading used extends the Q4_0
 * rule to two levels:
 *   sc_j = -x_max,j / 32 (x_max,j the signed value of largest magnitude in
 *          group j, first one on ties), d = max_j |sc_j| / 127 (fp16),
 *   s_j  = clamp(round(sc_j / d), -127, 127),
 *   q    = clamp(round(x / (d16 * s_j)), -32, 31), stored as u = q + 32,
 * with the stored d16 for the codes (round = half away from zero). Bit
 * order, the Q4_K pairing (fields 32 elements apart) applied to both arrays:
 *   ql[32c + l] = (u[64c + l] & 15) | (u[64c + 32 + l] & 15) << 4, c < 4
 *   qh[32h + l] = sum_i (u[128h + 32i + l] >> 4) << 2i,            h < 2. */
static void q6_K_pack(const uint8_t *u, orc_block_q6_K *blk) {
    for (int c = 0; c < 4; ++c)
        for (int l = 0; l < 32; ++l)
            blk->ql[32 * c + l] = (uint8_t)((u[64 * c + l] & 15) | ((u[64 * c + 32 + l] & 15) << 4));
    for (int h = 0; h < 2; ++h) {
        for (int l = 0; l < 32; ++l) {
            uint8_t v = 0;
            for (int i = 0; i < 4; ++i) v = (uint8_t)(v | ((u[128 * h + 32 * i + l] >> 4) << (2 * i)));
            blk->qh[32 * h + l] = v;
        }
    }
}

void orc_quantize_row_q6_K(const float *x, void *blocks, int64_t k) {
    orc_block_q6_K *y = (orc_block_q6_K *)blocks;
    const int64_t nb = k / 256;
    for (int64_t b = 0; b < nb; ++b) {
        const float *xb = x + b * 256;
        float sc[16], max_sc = 0.0f;
        for (int j = 0; j < 16; ++j) {
            float amax = 0.0f, vmax = 0.0f;
            for (int i = 0; i < 16; ++i) {
                const float a = fabsf(xb[16 * j + i]);
                if (a > amax) {
                    amax = a;
                    vmax = xb[16 * j + i];
                }
            }
            sc[j] = vmax / -32.0f;
            if (fabsf(sc[j]) > max_sc) max_sc = fabsf(sc[j]);
        }
        const float d = max_sc / 127.0f;
        y[b].d = orc_fp32_to_fp16(d);
        const float d16 = orc_fp16_to_fp32(y[b].d);
        uint8_t u[256];
        for (int j = 0; j < 16; ++j) {
            const int s = d > 0.0f ? clampi((int)rha(sc[j] / d), -127, 127) : 0;
            y[b].scales[j] = (int8_t)s;
            const float D = d16 * (float)s;
            for (int i = 0; i < 16; ++i) {
                int q = 0;
                if (D != 0.0f) q = clampi((int)rha(xb[16 * j + i] / D), -32, 31);
                u[16 * j + i] = (uint8_t)(q + 32);
            }
        }
        q6_K_pack(u, &y[b]);
    }
}

void orc_quantize_rows(int type, const float *x, void *blocks, int64_t rows, int64_t k,
                       int nthreads) {
    const size_t row_bytes = orc_block_bytes(type) * (size_t)(k / orc_block_elems(type));
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(static) num_threads(nthreads)
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * k;
        void *yr = (uint8_t *)blocks + (size_t)r * row_bytes;
        switch (type) {
        case ORC_Q4_0: orc_quantize_row_q4_0(xr, yr, k); break;
        case ORC_Q4_K: orc_quantize_row_q4_K(xr, yr, k); break;
        case ORC_Q8_0: orc_quantize_row_q8_0(xr, yr, k); break;
        case ORC_Q8_K: orc_quantize_row_q8_K(xr, yr, k); break;
        case ORC_Q6_K: orc_quantize_row_q6_K(xr, yr, k); break;
        default: break;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Dequantizers ([P1] formulas; [P4] "量化: 热路径是点积" notes these are     */
/* tools, not the hot path).                                                 */
/* ------------------------------------------------------------------------ */

/* Unpacked view of one weight/activation element, shared by both dequantizers
 * so that the fp32 and fp64 versions read the same fields. */
static void q4_K_fields(const orc_block_q4_K *blk, int i, int *q, int *s, int *m) {
    const int c = i / 64, l = i % 64;
    const uint8_t byte = blk->qs[32 * c + (l % 32)];
    *q = l < 32 ? (byte & 0x0F) : (byte >> 4);
    uint8_t sj, mj;
    orc_get_scale_min_k4(i / 32, blk->scales, &sj, &mj);
    *s = sj;
    *m = mj;
}

/* Signed 6-bit code of element i (-32..31), read back from ql and qh. */
static int q6_K_code(const orc_block_q6_K *blk, int i) {
    const int c = i / 64, l = i % 64, h = i / 128, r = i % 128;
    const uint8_t lo_byte = blk->ql[32 * c + (l % 32)];
    const int lo = l < 32 ? (lo_byte & 15) : (lo_byte >> 4);
    const int hi = (blk->qh[32 * h + (r % 32)] >> (2 * (r / 32))) & 3;
    return (lo | (hi << 4)) - 32;
}

static int q4_0_code(const orc_block_q4_0 *blk, int i) {
    return i < 16 ? (blk->qs[i] & 0x0F) : (blk->qs[i - 16] >> 4);
}

void orc_dequantize_row(int type, const void *blocks, float *y, int64_t k) {
    if (type == ORC_Q4_0) {
        const orc_block_q4_0 *x = (const orc_block_q4_0 *)blocks;
        for (int64_t b = 0; b < k / 32; ++b) {
            const float d = orc_fp16_to_fp32(x[b].d);
            for (int i = 0; i < 32; ++i) y[b * 32 + i] = d * (float)(q4_0_code(&x[b], i) - 8);
        }
    } else if (type == ORC_Q4_K) {
        const orc_block_q4_K *x = (const orc_block_q4_K *)blocks;
        for (int64_t b = 0; b < k / 256; ++b) {
            const float d = orc_fp16_to_fp32(x[b].d);
            const float dmin = orc_fp16_to_fp32(x[b].dmin);
            for (int i = 0; i < 256; ++i) {
                int q, s, m;
                q4_K_fields(&x[b], i, &q, &s, &m);
                y[b * 256 + i] = d * (float)s * (float)q - dmin * (float)m;
            }
        }
    } else if (type == ORC_Q6_K) {
        const orc_block_q6_K *x = (const orc_block_q6_K *)blocks;
        for (int64_t b = 0; b < k / 256; ++b) {
            const float d = orc_fp16_to_fp32(x[b].d);
            for (int i = 0; i < 256; ++i)
                y[b * 256 + i] = d * (float)x[b].scales[i / 16] * (float)q6_K_code(&x[b], i);
        }
    } else if (type == ORC_Q8_0) {
        const orc_block_q8_0 *x = (const orc_block_q8_0 *)blocks;
        for (int64_t b = 0; b < k / 32; ++b) {
            const float d = orc_fp16_to_fp32(x[b].d);
            for (int i = 0; i < 32; ++i) y[b * 32 + i] = d * (float)x[b].qs[i];
        }
    } else if (type == ORC_Q8_K) {
        const orc_block_q8_K *x = (const orc_block_q8_K *)blocks;
        for (int64_t b = 0; b < k / 256; ++b) {
            for (int i = 0; i < 256; ++i) y[b * 256 + i] = x[b].d * (float)x[b].qs[i];
        }
    }
}

void orc_dequantize_row_f64(int type, const void *blocks, double *y, int64_t k) {
    if (type == ORC_Q4_0) {
        const orc_block_q4_0 *x = (const orc_block_q4_0 *)blocks;
        for (int64_t b = 0; b < k / 32; ++b) {
            const double d = orc_fp16_to_fp32(x[b].d);
            for (int i = 0; i < 32; ++i) y[b * 32 + i] = d * (double)(q4_0_code(&x[b], i) - 8);
        }
    } else if (type == ORC_Q4_K) {
        const orc_block_q4_K *x = (const orc_block_q4_K *)blocks;
        for (int64_t b = 0; b < k / 256; ++b) {
            const double d = orc_fp16_to_fp32(x[b].d);
            const double dmin = orc_fp16_to_fp32(x[b].dmin);
            for (int i = 0; i < 256; ++i) {
                int q, s, m;
                q4_K_fields(&x[b], i, &q, &s, &m);
                y[b * 256 + i] = d * (double)s * (double)q - dmin * (double)m;
            }
        }
    } else if (type == ORC_Q6_K) {
        const orc_block_q6_K *x = (const orc_block_q6_K *)blocks;
        for (int64_t b = 0; b < k / 256; ++b) {
            const double d = orc_fp16_to_fp32(x[b].d);
            for (int i = 0; i < 256; ++i)
                y[b * 256 + i] = d * (double)x[b].scales[i / 16] * (double)q6_K_code(&x[b], i);
        }
    } else if (type == ORC_Q8_0) {
        const orc_block_q8_0 *x = (const orc_block_q8_0 *)blocks;
        for (int64_t b = 0; b < k / 32; ++b) {
            const double d = orc_fp16_to_fp32(x[b].d);
            for (int i = 0; i < 32; ++i) y[b * 32 + i] = d * (double)x[b].qs[i];
        }
    } else if (type == ORC_Q8_K) {
        const orc_block_q8_K *x = (const orc_block_q8_K *)blocks;
        for (int64_t b = 0; b < k / 256; ++b) {
            for (int i = 0; i < 256; ++i) y[b * 256 + i] = (double)x[b].d * (double)x[b].qs[i];
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Integer block sums and the vec_dot ([P1] "正确性", "通用实现").             */
/* sum_i w_i a_i = d d_a s sum_i q_i y_i - dmin d_a m sum_i y_i per sub-block, */
/* with sum_i y_i taken from the activation's bsums.                          */
/* ------------------------------------------------------------------------ */
void orc_block_sums_q4_0(int64_t k, const void *w, const void *a, int32_t *isum) {
    const orc_block_q4_0 *x = (const orc_block_q4_0 *)w;
    const orc_block_q8_0 *y = (const orc_block_q8_0 *)a;
    for (int64_t b = 0; b < k / 32; ++b) {
        int32_t s = 0;
        for (int l = 0; l < 16; ++l) {
            s += ((x[b].qs[l] & 0x0F) - 8) * y[b].qs[l];
            s += ((x[b].qs[l] >> 4) - 8) * y[b].qs[l + 16];
        }
        isum[b] = s;
    }
}

void orc_block_sums_q4_K(int64_t k, const void *w, const void *a, int32_t *S, int32_t *isum,
                         int32_t *msum) {
    const orc_block_q4_K *x = (const orc_block_q4_K *)w;
    const orc_block_q8_K *y = (const orc_block_q8_K *)a;
    for (int64_t b = 0; b < k / 256; ++b) {
        int32_t Sj[8];
        for (int c = 0; c < 4; ++c) {
            int32_t lo = 0, hi = 0;
            for (int l = 0; l < 32; ++l) {
                lo += (x[b].qs[32 * c + l] & 0x0F) * y[b].qs[64 * c + l];
                hi += (x[b].qs[32 * c + l] >> 4) * y[b].qs[64 * c + 32 + l];
            }
            Sj[2 * c] = lo;
            Sj[2 * c + 1] = hi;
        }
        int32_t is = 0, ms = 0;
        for (int j = 0; j < 8; ++j) {
            uint8_t sj, mj;
            orc_get_scale_min_k4(j, x[b].scales, &sj, &mj);
            is += (int32_t)sj * Sj[j];
            ms += (int32_t)mj * ((int32_t)y[b].bsums[2 * j] + (int32_t)y[b].bsums[2 * j + 1]);
            if (S) S[b * 8 + j] = Sj[j];
        }
        if (isum) isum[b] = is;
        if (msum) msum[b] = ms;
    }
}

/* Q6_K x Q8_K ([P1] "更低的比特": no min term, so no bsums): per super-block
 * S_j = sum_{i in group j} q_i y_i over the 16 elements of group j, and
 * isum = sum_j s_j S_j; the dot adds d_a d isum. */
void orc_block_sums_q6_K(int64_t k, const void *w, const void *a, int32_t *S, int32_t *isum) {
    const orc_block_q6_K *x = (const orc_block_q6_K *)w;
    const orc_block_q8_K *y = (const orc_block_q8_K *)a;
    for (int64_t b = 0; b < k / 256; ++b) {
        int32_t is = 0;
        for (int j = 0; j < 16; ++j) {
            int32_t Sj = 0;
            for (int i = 0; i < 16; ++i) Sj += q6_K_code(&x[b], 16 * j + i) * y[b].qs[16 * j + i];
            is += (int32_t)x[b].scales[j] * Sj;
            if (S) S[b * 16 + j] = Sj;
        }
        if (isum) isum[b] = is;
    }
}

float orc_vec_dot_q6_K_q8_K(int64_t k, const void *w, const void *a) {
    const orc_block_q6_K *x = (const orc_block_q6_K *)w;
    const orc_block_q8_K *y = (const orc_block_q8_K *)a;
    float acc = 0.0f;
    for (int64_t b = 0; b < k / 256; ++b) {
        int32_t isum;
        orc_block_sums_q6_K(256, &x[b], &y[b], NULL, &isum);
        acc += (y[b].d * orc_fp16_to_fp32(x[b].d)) * (float)isum;
    }
    return acc;
}

float orc_vec_dot_q4_0_q8_0(int64_t k, const void *w, const void *a) {
    const orc_block_q4_0 *x = (const orc_block_q4_0 *)w;
    const orc_block_q8_0 *y = (const orc_block_q8_0 *)a;
    float acc = 0.0f;
    for (int64_t b = 0; b < k / 32; ++b) {
        int32_t isum;
        orc_block_sums_q4_0(32, &x[b], &y[b], &isum);
        acc += (orc_fp16_to_fp32(x[b].d) * orc_fp16_to_fp32(y[b].d)) * (float)isum;
    }
    return acc;
}

float orc_vec_dot_q4_K_q8_K(int64_t k, const void *w, const void *a) {
    const orc_block_q4_K *x = (const orc_block_q4_K *)w;
    const orc_block_q8_K *y = (const orc_block_q8_K *)a;
    float acc = 0.0f;
    for (int64_t b = 0; b < k / 256; ++b) {
        int32_t isum, msum;
        orc_block_sums_q4_K(256, &x[b], &y[b], NULL, &isum, &msum);
        const float t1 = (y[b].d * orc_fp16_to_fp32(x[b].d)) * (float)isum;
        const float t2 = (y[b].d * orc_fp16_to_fp32(x[b].dmin)) * (float)msum;
        acc += t1 - t2;
    }
    return acc;
}

double orc_vec_dot_f64(int wtype, int64_t k, const void *w, const void *a) {
    double acc = 0.0;
    if (wtype == ORC_Q4_0) {
        const orc_block_q4_0 *x = (const orc_block_q4_0 *)w;
        const orc_block_q8_0 *y = (const orc_block_q8_0 *)a;
        for (int64_t b = 0; b < k / 32; ++b) {
            int32_t isum;
            orc_block_sums_q4_0(32, &x[b], &y[b], &isum);
            acc += (double)orc_fp16_to_fp32(x[b].d) * (double)orc_fp16_to_fp32(y[b].d) *
                   (double)isum;
        }
    } else if (wtype == ORC_Q4_K) {
        const orc_block_q4_K *x = (const orc_block_q4_K *)w;
        const orc_block_q8_K *y = (const orc_block_q8_K *)a;
        for (int64_t b = 0; b < k / 256; ++b) {
            int32_t isum, msum;
            orc_block_sums_q4_K(256, &x[b], &y[b], NULL, &isum, &msum);
            acc += (double)y[b].d * (double)orc_fp16_to_fp32(x[b].d) * (double)isum -
                   (double)y[b].d * (double)orc_fp16_to_fp32(x[b].dmin) * (double)msum;
        }    } else if (wtype == ORC_Q6_K) {
        const orc_block_q6_K *x = (const orc_block_q6_K *)w;
        const orc_block_q8_K *y = (const orc_block_q8_K *)a;
        for (int64_t b = 0; b < k / 256; ++b) {
            int32_t isum;
            orc_block_sums_q6_K(256, &x[b], &y[b], NULL, &isum);
            acc += (double)y[b].d * (double)orc_fp16_to_fp32(x[b].d) * (double)isum;
        }
    }
    return acc;
}

/* ------------------------------------------------------------------------ */
/* mul_mat: Y[m, n] = sum_k W[n, k] X[m, k] ([P1] "mul_mat: 一次矩阵乘").      */
/* ------------------------------------------------------------------------ */
void orc_mul_mat_q8(int wtype, const void *W, int64_t N, int64_t K, const void *Xq, int64_t M,
                    const int64_t *rows, int64_t nrows, float *Y32, double *Y64, double *den,
                    int nthreads) {
    const int atype = wtype == ORC_Q4_0 ? ORC_Q8_0 : ORC_Q8_K;
    const size_t wrow = orc_block_bytes(wtype) * (size_t)(K / orc_block_elems(wtype));
    const size_t arow = orc_block_bytes(atype) * (size_t)(K / orc_block_elems(atype));
    if (!rows) nrows = N;
    if (nthreads < 1) nthreads = 1;
    const int need_f64 = (Y64 != NULL) || (den != NULL);
#pragma omp parallel num_threads(nthreads)
    {
        double *wd = NULL, *ad = NULL;
        if (need_f64) {
            wd = (double *)malloc(sizeof(double) * (size_t)K);
            ad = (double *)malloc(sizeof(double) * (size_t)K);
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < nrows; ++r) {
            const int64_t n = rows ? rows[r] : r;
            const uint8_t *wr = (const uint8_t *)W + (size_t)n * wrow;
            if (need_f64) orc_dequantize_row_f64(wtype, wr, wd, K);
            for (int64_t m = 0; m < M; ++m) {
                const uint8_t *ar = (const uint8_t *)Xq + (size_t)m * arow;
                if (Y32) {
                    Y32[m * nrows + r] = wtype == ORC_Q4_0   ? orc_vec_dot_q4_0_q8_0(K, wr, ar)
                                         : wtype == ORC_Q6_K ? orc_vec_dot_q6_K_q8_K(K, wr, ar)
                                                             : orc_vec_dot_q4_K_q8_K(K, wr, ar);
                }
                if (need_f64) {
                    orc_dequantize_row_f64(atype, ar, ad, K);
                    double s = 0.0, sa = 0.0;
                    for (int64_t kk = 0; kk < K; ++kk) {
                        s += wd[kk] * ad[kk];
                        sa += fabs(wd[kk] * ad[kk]);
                    }
                    if (Y64) Y64[m * nrows + r] = s;
                    if (den) den[m * nrows + r] = sa;
                }
            }
        }
        free(wd);
        free(ad);
    }
}

/* ------------------------------------------------------------------------ */
/* W4A16 ([P3] "从数学表达式到真实存储", "位级打包").                          */
/* ------------------------------------------------------------------------ */
void orc_w4a16_pack(const uint8_t *q, uint32_t *qweight, int64_t N, int64_t K) {
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t c = 0; c < K / 8; ++c) {
            uint32_t u = 0;
            for (int i = 0; i < 8; ++i) u += ((uint32_t)q[n * K + 8 * c + i] & 15u) << (4 * i);
            qweight[n * (K / 8) + c] = u;
        }
    }
}

void orc_w4a16_unpack(const uint32_t *qweight, uint8_t *q, int64_t N, int64_t K) {
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t kk = 0; kk < K; ++kk) {
            const uint32_t u = qweight[n * (K / 8) + kk / 8];
            q[n * K + kk] = (uint8_t)((u >> (4 * (kk % 8))) & 15u);
        }
    }
}

/* Zero points packed like the codes ([P3] "从数学表达式到真实存储": a zero
 * point packed in low bits needs one more bit extraction; "位级打包" gives the
 * nibble order): row n's groups 8c .. 8c+7 sit in word c, group g at bits
 * 4 (g mod 8) .. 4 (g mod 8) + 3; a row has ceil(ng / 8) words. */
void orc_w4a16_unpack_zeros(const uint32_t *zp, uint8_t *z, int64_t N, int64_t ng) {
    const int64_t words = (ng + 7) / 8;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t g = 0; g < ng; ++g)
            z[n * ng + g] = (uint8_t)((zp[n * words + g / 8] >> (4 * (g % 8))) & 15u);
}

void orc_w4a16_matmul(const uint32_t *qweight, const uint16_t *scales, const uint8_t *zeros,
                      int64_t G, const uint16_t *A, int64_t M, int64_t N, int64_t K,
                      const int64_t *rows, int64_t nrows, uint16_t *C16, double *C64, double *den,
                      int nthreads) {
    const int64_t ng = K / G;
    if (!rows) nrows = N;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        double *wh = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
        for (int64_t r = 0; r < nrows; ++r) {
            const int64_t n = rows ? rows[r] : r;
            for (int64_t kk = 0; kk < K; ++kk) {
                const int64_t g = kk / G;
                const uint32_t u = qweight[n * (K / 8) + kk / 8];
                const int q = (int)((u >> (4 * (kk % 8))) & 15u);
                const int z = zeros[n * ng + g];
                wh[kk] = (double)orc_fp16_to_fp32(scales[n * ng + g]) * (double)(q - z);
            }
            for (int64_t m = 0; m < M; ++m) {
                double s = 0.0, sa = 0.0;
                for (int64_t kk = 0; kk < K; ++kk) {
                    const double t = (double)orc_fp16_to_fp32(A[m * K + kk]) * wh[kk];
                    s += t;
                    sa += fabs(t);
                }
                if (C64) C64[m * nrows + r] = s;
                if (den) den[m * nrows + r] = sa;
                if (C16) C16[m * nrows + r] = orc_fp64_to_fp16(s);
            }
        }
        free(wh);
    }
}

/* Non-uniform 4-bit codes ([P3] "从数学表达式到真实存储": for NF4-like
 * formats q is an index into a code table, W-hat = s * LUT(q), no zero
 * point). lut holds the 16 table values as fp16 bit patterns. Outputs as
 * orc_w4a16_matmul. */
void orc_w4a16_lut_matmul(const uint32_t *qweight, const uint16_t *scales, const uint16_t *lut,
                          int64_t G, const uint16_t *A, int64_t M, int64_t N, int64_t K,
                          const int64_t *rows, int64_t nrows, uint16_t *C16, double *C64,
                          double *den, int nthreads) {
    const int64_t ng = K / G;
    if (!rows) nrows = N;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        double *wh = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
        for (int64_t r = 0; r < nrows; ++r) {
            const int64_t n = rows ? rows[r] : r;
            for (int64_t kk = 0; kk < K; ++kk) {
                const int64_t g = kk / G;
                const uint32_t u = qweight[n * (K / 8) + kk / 8];
                const int q = (int)((u >> (4 * (kk % 8))) & 15u);
                wh[kk] = (double)orc_fp16_to_fp32(scales[n * ng + g]) * (double)orc_fp16_to_fp32(lut[q]);
            }
            for (int64_t m = 0; m < M; ++m) {
                double s = 0.0, sa = 0.0;
                for (int64_t kk = 0; kk < K; ++kk) {
                    const double t = (double)orc_fp16_to_fp32(A[m * K + kk]) * wh[kk];
                    s += t;
                    sa += fabs(t);
                }
                if (C64) C64[m * nrows + r] = s;
                if (den) den[m * nrows + r] = sa;
                if (C16) C16[m * nrows + r] = orc_fp64_to_fp16(s);
            }
        }
        free(wh);
    }
}
