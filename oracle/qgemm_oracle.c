/*
 * qgemm_oracle.c -- plain, slow CPU oracle for the block-scaled quantized matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may link, load or call
 * this file; only the test suite, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header, table or constant with the CUDA path.
 *
 * What it computes (page citations name the page's title and section):
 *   - "TensorOps: quantized matmul, cooperative tensors, and the neural accelerator",
 *     section "Scale planes: one MTLTensor = data + scales": one tensor is a data plane plus an
 *     auxiliary plane of block scales; a 32x1 block means 32 consecutive data elements (along the
 *     contiguous dimension) share one scale.
 *   - same page, section "Kernel-phase findings", fact 2: the scale type is FP8 E8M0 (UE8M0,
 *     a power of two), block sizes 32 (inner) and 1 (outer).
 *   - same page, fact 5 of "VALIDATED ON M4 MAX": int4 is two's complement, two per byte, the
 *     low nibble holds the even linear index.
 *   - "Optimize custom machine learning operations with Metal tensors" (WWDC26 session 330
 *     summary), section "Shader MXFP8 tensor types": the data plane type is FP8 E4M3.
 *   - "Running inline ML operations in a shader with Metal 4": the product is checked against
 *     a CPU reference implementation; matmul2d in multiply mode overwrites C with A*B.
 *   - same summary, section on the quantized data types: OS 27 adds 4-bit and 8-bit floating-point
 *     data planes ("fp4, fp8, int2 native" in the TensorOps page's table).
 * Readings where the pages are silent:
 *   - fp4 is the OCP MX FP4 element E2M1 (sign, 2 exponent bits with bias 1, 1 mantissa bit; no
 *     infinity or NaN; largest magnitude 6), packed two per byte with the low nibble holding the
 *     even index (the pages' int4 rule), with the same UE8M0 block-32 scale plane.
 *   - E4M3 is the OCP 8-bit E4M3 encoding (bias 7, no infinity, S.1111.111 is NaN).
 *   - UE8M0 byte e means 2^(e-127); e = 255 is NaN.
 *   - The exact product sum_k deq(A)[m,k]*deq(B)[n,k] is formed in fp64; the reported output is
 *     that value rounded to IEEE binary16 with round-to-nearest-even, overflow to +-inf.
 *
 *   - "TensorOps: quantized matmul ...", sections "Revised kernel strategy" and "M2 = block-32
 *     fp16 scaling" (the custom-format escape hatch: int4 weights with arbitrary fp16 scales per
 *     block of 32 along K, which the native E8M0 scale plane cannot carry): each weight of a
 *     block is dequantised into half precision as its int4 value times the block's fp16 scale,
 *     and the half x half product is accumulated.  Reading: that dequantised weight is the fp16
 *     round-to-nearest-even of the exact product q * s (one rounding, as a half multiply gives);
 *     the product is then formed exactly from those weights.
 *   - "TensorOps: quantized matmul ...", section "FlashAttention on TensorOps (the recipe)", and
 *     "Optimize custom machine learning operations with Metal tensors", section on FlashAttention
 *     with cooperative tensors: fused attention multiplies Q by K^T, takes each row's maximum
 *     (initial value -infinity), exponentiates each score minus its row maximum, and multiplies
 *     the result by V.  Readings: the softmax is normalised (each row of exp(s - max) divided by
 *     its sum, which is what softmax means in that text); the scores carry a caller-given scale
 *     (1/sqrt(d) for scaled dot-product attention); no mask (the recipe shows none).
 * Every function here follows the plain definition: decode each element, multiply by its
 * block's scale, sum the products in index order.  No blocking, no reordering.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* dtype codes private to the oracle */
enum { ORC_F16 = 0, ORC_E4M3 = 1, ORC_INT8 = 2, ORC_INT4 = 3, ORC_E2M1 = 4 };

/* OCP FP8 E4M3: sign(1) exponent(4, bias 7) mantissa(3).  Exponent field 0 is subnormal
 * (m * 2^-9); exponent 15 with mantissa 7 is NaN; there is no infinity. */
double orc_e4m3(uint8_t b) {
    int s = (b >> 7) & 1;
    int e = (b >> 3) & 15;
    int m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* OCP FP4 E2M1 (low 4 bits of nib): sign(1) exponent(2, bias 1) mantissa(1).  Exponent field 0
 * is subnormal (m * 2^-1); no infinity, no NaN. */
double orc_e2m1(uint8_t nib) {
    int s = (nib >> 3) & 1;
    int e = (nib >> 1) & 3;
    int m = nib & 1;
    double v = (e == 0) ? ldexp((double)m, -1) : ldexp(1.0 + (double)m / 2.0, e - 1);
    return s ? -v : v;
}

/* UE8M0 block scale: unsigned exponent only, value 2^(e-127); 0xFF is NaN. */
double orc_ue8m0(uint8_t e) {
    if (e == 255) return NAN;
    return ldexp(1.0, (int)e - 127);
}

/* IEEE binary16 bits -> value. */
double orc_f16(uint16_t h) {
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 31) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m, -24);
    else v = ldexp(1.0 + (double)m / 1024.0, e - 15);
    return s ? -v : v;
}

/* value -> IEEE binary16 bits, round to nearest, ties to even; magnitudes that round past the
 * largest finite value (65504) become infinity. */
uint16_t orc_f16_rn(double x) {
    uint16_t sign;
    double a, q;
    int E, e;
    if (isnan(x)) return 0x7E00;
    sign = signbit(x) ? 0x8000 : 0;
    a = fabs(x);
    if (isinf(a)) return sign | 0x7C00;
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: integer multiples of 2^-24 */
        q = rint(ldexp(a, 24));           /* exact scaling, then round half to even */
        return sign | (uint16_t)q;        /* q == 1024 is the smallest normal, bit-for-bit */
    }
    frexp(a, &E);                         /* a = f * 2^E, f in [0.5, 1) */
    e = E - 1;                            /* a = (1 + frac) * 2^e */
    q = rint((ldexp(a, -e) - 1.0) * 1024.0);
    if (q == 1024.0) { q = 0.0; e += 1; }
    if (e + 15 >= 31) return sign | 0x7C00;
    return sign | (uint16_t)(((e + 15) << 10) | (int)q);
}

static int orc_int8_val(uint8_t b) {
    int v = (int)b;
    return v >= 128 ? v - 256 : v;
}

/* element k of a packed int4 row: byte k/2, low nibble for even k, high nibble for odd k */
static int orc_int4_val(const uint8_t *row, int64_t k) {
    int byte = row[k >> 1];
    int nib = (k & 1) ? (byte >> 4) & 15 : byte & 15;
    return nib >= 8 ? nib - 16 : nib;
}

int orc_int4_get(const uint8_t *row, int64_t k) { return orc_int4_val(row, k); }

/* element k of a packed E2M1 row: byte k/2, low nibble for even k, high nibble for odd k */
static double orc_e2m1_val(const uint8_t *row, int64_t k) {
    int byte = row[k >> 1];
    return orc_e2m1((uint8_t)((k & 1) ? (byte >> 4) & 15 : byte & 15));
}
int orc_int8_get(uint8_t b) { return orc_int8_val(b); }

/* Decoded value of element (r, j) of a [rows, k] plane, scale included. */
static double orc_element(int dtype, const uint8_t *data, int64_t ld, const uint8_t *scales,
                          int64_t lds, int64_t r, int64_t j) {
    const uint8_t *row = data + r * ld;
    double q, s;
    uint16_t h;
    switch (dtype) {
    case ORC_F16:
        memcpy(&h, row + 2 * j, 2);
        return orc_f16(h);
    case ORC_E4M3: q = orc_e4m3(row[j]); break;
    case ORC_INT8: q = (double)orc_int8_val(row[j]); break;
    case ORC_INT4: q = (double)orc_int4_val(row, j); break;
    case ORC_E2M1: q = orc_e2m1_val(row, j); break;
    default: return NAN;
    }
    s = orc_ue8m0(scales[r * lds + j / 32]);   /* block of 32 along k, one row per block row */
    return q * s;
}

/* int4 weights with fp16 block scales (the M2 recipe): out[i*k + j] = value of
 * fp16_rn(int4(W[r, j]) * fp16(S[r, j / 32])) for r = rows_idx[i]; S is [rows, k/32] fp16 bits
 * with a row stride of lds elements. */
void orc_dequant_int4_f16s(int64_t nrows, int64_t k, const uint8_t *data, int64_t ld,
                           const uint16_t *scales, int64_t lds, const int64_t *rows_idx,
                           double *out) {
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < nrows; ++i) {
        int64_t r = rows_idx ? rows_idx[i] : i;
        const uint8_t *row = data + r * ld;
        int64_t j;
        for (j = 0; j < k; ++j) {
            double exact = (double)orc_int4_val(row, j) * orc_f16(scales[r * lds + j / 32]);
            out[i * k + j] = orc_f16(orc_f16_rn(exact));
        }
    }
}

/* out[i*k + j] = decoded element (rows_idx[i], j).  rows_idx == NULL means rows 0..nrows-1. */
void orc_dequant(int dtype, int64_t nrows, int64_t k, const uint8_t *data, int64_t ld,
                 const uint8_t *scales, int64_t lds, const int64_t *rows_idx, double *out) {
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < nrows; ++i) {
        int64_t r = rows_idx ? rows_idx[i] : i;
        int64_t j;
        for (j = 0; j < k; ++j) out[i * k + j] = orc_element(dtype, data, ld, scales, lds, r, j);
    }
}

/* fp16 matrix stored [k, cols] row-major (leading dimension ld elements), read transposed:
 * out[i*k + j] = value(B[j, cols_idx[i]]).  This is the right operand of the fp16 GEMM. */
void orc_dequant_f16_kn(int64_t ncols, int64_t k, const uint16_t *b, int64_t ld,
                        const int64_t *cols_idx, double *out) {
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < ncols; ++i) {
        int64_t c = cols_idx ? cols_idx[i] : i;
        int64_t j;
        for (j = 0; j < k; ++j) out[i * k + j] = orc_f16(b[j * ld + c]);
    }
}

/* C[i, n] = sum_j A[i, j] * B[n, j]; D[i, n] = sum_j |A[i, j] * B[n, j]|, in fp64, j ascending.
 * A is [ma, k], B is [nb, k], both row-major fp64. */
void orc_dot_rows(int64_t ma, int64_t nb, int64_t k, const double *A, const double *B, double *C,
                  double *D) {
    int64_t i;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = 0; i < ma; ++i) {
        const double *a = A + i * k;
        int64_t n;
        for (n = 0; n < nb; ++n) {
            const double *b = B + n * k;
            double c = 0.0, d = 0.0;
            int64_t j;
            for (j = 0; j < k; ++j) {
                double p = a[j] * b[j];
                c += p;
                d += fabs(p);
            }
            C[i * nb + n] = c;
            D[i * nb + n] = d;
        }
    }
}

/* Decode-as-you-go product for a long right operand (the decode GEMV): for every row n of the
 * quantized plane W [nw, k], decode it and dot it with each of the ma fp64 rows of X.
 * C and D are [ma, nw]. */
void orc_dot_quant(int64_t ma, int64_t nw, int64_t k, const double *X, int dtype,
                   const uint8_t *w, int64_t ldw, const uint8_t *sw, int64_t ldsw, double *C,
                   double *D) {
    int64_t n;
#pragma omp parallel for schedule(dynamic, 16)
    for (n = 0; n < nw; ++n) {
        int64_t i;
        for (i = 0; i < ma; ++i) {
            const double *x = X + i * k;
            double c = 0.0, d = 0.0;
            int64_t j;
            for (j = 0; j < k; ++j) {
                double p = x[j] * orc_element(dtype, w, ldw, sw, ldsw, n, j);
                c += p;
                d += fabs(p);
            }
            C[i * nw + n] = c;
            D[i * nw + n] = d;
        }
    }
}

/* bits[i] = fp16 round-to-nearest-even of x[i] */
void orc_f16_rn_array(int64_t count, const double *x, uint16_t *bits) {
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < count; ++i) bits[i] = orc_f16_rn(x[i]);
}

/* Fused attention, one output row per (head, query) pair listed in heads[i], qrows[i]:
 *   s_j = scale * sum_c Q[h, r, c] K[h, j, c]        (j = 0 .. Lk-1)
 *   m = max_j s_j;  p_j = exp(s_j - m);  l = sum_j p_j
 *   O[i, c] = sum_j p_j V[h, j, c] / l;   Dm[i, c] = sum_j p_j |V[h, j, c]| / l
 * Q, K, V are fp16 bits laid out [BH][L][d] with the given head and row strides (elements).
 * Dm is the magnitude the tolerance is normalised by. */
void orc_attention(int64_t n, const int64_t *heads, const int64_t *qrows, int64_t Lk, int64_t d,
                   const uint16_t *Q, int64_t q_hs, int64_t q_rs, const uint16_t *K, int64_t k_hs,
                   int64_t k_rs, const uint16_t *V, int64_t v_hs, int64_t v_rs, double scale,
                   double *O, double *Dm) {
    int64_t i;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = 0; i < n; ++i) {
        const uint16_t *q = Q + heads[i] * q_hs + qrows[i] * q_rs;
        double *s = (double *)malloc((size_t)Lk * sizeof(double));
        double m = -INFINITY, l = 0.0;
        int64_t j, c;
        for (j = 0; j < Lk; ++j) {
            const uint16_t *k = K + heads[i] * k_hs + j * k_rs;
            double dot = 0.0;
            for (c = 0; c < d; ++c) dot += orc_f16(q[c]) * orc_f16(k[c]);
            s[j] = scale * dot;
            if (s[j] > m) m = s[j];
        }
        for (j = 0; j < Lk; ++j) {
            s[j] = exp(s[j] - m);
            l += s[j];
        }
        for (c = 0; c < d; ++c) {
            double o = 0.0, a = 0.0;
            for (j = 0; j < Lk; ++j) {
                double v = orc_f16(V[heads[i] * v_hs + j * v_rs + c]);
                o += s[j] * v;
                a += s[j] * fabs(v);
            }
            O[i * d + c] = o / l;
            Dm[i * d + c] = a / l;
        }
        free(s);
    }
}

/* tables for the pin tests: all 256 codes of each 8-bit format */
void orc_e4m3_table(double *out) {
    int b;
    for (b = 0; b < 256; ++b) out[b] = orc_e4m3((uint8_t)b);
}

void orc_e2m1_table(double *out) {
    int b;
    for (b = 0; b < 16; ++b) out[b] = orc_e2m1((uint8_t)b);
}

void orc_ue8m0_table(double *out) {
    int b;
    for (b = 0; b < 256; ++b) out[b] = orc_ue8m0((uint8_t)b);
}
