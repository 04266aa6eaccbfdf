/*
 * w4_oracle.c -- CPU oracle for the fused int4 dequantize-matmul.
 *
 * TEST INFRASTRUCTURE ONLY (see w4_oracle.h): used by tests/, the package
 * smoke check and the benchmark's CPU-baseline leg; never by the product.
 *
 * Build:  cc -O2 -std=c11 -ffp-contract=off -fPIC -shared w4_oracle.c -lm
 *         (add -fopenmp for the row-parallel timing build).
 *
 * W4_ORACLE_MUTANT=n plants one known mistake (a "mutant") so the tests can
 * show that the pins catch it.  The list mirrors the pitfalls table of
 * "Fused int4 and int8 dequantize-matmul in C" (section 5, mutants s01-s12)
 * and adds mistakes specific to the biased-Q4 / Q8 contracts:
 *    1 signed nibble read as unsigned            (s01)
 *    2 high nibble taken as the even column      (s02)
 *    3 group scales indexed by group only        (s03)
 *    4 group partial not reset per group         (s04)
 *    5 f16 scale decoded as bfloat16             (s05)
 *    6 every group reads the first group's codes (s06)
 *    7 per-row weight scale indexed by m         (s07)
 *    8 weight scale forgotten                    (s08)
 *    9 special summation order when M == 1       (s09)
 *   10 group that does not divide K accepted     (s10)
 *   11 NULL weights not checked                 (s11: the read crashes; its
 *      pin runs in a child process)
 *   12 last output row dropped when N % 8 != 0   (s12)
 *   13 +8 bias correction dropped
 *   14 ties rounded away from zero
 *   15 Q8 scale divides by 128 instead of 127
 *   16 odd-K pad nibble written as a raw 0
 *   17 Q4 scale divides by 8 instead of 7
 *   18 interleave puts channel d+32 in the low nibble
 *   19 amax taken as the signed maximum
 *   20 f16 subnormals decoded with an implicit leading 1
 *   21 interleave pairs channels 2d and 2d+1 in byte d
 *   22 bias correction uses 7 instead of 8
 *   23 activation bf16 decoded as f16
 *   24 grouped W4A8 zero point indexed by group only
 *   25 grouped W4A8 zero points ignored (the constant 8 used)
 *   26 Q8 weight matrix quantised with 128 in place of 127
 *   27 Q8 weight matrix row n quantised from row n - 1
 *   28 bf16 prefill dequantisation rounded through f16 instead
 *   29 bf16 prefill dequantisation truncated instead of rounded to even
 *   30 inline-scale block stores its f16 scale big-endian
 *   31 inline-scale reader takes the codes from the block's first byte
 *   32 W8A16 codes read as unsigned bytes
 *   33 int8 dot reads the second operand as unsigned
 *   34 interleave reader swaps the two channels of a byte
 *   35 interleave reader drops the odd-K pad nibble
 *   36 W8A32 codes read as unsigned bytes
 */
#pragma STDC FP_CONTRACT OFF

#include "w4_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifndef W4_ORACLE_MUTANT
#define W4_ORACLE_MUTANT 0
#endif
#define MUT(n) (W4_ORACLE_MUTANT == (n))

int ref_mutant_id(void) { return W4_ORACLE_MUTANT; }

/* ------------------------------------------------------------------------ */
/* Element decoders                                                          */
/* ------------------------------------------------------------------------ */

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits.  Normal:
 * (1024 + m) * 2^(e - 25); subnormal (e = 0): m * 2^-24.  Every binary16
 * value is exact in f32 ("Fused int4 ..." 2.2: "raw bit patterns of IEEE
 * half precision", decoded as half, not as bfloat16). */
float ref_f16_to_f32(uint16_t h) {
#if MUT(5)
    return ref_bf16_to_f32(h);
#else
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1F;
    const int m = h & 0x3FF;
    double v;
    if (e == 0) {
#if MUT(20)
        v = ldexp((double)(1024 + m), -25);
#else
        v = ldexp((double)m, -24);
#endif
    } else if (e == 31) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + m), e - 25);
    }
    return (float)(sign ? -v : v);
#endif
}

float ref_bf16_to_f32(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

uint16_t ref_f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
    const uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* Activation decoder for the W4A16 contract (bf16 x). */
static float act_bf16(uint16_t b) {
#if MUT(23)
    return ref_f16_to_f32(b);
#else
    return ref_bf16_to_f32(b);
#endif
}

/* Signed 4-bit two's complement: u when u < 8, u - 16 otherwise. */
int ref_nibble_signed(unsigned u) {
    u &= 0xF;
#if MUT(1)
    return (int)u;
#else
    return (int)u - (int)((u & 8u) << 1);
#endif
}

/* Biased by +8 ("Packing": [-7, 7] stored as [1, 15]). */
int ref_nibble_biased(unsigned u) { return (int)(u & 0xF) - 8; }

/* Raw nibble of column k in a packed row: byte k/2, low nibble for even k. */
static unsigned nib(const uint8_t *row, int64_t k) {
    const uint8_t b = row[k >> 1];
#if MUT(2)
    return (k & 1) ? (b & 0xFu) : (b >> 4);
#else
    return (k & 1) ? (b >> 4) : (b & 0xFu);
#endif
}

/* ------------------------------------------------------------------------ */
/* Quantizers                                                                */
/* ------------------------------------------------------------------------ */

/* The symmetric recipe ([int8] summary: scale = max|row| / 127, ties to
 * even, codes in [-127, 127]; [int4] contract: the same shape with 7, -8
 * never emitted).  Division is one f32 IEEE division; rint rounds in the
 * default round-to-nearest-even mode; the clamp keeps the range symmetric. */
void ref_quantize_row(const float *v, int64_t K, int Q, int8_t *q, float *s_out) {
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
#if MUT(19)
        const float a = v[k];
#else
        const float a = fabsf(v[k]);
#endif
        if (a > amax) amax = a;
    }
    float Qf = (float)Q;
#if MUT(17)
    if (Q == 7) Qf = 8.0f;
#endif
#if MUT(15)
    if (Q == 127) Qf = 128.0f;
#endif
    const float s = amax / Qf;
    *s_out = s;
    if (s == 0.0f) {
        for (int64_t k = 0; k < K; ++k) q[k] = 0;
        return;
    }
    const int lo = -Q;
    for (int64_t k = 0; k < K; ++k) {
        const float t = v[k] / s;
#if MUT(14)
        float r = roundf(t);
#else
        float r = rintf(t);
#endif
        if (r > (float)Q) r = (float)Q;
        if (r < (float)lo) r = (float)lo;
        q[k] = (int8_t)(int)r;
    }
}

int ref_quantize_row_q8(const float *x, int64_t M, int64_t K, int8_t *q, float *sx, int32_t *rowsum) {
    if (M < 0 || K < 0) return REF_EINVAL;
    if (M == 0) return REF_OK;
    if (!sx || (K > 0 && (!x || !q))) return REF_EINVAL;
    for (int64_t m = 0; m < M; ++m) {
        ref_quantize_row(x + m * K, K, 127, q + m * K, &sx[m]);
        if (rowsum) {
            int32_t acc = 0;
            for (int64_t k = 0; k < K; ++k) acc += q[m * K + k];
            rowsum[m] = acc;
        }
    }
    return REF_OK;
}

int ref_quantize_matrix_q4(const float *W, int64_t N, int64_t K, uint8_t *packed, float *sw) {
    if (N < 0 || K < 0) return REF_EINVAL;
    if (N == 0) return REF_OK;
    if (!sw || (K > 0 && (!W || !packed))) return REF_EINVAL;
    const int64_t Kb = (K + 1) / 2;
    int8_t *q = (int8_t *)malloc((size_t)(K > 0 ? K : 1));
    if (!q) return REF_EINVAL;
    for (int64_t n = 0; n < N; ++n) {
        ref_quantize_row(W + n * K, K, 7, q, &sw[n]);
        for (int64_t b = 0; b < Kb; ++b) {
            const unsigned lo = (unsigned)(q[2 * b] + 8);
#if MUT(16)
            const unsigned pad = 0u;
#else
            const unsigned pad = 8u; /* the biased zero */
#endif
            const unsigned hi = (2 * b + 1 < K) ? (unsigned)(q[2 * b + 1] + 8) : pad;
            packed[n * Kb + b] = (uint8_t)(lo | (hi << 4));
        }
    }
    free(q);
    return REF_OK;
}

int ref_quantize_matrix_q8(const float *W, int64_t N, int64_t K, int8_t *q, float *sw) {
    if (N < 0 || K < 0) return REF_EINVAL;
    if (N == 0) return REF_OK;
    if (!sw || (K > 0 && (!W || !q))) return REF_EINVAL;
    for (int64_t n = 0; n < N; ++n) {
#if MUT(26)
        ref_quantize_row(W + n * K, K, 128, q + n * K, &sw[n]);
#elif MUT(27)
        ref_quantize_row(W + (n > 0 ? n - 1 : 0) * K, K, 127, q + n * K, &sw[n]);
#else
        ref_quantize_row(W + n * K, K, 127, q + n * K, &sw[n]);
#endif
    }
    return REF_OK;
}

/* ------------------------------------------------------------------------ */
/* Dots                                                                      */
/* ------------------------------------------------------------------------ */

/* [int4] dot_i32_q4 / "Packing": storing u = q + 8 makes the unpack a
 * shift-and-mask, and sum x*q = sum x*u - 8 * sum x. */
int32_t ref_dot_i32_q4(const int8_t *xq, const uint8_t *wrow, int64_t K) {
    int32_t sxu = 0, sx = 0;
    for (int64_t k = 0; k < K; ++k) {
        sxu += (int32_t)xq[k] * (int32_t)nib(wrow, k);
        sx += xq[k];
    }
#if MUT(13)
    return sxu;
#elif MUT(22)
    return sxu - 7 * sx;
#else
    return sxu - 8 * sx;
#endif
}

int64_t ref_dot_naive_q4(const int8_t *xq, const uint8_t *wrow, int64_t K) {
    int64_t acc = 0;
    for (int64_t k = 0; k < K; ++k) acc += (int64_t)xq[k] * (int64_t)ref_nibble_biased(nib(wrow, k));
    return acc;
}

int32_t ref_dot_i32(const int8_t *a, const int8_t *b, int64_t K) {
    int32_t acc = 0;
#if MUT(33)
    for (int64_t k = 0; k < K; ++k) acc += (int32_t)a[k] * (int32_t)(uint8_t)b[k];
#else
    for (int64_t k = 0; k < K; ++k) acc += (int32_t)a[k] * (int32_t)b[k];
#endif
    return acc;
}

/* ------------------------------------------------------------------------ */
/* Linears                                                                   */
/* ------------------------------------------------------------------------ */

static int64_t rows_done(int64_t N) {
#if MUT(12)
    return (N % 8) ? N - 1 : N;
#else
    return N;
#endif
}

/* Both scales applied once per element after exact accumulation, in one
 * fixed order ([int8] summary): activation scale first, then the weight
 * scale, each an f32 multiply rounded to nearest even (no fused multiply-add). */
static float epilogue(int32_t acc, float sxm, float swn) {
    float y = (float)acc;
    y = y * sxm;
#if MUT(8)
    (void)swn;
#else
    y = y * swn;
#endif
    return y;
}

int ref_linear_q4(const int8_t *xq, const float *sx, const uint8_t *w, const float *sw,
                  float *y, int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0) return REF_EINVAL;
    if (M == 0 || N == 0) return REF_OK;
    if (!y || !sx || !sw || (K > 0 && (!xq || !w))) return REF_EINVAL;
    const int64_t Kb = (K + 1) / 2;
    const int64_t Nd = rows_done(N);
#pragma omp parallel for schedule(static, 8)
    for (int64_t n = 0; n < Nd; ++n)
        for (int64_t m = 0; m < M; ++m) {
            const int32_t acc = ref_dot_i32_q4(xq + m * K, w + n * Kb, K);
            y[m * N + n] = epilogue(acc, sx[m], sw[n]);
        }
    return REF_OK;
}

int ref_linear_q8(const int8_t *xq, const float *sx, const int8_t *wq, const float *sw,
                  float *y, int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0) return REF_EINVAL;
    if (M == 0 || N == 0) return REF_OK;
    if (!y || !sx || !sw || (K > 0 && (!xq || !wq))) return REF_EINVAL;
    const int64_t Nd = rows_done(N);
#pragma omp parallel for schedule(static, 8)
    for (int64_t n = 0; n < Nd; ++n)
        for (int64_t m = 0; m < M; ++m) {
            const int32_t acc = ref_dot_i32(xq + m * K, wq + n * K, K);
#if MUT(7)
            const float swn = sw[m < N ? m : N - 1];
#else
            const float swn = sw[n];
#endif
            y[m * N + n] = epilogue(acc, sx[m], swn);
        }
    return REF_OK;
}

/* linear_w8a16 (docs.rs ftts_kernels::int8, linear_w8a16: f32 activations
 * times a QuantizedMatrix, f32 out) as the tolerance reference:
 *   y64[m][n] = sw[n] * sum_k x[m][k] * q[n][k]   in double (every product exact),
 *   abs64     = |sw[n]| * sum_k |x[m][k] * q[n][k]|. */
int ref_linear_w8a16_exact(const float *x, const int8_t *wq, const float *sw, double *y64, double *abs64,
                           int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0) return REF_EINVAL;
    if (M == 0 || N == 0) return REF_OK;
    if (!y64 || !sw || (K > 0 && (!x || !wq))) return REF_EINVAL;
    const int64_t Nd = rows_done(N);
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < Nd; ++n) {
            double acc = 0.0, aacc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
#if MUT(32)
                const double p = (double)x[m * K + k] * (double)(uint8_t)wq[n * K + k];
#else
                const double p = (double)x[m * K + k] * (double)wq[n * K + k];
#endif
                acc += p;
                aacc += fabs(p);
            }
#if MUT(8)
            const double swn = 1.0;
#elif MUT(7)
            const double swn = (double)sw[m < N ? m : N - 1];
#else
            const double swn = (double)sw[n];
#endif
            y64[m * N + n] = swn * acc;
            if (abs64) abs64[m * N + n] = fabs(swn) * aacc;
        }
    return REF_OK;
}

int ref_linear_w8a32(const float *x, const int8_t *wq, const float *s, float *y,
                     int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0) return REF_EINVAL;
    if (M == 0 || N == 0) return REF_OK;
    if (!y || !s || (K > 0 && (!x || !wq))) return REF_EINVAL;
    const int64_t Nd = rows_done(N);
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < Nd; ++n) {
            float acc = 0.0f;
#if MUT(36)
            for (int64_t k = 0; k < K; ++k) acc = acc + x[m * K + k] * (float)(uint8_t)wq[n * K + k];
#else
            for (int64_t k = 0; k < K; ++k) acc = acc + x[m * K + k] * (float)wq[n * K + k];
#endif
#if MUT(8)
            y[m * N + n] = acc;
#elif MUT(7)
            y[m * N + n] = s[m < N ? m : N - 1] * acc;
#else
            y[m * N + n] = s[n] * acc;
#endif
        }
    return REF_OK;
}

/* Shape rules of "Fused int4 ..." section 2.2 / 4, with odd K accepted as
 * an extension: Kp = K rounded up to even is what the bytes describe, the
 * pad nibble is never read (x has no element K). */
static int w4a16_check(const void *x, const void *w, const void *s, const void *y,
                       int64_t M, int64_t N, int64_t K, int64_t G) {
    if (M < 0 || N < 0 || K < 0) return REF_EINVAL;
    const int64_t Kp = K + (K & 1);
#if MUT(10)
    if (G <= 0) return REF_ESHAPE;
#else
    if (G <= 0 || (G & 1) || (Kp % G) != 0) return REF_ESHAPE;
#endif
    if (M == 0 || N == 0) return REF_OK;
#if MUT(11)
    if (!y || (K > 0 && (!x || !s))) return REF_EINVAL;
#else
    if (!y || (K > 0 && (!x || !w || !s))) return REF_EINVAL;
#endif
    return -1; /* proceed */
}

static double scale_of(const uint16_t *s, int64_t n, int64_t ng, int64_t g) {
#if MUT(3)
    (void)n; (void)ng;
    return (double)ref_f16_to_f32(s[g]);
#else
    return (double)ref_f16_to_f32(s[n * ng + g]);
#endif
}

/* Column index of position i of group g (mutant 6 reads group 0 everywhere). */
static int64_t col_of(int64_t g, int64_t G, int64_t i) {
#if MUT(6)
    (void)g;
    return i;
#else
    return g * G + i;
#endif
}

/* y = sum_g s[n,g] * partial_g, partial_g = sum_{k in g} x[m,k] * q[n,k]
 * ("Fused int4 ..." 2.3).  Each x*q is an exact double (8 + 4 bits), each
 * partial a sum of at most G such products, each s*partial exact enough that
 * the only rounding is double addition. */
int ref_linear_w4a16_exact(const uint16_t *x, const uint8_t *w, const uint16_t *s,
                           double *y64, double *abs64, int64_t M, int64_t N, int64_t K, int64_t G) {
    const int rc = w4a16_check(x, w, s, y64, M, N, K, G);
    if (rc >= 0) return rc;
    const int64_t Kb = (K + 1) / 2, Kp = K + (K & 1), ng = Kp / G;
    const int64_t Nd = rows_done(N);
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < Nd; ++n) {
            const uint8_t *row = w + n * Kb;
            double acc = 0.0, aacc = 0.0, part = 0.0, apart = 0.0;
            for (int64_t g = 0; g < ng; ++g) {
#if !MUT(4)
                part = 0.0;
                apart = 0.0;
#endif
                for (int64_t i = 0; i < G; ++i) {
                    const int64_t k = col_of(g, G, i);
                    if (k >= K) continue;
                    const double p = (double)act_bf16(x[m * K + k]) * (double)ref_nibble_signed(nib(row, k));
                    part += p;
                    apart += fabs(p);
                }
                const double sg = scale_of(s, n, ng, g);
                acc += sg * part;
                aacc += fabs(sg) * apart;
            }
            y64[m * N + n] = acc;
            if (abs64) abs64[m * N + n] = aacc;
        }
    return REF_OK;
}

/* Grouped asymmetric W4A8 (vllm-omni "The 4-bit CPU path", "W4A8 --
 * _C::int4_scaled_mm_cpu": GPTQ-style weights with the checkpoint's zero
 * points, the constant 8 only when none are given; int8 activations):
 *   acc_g   = sum over k in group g (k < K) of xq[m][k] * (u[n][k] - z[n][g])   (exact integer)
 *   y64     = sx[m] * sum_g acc_g * s[n][g]                                      (double)
 *   abs64   = sum over k of |xq[m][k] * sx[m] * (u[n][k] - z[n][g]) * s[n][g]|   (tolerance denominator)
 * u are the raw stored nibbles (low nibble = even column), s f16 [N][Kp/G],
 * z one byte per group [N][Kp/G].  Every product acc_g * s_g is exact in
 * double; only the sum over groups rounds. */
static int64_t zero_of(const uint8_t *z, int64_t n, int64_t ng, int64_t g) {
#if MUT(24)
    (void)n; (void)ng;
    return z[g];
#elif MUT(25)
    (void)z; (void)n; (void)ng; (void)g;
    return 8;
#else
    return z[n * ng + g];
#endif
}

int ref_linear_q4_group(const int8_t *xq, const float *sx, const uint8_t *w, const uint16_t *s, const uint8_t *z,
                        double *y64, double *abs64, int64_t M, int64_t N, int64_t K, int64_t G) {
    const int rc = w4a16_check(xq, w, s, y64, M, N, K, G);
    if (rc >= 0) return rc;
    if (!sx || !z) return REF_EINVAL;
    const int64_t Kb = (K + 1) / 2, Kp = K + (K & 1), ng = Kp / G;
    const int64_t Nd = rows_done(N);
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < Nd; ++n) {
            const uint8_t *row = w + n * Kb;
            double acc = 0.0, aacc = 0.0;
            for (int64_t g = 0; g < ng; ++g) {
                const int64_t zz = zero_of(z, n, ng, g);
                int64_t ig = 0, ia = 0;
                for (int64_t i = 0; i < G; ++i) {
                    const int64_t k = col_of(g, G, i);
                    if (k >= K) continue;
                    const int64_t p = (int64_t)xq[m * K + k] * ((int64_t)nib(row, k) - zz);
                    ig += p;
                    ia += p < 0 ? -p : p;
                }
                const double sg = scale_of(s, n, ng, g);
                acc += (double)ig * sg;
                aacc += (double)ia * fabs(sg);
            }
            y64[m * N + n] = (double)sx[m] * acc;
            if (abs64) abs64[m * N + n] = fabs((double)sx[m]) * aacc;
        }
    return REF_OK;
}

/* Inline-scale block format, written from the description in "Fused int4
 * and int8 dequantize-matmul in C" (Going further: "blocks of 32 with the scale
 * stored inline next to the codes"): row n is nb = Kp / 32 blocks of 18 bytes,
 * bytes 0-1 the block's f16 scale (little-endian), bytes 2-17 the signed
 * nibbles of columns 32b .. 32b+31, low nibble = even column.  The same
 * numbers as group-wise W4A16 with G = 32; only the bytes move. */
int ref_blocks_b32(const uint8_t *w, const uint16_t *s, uint8_t *blocks, int64_t N, int64_t K) {
    if (N < 0 || K < 0) return REF_EINVAL;
    const int64_t Kp = K + (K & 1);
    if (Kp % 32) return REF_ESHAPE;
    if (N == 0 || K == 0) return REF_OK;
    if (!w || !s || !blocks) return REF_EINVAL;
    const int64_t nb = Kp / 32, Kb = Kp / 2;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < nb; ++b) {
            uint8_t *blk = blocks + (n * nb + b) * 18;
            const uint16_t sc = s[n * nb + b];
#if MUT(30)
            blk[0] = (uint8_t)(sc >> 8);
            blk[1] = (uint8_t)(sc & 0xFF);
#else
            blk[0] = (uint8_t)(sc & 0xFF);
            blk[1] = (uint8_t)(sc >> 8);
#endif
            for (int64_t j = 0; j < 16; ++j) blk[2 + j] = w[n * Kb + 16 * b + j];
        }
    return REF_OK;
}

/* Group-wise W4A16 read from the inline-scale blocks: every step of
 * ref_linear_w4a16_exact (G = 32), the codes and scale of group b taken from
 * block b of the row. */
int ref_linear_w4a16_b32_exact(const uint16_t *x, const uint8_t *blocks, double *y64, double *abs64,
                               int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0) return REF_EINVAL;
    const int64_t Kp = K + (K & 1);
    if (Kp % 32) return REF_ESHAPE;
    if (M == 0 || N == 0) return REF_OK;
    if (!y64 || (K > 0 && (!x || !blocks))) return REF_EINVAL;
    const int64_t nb = Kp / 32;
    const int64_t Nd = rows_done(N);
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < Nd; ++n) {
            double acc = 0.0, aacc = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t *blk = blocks + (n * nb + b) * 18;
                const double sg = (double)ref_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
                double part = 0.0, apart = 0.0;
                for (int64_t i = 0; i < 32; ++i) {
                    const int64_t k = 32 * b + i;
                    if (k >= K) continue;
#if MUT(31)
                    const double p = (double)act_bf16(x[m * K + k]) * (double)ref_nibble_signed(nib(blk, i));
#else
                    const double p = (double)act_bf16(x[m * K + k]) * (double)ref_nibble_signed(nib(blk + 2, i));
#endif
                    part += p;
                    apart += fabs(p);
                }
                acc += sg * part;
                aacc += fabs(sg) * apart;
            }
            y64[m * N + n] = acc;
            if (abs64) abs64[m * N + n] = aacc;
        }
    return REF_OK;
}

/* The pages' own f32 order ("Fused int4 ..." 2.4): 8 independent lanes per
 * group, lane l accumulating positions l, l+8, ... in increasing order; the
 * lanes combine in the fixed tree; the output accumulates s_g * partial_g in
 * increasing g.  Every step depends only on (m, n). */
int ref_linear_w4a16_lanes(const uint16_t *x, const uint8_t *w, const uint16_t *s,
                           float *y, int64_t M, int64_t N, int64_t K, int64_t G) {
    const int rc = w4a16_check(x, w, s, y, M, N, K, G);
    if (rc >= 0) return rc;
    const int64_t Kb = (K + 1) / 2, Kp = K + (K & 1), ng = Kp / G;
    const int64_t Nd = rows_done(N);
#pragma omp parallel for schedule(static, 8)
    for (int64_t n = 0; n < Nd; ++n)
        for (int64_t m = 0; m < M; ++m) {
            const uint8_t *row = w + n * Kb;
            float out = 0.0f;
            float lane[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            for (int64_t g = 0; g < ng; ++g) {
#if !MUT(4)
                for (int l = 0; l < 8; ++l) lane[l] = 0.0f;
#endif
                float partial;
#if MUT(9)
                if (M == 1) {
                    float seq = 0.0f;
                    for (int64_t i = 0; i < G; ++i) {
                        const int64_t k = col_of(g, G, i);
                        if (k < K) seq = seq + act_bf16(x[m * K + k]) * (float)ref_nibble_signed(nib(row, k));
                    }
                    partial = seq;
                } else
#endif
                {
                    for (int64_t i = 0; i < G; ++i) {
                        const int64_t k = col_of(g, G, i);
                        if (k >= K) continue;
                        const float prod = act_bf16(x[m * K + k]) * (float)ref_nibble_signed(nib(row, k));
                        lane[i & 7] = lane[i & 7] + prod;
                    }
                    partial = ((lane[0] + lane[1]) + (lane[2] + lane[3])) +
                              ((lane[4] + lane[5]) + (lane[6] + lane[7]));
                }
                const float sg = (float)scale_of(s, n, ng, g);
                out = out + sg * partial;
            }
            y[m * N + n] = out;
        }
    return REF_OK;
}

#if MUT(28)
/* Planted mistake only: f32 -> binary16, round to nearest even (normals;
 * the products used here never underflow binary16's normal range). */
static uint16_t f32_to_f16_rne_mutant(float f) {
    if (f == 0.0f) return 0;
    int e;
    const double m = frexp(fabs((double)f), &e); /* |f| = m * 2^e, m in [0.5, 1) */
    double r = rint(ldexp(m, 11));               /* 11 significant bits */
    if (r == 2048.0) { r = 1024.0; ++e; }
    const unsigned bits = (unsigned)((e - 1 + 15) << 10) | ((unsigned)r - 1024u);
    return (uint16_t)(bits | (f < 0 ? 0x8000u : 0u));
}
#endif

/* The prefill reading: each weight dequantized once to bf16,
 * w = bf16_rne(f32(q) * f32(s)) (the product is exact in f32), then summed
 * against x in double. */
int ref_linear_w4a16_bf16dequant(const uint16_t *x, const uint8_t *w, const uint16_t *s,
                                 double *y64, int64_t M, int64_t N, int64_t K, int64_t G) {
    const int rc = w4a16_check(x, w, s, y64, M, N, K, G);
    if (rc >= 0) return rc;
    const int64_t Kb = (K + 1) / 2, Kp = K + (K & 1), ng = Kp / G;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            const uint8_t *row = w + n * Kb;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const float sg = (float)scale_of(s, n, ng, k / G);
                const float wq = (float)ref_nibble_signed(nib(row, k)) * sg;
#if MUT(28)
                const float wb = ref_f16_to_f32(f32_to_f16_rne_mutant(wq));
#elif MUT(29)
                uint32_t wu;
                memcpy(&wu, &wq, sizeof wu);
                const float wb = ref_bf16_to_f32((uint16_t)(wu >> 16));
#else
                const float wb = ref_bf16_to_f32(ref_f32_to_bf16_rne(wq));
#endif
                acc += (double)act_bf16(x[m * K + k]) * (double)wb;
            }
            y64[m * N + n] = acc;
        }
    return REF_OK;
}

/* ------------------------------------------------------------------------ */
/* Interleaved [N/64][K][32 B] layout                                        */
/* ------------------------------------------------------------------------ */

/* "The weight layout, measured": per 64-channel block and per k, 32 bytes;
 * byte d carries channel d in its low nibble and channel d + 32 in its high
 * nibble, the same permutation for every k and every block. */
int ref_pack_interleaved_n64(const uint8_t *w_rm, uint8_t *w_il, int64_t N, int64_t K) {
    if (N < 0 || K < 0) return REF_EINVAL;
    if (N % 64) return REF_ESHAPE;
    if (N == 0 || K == 0) return REF_OK;
    if (!w_rm || !w_il) return REF_EINVAL;
    const int64_t Kb = (K + 1) / 2;
    for (int64_t b = 0; b < N / 64; ++b)
        for (int64_t k = 0; k < K; ++k)
            for (int d = 0; d < 32; ++d) {
#if MUT(18)
                const unsigned lo = nib(w_rm + (64 * b + d + 32) * Kb, k);
                const unsigned hi = nib(w_rm + (64 * b + d) * Kb, k);
#elif MUT(21)
                const unsigned lo = nib(w_rm + (64 * b + 2 * d) * Kb, k);
                const unsigned hi = nib(w_rm + (64 * b + 2 * d + 1) * Kb, k);
#else
                const unsigned lo = nib(w_rm + (64 * b + d) * Kb, k);
                const unsigned hi = nib(w_rm + (64 * b + d + 32) * Kb, k);
#endif
                w_il[(b * K + k) * 32 + d] = (uint8_t)(lo | (hi << 4));
            }
    return REF_OK;
}

int ref_unpack_interleaved_n64(const uint8_t *w_il, uint8_t *w_rm, int64_t N, int64_t K, unsigned pad) {
    if (N < 0 || K < 0) return REF_EINVAL;
    if (N % 64) return REF_ESHAPE;
    if (N == 0 || K == 0) return REF_OK;
    if (!w_rm || !w_il) return REF_EINVAL;
    const int64_t Kb = (K + 1) / 2;
    memset(w_rm, 0, (size_t)(N * Kb));
    for (int64_t b = 0; b < N / 64; ++b)
        for (int64_t k = 0; k < K; ++k)
            for (int d = 0; d < 32; ++d) {
                const uint8_t byte = w_il[(b * K + k) * 32 + d];
#if MUT(34)
                const int64_t n0 = 64 * b + d + 32, n1 = 64 * b + d;
#else
                const int64_t n0 = 64 * b + d, n1 = 64 * b + d + 32;
#endif
                const unsigned sh = (unsigned)(k & 1) * 4u;
                w_rm[n0 * Kb + k / 2] |= (uint8_t)((byte & 0xFu) << sh);
                w_rm[n1 * Kb + k / 2] |= (uint8_t)((byte >> 4) << sh);
            }
#if MUT(35)
    (void)pad;
#else
    if (K & 1)
        for (int64_t n = 0; n < N; ++n) w_rm[n * Kb + Kb - 1] |= (uint8_t)((pad & 0xFu) << 4);
#endif
    return REF_OK;
}
