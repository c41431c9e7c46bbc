/*
 * oracle.c -- plain, slow, obviously-correct CPU reference for the GGUF
 * block-quantised weight x f32 activation matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the bench's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * Build: gcc -std=c99 -O2 -fno-fast-math -ffp-contract=off -shared -fPIC
 * (no FMA contraction, no fast-math: the activation quantiser below is
 * defined in IEEE binary32 arithmetic and must be computed exactly so).
 * The same file built with -fopenmp runs the output rows of the matvec, the
 * block dots and the MMQ reference on all cores (one thread per row at a time,
 * each row's arithmetic and summation order exactly as in the plain build, so
 * both builds return the same bits); without -fopenmp the pragmas are ignored.
 *
 * What it computes, and the passage each function follows:
 *
 *  - f16 -> double: IEEE 754 binary16 decoding, subnormals and signed zero
 *    included (the block scales d and dmin are binary16); bf16 -> double likewise
 *    (the upper half of a binary32).  f16 and bf16 weight rows (the f16/bf16 kernels
 *    of "CUDA Backend Design" §4.4) are K such elements, with no integer form.
 *  - dequantisation of one weight row, per the GGUF block layouts whose byte
 *    ratios the minfer "CUDA Backend Design" page gives in §2.3 (q8_0 34 bytes
 *    per 32 elements, q4_K 144 per 256, q6_K 210 per 256; q4_0 and q5_K, among
 *    the types the page's weight gate admits in §4.6, 18 per 32 and 176 per 256)
 *    and whose field
 *    layout is the public ggml block format, restated in prose in the header
 *    of each function below.
 *  - the decode matvec reference y[b][n] = sum_k w[n][k] * x[b][k] in double,
 *    k in increasing order ("CUDA Backend Design" §4.4: f32 activations, the
 *    quantised matmul family), with the per-row bound sum_k |w||x|.
 *  - the activation quantiser (per row, per 32-element block: amax, scale =
 *    amax/127, q = round-half-even(x/scale)) in binary32, following the
 *    Q8_0 quantiser steps of "Architecture Execution Plan" C4 S2b design
 *    decision 4 with the scale kept in f32 (the plainest reading of the
 *    prefill-MMQ statement "scale = max|x|/127").
 *  - the per-block integer dots D[m][n][b] = sum_{k in block b} W_int[n][k] *
 *    q[m][k] in int64, where W_int is the block's integer weight (q8_0: the
 *    int8 quant; q4_K: sub-block scale times 4-bit quant; q6_K: 16-element
 *    sub-scale times (6-bit quant - 32)).
 *  - the prefill MMQ reference y[m][n] = sum_k w[n][k] * (scale[m][b] *
 *    q[m][k]) in double, with the bound sum_k |w| |scale*q| ("CUDA Backend
 *    Design" §4.4: prefill quantises A into per-32 int8 blocks).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads the row loops below use: 1 in the plain build. */
int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Sets the thread count of the row loops (OpenMP build; a no-op otherwise). */
void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

#define OR_F16 1
#define OR_BF16 30
#define OR_Q4_0 2
#define OR_Q4_1 3
#define OR_Q5_0 6
#define OR_Q5_1 7
#define OR_Q8_0 8
#define OR_Q4_K 12
#define OR_Q5_K 13
#define OR_Q6_K 14

/* ---- IEEE binary16 -> double ------------------------------------------ */
/* sign 1 bit, exponent 5 bits (bias 15), fraction 10 bits.  exponent 0:
 * subnormal fraction * 2^-24; exponent 31: infinity / NaN. */
double oracle_f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25);
    }
    return sign ? -v : v;
}

/* ---- bfloat16 -> double --------------------------------------------------
 * sign 1 bit, exponent 8 bits (bias 127), fraction 7 bits (the upper half of a
 * binary32).  exponent 0: subnormal fraction * 2^-133; exponent 255: inf / NaN. */
double oracle_bf16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 255;
    int f = h & 127;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133);
    } else if (e == 255) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(128 + f), e - 134);
    }
    return sign ? -v : v;
}

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* f16 / bf16 weights: one 2-byte little-endian element per "block", no integer form */
static int is_float_type(int type) { return type == OR_F16 || type == OR_BF16; }

int oracle_block_elems(int type)
{
    switch (type) {
    case OR_F16: return 1;
    case OR_BF16: return 1;
    case OR_Q4_0: return 32;
    case OR_Q4_1: return 32;
    case OR_Q5_0: return 32;
    case OR_Q5_1: return 32;
    case OR_Q8_0: return 32;
    case OR_Q4_K: return 256;
    case OR_Q5_K: return 256;
    case OR_Q6_K: return 256;
    default: return 0;
    }
}

int oracle_block_bytes(int type)
{
    switch (type) {
    case OR_F16: return 2;
    case OR_BF16: return 2;
    case OR_Q4_0: return 18;
    case OR_Q4_1: return 20;
    case OR_Q5_0: return 22;
    case OR_Q5_1: return 24;
    case OR_Q8_0: return 34;
    case OR_Q4_K: return 144;
    case OR_Q5_K: return 176;
    case OR_Q6_K: return 210;
    default: return 0;
    }
}

/* q4_K 6-bit sub-block scale and min, j = 0..7, from the 12 packed bytes.
 * j < 4 : scale = s[j] & 63,                       min = s[j+4] & 63
 * j >= 4: scale = (s[j+4] & 15) | (s[j-4] >> 6) << 4, min = (s[j+4] >> 4) | (s[j] >> 6) << 4 */
void oracle_q4_k_scale_min(const uint8_t *s12, int j, int *sc, int *mn)
{
    if (j < 4) {
        *sc = s12[j] & 63;
        *mn = s12[j + 4] & 63;
    } else {
        *sc = (s12[j + 4] & 15) | ((s12[j - 4] >> 6) << 4);
        *mn = (s12[j + 4] >> 4) | ((s12[j] >> 6) << 4);
    }
}

/* Integer weight of element e of one block, and the block-level scales.
 * The dequantised weight is  w = dscale * wint - dmin_term, where
 *   q4_0: wint = nib(e) - 8,           dscale = d, dmin_term = 0
 *   q4_1: wint = nib(e),               dscale = d, dmin_term = -m   (w = d*nib + m)
 *   q5_0: wint = q5(e) - 16,           dscale = d, dmin_term = 0
 *   q5_1: wint = q5(e),                dscale = d, dmin_term = -m   (w = d*q5 + m)
 *   q8_0: wint = q[e],                 dscale = d, dmin_term = 0
 *   q4_K: wint = sc_j * nib(e),        dscale = d, dmin_term = dmin * m_j
 *   q5_K: wint = sc_j * q5(e),         dscale = d, dmin_term = dmin * m_j
 *   q6_K: wint = sc[16-group] * (q-32), dscale = d, dmin_term = 0
 * q4_0 (d f16 at 0, 16 quant bytes at 2): element e = 16h + j, nib = (qs[j] >> 4h) & 15.
 * q4_1 (d, m f16 at 0 and 2, 16 quant bytes at 4): nibbles as q4_0.
 * q5_0 (d f16 at 0, fifth-bit word qh (u32, little-endian) at 2, 16 quant bytes at 6):
 *   q5 = nib(e) | ((qh >> e) & 1) << 4, nibbles as q4_0.
 * q5_1 (d, m f16 at 0 and 2, qh at 4, 16 quant bytes at 8): as q5_0.
 * q5_K (d, dmin f16 at 0 and 2, 12 scale bytes at 4 packed as in q4_K, 32 high-bit
 *   bytes at 16, 128 quant bytes at 48): element e = 64c + 32h + l,
 *   q5 = ((qs[32c+l] >> 4h) & 15) | ((qh[l] >> (2c + h)) & 1) << 4, j = 2c + h.
 * q4_K element e = 64c + 32h + l: nib = (qs[32c+l] >> 4h) & 15, j = 2c + h.
 * q6_K element e = 128h + 32r + l:
 *   lo4 = ql[64h + 32(r%2) + l], low nibble for r < 2, high nibble for r >= 2
 *   hi2 = (qh[32h + l] >> 2r) & 3,  q = lo4 | hi2 << 4
 *   sub-scale index 8h + 2r + l/16. */
static void block_elem(int type, const uint8_t *blk, int e, int64_t *wint, int *mterm)
{
    *mterm = 0;
    if (type == OR_Q8_0) {
        *wint = (int8_t)blk[2 + e];
    } else if (type == OR_Q4_0) {
        int h = e / 16, j = e % 16;
        *wint = ((blk[2 + j] >> (4 * h)) & 15) - 8;
    } else if (type == OR_Q4_1) {
        int h = e / 16, j = e % 16;
        *wint = (blk[4 + j] >> (4 * h)) & 15;
        *mterm = -1;
    } else if (type == OR_Q5_0 || type == OR_Q5_1) {
        int h = e / 16, j = e % 16, qo = type == OR_Q5_0 ? 6 : 8, ho = type == OR_Q5_0 ? 2 : 4;
        uint32_t qh = (uint32_t)blk[ho] | ((uint32_t)blk[ho + 1] << 8) |
                      ((uint32_t)blk[ho + 2] << 16) | ((uint32_t)blk[ho + 3] << 24);
        int q5 = ((blk[qo + j] >> (4 * h)) & 15) | (int)(((qh >> e) & 1) << 4);
        *wint = type == OR_Q5_0 ? q5 - 16 : q5;
        *mterm = type == OR_Q5_0 ? 0 : -1;
    } else if (type == OR_Q5_K) {
        int c = e / 64, h = (e / 32) % 2, l = e % 32;
        int q5 = ((blk[48 + 32 * c + l] >> (4 * h)) & 15) | (((blk[16 + l] >> (2 * c + h)) & 1) << 4);
        int sc, mn;
        oracle_q4_k_scale_min(blk + 4, 2 * c + h, &sc, &mn);
        *wint = (int64_t)sc * q5;
        *mterm = mn;
    } else if (type == OR_Q4_K) {
        int c = e / 64, h = (e / 32) % 2, l = e % 32;
        int nib = (blk[16 + 32 * c + l] >> (4 * h)) & 15;
        int sc, mn;
        oracle_q4_k_scale_min(blk + 4, 2 * c + h, &sc, &mn);
        *wint = (int64_t)sc * nib;
        *mterm = mn;
    } else { /* OR_Q6_K */
        int h = e / 128, r = (e / 32) % 4, l = e % 32;
        int qlb = blk[64 * h + 32 * (r % 2) + l];
        int lo4 = (r < 2) ? (qlb & 15) : (qlb >> 4);
        int hi2 = (blk[128 + 32 * h + l] >> (2 * r)) & 3;
        int q = lo4 | (hi2 << 4);
        int sc = (int8_t)blk[192 + 8 * h + 2 * r + l / 16];
        *wint = (int64_t)sc * (q - 32);
    }
}

static double block_d(int type, const uint8_t *blk)
{
    if (type == OR_Q8_0 || type == OR_Q4_0 || type == OR_Q4_1 || type == OR_Q5_0 ||
        type == OR_Q5_1)
        return oracle_f16_to_double(rd16(blk));
    if (type == OR_Q4_K || type == OR_Q5_K) return oracle_f16_to_double(rd16(blk));
    return oracle_f16_to_double(rd16(blk + 208));
}

static double block_dmin(int type, const uint8_t *blk)
{
    /* q4_K, q5_K: dmin; q4_1, q5_1: the additive min m (paired with mterm = -1) */
    return (type == OR_Q4_K || type == OR_Q5_K || type == OR_Q4_1 || type == OR_Q5_1)
               ? oracle_f16_to_double(rd16(blk + 2))
               : 0.0;
}

static int valid_shape(int type, int64_t K)
{
    int be = oracle_block_elems(type);
    return be > 0 && K > 0 && K % be == 0;
}

/* Dequantise one row of K elements (row = K/blk blocks, contiguous). */
int oracle_dequant_row(int type, const uint8_t *row, int64_t K, double *out)
{
    if (!valid_shape(type, K)) return -1;
    if (is_float_type(type)) {
        for (int64_t k = 0; k < K; ++k)
            out[k] = type == OR_F16 ? oracle_f16_to_double(rd16(row + 2 * k))
                                    : oracle_bf16_to_double(rd16(row + 2 * k));
        return 0;
    }
    int be = oracle_block_elems(type), bb = oracle_block_bytes(type);
    for (int64_t b = 0; b < K / be; ++b) {
        const uint8_t *blk = row + b * bb;
        double d = block_d(type, blk), dmin = block_dmin(type, blk);
        for (int e = 0; e < be; ++e) {
            int64_t wint;
            int mterm;
            block_elem(type, blk, e, &wint, &mterm);
            out[b * be + e] = d * (double)wint - dmin * (double)mterm;
        }
    }
    return 0;
}

/* Integer weights of one row (the W_int of the block dots). */
int oracle_int_weights_row(int type, const uint8_t *row, int64_t K, int64_t *out)
{
    if (!valid_shape(type, K) || is_float_type(type)) return -1;
    int be = oracle_block_elems(type), bb = oracle_block_bytes(type);
    for (int64_t b = 0; b < K / be; ++b) {
        for (int e = 0; e < be; ++e) {
            int mterm;
            block_elem(type, row + b * bb, e, &out[b * be + e], &mterm);
        }
    }
    return 0;
}

/* Decode matvec for rows n0 <= n < n1 of W (N x K), all B activation rows.
 * y[b*(n1-n0) + (n-n0)] = sum_k w[n][k] x[b][k]; bound likewise = sum |w||x|. */
int oracle_matvec(int type, const uint8_t *W, int64_t N, int64_t K, const float *x, int B,
                  int64_t n0, int64_t n1, double *y, double *bound)
{
    if (!valid_shape(type, K) || n0 < 0 || n1 > N || n0 > n1 || B < 1) return -1;
    int64_t rowbytes = K / oracle_block_elems(type) * oracle_block_bytes(type);
    int err = 0;
#pragma omp parallel
    {
        double *w = (double *)malloc((size_t)K * sizeof(double));
        if (!w) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 8)
        for (int64_t n = n0; n < n1; ++n) {
            if (!w) continue;
            oracle_dequant_row(type, W + n * rowbytes, K, w);
            for (int b = 0; b < B; ++b) {
                double acc = 0.0, bnd = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    double xv = (double)x[(int64_t)b * K + k];
                    acc += w[k] * xv;
                    bnd += fabs(w[k]) * fabs(xv);
                }
                y[(int64_t)b * (n1 - n0) + (n - n0)] = acc;
                bound[(int64_t)b * (n1 - n0) + (n - n0)] = bnd;
            }
        }
        free(w);
    }
    return err;
}

/* Activation quantiser, binary32 throughout.  For row m and 32-element block
 * b (elements 32b .. 32b+31):
 *   amax  = max |x|                         (fabsf: exact)
 *   s     = amax / 127.0f                   (correctly rounded f32 division)
 *   if s == 0 (amax == 0, or the division underflows): q = 0, S = 0
 *   else q = nearbyintf(x / s)              (f32 division, round half to even)
 *        clamped to [-127, 127],  S = sum q (int32)
 * qs[m*K + k], scale[m*(K/32) + b], bsum[m*(K/32) + b]. */
int oracle_quantize_act(const float *x, int64_t M, int64_t K, int8_t *qs, float *scale,
                        int32_t *bsum)
{
    if (M < 0 || K <= 0 || K % 32) return -1;
    int64_t nb = K / 32;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *xb = x + m * K + 32 * b;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                float a = fabsf(xb[i]);
                if (a > amax) amax = a;
            }
            volatile float s = amax / 127.0f;
            int32_t S = 0;
            for (int i = 0; i < 32; ++i) {
                int q = 0;
                if (s != 0.0f) {
                    volatile float v = xb[i] / s;
                    float r = nearbyintf(v);
                    if (r > 127.0f) r = 127.0f;
                    if (r < -127.0f) r = -127.0f;
                    q = (int)r;
                }
                qs[m * K + 32 * b + i] = (int8_t)q;
                S += q;
            }
            scale[m * nb + b] = s;
            bsum[m * nb + b] = S;
        }
    }
    return 0;
}

/* Per-block integer dots for the listed activation rows (mrows[0..nm)) and
 * weight rows n0 <= n < n1:
 *   D[(i*(n1-n0) + (n-n0))*(K/32) + b] = sum_{k=32b}^{32b+31} W_int[n][k] q[mrows[i]][k]. */
int oracle_blockdots(int type, const uint8_t *W, int64_t N, int64_t K, const int8_t *qs,
                     int64_t M, const int64_t *mrows, int64_t nm, int64_t n0, int64_t n1,
                     int64_t *D)
{
    if (!valid_shape(type, K) || is_float_type(type) || K % 32 || n0 < 0 || n1 > N || n0 > n1)
        return -1;
    int64_t rowbytes = K / oracle_block_elems(type) * oracle_block_bytes(type);
    int64_t nb = K / 32;
    for (int64_t i = 0; i < nm; ++i)
        if (mrows[i] < 0 || mrows[i] >= M) return -1;
    int err = 0;
#pragma omp parallel
    {
        int64_t *wi = (int64_t *)malloc((size_t)K * sizeof(int64_t));
        if (!wi) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 8)
        for (int64_t n = n0; n < n1; ++n) {
            if (!wi) continue;
            oracle_int_weights_row(type, W + n * rowbytes, K, wi);
            for (int64_t i = 0; i < nm; ++i) {
                int64_t m = mrows[i];
                for (int64_t b = 0; b < nb; ++b) {
                    int64_t acc = 0;
                    for (int64_t k = 32 * b; k < 32 * b + 32; ++k) acc += wi[k] * (int64_t)qs[m * K + k];
                    D[(i * (n1 - n0) + (n - n0)) * nb + b] = acc;
                }
            }
        }
        free(wi);
    }
    return err;
}

/* Prefill MMQ reference for activation rows mrows[0..nm) and weight rows
 * n0 <= n < n1:  y = sum_k w[n][k] * (double)scale[m][k/32] * q[m][k],
 * bound = sum_k |w[n][k]| * |scale * q|.  Output index i*(n1-n0) + (n-n0). */
int oracle_mmq(int type, const uint8_t *W, int64_t N, int64_t K, const int8_t *qs,
               const float *scale, int64_t M, const int64_t *mrows, int64_t nm, int64_t n0,
               int64_t n1, double *y, double *bound)
{
    if (!valid_shape(type, K) || K % 32 || n0 < 0 || n1 > N || n0 > n1 || nm < 0) return -1;
    int64_t rowbytes = K / oracle_block_elems(type) * oracle_block_bytes(type);
    int64_t nb = K / 32;
    for (int64_t i = 0; i < nm; ++i)
        if (mrows[i] < 0 || mrows[i] >= M) return -1;
    double *xh = (double *)malloc((size_t)(nm > 0 ? nm : 1) * (size_t)K * sizeof(double));
    if (!xh) return -2;
    /* the dequantised activations x^ = scale * q, one row per listed m */
    for (int64_t i = 0; i < nm; ++i)
        for (int64_t k = 0; k < K; ++k)
            xh[i * K + k] = (double)scale[mrows[i] * nb + k / 32] * (double)qs[mrows[i] * K + k];
    int err = 0;
#pragma omp parallel
    {
        double *w = (double *)malloc((size_t)K * sizeof(double));
        if (!w) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 8)
        for (int64_t n = n0; n < n1; ++n) {
            if (!w) continue;
            oracle_dequant_row(type, W + n * rowbytes, K, w);
            for (int64_t i = 0; i < nm; ++i) {
                double acc = 0.0, bnd = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    acc += w[k] * xh[i * K + k];
                    bnd += fabs(w[k]) * fabs(xh[i * K + k]);
                }
                y[i * (n1 - n0) + (n - n0)] = acc;
                bound[i * (n1 - n0) + (n - n0)] = bnd;
            }
        }
        free(w);
    }
    free(xh);
    return err;
}
