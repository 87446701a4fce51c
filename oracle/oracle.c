/*
 * oracle.c -- the plain, slow, obviously correct CPU definition of what the
 * block-quantized weight path computes.  TEST INFRASTRUCTURE ONLY: it is
 * loaded by tests/, by the smoke check and by the CPU baseline leg of the
 * benchmark; the product library never links, loads or calls it, and it
 * shares no code, header, table or constant with the CUDA sources.
 *
 * Compile with -O2 -ffp-contract=off -fno-fast-math (no FMA contraction, no
 * reassociation): every float operation below is the IEEE operation it reads
 * as.  OpenMP, when enabled, only splits independent rows between threads;
 * each output element is computed by the same sequence of operations for any
 * thread count.
 *
 * Sources (page titles and sections):
 *  - "llama_cpp 0.12.1 -> 0.12.2" (my.diffend.io diff of the vendored
 *    ggml-cuda.cu): the hunks adding dequantize_block_q4_0,
 *    dequantize_block_q4_1 and dequantize_block_q8_0_f16, and the
 *    ggml_get_to_fp16_cuda / ggml_get_to_fp32_cuda dispatch hunk.
 *  - The block formats as the method statement spells them out: Q4_0 is an
 *    fp16 scale d followed by 16 nibble bytes, w = d*(q-8), low nibbles give
 *    elements 0-15 and high nibbles elements 16-31; Q4_1 is fp16 d and m then
 *    16 nibble bytes, w = d*q + m; Q8_0 is fp16 d then 32 int8, w = d*q.
 *
 * Readings taken where the pages leave a step open (all restated in the
 * design notes):
 *  - Q4_0: the kernel writes d*q + (-8*d); the format statement writes
 *    d*(q-8).  Both are the exact real number d*(q-8) here, because an fp16
 *    d (11 significant bits) times an integer of magnitude <= 16 is exact in
 *    fp32, so the oracle evaluates d*(q-8) directly.
 *  - Q4_1: the product d*q is rounded to fp32, then the sum with m is
 *    rounded to fp32 (two IEEE operations, no fused multiply-add).
 *  - f16 outputs: the fp32 value is computed first, then rounded to fp16
 *    with round-to-nearest-even (the kernels' implicit dst_t conversion).
 *  - GEMV / GEMM: the result is the plain dot product, accumulated in
 *    double in increasing k and rounded once to fp32.
 *  - Block byte layout: Q4_0 = [d:2][qs:16] (18 B), Q4_1 = [d:2][m:2][qs:16]
 *    (20 B, the half2 dm pair), Q8_0 = [d:2][qs:32] (34 B), little-endian
 *    fp16; a row of ncols weights is ncols/32 consecutive blocks and rows
 *    are consecutive.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_FMT_Q4_0 0
#define ORACLE_FMT_Q4_1 1
#define ORACLE_FMT_Q8_0 2

/* ---------------------------------------------------------------- fp16 */

/* IEEE-754 binary16 -> binary32, bit by bit: sign, 5-bit exponent (bias
 * 15), 10-bit fraction.  Exponent 0 is zero/subnormal (fraction * 2^-24),
 * exponent 31 is infinity (fraction 0) or NaN. */
float oracle_fp16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);
    } else if (expo == 31) {
        if (frac == 0) {
            v = INFINITY;
        } else {
            /* keep the payload: a quiet NaN with the fraction in the top bits */
            uint32_t bits = ((uint32_t)sign << 31) | 0x7f800000u | 0x00400000u |
                            ((uint32_t)frac << 13);
            float f;
            memcpy(&f, &bits, 4);
            return f;
        }
    } else {
        v = ldexp((double)(1024 + frac), expo - 25);
    }
    return (float)(sign ? -v : v);
}

/* binary32 -> binary16, round to nearest, ties to even.  Overflow goes to
 * infinity, results below 2^-14 become subnormal (or zero), NaN stays NaN
 * (quiet, sign kept, top fraction bits kept). */
uint16_t oracle_f32_to_fp16(float f)
{
    uint32_t x;
    memcpy(&x, &f, 4);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t ax = x & 0x7fffffffu;

    if (ax > 0x7f800000u) {                       /* NaN */
        return (uint16_t)(sign | 0x7e00u | ((ax >> 13) & 0x3ffu));
    }
    if (ax == 0x7f800000u) {                      /* infinity */
        return (uint16_t)(sign | 0x7c00u);
    }
    /* Half-way point between the largest fp16 (65504) and the next power of
     * two (65536, not representable): 65520 = 0x477ff000.  At and above it,
     * round-to-nearest-even gives infinity. */
    if (ax >= 0x477ff000u) {
        return (uint16_t)(sign | 0x7c00u);
    }
    if (ax < 0x38800000u) {                       /* |f| < 2^-14: subnormal range */
        float af;
        memcpy(&af, &ax, 4);
        double v = (double)af * 16777216.0;       /* units of 2^-24, exact */
        double fl = floor(v);
        double rem = v - fl;
        if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) == 1.0)) {
            fl += 1.0;
        }
        /* fl <= 1024; 1024 is the smallest normal, whose bit pattern is 0x400 */
        return (uint16_t)(sign | (uint16_t)fl);
    }
    /* normal range: rebias the exponent, keep 10 fraction bits, round the
     * 13 dropped bits to nearest even (a carry may bump the exponent) */
    uint32_t e = (ax >> 23) - 127 + 15;
    uint32_t m = ax & 0x7fffffu;
    uint32_t h = (e << 10) | (m >> 13);
    uint32_t dropped = m & 0x1fffu;
    if (dropped > 0x1000u || (dropped == 0x1000u && (h & 1u))) {
        h += 1u;
    }
    return (uint16_t)(sign | h);
}

/* bfloat16 -> binary32: bfloat16 is the top half of a binary32. */
float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, 4);
    return f;
}

static uint16_t load_u16le(const uint8_t *p)
{
    return (uint16_t)(p[0] | (p[1] << 8));
}

/* ------------------------------------------------------ block decoding */

int oracle_block_bytes(int fmt)
{
    switch (fmt) {
    case ORACLE_FMT_Q4_0: return 18;
    case ORACLE_FMT_Q4_1: return 20;
    case ORACLE_FMT_Q8_0: return 34;
    default: return -1;
    }
}

/* Dequantize one 32-weight block to fp32.
 * Q4_0: element j (<16) is the low nibble of qs[j], element j+16 its high
 *       nibble; w = d * (q - 8).
 * Q4_1: same nibble order; w = d*q + m, two roundings.
 * Q8_0: element j is the signed byte qs[j]; w = d * q. */
static void dequant_block(int fmt, const uint8_t *blk, float w[32])
{
    if (fmt == ORACLE_FMT_Q4_0) {
        float d = oracle_fp16_to_f32(load_u16le(blk));
        const uint8_t *qs = blk + 2;
        for (int j = 0; j < 16; ++j) {
            int lo = qs[j] & 0x0f;
            int hi = qs[j] >> 4;
            w[j]      = d * (float)(lo - 8);
            w[j + 16] = d * (float)(hi - 8);
        }
    } else if (fmt == ORACLE_FMT_Q4_1) {
        float d = oracle_fp16_to_f32(load_u16le(blk));
        float m = oracle_fp16_to_f32(load_u16le(blk + 2));
        const uint8_t *qs = blk + 4;
        for (int j = 0; j < 16; ++j) {
            int lo = qs[j] & 0x0f;
            int hi = qs[j] >> 4;
            float plo = d * (float)lo;
            float phi = d * (float)hi;
            w[j]      = plo + m;
            w[j + 16] = phi + m;
        }
    } else {
        float d = oracle_fp16_to_f32(load_u16le(blk));
        const uint8_t *qs = blk + 2;
        for (int j = 0; j < 32; ++j) {
            int q = (int)(int8_t)qs[j];
            w[j] = d * (float)q;
        }
    }
}

/* Dequantize row r (ncols weights, ncols % 32 == 0) into w[ncols]. */
static void dequant_row(int fmt, const uint8_t *W, int64_t ncols, int64_t r, float *w)
{
    int bb = oracle_block_bytes(fmt);
    int64_t nb = ncols / 32;
    const uint8_t *row = W + r * nb * bb;
    for (int64_t b = 0; b < nb; ++b) {
        dequant_block(fmt, row + b * bb, w + b * 32);
    }
}

static int check_args(int fmt, int64_t nrows, int64_t ncols)
{
    if (oracle_block_bytes(fmt) < 0) return -1;
    if (nrows < 0 || ncols < 0 || ncols % 32 != 0) return -1;
    return 0;
}

/* ------------------------------------------------------------- threads */

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ----------------------------------------------------------- dequantize */

/* out is [nrows][ncols] row-major; out_f16 == 0 writes fp32, otherwise fp16
 * bit patterns (round-to-nearest-even of the fp32 value). */
int oracle_dequant(int fmt, const uint8_t *W, int64_t nrows, int64_t ncols,
                   int out_f16, void *out)
{
    if (check_args(fmt, nrows, ncols)) return -1;
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < nrows; ++r) {
        float *w = (float *)malloc(sizeof(float) * (size_t)(ncols > 0 ? ncols : 1));
        dequant_row(fmt, W, ncols, r, w);
        if (out_f16) {
            uint16_t *o = (uint16_t *)out + r * ncols;
            for (int64_t k = 0; k < ncols; ++k) o[k] = oracle_f32_to_fp16(w[k]);
        } else {
            float *o = (float *)out + r * ncols;
            for (int64_t k = 0; k < ncols; ++k) o[k] = w[k];
        }
        free(w);
    }
    return 0;
}

/* ----------------------------------------------------------------- GEMV */

/* y[b][r] = fp32( sum_k double(w[r][k]) * double(x[b][k]) ), k increasing.
 * x is [batch][ncols], y is [batch][nrows].  If absdot is not NULL it
 * receives sum_k |w[r][k] * x[b][k]| (double), the scale of the error bound. */
int oracle_gemv(int fmt, const uint8_t *W, const float *x, float *y,
                int64_t nrows, int64_t ncols, int64_t batch, double *absdot)
{
    if (check_args(fmt, nrows, ncols) || batch < 0) return -1;
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < nrows; ++r) {
        float *w = (float *)malloc(sizeof(float) * (size_t)(ncols > 0 ? ncols : 1));
        dequant_row(fmt, W, ncols, r, w);
        for (int64_t b = 0; b < batch; ++b) {
            const float *xb = x + b * ncols;
            double acc = 0.0, aacc = 0.0;
            for (int64_t k = 0; k < ncols; ++k) {
                double p = (double)w[k] * (double)xb[k];
                acc += p;
                aacc += fabs(p);
            }
            y[b * nrows + r] = (float)acc;
            if (absdot) absdot[b * nrows + r] = aacc;
        }
        free(w);
    }
    return 0;
}

/* The same definition on a chosen subset of rows: for i < nsel,
 * ysel[b*nsel + i] = y[b][rows[i]] (and absdot likewise). */
int oracle_gemv_rows(int fmt, const uint8_t *W, const float *x,
                     int64_t nrows, int64_t ncols, int64_t batch,
                     const int64_t *rows, int64_t nsel, float *ysel, double *absdot)
{
    if (check_args(fmt, nrows, ncols) || batch < 0 || nsel < 0) return -1;
    for (int64_t i = 0; i < nsel; ++i) {
        if (rows[i] < 0 || rows[i] >= nrows) return -1;
    }
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < nsel; ++i) {
        float *w = (float *)malloc(sizeof(float) * (size_t)(ncols > 0 ? ncols : 1));
        dequant_row(fmt, W, ncols, rows[i], w);
        for (int64_t b = 0; b < batch; ++b) {
            const float *xb = x + b * ncols;
            double acc = 0.0, aacc = 0.0;
            for (int64_t k = 0; k < ncols; ++k) {
                double p = (double)w[k] * (double)xb[k];
                acc += p;
                aacc += fabs(p);
            }
            ysel[b * nsel + i] = (float)acc;
            if (absdot) absdot[b * nsel + i] = aacc;
        }
        free(w);
    }
    return 0;
}

/* ----------------------------------------------------------------- GEMM */

/* Prefill matmul: Y[m][n] = fp32( sum_k double(w[n][k]) * double(bf16(X[m][k])) ).
 * X is [mrows][ncols] bfloat16 bit patterns, Y is [mrows][nrows] fp32. */
int oracle_gemm(int fmt, const uint8_t *W, const uint16_t *X, float *Y,
                int64_t nrows, int64_t ncols, int64_t mrows, double *absdot)
{
    if (check_args(fmt, nrows, ncols) || mrows < 0) return -1;
    int64_t n;
#pragma omp parallel for schedule(static)
    for (n = 0; n < nrows; ++n) {
        float *w = (float *)malloc(sizeof(float) * (size_t)(ncols > 0 ? ncols : 1));
        dequant_row(fmt, W, ncols, n, w);
        for (int64_t m = 0; m < mrows; ++m) {
            const uint16_t *xm = X + m * ncols;
            double acc = 0.0, aacc = 0.0;
            for (int64_t k = 0; k < ncols; ++k) {
                double p = (double)w[k] * (double)oracle_bf16_to_f32(xm[k]);
                acc += p;
                aacc += fabs(p);
            }
            Y[m * nrows + n] = (float)acc;
            if (absdot) absdot[m * nrows + n] = aacc;
        }
        free(w);
    }
    return 0;
}

/* The same definition on chosen (m, n) entries: out[i] = Y[mi[i]][ni[i]]. */
int oracle_gemm_entries(int fmt, const uint8_t *W, const uint16_t *X,
                        int64_t nrows, int64_t ncols, int64_t mrows,
                        const int64_t *mi, const int64_t *ni, int64_t cnt,
                        float *out, double *absdot)
{
    if (check_args(fmt, nrows, ncols) || mrows < 0 || cnt < 0) return -1;
    for (int64_t i = 0; i < cnt; ++i) {
        if (mi[i] < 0 || mi[i] >= mrows || ni[i] < 0 || ni[i] >= nrows) return -1;
    }
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < cnt; ++i) {
        float *w = (float *)malloc(sizeof(float) * (size_t)(ncols > 0 ? ncols : 1));
        dequant_row(fmt, W, ncols, ni[i], w);
        const uint16_t *xm = X + mi[i] * ncols;
        double acc = 0.0, aacc = 0.0;
        for (int64_t k = 0; k < ncols; ++k) {
            double p = (double)w[k] * (double)oracle_bf16_to_f32(xm[k]);
            acc += p;
            aacc += fabs(p);
        }
        out[i] = (float)acc;
        if (absdot) absdot[i] = aacc;
        free(w);
    }
    return 0;
}

/* ----------------------------------------------- expert-selected GEMV */

/* The pages name the expert-selecting matrix product (ggml_cuda_mul_mat_id,
 * GGML_OP_MUL_MAT_ID, and the ffn_(up|gate|down)_exps weight names of the
 * tensor-parallel split rules) without printing what it computes.  Reading:
 * W holds n_expert matrices of nrows x ncols one after the other (each in
 * the row layout above); output column b uses expert ids[b] and activation
 * row b / x_group (x_group = experts per token when a token's experts share
 * its activations, as in the up and gate projections; 1 when each column
 * has its own, as in the down projection):
 *   y[b][r] = fp32( sum_k double(w_{ids[b]}[r][k]) * double(x[b / x_group][k]) ),
 * the GEMV definition above on the selected matrix.  An id outside
 * [0, n_expert), or batch not a multiple of x_group, is an error (-1). */
int oracle_gemv_id(int fmt, const uint8_t *W, int64_t n_expert, const int32_t *ids, const float *x,
                   int64_t x_group, float *y, int64_t nrows, int64_t ncols, int64_t batch, double *absdot)
{
    if (check_args(fmt, nrows, ncols) || batch < 0 || n_expert < 1 || x_group < 1 || batch % x_group)
        return -1;
    for (int64_t b = 0; b < batch; ++b) {
        if (ids[b] < 0 || ids[b] >= n_expert) return -1;
    }
    const int64_t ebytes = nrows * (ncols / 32) * oracle_block_bytes(fmt);
    for (int64_t b = 0; b < batch; ++b) {
        const uint8_t *We = W + ids[b] * ebytes;
        int64_t r;
#pragma omp parallel for schedule(static)
        for (r = 0; r < nrows; ++r) {
            float *w = (float *)malloc(sizeof(float) * (size_t)(ncols > 0 ? ncols : 1));
            dequant_row(fmt, We, ncols, r, w);
            const float *xb = x + (b / x_group) * ncols;
            double acc = 0.0, aacc = 0.0;
            for (int64_t k = 0; k < ncols; ++k) {
                double pr = (double)w[k] * (double)xb[k];
                acc += pr;
                aacc += fabs(pr);
            }
            y[b * nrows + r] = (float)acc;
            if (absdot) absdot[b * nrows + r] = aacc;
            free(w);
        }
    }
    return 0;
}

/* ------------------------------------------- quantized activations (q8_1) */

/* The pages name the second GEMV family, mul_mat_vec_q, whose activations are
 * first converted to int8 blocks ("convert_src1_to_q8_1" in
 * ggml_cuda_op_mul_mat, and the ggml_cuda_op_mul_mat_vec_q signature on the
 * "llama_cpp 0.12.1 -> 0.12.2" page) and contracted with byte-wise integer
 * dot products (the __dp4a note beside MIN_CC_DP4A).  The pages print
 * neither the block layout nor the quantizer, so both are a reading:
 *  - x is cut into blocks of 32 consecutive values of one batch column;
 *  - amax = max |x_i| over the block, d = amax / 127 (one fp32 division);
 *  - q_i = x_i / d (fp32 division) rounded to the nearest integer, ties to
 *    even, then clamped to [-127, 127]; q_i = 0 when d == 0;
 *  - a block that holds a NaN or an infinity gets d = NaN and q_i = 0;
 *  - s = sum_i q_i, an exact integer.
 * q is [batch][ncols] int8, d and s are [batch][ncols/32]. */
static int round_half_even(float t)
{
    double f = floor((double)t);
    double frac = (double)t - f;
    if (frac > 0.5 || (frac == 0.5 && fmod(f, 2.0) != 0.0)) f += 1.0;
    return (int)f;
}

int oracle_quantize_q8_1(const float *x, int64_t ncols, int64_t batch,
                         int8_t *q, float *d, int32_t *s)
{
    if (ncols < 0 || ncols % 32 != 0 || batch < 0) return -1;
    int64_t nb = ncols / 32;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t j = 0; j < nb; ++j) {
            const float *xb = x + b * ncols + j * 32;
            int8_t *qb = q + b * ncols + j * 32;
            float amax = 0.0f;
            int finite = 1;
            for (int i = 0; i < 32; ++i) {
                float a = fabsf(xb[i]);
                if (!isfinite(a)) finite = 0;
                else if (a > amax) amax = a;
            }
            float dd = finite ? amax / 127.0f : NAN;
            int32_t sum = 0;
            for (int i = 0; i < 32; ++i) {
                int v = 0;
                if (finite && dd != 0.0f) {
                    v = round_half_even(xb[i] / dd);
                    if (v > 127) v = 127;
                    if (v < -127) v = -127;
                }
                qb[i] = (int8_t)v;
                sum += v;
            }
            d[b * nb + j] = dd;
            s[b * nb + j] = sum;
        }
    }
    return 0;
}

/* The GEMV over quantized activations: with xhat[b][k] = d[b][k/32] * q[b][k]
 * (exact in double),
 *   y[b][r] = fp32( sum_k double(w[r][k]) * xhat[b][k] ), k increasing,
 * the same plain dot product as oracle_gemv with x replaced by its q8_1
 * reconstruction.  absdot receives sum_k |w[r][k] * xhat[b][k]|. */
int oracle_gemv_q8_1(int fmt, const uint8_t *W, const int8_t *q, const float *d,
                     float *y, int64_t nrows, int64_t ncols, int64_t batch,
                     double *absdot)
{
    if (check_args(fmt, nrows, ncols) || batch < 0) return -1;
    int64_t nb = ncols / 32;
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < nrows; ++r) {
        float *w = (float *)malloc(sizeof(float) * (size_t)(ncols > 0 ? ncols : 1));
        dequant_row(fmt, W, ncols, r, w);
        for (int64_t b = 0; b < batch; ++b) {
            double acc = 0.0, aacc = 0.0;
            for (int64_t k = 0; k < ncols; ++k) {
                double xhat = (double)d[b * nb + k / 32] * (double)q[b * ncols + k];
                double p = (double)w[k] * xhat;
                acc += p;
                aacc += fabs(p);
            }
            y[b * nrows + r] = (float)acc;
            if (absdot) absdot[b * nrows + r] = aacc;
        }
        free(w);
    }
    return 0;
}

/* ------------------------------------------------ array forms (for tests) */

void oracle_fp16_to_f32_array(const uint16_t *h, float *f, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) f[i] = oracle_fp16_to_f32(h[i]);
}

void oracle_f32_to_fp16_array(const float *f, uint16_t *h, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) h[i] = oracle_f32_to_fp16(f[i]);
}

void oracle_bf16_to_f32_array(const uint16_t *b, float *f, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) f[i] = oracle_bf16_to_f32(b[i]);
}
