/*
 * mx_oracle.c -- plain, slow, single-threaded CPU oracle for MXFP4 encoding
 * and the block-scaled contraction.  TEST INFRASTRUCTURE ONLY (see header).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no fast-math:
 * every fp32 operation below must round exactly once, to nearest-even).
 *
 * The method being checked (cited by page and section):
 *  - [36kr] "Was ist MXFP4?" / [htx] "Apa itu MXFP4": a tensor is cut into
 *    blocks of 32 elements; each block gets one shared E8M0 exponent equal to
 *    the block's largest exponent, and each element is an FP4 value obtained
 *    by rounding to the nearest representable 4-bit float.  The page's
 *    reconstruction formula did not survive extraction; the reading used is
 *    x_hat = 2^s * Q(x / 2^s) with s = floor(log2 amax) - 2, i.e. the block's
 *    largest exponent minus the largest E2M1 exponent (2) as in the OCP MX
 *    standard named in [36kr] "Fazit".
 *  - [show] section 2.2: FP4 is 1 sign, 2 exponent, 1 mantissa bit (E2M1).
 *  - [36kr] "Fehlerdiagnoseexperiment": the Wgrad GEMM dW = dY^T X; the
 *    deterministic Hadamard rotation (same orthogonal transform every step)
 *    and the two randomised ablations (stochastic rounding with zero-mean
 *    error; Hadamard with random sign flip) applied before quantisation.
 *  - [36kr] "Ende-zu-Ende-Effizienz" figure caption: "H16" names the
 *    Hadamard block size used for the deterministic rotation.
 */
#include "mx_oracle.h"

#include <float.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Philox4x32-10, written from the description in Salmon et al., SC'11:      */
/* each round multiplies words 0 and 2 by two odd 32-bit constants, splits   */
/* the 64-bit products into hi/lo halves, and mixes the highs with words 1,  */
/* 3 and the round key; the key is bumped by two Weyl constants between      */
/* rounds.                                                                   */
/* ------------------------------------------------------------------------ */
static const uint32_t PHILOX_MUL_A = 0xD2511F53u;
static const uint32_t PHILOX_MUL_B = 0xCD9E8D57u;
static const uint32_t PHILOX_WEYL_A = 0x9E3779B9u; /* golden ratio */
static const uint32_t PHILOX_WEYL_B = 0xBB67AE85u; /* sqrt(3) - 1  */

void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += PHILOX_WEYL_A;
            k1 += PHILOX_WEYL_B;
        }
        uint64_t pa = (uint64_t)PHILOX_MUL_A * (uint64_t)x0;
        uint64_t pb = (uint64_t)PHILOX_MUL_B * (uint64_t)x2;
        uint32_t n0 = (uint32_t)(pb >> 32) ^ x1 ^ k0;
        uint32_t n1 = (uint32_t)pb;
        uint32_t n2 = (uint32_t)(pa >> 32) ^ x3 ^ k1;
        uint32_t n3 = (uint32_t)pa;
        x0 = n0; x1 = n1; x2 = n2; x3 = n3;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* One 128-bit block of the stream (seed, tag): key = the seed's two 32-bit
 * halves (low first), counter = (n low, n high, tag low, tag high). */
static void philox_block(uint64_t seed, uint64_t tag, uint64_t n, uint32_t out[4])
{
    uint32_t ctr[4] = {(uint32_t)n, (uint32_t)(n >> 32), (uint32_t)tag, (uint32_t)(tag >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    oracle_philox4x32_10(ctr, key, out);
}

/* Sign vector: block n = t/128 of the stream (seed, 0) gives 128 bits;
 * position t uses bit (t mod 32) of word ((t mod 128) / 32).
 * Bit 1 means d_t = -1. */
int oracle_sign(uint64_t seed, int64_t t)
{
    uint32_t out[4];
    philox_block(seed, 0, (uint64_t)t / 128u, out);
    unsigned b = (unsigned)((uint64_t)t % 128u);
    return ((out[b / 32] >> (b % 32)) & 1u) ? -1 : +1;
}

/* SR draw: block n = e/4 of the stream (seed, tag) gives four 32-bit words;
 * element e uses word (e mod 4) >> 8. */
uint32_t oracle_sr_u24(uint64_t seed, uint64_t tag, uint64_t e)
{
    uint32_t out[4];
    philox_block(seed, tag, e / 4u, out);
    return out[e % 4u] >> 8;
}

/* ------------------------------------------------------------------------ */
/* Hadamard rotation ([36kr] "Fehlerdiagnoseexperiment": an orthogonal       */
/* Hadamard transform applied before quantisation; block size n, "H16").   */
/* ------------------------------------------------------------------------ */
static float inv_sqrt_n_f32(int n)
{
    /* fp32 value nearest to 1/sqrt(n): exact power of two for n = 4^k. */
    return (float)(1.0 / sqrt((double)n));
}

void oracle_fwht_f32(float *x, int n)
{
    for (int h = 1; h < n; h *= 2) {
        for (int i = 0; i < n; i += 2 * h) {
            for (int j = i; j < i + h; ++j) {
                float a = x[j];
                float b = x[j + h];
                x[j] = a + b;
                x[j + h] = a - b;
            }
        }
    }
    float c = inv_sqrt_n_f32(n);
    for (int i = 0; i < n; ++i)
        x[i] = x[i] * c;
}

static int popcount_u32(uint32_t v)
{
    int c = 0;
    while (v) {
        c += (int)(v & 1u);
        v >>= 1;
    }
    return c;
}

void oracle_hadamard_f64(const double *x, int n, double *y)
{
    double c = 1.0 / sqrt((double)n);
    for (int i = 0; i < n; ++i) {
        double acc = 0.0;
        for (int j = 0; j < n; ++j) {
            double h = (popcount_u32((uint32_t)(i & j)) & 1) ? -1.0 : 1.0;
            acc += h * x[j];
        }
        y[i] = c * acc;
    }
}

/* ------------------------------------------------------------------------ */
/* Shared scale and element rounding.                                        */
/* ------------------------------------------------------------------------ */
/* E8M0 block exponent: floor(log2 amax) minus the element format's largest
 * exponent (emax), clamped to the byte's range; 0xFF marks a non-finite block. */
static uint8_t scale_byte_emax(float amax, int emax)
{
    if (isnan(amax) || isinf(amax))
        return 0xFF;
    if (amax == 0.0f)
        return 0x00;
    int e;
    (void)frexp((double)amax, &e);    /* amax = m * 2^e, m in [0.5, 1) */
    int s = (e - 1) - emax;           /* floor(log2 amax) - emax */
    if (s < -127)
        s = -127;
    if (s > 127)
        s = 127;
    return (uint8_t)(s + 127);
}

uint8_t oracle_scale_byte(float amax)
{
    return scale_byte_emax(amax, 2);  /* E2M1: largest value 6 = 1.5 * 2^2 */
}

uint8_t oracle_scale_byte_e4m3(float amax)
{
    return scale_byte_emax(amax, 8);  /* E4M3: largest value 448 = 1.75 * 2^8 */
}

/* The eight non-negative E2M1 magnitudes, listed by code 0..7
 * (exponent bias 1; exponent field 0 is subnormal with value m * 0.5). */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

uint8_t oracle_e2m1_rne(float v)
{
    double a = fabs((double)v);
    if (a >= E2M1_MAG[7])              /* saturate: beyond the grid, 6 is nearest */
        return (uint8_t)((signbit(v) ? 8 : 0) | 7);
    int best = 0;
    double best_d = fabs(a - E2M1_MAG[0]);
    for (int c = 1; c < 8; ++c) {
        double d = fabs(a - E2M1_MAG[c]);
        /* strictly nearer wins; on an exact tie the even code wins */
        if (d < best_d || (d == best_d && (c % 2) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)((signbit(v) ? 8 : 0) | best);
}

uint8_t oracle_e2m1_sr(float v, uint32_t u24)
{
    double a = fabs((double)v);
    int code;
    if (a >= E2M1_MAG[7]) {
        code = 7;
    } else {
        int lo = 0;
        while (lo < 6 && E2M1_MAG[lo + 1] <= a)
            ++lo;
        double frac = (a - E2M1_MAG[lo]) / (E2M1_MAG[lo + 1] - E2M1_MAG[lo]);
        code = ((double)u24 < frac * 16777216.0) ? lo + 1 : lo;
    }
    return (uint8_t)((signbit(v) ? 8 : 0) | code);
}

double oracle_e2m1_value(uint8_t code)
{
    double m = E2M1_MAG[code & 7u];
    return (code & 8u) ? -m : m;
}

/* E4M3 (OCP 8-bit float, the "FP8 (E4M3)" of [show] section 2.2): sign in
 * bit 7, exponent field bits 6..3 with bias 7, mantissa bits 2..0.  Exponent
 * field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there is no infinity,
 * so the largest finite magnitude is 1.75 * 2^8 = 448. */
double oracle_e4m3_value(uint8_t code)
{
    int e = (code >> 3) & 0xF, m = code & 7;
    if (e == 15 && m == 7)
        return NAN;
    double mag = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return (code & 0x80u) ? -mag : mag;
}

uint8_t oracle_e4m3_rne(float v)
{
    double a = fabs((double)v);
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    if (a >= 448.0)                    /* saturate: beyond the grid, 448 is nearest */
        return (uint8_t)(sign | 0x7E);
    int best = 0;
    double best_d = a;
    for (int c = 1; c <= 0x7E; ++c) {  /* every non-negative finite code */
        double d = fabs(a - oracle_e4m3_value((uint8_t)c));
        /* strictly nearer wins; on an exact tie the even code wins */
        if (d < best_d || (d == best_d && (c % 2) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sign | best);
}

void oracle_scale_bytes_e4m3(const float *amax, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_scale_byte_e4m3(amax[i]);
}

void oracle_e4m3_rne_vec(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_rne(v[i]);
}

/* NVFP4 (E2M1 elements, blocks of 16, UE4M3 block scale, fp32 tensor
 * scale): the tensor's encode scale maps its largest magnitude onto the
 * largest value a block can hold, 448 (E4M3) * 6 (E2M1) = 2688. */
float oracle_nvfp4_tensor_scale(float amax)
{
    if (!(amax > 0.0f) || !isfinite(amax))
        return 1.0f;
    float s = 2688.0f / amax;          /* fp32 division, rounded to nearest */
    if (isinf(s))
        s = FLT_MAX;
    return s;
}

/* Block scale code: the block's decode scale amax/6 in the tensor's encoded
 * units, rounded to nearest-even E4M3 (saturating at 448; always >= 0). */
uint8_t oracle_nvfp4_block_scale(float block_amax, float s_enc)
{
    float t = block_amax / 6.0f;
    float u = t * s_enc;
    return oracle_e4m3_rne(u);
}

void oracle_scale_bytes(const float *amax, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_scale_byte(amax[i]);
}

void oracle_e2m1_rne_vec(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e2m1_rne(v[i]);
}

void oracle_e2m1_sr_vec(const float *v, const uint32_t *u24, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e2m1_sr(v[i], u24[i]);
}

/* ------------------------------------------------------------------------ */
/* One contraction line: rotate, then encode.                                */
/* ------------------------------------------------------------------------ */
static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static int valid_rot_block(int n)
{
    return n == 16 || n == 32 || n == 64 || n == 128 || n == 256;
}

int oracle_rotate_line(const uint16_t *line_bf16, int64_t stride, int64_t L, int64_t t0,
                       int rot, int rot_block, uint64_t seed, int precise, float *out)
{
    (void)t0;
    if (rot == ORACLE_ROT_NONE) {
        for (int64_t t = 0; t < L; ++t)
            out[t] = bf16_to_f32(line_bf16[t * stride]);
        return 0;
    }
    if (!valid_rot_block(rot_block) || L % rot_block != 0)
        return -1;
    int n = rot_block;
    float *xf = (float *)malloc(sizeof(float) * (size_t)n);
    double *xd = (double *)malloc(sizeof(double) * (size_t)n);
    double *yd = (double *)malloc(sizeof(double) * (size_t)n);
    for (int64_t b0 = 0; b0 < L; b0 += n) {
        for (int i = 0; i < n; ++i) {
            float x = bf16_to_f32(line_bf16[(b0 + i) * stride]);
            if (rot == ORACLE_ROT_HADAMARD_RAND && oracle_sign(seed, t0 + b0 + i) < 0)
                x = -x;
            xf[i] = x;
            xd[i] = (double)x;
        }
        if (precise) {
            oracle_hadamard_f64(xd, n, yd);
            for (int i = 0; i < n; ++i)
                out[b0 + i] = (float)yd[i];
        } else {
            oracle_fwht_f32(xf, n);
            for (int i = 0; i < n; ++i)
                out[b0 + i] = xf[i];
        }
    }
    free(xf);
    free(xd);
    free(yd);
    return 0;
}

static void encode_line(const float *r, int64_t L, int rnd, uint64_t seed, uint64_t sr_tag,
                        uint64_t line_index, uint8_t *codes, uint8_t *scales)
{
    for (int64_t b = 0; b < L / 32; ++b) {
        const float *blk = r + b * 32;
        float amax = 0.0f;
        int nonfinite = 0;
        for (int i = 0; i < 32; ++i) {
            float a = fabsf(blk[i]);
            if (!isfinite(a))
                nonfinite = 1;
            else if (a > amax)
                amax = a;
        }
        uint8_t sb = nonfinite ? (uint8_t)0xFF : oracle_scale_byte(amax);
        scales[b] = sb;
        uint8_t q[32];
        if (sb == 0xFF) {
            memset(q, 0, sizeof q);
        } else {
            int s = (int)sb - 127;
            float inv = ldexpf(1.0f, -s);          /* exact power of two */
            for (int i = 0; i < 32; ++i) {
                float v = blk[i] * inv;            /* fp32, exact unless subnormal */
                if (rnd == ORACLE_ROUND_SR) {
                    uint64_t e = line_index * (uint64_t)L + (uint64_t)(b * 32 + i);
                    q[i] = oracle_e2m1_sr(v, oracle_sr_u24(seed, sr_tag, e));
                } else {
                    q[i] = oracle_e2m1_rne(v);
                }
            }
        }
        for (int i = 0; i < 16; ++i)
            codes[b * 16 + i] = (uint8_t)((q[2 * i] & 0xFu) | ((q[2 * i + 1] & 0xFu) << 4));
    }
}

/* MXFP8 line: the same blocks of 32 and E8M0 exponent rule as MXFP4 with
 * E4M3's emax (8), each element rounded to nearest-even E4M3 (saturating),
 * one byte per element. */
static void encode_line_e4m3(const float *r, int64_t L, uint8_t *codes, uint8_t *scales)
{
    for (int64_t b = 0; b < L / 32; ++b) {
        const float *blk = r + b * 32;
        float amax = 0.0f;
        int nonfinite = 0;
        for (int i = 0; i < 32; ++i) {
            float a = fabsf(blk[i]);
            if (!isfinite(a))
                nonfinite = 1;
            else if (a > amax)
                amax = a;
        }
        uint8_t sb = nonfinite ? (uint8_t)0xFF : oracle_scale_byte_e4m3(amax);
        scales[b] = sb;
        if (sb == 0xFF) {
            memset(codes + b * 32, 0, 32);
            continue;
        }
        int s = (int)sb - 127;
        float inv = ldexpf(1.0f, -s);              /* exact power of two, normal */
        for (int i = 0; i < 32; ++i)
            codes[b * 32 + i] = oracle_e4m3_rne(blk[i] * inv);
    }
}

/* NVFP4 line: blocks of 16; the block scale as above; each element x becomes
 * the nearest-even E2M1 code of x * q with q = s_enc / sf (fp32, at most
 * FLT_MAX), so that x ~ e2m1 * sf / s_enc.  A block holding Inf/NaN gets the
 * E4M3 NaN code 0x7F and zero codes; a block whose scale rounds to zero gets
 * zero codes. */
static void encode_line_nvfp4(const float *r, int64_t L, float s_enc, uint8_t *codes,
                              uint8_t *scales)
{
    for (int64_t b = 0; b < L / 16; ++b) {
        const float *blk = r + b * 16;
        float amax = 0.0f;
        int nonfinite = 0;
        for (int i = 0; i < 16; ++i) {
            float a = fabsf(blk[i]);
            if (!isfinite(a))
                nonfinite = 1;
            else if (a > amax)
                amax = a;
        }
        uint8_t q[16];
        memset(q, 0, sizeof q);
        uint8_t sf = nonfinite ? (uint8_t)0x7F : oracle_nvfp4_block_scale(amax, s_enc);
        scales[b] = sf;
        if (!nonfinite && sf != 0) {
            float m = s_enc / (float)oracle_e4m3_value(sf);
            if (isinf(m))
                m = FLT_MAX;
            for (int i = 0; i < 16; ++i)
                q[i] = oracle_e2m1_rne(blk[i] * m);
        }
        for (int i = 0; i < 8; ++i)
            codes[b * 8 + i] = (uint8_t)((q[2 * i] & 0xFu) | ((q[2 * i + 1] & 0xFu) << 4));
    }
}

static int quantize_impl(int fmt, const uint16_t *src, int64_t rows, int64_t cols,
                         int contract, int rot, int rot_block, int rnd, uint64_t seed,
                         uint64_t sr_tag, const int64_t *lines, int64_t nlines, int precise,
                         uint8_t *codes, uint8_t *scales);
static int quantize_core(int fmt, const uint16_t *src, int64_t rows, int64_t cols,
                         int contract, int rot, int rot_block, int rnd, uint64_t seed,
                         uint64_t sr_tag, const int64_t *lines, int64_t nlines, int precise,
                         float s_enc, uint8_t *codes, uint8_t *scales, float *amax_out);

int oracle_quantize_nvfp4(const uint16_t *src, int64_t rows, int64_t cols, int contract,
                          int rot, int rot_block, uint64_t seed, const int64_t *lines,
                          int64_t nlines, int precise, uint8_t *codes, uint8_t *scales,
                          float *tensor_amax, float *s_enc)
{
    /* Pass 1: the largest finite magnitude of the (rotated) tensor, over
     * every line; pass 2: the requested lines, encoded with its scale. */
    float amax = 0.0f;
    int rc = quantize_core(ORACLE_FMT_NVFP4, src, rows, cols, contract, rot, rot_block,
                           ORACLE_ROUND_RNE, seed, 0, NULL, 0, precise, 1.0f, NULL, NULL, &amax);
    if (rc != 0)
        return rc;
    float se = oracle_nvfp4_tensor_scale(amax);
    if (tensor_amax)
        *tensor_amax = amax;
    if (s_enc)
        *s_enc = se;
    return quantize_core(ORACLE_FMT_NVFP4, src, rows, cols, contract, rot, rot_block,
                         ORACLE_ROUND_RNE, seed, 0, lines, nlines, precise, se, codes, scales,
                         NULL);
}

int oracle_quantize(const uint16_t *src, int64_t rows, int64_t cols, int contract,
                    int rot, int rot_block, int rnd, uint64_t seed, uint64_t sr_tag,
                    const int64_t *lines, int64_t nlines, int precise,
                    uint8_t *codes, uint8_t *scales)
{
    return quantize_impl(ORACLE_FMT_MXFP4, src, rows, cols, contract, rot, rot_block, rnd,
                         seed, sr_tag, lines, nlines, precise, codes, scales);
}

int oracle_quantize_mxfp8(const uint16_t *src, int64_t rows, int64_t cols, int contract,
                          int rot, int rot_block, uint64_t seed, const int64_t *lines,
                          int64_t nlines, int precise, uint8_t *codes, uint8_t *scales)
{
    return quantize_impl(ORACLE_FMT_MXFP8, src, rows, cols, contract, rot, rot_block,
                         ORACLE_ROUND_RNE, seed, 0, lines, nlines, precise, codes, scales);
}

static int quantize_impl(int fmt, const uint16_t *src, int64_t rows, int64_t cols,
                         int contract, int rot, int rot_block, int rnd, uint64_t seed,
                         uint64_t sr_tag, const int64_t *lines, int64_t nlines, int precise,
                         uint8_t *codes, uint8_t *scales)
{
    if (!codes || !scales)
        return -1;
    return quantize_core(fmt, src, rows, cols, contract, rot, rot_block, rnd, seed, sr_tag,
                         lines, nlines, precise, 1.0f, codes, scales, NULL);
}

/* Rotates every requested line and encodes it in format fmt; with amax_out
 * set (and no outputs) it only records the largest finite magnitude of the
 * rotated lines. */
static int quantize_core(int fmt, const uint16_t *src, int64_t rows, int64_t cols,
                         int contract, int rot, int rot_block, int rnd, uint64_t seed,
                         uint64_t sr_tag, const int64_t *lines, int64_t nlines, int precise,
                         float s_enc, uint8_t *codes, uint8_t *scales, float *amax_out)
{
    if (!src || rows <= 0 || cols <= 0)
        return -1;
    if (!amax_out && (!codes || !scales))
        return -1;
    if (contract != ORACLE_CONTRACT_ROWS && contract != ORACLE_CONTRACT_COLS)
        return -1;
    if (rot < ORACLE_ROT_NONE || rot > ORACLE_ROT_HADAMARD_RAND)
        return -1;
    if (rnd != ORACLE_ROUND_RNE && rnd != ORACLE_ROUND_SR)
        return -1;
    int64_t L = (contract == ORACLE_CONTRACT_ROWS) ? rows : cols;
    int64_t nl = (contract == ORACLE_CONTRACT_ROWS) ? cols : rows;
    if (L % 32 != 0)
        return -1;
    if (rot != ORACLE_ROT_NONE && (!valid_rot_block(rot_block) || L % rot_block != 0))
        return -1;
    int64_t count = lines ? nlines : nl;
    float *r = (float *)malloc(sizeof(float) * (size_t)L);
    for (int64_t k = 0; k < count; ++k) {
        int64_t line = lines ? lines[k] : k;
        if (line < 0 || line >= nl) {
            free(r);
            return -1;
        }
        const uint16_t *base;
        int64_t stride;
        if (contract == ORACLE_CONTRACT_ROWS) {
            base = src + line;
            stride = cols;
        } else {
            base = src + line * cols;
            stride = 1;
        }
        if (oracle_rotate_line(base, stride, L, 0, rot, rot_block, seed, precise, r) != 0) {
            free(r);
            return -1;
        }
        if (amax_out) {
            for (int64_t t = 0; t < L; ++t)
                if (isfinite(r[t]) && fabsf(r[t]) > *amax_out)
                    *amax_out = fabsf(r[t]);
        } else if (fmt == ORACLE_FMT_NVFP4)
            encode_line_nvfp4(r, L, s_enc, codes + k * (L / 2), scales + k * (L / 16));
        else if (fmt == ORACLE_FMT_MXFP8)
            encode_line_e4m3(r, L, codes + k * L, scales + k * (L / 32));
        else
            encode_line(r, L, rnd, seed, sr_tag, (uint64_t)line, codes + k * (L / 2),
                        scales + k * (L / 32));
    }
    free(r);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Decoding and the contraction ([36kr] "Fehlerdiagnoseexperiment": Fprop    */
/* Y = X W^T, Dgrad dX = dY W, Wgrad dW = dY^T X; all three are C = A B^T     */
/* over operands encoded along the contraction dimension).                   */
/* ------------------------------------------------------------------------ */
/* Bytes of codes per encoded line of k elements. */
static int64_t code_row_bytes(int fmt, int64_t k)
{
    return fmt == ORACLE_FMT_MXFP8 ? k : k / 2;
}

static double decode(int fmt, const uint8_t *codes, const uint8_t *scales, int64_t row,
                     int64_t k, int64_t t, double s_enc)
{
    if (fmt == ORACLE_FMT_NVFP4) {
        uint8_t sf = scales[row * (k / 16) + t / 16];
        uint8_t byte = codes[row * (k / 2) + t / 2];
        uint8_t code = (t % 2 == 0) ? (uint8_t)(byte & 0xFu) : (uint8_t)(byte >> 4);
        return oracle_e2m1_value(code) * oracle_e4m3_value(sf) / s_enc;
    }
    uint8_t sb = scales[row * (k / 32) + t / 32];
    if (sb == 0xFF)
        return NAN;
    double v;
    if (fmt == ORACLE_FMT_MXFP8) {
        v = oracle_e4m3_value(codes[row * k + t]);
    } else {
        uint8_t byte = codes[row * (k / 2) + t / 2];
        uint8_t code = (t % 2 == 0) ? (uint8_t)(byte & 0xFu) : (uint8_t)(byte >> 4);
        v = oracle_e2m1_value(code);
    }
    return ldexp(v, (int)sb - 127);
}

void oracle_dequantize_fmt(int fmt, const uint8_t *codes, const uint8_t *scales, int64_t mn,
                           int64_t k, double s_enc, double *out)
{
    for (int64_t i = 0; i < mn; ++i)
        for (int64_t t = 0; t < k; ++t)
            out[i * k + t] = decode(fmt, codes, scales, i, k, t, s_enc);
}

void oracle_dequantize(const uint8_t *codes, const uint8_t *scales, int64_t mn, int64_t k,
                       double *out)
{
    oracle_dequantize_fmt(ORACLE_FMT_MXFP4, codes, scales, mn, k, 1.0, out);
}

void oracle_gemm_entries_fmt(int fmt, const uint8_t *Aq, const uint8_t *As, double a_senc,
                             const uint8_t *Bq, const uint8_t *Bs, double b_senc, int64_t K,
                             const int64_t *ii, const int64_t *jj, int64_t n, double *C,
                             double *Cabs)
{
    for (int64_t p = 0; p < n; ++p) {
        double acc = 0.0, acc_abs = 0.0;
        for (int64_t t = 0; t < K; ++t) {
            double a = decode(fmt, Aq, As, ii[p], K, t, a_senc);
            double b = decode(fmt, Bq, Bs, jj[p], K, t, b_senc);
            acc += a * b;
            acc_abs += fabs(a) * fabs(b);
        }
        C[p] = acc;
        Cabs[p] = acc_abs;
    }
}

void oracle_gemm_entries(const uint8_t *Aq, const uint8_t *As, const uint8_t *Bq,
                         const uint8_t *Bs, int64_t K, const int64_t *ii, const int64_t *jj,
                         int64_t n, double *C, double *Cabs)
{
    oracle_gemm_entries_fmt(ORACLE_FMT_MXFP4, Aq, As, 1.0, Bq, Bs, 1.0, K, ii, jj, n, C, Cabs);
}

void oracle_gemm_rows_fmt(int fmt, const uint8_t *Aq, const uint8_t *As, double a_senc,
                          const uint8_t *Bq, const uint8_t *Bs, double b_senc, int64_t M,
                          int64_t N, int64_t K, int64_t m0, int64_t m1, double *C, double *Cabs)
{
    (void)M;
    double *a = (double *)malloc(sizeof(double) * (size_t)K);
    double *b = (double *)malloc(sizeof(double) * (size_t)N * (size_t)K);
    const int64_t block = fmt == ORACLE_FMT_NVFP4 ? 16 : 32;
    oracle_dequantize_fmt(fmt, Bq, Bs, N, K, b_senc, b);
    for (int64_t i = m0; i < m1; ++i) {
        oracle_dequantize_fmt(fmt, Aq + i * code_row_bytes(fmt, K), As + i * (K / block), 1, K,
                              a_senc, a);
        for (int64_t j = 0; j < N; ++j) {
            const double *bj = b + j * K;
            double acc = 0.0, acc_abs = 0.0;
            for (int64_t t = 0; t < K; ++t) {
                acc += a[t] * bj[t];
                acc_abs += fabs(a[t]) * fabs(bj[t]);
            }
            C[(i - m0) * N + j] = acc;
            Cabs[(i - m0) * N + j] = acc_abs;
        }
    }
    free(a);
    free(b);
}

void oracle_gemm_rows(const uint8_t *Aq, const uint8_t *As, const uint8_t *Bq,
                      const uint8_t *Bs, int64_t M, int64_t N, int64_t K, int64_t m0,
                      int64_t m1, double *C, double *Cabs)
{
    oracle_gemm_rows_fmt(ORACLE_FMT_MXFP4, Aq, As, 1.0, Bq, Bs, 1.0, M, N, K, m0, m1, C, Cabs);
}
