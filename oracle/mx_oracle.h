/*
 * mx_oracle.h -- plain CPU oracle for the MXFP4 weight-gradient path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference arm of bench.py may load or call this library.
 * The product (mxfp4_precision_gb300/) never links, imports or executes it,
 * and shares no code, header or table with it.
 *
 * Sources followed (cited by page title and section):
 *   [36kr]  "Neue Studie von AMD durchbricht die bestehende Erkenntnis: Die
 *           Instabilitaet von FP4-Training liegt nicht an unzureichender
 *           Zufaelligkeit" (eu.36kr.com), sections "Was ist MXFP4?",
 *           "Fehlerdiagnoseexperiment", "Ende-zu-Ende-Effizienz".
 *   [htx]   the Indonesian rendering of the same article (htx.com), sections
 *           "Apa itu MXFP4", "Eksperimen Investigasi".
 *   [show]  "AMD颠覆认知：FP4不稳定性的真正原因" (showapi.com), section 2.2
 *           (FP4 = 1 sign, 2 exponent, 1 mantissa bit).
 *   OCP Microscaling (MX) standard, named in [36kr] "Fazit": E8M0 scale
 *           (bias 127), E2M1 element (bias 1, max 6, no Inf/NaN); its 8-bit
 *           member MXFP8 (E4M3 element, bias 7, max 448) is the block-scaled
 *           form of the FP8 baseline of [36kr] "Ende-zu-Ende-Effizienz".
 *   Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
 *           Easy as 1, 2, 3", SC'11.
 *
 * Every routine is single-threaded and written for readability, not speed.
 */
#ifndef MX_ORACLE_H
#define MX_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Philox4x32 with 10 rounds (Salmon et al. SC'11): out = philox(ctr, key). */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* Random sign d_t in {+1,-1} for absolute contraction position t: stream
 * (seed, tag 0), block t/128, bit t mod 128.
 * Reading of [36kr] "Fehlerdiagnoseexperiment" (Hadamard with random sign flip). */
int oracle_sign(uint64_t seed, int64_t t);

/* 24-bit stochastic-rounding draw for flat element index e: stream (seed, tag),
 * block e/4, word e mod 4, top 24 bits.  A stream (seed, tag) is Philox4x32-10
 * with key (seed low, seed high) and counter (block low, block high, tag low,
 * tag high). */
uint32_t oracle_sr_u24(uint64_t seed, uint64_t tag, uint64_t e);

/* Canonical fp32 Walsh-Hadamard of one block of n floats, in place:
 * butterfly stages h = 1, 2, ..., n/2 (Sylvester / natural order), each
 * (a, b) -> (a + b, a - b) rounded to fp32, then one fp32 multiply by the
 * fp32 value nearest to 1/sqrt(n). */
void oracle_fwht_f32(float *x, int n);

/* Mathematical rotation in double: y = n^(-1/2) * H_n * x with the dense
 * Sylvester matrix H_n[i][j] = (-1)^popcount(i & j). */
void oracle_hadamard_f64(const double *x, int n, double *y);

/* E8M0 shared-scale byte for a block whose largest magnitude is amax:
 * s = floor(log2 amax) - 2 clamped to [-127, 127], byte = s + 127;
 * amax == 0 -> 0x00; non-finite amax -> 0xFF. */
uint8_t oracle_scale_byte(float amax);

/* E2M1 code of v (already divided by the block scale), round to nearest,
 * ties to the even code, saturating at +-6, sign of v kept. */
uint8_t oracle_e2m1_rne(float v);

/* E2M1 code of v with stochastic rounding: round away from the lower grid
 * neighbour iff u24 < frac * 2^24, frac = (|v| - lo) / (hi - lo). */
uint8_t oracle_e2m1_sr(float v, uint32_t u24);

/* Exact value of a 4-bit E2M1 code (bit 3 = sign). */
double oracle_e2m1_value(uint8_t code);

/* Vector helpers over the scalar routines above (for exhaustive tests). */
void oracle_scale_bytes(const float *amax, int64_t n, uint8_t *out);
void oracle_e2m1_rne_vec(const float *v, int64_t n, uint8_t *out);
void oracle_e2m1_sr_vec(const float *v, const uint32_t *u24, int64_t n, uint8_t *out);

/* Rotation mode / rounding mode / contraction direction. */
enum { ORACLE_FMT_MXFP4 = 0, ORACLE_FMT_MXFP8 = 1, ORACLE_FMT_NVFP4 = 2 };
enum { ORACLE_ROT_NONE = 0, ORACLE_ROT_HADAMARD_DET = 1, ORACLE_ROT_HADAMARD_RAND = 2 };
enum { ORACLE_ROUND_RNE = 0, ORACLE_ROUND_SR = 1 };
enum { ORACLE_CONTRACT_ROWS = 0, ORACLE_CONTRACT_COLS = 1 };

/* Rotated fp32 values of one contraction line (length L) of a bf16 matrix.
 * precise == 0: canonical fp32 FWHT (the bit-exact contract);
 * precise == 1: dense double product rounded once to fp32 (diagnostic). */
int oracle_rotate_line(const uint16_t *line_bf16, int64_t stride, int64_t L, int64_t t0,
                       int rot, int rot_block, uint64_t seed, int precise, float *out);

/* E8M0 byte for a block whose largest magnitude is amax, MXFP8 rule:
 * floor(log2 amax) - 8 (E4M3's largest exponent), clamped to [-127, 127],
 * biased by 127; 0 for amax == 0; 0xFF for a non-finite amax. */
uint8_t oracle_scale_byte_e4m3(float amax);

/* Nearest E4M3 code to v (ties to the even code, |v| >= 448 saturates to
 * 448, the sign of v kept, zero included).  Value of an E4M3 code (NaN for
 * S.1111.111). */
uint8_t oracle_e4m3_rne(float v);
double oracle_e4m3_value(uint8_t code);
void oracle_scale_bytes_e4m3(const float *amax, int64_t n, uint8_t *out);
void oracle_e4m3_rne_vec(const float *v, int64_t n, uint8_t *out);

/* MXFP4-encode a bf16 matrix src[rows][cols] (row-major).
 *  contract == ROWS: blocks of 32 run down each column; line c = column c,
 *      codes[c][rows/2], scales[c][rows/32]  (transposed, contraction-major).
 *  contract == COLS: blocks run along each row; line r = row r,
 *      codes[r][cols/2], scales[r][cols/32].
 * Codes: element 2i in bits [3:0], element 2i+1 in bits [7:4].
 * Scales: canonical layout, one E8M0 byte per block.
 * SR draws use stream (seed, sr_tag) and flat index line*L + t.
 * Only the lines listed in `lines` (nlines of them) are produced when lines
 * is non-NULL; outputs are then [nlines][...] in that order.
 * Returns 0, or -1 on bad arguments. */
int oracle_quantize(const uint16_t *src, int64_t rows, int64_t cols, int contract,
                    int rot, int rot_block, int rnd, uint64_t seed, uint64_t sr_tag,
                    const int64_t *lines, int64_t nlines, int precise,
                    uint8_t *codes, uint8_t *scales);

/* MXFP8-encode a bf16 matrix: the line selection, rotation and canonical
 * scale layout of oracle_quantize, E4M3 elements rounded to nearest-even,
 * one code byte per element: codes[line][L].  Returns 0, or -1 on bad
 * arguments. */
int oracle_quantize_mxfp8(const uint16_t *src, int64_t rows, int64_t cols, int contract,
                          int rot, int rot_block, uint64_t seed, const int64_t *lines,
                          int64_t nlines, int precise, uint8_t *codes, uint8_t *scales);

/* NVFP4 (the prior-work format named in [36kr]'s introduction; NVIDIA's
 * definition): E2M1 elements in blocks of 16 along the contraction, one
 * UE4M3 scale per block and one fp32 encode scale per tensor.
 *   tensor scale  s_enc = 2688 / amax (fp32; 448 * 6, the largest block
 *                 value), FLT_MAX if that overflows, 1 if amax is 0;
 *   block scale   sf = E4M3 nearest-even of fl(fl(block_amax / 6) * s_enc);
 *   element       E2M1 nearest-even of fl(x * fl(s_enc / sf)) (the factor at
 *                 most FLT_MAX); decoded value e2m1 * sf / s_enc.
 * A block with Inf/NaN gets sf = 0x7F (NaN) and zero codes; sf = 0 gives
 * zero codes. */
float oracle_nvfp4_tensor_scale(float amax);
uint8_t oracle_nvfp4_block_scale(float block_amax, float s_enc);

/* NVFP4-encode a bf16 matrix (rotation and line selection as in
 * oracle_quantize): the tensor amax is taken over every (rotated) line, then
 * the requested lines are encoded.  codes [line][L/2] (two per byte, as
 * MXFP4), scales canonical [line][L/16]; the tensor amax and s_enc are
 * returned through the two pointers (either may be NULL). */
int oracle_quantize_nvfp4(const uint16_t *src, int64_t rows, int64_t cols, int contract,
                          int rot, int rot_block, uint64_t seed, const int64_t *lines,
                          int64_t nlines, int precise, uint8_t *codes, uint8_t *scales,
                          float *tensor_amax, float *s_enc);

/* Decode, the contraction over listed entries and over a row range, for
 * every format (fmt = ORACLE_FMT_*): codes are [mn][k/2] for MXFP4 and
 * NVFP4, [mn][k] for MXFP8; canonical scales [mn][k/32] (MX) or [mn][k/16]
 * (NVFP4).  s_enc / a_senc / b_senc: the NVFP4 tensor scales (ignored for
 * the MX formats). */
void oracle_dequantize_fmt(int fmt, const uint8_t *codes, const uint8_t *scales, int64_t mn,
                           int64_t k, double s_enc, double *out);
void oracle_gemm_entries_fmt(int fmt, const uint8_t *Aq, const uint8_t *As, double a_senc,
                             const uint8_t *Bq, const uint8_t *Bs, double b_senc, int64_t K,
                             const int64_t *ii, const int64_t *jj, int64_t n, double *C,
                             double *Cabs);
void oracle_gemm_rows_fmt(int fmt, const uint8_t *Aq, const uint8_t *As, double a_senc,
                          const uint8_t *Bq, const uint8_t *Bs, double b_senc, int64_t M,
                          int64_t N, int64_t K, int64_t m0, int64_t m1, double *C, double *Cabs);

/* Decode codes[mn][k/2] + canonical scales[mn][k/32] into double out[mn][k]. */
void oracle_dequantize(const uint8_t *codes, const uint8_t *scales, int64_t mn, int64_t k,
                       double *out);

/* C[i][j] = sum_t a[i][t] * b[j][t] over decoded operands, in double, for
 * the n requested (i, j) pairs; also Cabs = sum_t |a| |b|. */
void oracle_gemm_entries(const uint8_t *Aq, const uint8_t *As, const uint8_t *Bq,
                         const uint8_t *Bs, int64_t K, const int64_t *ii, const int64_t *jj,
                         int64_t n, double *C, double *Cabs);

/* Full C[M][N] (and Cabs) for rows [m0, m1) of A; decoded row by row. */
void oracle_gemm_rows(const uint8_t *Aq, const uint8_t *As, const uint8_t *Bq,
                      const uint8_t *Bs, int64_t M, int64_t N, int64_t K, int64_t m0,
                      int64_t m1, double *C, double *Cabs);

#ifdef __cplusplus
}
#endif
#endif
