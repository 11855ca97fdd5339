// mx_encode.cuh -- device building blocks of the MXFP4 encoders: Philox4x32-10
// draws, Hadamard butterflies, block amax and shared exponent, E2M1 rounding
// and packing, and the tiled scale layout.  Shared by the stand-alone
// encoders (mx_quant.cu) and the encoder warps of the fused Wgrad GEMM
// (mx_gemm.cu), so that both produce the same bits.
//
// What is computed ("Neue Studie von AMD durchbricht die bestehende
// Erkenntnis", eu.36kr.com, sections "Was ist MXFP4?" and
// "Fehlerdiagnoseexperiment"): along the contraction dimension, an optional
// block Hadamard rotation (deterministic, or after a random sign flip), then
// blocks of 32 elements share one E8M0 exponent (the block's largest exponent
// minus 2, the largest E2M1 exponent) and each element is rounded to E2M1
// (nearest-even, or stochastically) and packed two per byte.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mx {
namespace enc {

// ---------------------------------------------------------------- Philox4x32-10
// Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11).  Each
// round is two 32 x 32 -> 64-bit products (one wide multiply each).
__device__ __forceinline__ void philox4x32_10(uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3,
                                              uint32_t k0, uint32_t k1, uint32_t (&o)[4]) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint64_t pa = static_cast<uint64_t>(0xD2511F53u) * x0;
        const uint64_t pb = static_cast<uint64_t>(0xCD9E8D57u) * x2;
        const uint32_t n0 = static_cast<uint32_t>(pb >> 32) ^ x1 ^ k0;
        const uint32_t n2 = static_cast<uint32_t>(pa >> 32) ^ x3 ^ k1;
        x0 = n0;
        x1 = static_cast<uint32_t>(pb);
        x2 = n2;
        x3 = static_cast<uint32_t>(pa);
    }
    o[0] = x0;
    o[1] = x1;
    o[2] = x2;
    o[3] = x3;
}

// Block n of the random stream (seed, tag): key = the seed's 32-bit halves
// (low first), counter = (n low, n high, tag low, tag high).  The random
// signs are stream (seed, 0), the SR draws of operand A (seed, 1) and of B
// (seed, 2).
__device__ __forceinline__ void philox_block(uint64_t seed, uint64_t tag, uint64_t n,
                                             uint32_t (&o)[4]) {
    philox4x32_10(static_cast<uint32_t>(n), static_cast<uint32_t>(n >> 32),
                  static_cast<uint32_t>(tag), static_cast<uint32_t>(tag >> 32),
                  static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32), o);
}

// 32 consecutive 24-bit SR draws for flat indices e0 .. e0+31 (e0 % 4 == 0):
// element e takes the top 24 bits of word e % 4 of block e / 4.
__device__ __forceinline__ void sr_draws32(uint64_t seed, uint64_t tag, uint64_t e0,
                                           uint32_t (&u)[32]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        uint32_t o[4];
        philox_block(seed, tag, e0 / 4 + q, o);
#pragma unroll
        for (int j = 0; j < 4; ++j) u[4 * q + j] = o[j] >> 8;
    }
}

// 128 random sign bits of tokens 128*n .. 128*n+127: bit t % 32 of word
// (t % 128) / 32 (bit set -> d = -1).
__device__ __forceinline__ void sign_block128(uint64_t seed, uint64_t n, uint32_t (&o)[4]) {
    philox_block(seed, 0, n, o);
}

__device__ __forceinline__ void apply_signs(float (&x)[32], uint32_t bits) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
        x[i] = __uint_as_float(__float_as_uint(x[i]) ^ (((bits >> i) & 1u) << 31));
}

// ---------------------------------------------------------------- Hadamard
// In-register butterfly stages of stride 1 .. min(N,32)/2 on 32 values.
template <int N>
__device__ __forceinline__ void fwht_in_thread(float (&x)[32]) {
    constexpr int H = N < 32 ? N : 32;
#pragma unroll
    for (int h = 1; h < H; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            if ((i & h) == 0) {
                const float a = x[i], b = x[i + h];
                x[i] = __fadd_rn(a, b);
                x[i + h] = __fsub_rn(a, b);
            }
        }
    }
}

// fp32 value nearest to 1/sqrt(N).
template <int N>
__device__ __forceinline__ float hadamard_norm() {
    if (N == 16) return 0.25f;
    if (N == 32) return __uint_as_float(0x3E3504F3u);
    if (N == 64) return 0.125f;
    if (N == 128) return __uint_as_float(0x3DB504F3u);
    return 0.0625f;
}

template <int N>
__device__ __forceinline__ void scale_by_norm(float (&x)[32]) {
    const float c = hadamard_norm<N>();
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = __fmul_rn(x[i], c);
}

// ---------------------------------------------------------------- encoding
// E2M1 with stochastic rounding: lower grid neighbour lo, step to the next;
// round up iff u24 < (|v| - lo) / step * 2^24.  Taken on the bits of |v|:
// from 1 up, a binade holds two grid points (the leading mantissa bit picks
// one) and (|v| - lo) / step * 2^24 is 4x the 22 mantissa bits below it, so
// the decision u24 / 4 < those bits is the carry out of adding their
// complement 2^22 - 1 - u24 / 4; in [0.5, 1) it is 2x the 23 mantissa bits
// against u24 / 2.  Below 0.5 the threshold |v| * 2^25 is compared in fp32
// (exact).  |v| >= 6 and Inf give 6, NaN gives zero.
__device__ __forceinline__ uint32_t e2m1_sr_code(float v, uint32_t u24) {
    const uint32_t b = __float_as_uint(v);
    const uint32_t sign = (b >> 28) & 8u;
    const uint32_t m = b & 0x7FFFFFFFu;
    uint32_t c;
    if (m >= 0x3F800000u) {         // |v| >= 1: codes 2 (1.0) .. 7 (6.0)
        c = ((m + (~(u24 >> 2) & 0x3FFFFFu)) >> 22) - 0xFCu;
        if (m >= 0x40C00000u) c = m > 0x7F800000u ? 0u : 7u;
    } else if (m >= 0x3F000000u) {  // [0.5, 1): code 1 (0.5) or 2 (1.0)
        c = ((m + (~(u24 >> 1) & 0x7FFFFFu)) >> 23) - 0x7Du;
    } else {                        // [0, 0.5): code 0 or 1 (0.5)
        c = static_cast<float>(u24) < __fmul_rn(__uint_as_float(m), 33554432.0f) ? 1u : 0u;
    }
    return sign | c;
}

// Pack e2m1(v[2j]) into the low nibble and e2m1(v[2j+1]) into the high nibble
// of byte j; four bytes per call (round to nearest even, saturating).
__device__ __forceinline__ uint32_t cvt_e2m1x8(float v0, float v1, float v2, float v3, float v4,
                                               float v5, float v6, float v7) {
    uint32_t out;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(out)
        : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
    return out;
}

// ---------------------------------------------------------------- paired lanes
// Two channels processed in lockstep travel as one 64-bit register pair
// {channel 2l (low), channel 2l+1 (high)}; the f32x2 instructions round each
// half exactly like the scalar fp32 instruction would.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(uint64_t r, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// NaN-propagating maxima of magnitudes: a NaN anywhere in a block survives
// (max.NaN returns the canonical NaN, whose bits exceed every other magnitude).
__device__ __forceinline__ float absmax2_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(fabsf(a)), "f"(fabsf(b)));
    return r;
}
__device__ __forceinline__ float absmax3_nan(float a, float b, float c) {
    float r;
    asm("max.NaN.abs.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// max |v_i| over 32 values as a tree of three-input maxima (17 instructions).
__device__ __forceinline__ float block_amax32(const float (&v)[32]) {
    float t[11];
#pragma unroll
    for (int j = 0; j < 10; ++j) t[j] = absmax3_nan(v[3 * j], v[3 * j + 1], v[3 * j + 2]);
    t[10] = absmax2_nan(v[30], v[31]);
    float u[4];
#pragma unroll
    for (int j = 0; j < 3; ++j) u[j] = absmax3_nan(t[3 * j], t[3 * j + 1], t[3 * j + 2]);
    u[3] = absmax2_nan(t[9], t[10]);
    return absmax2_nan(absmax3_nan(u[0], u[1], u[2]), u[3]);
}

// Butterfly stages of stride 1 .. min(N,32)/2 on 32 channel pairs.
template <int N>
__device__ __forceinline__ void fwht_pairs(uint64_t (&x)[32]) {
    constexpr int H = N < 32 ? N : 32;
#pragma unroll
    for (int h = 1; h < H; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            if ((i & h) == 0) {
                const uint64_t a = x[i], b = x[i + h];
                x[i] = add2(a, b);
                x[i + h] = sub2(a, b);
            }
        }
    }
}

// Shared-exponent byte and its exact inverse power of two for a block amax.
__device__ __forceinline__ uint32_t scale_of(float amax, float &inv) {
    const uint32_t m = __float_as_uint(amax);
    const uint32_t e = m >> 23;                 // biased exponent (0: zero/subnormal)
    const uint32_t sb = e >= 2u ? e - 2u : 0u;  // floor(log2 amax) - 2 + 127, clamped at 0
    inv = __uint_as_float((254u - (sb > 253u ? 253u : sb)) << 23);  // 2^(127 - sb)
    return m >= 0x7F800000u ? 0xFFu : sb;       // Inf/NaN in the block: NaN scale
}

// Round-to-nearest encode of two channels' blocks held as pairs.  x holds the
// rotation's butterfly sums before the 1/sqrt(n) factor cn (cn = 1: none).
// Rounding is monotone, so the block amax of fl(x*cn) is fl(amax(x)*cn), and
// the scale comes out exactly as if every value had been normalised first.
// The normalised value is then divided by the scale's power of two; when the
// scale exponent keeps both fl(x*cn) and cn*2^-e away from the subnormal
// range, fl(fl(x*cn)*2^-e) == fl(x*(cn*2^-e)) (scaling by a power of two
// commutes with rounding in the normal range, and any value that lands below
// it encodes to a signed zero either way), so one multiply does both.
// Outside that range the two multiplies are done one after the other.
template <bool NORM>
__device__ __forceinline__ void encode_pair_rne(uint64_t (&x)[32], float cn, uint4 &q0, uint4 &q1,
                                                uint32_t &s0, uint32_t &s1) {
    float l[32], h[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) unpack2(x[i], l[i], h[i]);
    float m0 = block_amax32(l), m1 = block_amax32(h);
    if (NORM) {
        m0 = __fmul_rn(m0, cn);
        m1 = __fmul_rn(m1, cn);
    }
    float inv0, inv1;
    s0 = scale_of(m0, inv0);
    s1 = scale_of(m1, inv1);
    uint64_t mult = pack2(inv0, inv1);
    if (NORM) {
        // Scale bytes 4 .. 249 (or a NaN scale, whose codes are discarded).
        const bool fused = (s0 - 4u <= 245u || s0 == 0xFFu) && (s1 - 4u <= 245u || s1 == 0xFFu);
        if (fused) {
            mult = pack2(__fmul_rn(inv0, cn), __fmul_rn(inv1, cn));
        } else {
            const uint64_t cc = pack2(cn, cn);
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] = mul2(x[i], cc);
        }
    }
    float v0[32], v1[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) unpack2(mul2(x[i], mult), v0[i], v1[i]);
    uint32_t w0[4], w1[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        w0[j] = cvt_e2m1x8(v0[8 * j], v0[8 * j + 1], v0[8 * j + 2], v0[8 * j + 3], v0[8 * j + 4],
                           v0[8 * j + 5], v0[8 * j + 6], v0[8 * j + 7]);
        w1[j] = cvt_e2m1x8(v1[8 * j], v1[8 * j + 1], v1[8 * j + 2], v1[8 * j + 3], v1[8 * j + 4],
                           v1[8 * j + 5], v1[8 * j + 6], v1[8 * j + 7]);
    }
    q0 = s0 == 0xFFu ? make_uint4(0, 0, 0, 0) : make_uint4(w0[0], w0[1], w0[2], w0[3]);
    q1 = s1 == 0xFFu ? make_uint4(0, 0, 0, 0) : make_uint4(w1[0], w1[1], w1[2], w1[3]);
}

// Encode one block of 32 rotated values.  Returns the E8M0 byte; codes in q.
template <bool SR>
__device__ __forceinline__ uint32_t encode_block32(const float (&r)[32], uint4 &q,
                                                   const uint32_t *u24) {
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) m = max(m, __float_as_uint(r[i]) & 0x7FFFFFFFu);
    if (m >= 0x7F800000u) {  // Inf or NaN in the block: NaN scale, zero codes
        q = make_uint4(0, 0, 0, 0);
        return 0xFFu;
    }
    const uint32_t e = m >> 23;               // biased exponent of amax (0: zero/subnormal)
    const uint32_t sb = e >= 2u ? e - 2u : 0u;  // floor(log2 amax) - 2 + 127, clamped at 0
    const float inv = __uint_as_float((254u - sb) << 23);  // 2^(127 - sb), exact
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(r[i], inv);
    uint32_t w[4];
    if (SR) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t word = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) word |= e2m1_sr_code(v[8 * j + k], u24[8 * j + k]) << (4 * k);
            w[j] = word;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            w[j] = cvt_e2m1x8(v[8 * j], v[8 * j + 1], v[8 * j + 2], v[8 * j + 3], v[8 * j + 4],
                              v[8 * j + 5], v[8 * j + 6], v[8 * j + 7]);
    }
    q = make_uint4(w[0], w[1], w[2], w[3]);
    return sb;
}

// ---------------------------------------------------------------- MXFP8
// E8M0 byte of an MXFP8 block (E4M3 elements, largest exponent 8) and its
// exact inverse power of two: floor(log2 amax) - 8 + 127, clamped at 0.
__device__ __forceinline__ uint32_t scale_of_e4m3(float amax, float &inv) {
    const uint32_t m = __float_as_uint(amax);
    const uint32_t e = m >> 23;                 // biased exponent (0: zero/subnormal)
    const uint32_t sb = e >= 8u ? e - 8u : 0u;  // at most 247, so 2^(127 - sb) is normal
    inv = __uint_as_float((254u - sb) << 23);   // 2^(127 - sb)
    return m >= 0x7F800000u ? 0xFFu : sb;       // Inf/NaN in the block: NaN scale
}

// Four E4M3 codes (round to nearest even, saturating at +-448), v0 in the
// low byte.  The packed conversion puts its first source in the upper byte.
__device__ __forceinline__ uint32_t cvt_e4m3x4(float v0, float v1, float v2, float v3) {
    uint32_t out;
    asm("{\n\t.reg .b16 h0, h1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 h0, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 h1, %4, %3;\n\t"
        "mov.b32 %0, {h0, h1};\n\t}"
        : "=r"(out)
        : "f"(v0), "f"(v1), "f"(v2), "f"(v3));
    return out;
}

// MXFP8 encode of two channels' blocks of 32 held as pairs (no rotation):
// 32 code bytes per channel in q0 / q1.  The scaled value fl(x * 2^-s) is
// exact for every scale this rule yields unless it is an fp32 subnormal,
// which lies far below E4M3's smallest subnormal (2^-9) and rounds to a
// signed zero either way.
__device__ __forceinline__ void encode_pair_e4m3(const uint64_t (&x)[32], uint4 (&q0)[2],
                                                 uint4 (&q1)[2], uint32_t &s0, uint32_t &s1) {
    float l[32], h[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) unpack2(x[i], l[i], h[i]);
    float inv0, inv1;
    s0 = scale_of_e4m3(block_amax32(l), inv0);
    s1 = scale_of_e4m3(block_amax32(h), inv1);
    const uint64_t mult = pack2(inv0, inv1);
    float v0[32], v1[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) unpack2(mul2(x[i], mult), v0[i], v1[i]);
    uint32_t w0[8], w1[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        w0[j] = cvt_e4m3x4(v0[4 * j], v0[4 * j + 1], v0[4 * j + 2], v0[4 * j + 3]);
        w1[j] = cvt_e4m3x4(v1[4 * j], v1[4 * j + 1], v1[4 * j + 2], v1[4 * j + 3]);
    }
    const bool z0 = s0 == 0xFFu, z1 = s1 == 0xFFu;  // NaN scale: zero codes
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        q0[k] = z0 ? make_uint4(0, 0, 0, 0)
                   : make_uint4(w0[4 * k], w0[4 * k + 1], w0[4 * k + 2], w0[4 * k + 3]);
        q1[k] = z1 ? make_uint4(0, 0, 0, 0)
                   : make_uint4(w1[4 * k], w1[4 * k + 1], w1[4 * k + 2], w1[4 * k + 3]);
    }
}

// ---------------------------------------------------------------- NVFP4
// Value of an E4M3 code (sign ignored: block scales are non-negative; the
// NaN code never reaches this), exact in fp32.
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
    const uint32_t e = (c >> 3) & 15u, m = c & 7u;
    return e == 0u ? __uint2float_rn(m) * 0.001953125f            // m * 2^-9
                   : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// E4M3 code of a non-negative finite value, nearest even, saturating at 448.
__device__ __forceinline__ uint32_t f32_to_e4m3(float u) {
    uint16_t h;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(0.0f), "f"(u));
    return h & 0xFFu;
}

// Tensor encode scale of NVFP4 from the tensor's largest finite magnitude:
// 2688 / amax (448 * 6, the largest block value), FLT_MAX if that overflows,
// 1 for amax == 0.
__device__ __forceinline__ float nv_tensor_scale(float amax) {
    if (!(amax > 0.0f) || !(amax <= 3.402823466e38f)) return 1.0f;
    const float s = __fdiv_rn(2688.0f, amax);
    return s <= 3.402823466e38f ? s : 3.402823466e38f;
}

// NVFP4 encode of one block of 16 rotated values: returns the UE4M3 scale
// code (0x7F for a block holding Inf/NaN) and the 8 code bytes in q.
__device__ __forceinline__ uint32_t nv_encode_block16(const float *r, float s_enc, uint2 &q) {
    uint32_t mb = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) mb = max(mb, __float_as_uint(r[i]) & 0x7FFFFFFFu);
    if (mb >= 0x7F800000u) {
        q = make_uint2(0, 0);
        return 0x7Fu;
    }
    const float u = __fmul_rn(__fdiv_rn(__uint_as_float(mb), 6.0f), s_enc);
    const uint32_t sf = f32_to_e4m3(u);
    if (sf == 0u) {
        q = make_uint2(0, 0);
        return 0u;
    }
    float m = __fdiv_rn(s_enc, e4m3_to_f32(sf));
    m = m <= 3.402823466e38f ? m : 3.402823466e38f;
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(r[i], m);
    q = make_uint2(cvt_e2m1x8(v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7]),
                   cvt_e2m1x8(v[8], v[9], v[10], v[11], v[12], v[13], v[14], v[15]));
    return sf;
}

// Byte offset of the NVFP4 scale of (line, block of 16) in its tiled layout:
// 512-byte atoms of 128 lines x 4 blocks, `katoms` atoms per 128-line group.
__device__ __forceinline__ int64_t nv_scale_offset(int64_t line, int64_t block, int64_t katoms) {
    return ((line / 128) * katoms + block / 4) * 512 + (line % 32) * 16 + ((line % 128) / 32) * 4 +
           (block % 4);
}

// Stochastic-rounding encode of one block of 32 that draws its randomness 4
// elements at a time (one Philox call per 4, in the order of sr_draws32), so
// that only 4 draws are live at once: the same codes as encode_block32<true>
// fed by sr_draws32(seed, tag, e0, u).
__device__ __forceinline__ uint32_t encode_block32_sr(const float (&r)[32], uint4 &q,
                                                      uint64_t seed, uint64_t tag, uint64_t e0) {
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) m = max(m, __float_as_uint(r[i]) & 0x7FFFFFFFu);
    if (m >= 0x7F800000u) {  // Inf or NaN in the block: NaN scale, zero codes
        q = make_uint4(0, 0, 0, 0);
        return 0xFFu;
    }
    const uint32_t e = m >> 23;
    const uint32_t sb = e >= 2u ? e - 2u : 0u;            // floor(log2 amax) - 2 + 127, >= 0
    const float inv = __uint_as_float((254u - sb) << 23);  // 2^(127 - sb), exact
    uint32_t w[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        uint32_t word = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t o[4];
            philox_block(seed, tag, e0 / 4 + 2 * g + h, o);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                word |= e2m1_sr_code(__fmul_rn(r[8 * g + 4 * h + k], inv), o[k] >> 8)
                        << (4 * (4 * h + k));
        }
        w[g] = word;
    }
    q = make_uint4(w[0], w[1], w[2], w[3]);
    return sb;
}

__device__ __forceinline__ void st_global_16(void *p, uint4 v) {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Byte offset of the scale of (line, block) in the tiled layout.
__device__ __forceinline__ int64_t scale_offset(int64_t line, int64_t block, int64_t katoms) {
    return ((line / 128) * katoms + block / 4) * 512 + (line % 32) * 16 + ((line % 128) / 32) * 4 +
           (block % 4);
}


}  // namespace enc
}  // namespace mx
