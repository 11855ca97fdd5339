// mx_quant.cu -- rotate + MXFP4-encode kernels for sm_103a.
//
// What is computed ("Neue Studie von AMD durchbricht die bestehende
// Erkenntnis", eu.36kr.com, sections "Was ist MXFP4?" and
// "Fehlerdiagnoseexperiment"): along the contraction dimension, an optional
// block Hadamard rotation (deterministic, or after a random sign flip), then
// blocks of 32 elements share one E8M0 exponent (the block's largest exponent
// minus 2, the largest E2M1 exponent) and each element is rounded to E2M1
// (nearest-even, or stochastically) and packed two per byte.
//
// Two kernels, both persistent with a 3-deep TMA ring:
//   mxq_colwise  contraction down the rows of src[T][C] (Wgrad operands,
//                Dgrad's W): a 256-token x 64-channel tile is loaded by TMA;
//                each thread owns 2 adjacent channels x 32 tokens, so the
//                transpose is free (it reads a column pair from shared
//                memory) and the Hadamard up to 32 and the block amax stay in
//                registers.  Hadamard stages of stride >= 32 cross warps
//                through a shared-memory exchange.
//   mxq_rowwise  contraction along the rows of src[R][C] (Fprop operands,
//                Dgrad's dY): a 64-row x 256-column tile arrives as four
//                128-byte-swizzled TMA boxes; each thread owns 2 blocks of 32
//                of one row; Hadamard stages of stride 32/64 use warp
//                shuffles, stride 128 is in-thread.
// Fp32 arithmetic uses explicit round-to-nearest intrinsics so that the
// rotated values are bit-identical to the canonical butterfly order.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "mx_internal.h"
#include "mx_ptx.cuh"

namespace mx {
namespace {

constexpr int kStages = 3;
constexpr int kThreads = 256;
constexpr uint32_t kTileBytes = 32768;  // 256 x 64 bf16 (colwise) / 64 x 256 bf16 (rowwise)
constexpr uint32_t kScaleStage = 512;   // two half-atoms of scales per tile

struct QuantArgs {
    int64_t L;         // contraction length
    int64_t lines;     // number of encoded lines
    int64_t katoms;    // scale k-atoms per 128-line group
    uint8_t *codes;
    uint8_t *scales;
    uint64_t seed;
    uint64_t sr_tag;
    int *status;
    int tiles_inner;   // tiles along the fast tile axis
    int num_tiles;
};

// ---------------------------------------------------------------- Philox4x64-10
// Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11).
__device__ __forceinline__ void philox4x64_10(uint64_t c0, uint64_t k0, uint64_t k1,
                                              uint64_t (&o)[4]) {
    const uint64_t mul_a = 0xD2E7470EE14C6C93ull, mul_b = 0xCA5A826395121157ull;
    const uint64_t weyl_a = 0x9E3779B97F4A7C15ull, weyl_b = 0xBB67AE8584CAA73Bull;
    uint64_t x0 = c0, x1 = 0, x2 = 0, x3 = 0;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += weyl_a;
            k1 += weyl_b;
        }
        const uint64_t lo_a = mul_a * x0, hi_a = __umul64hi(mul_a, x0);
        const uint64_t lo_b = mul_b * x2, hi_b = __umul64hi(mul_b, x2);
        const uint64_t n0 = hi_b ^ x1 ^ k0, n2 = hi_a ^ x3 ^ k1;
        x0 = n0;
        x1 = lo_b;
        x2 = n2;
        x3 = lo_a;
    }
    o[0] = x0;
    o[1] = x1;
    o[2] = x2;
    o[3] = x3;
}

// 32 consecutive 24-bit SR draws for flat indices e0 .. e0+31 (e0 % 8 == 0).
__device__ __forceinline__ void sr_draws32(uint64_t seed, uint64_t tag, uint64_t e0,
                                           uint32_t (&u)[32]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint64_t o[4];
        philox4x64_10(e0 / 8 + q, seed, tag, o);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            u[8 * q + j] = static_cast<uint32_t>(o[j / 2] >> (32 * (j % 2))) >> 8;
    }
}

// 32 random sign bits for positions 32*chunk .. 32*chunk+31 of the 256-block
// `blk256` (bit i set -> d = -1).
__device__ __forceinline__ uint32_t sign_bits32(uint64_t seed, uint64_t blk256, int chunk) {
    uint64_t o[4];
    philox4x64_10(blk256, seed, 0, o);
    return static_cast<uint32_t>(o[chunk / 2] >> (32 * (chunk % 2)));
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
// round up iff u24 < (|v| - lo) / step * 2^24 (exact in fp32).
__device__ __forceinline__ uint32_t e2m1_sr_code(float v, uint32_t u24) {
    const uint32_t sign = (__float_as_uint(v) >> 28) & 8u;
    const float a = fabsf(v);
    if (a >= 6.0f) return sign | 7u;
    const uint32_t lo = (a >= 0.5f) + (a >= 1.0f) + (a >= 1.5f) + (a >= 2.0f) + (a >= 3.0f) +
                        (a >= 4.0f);
    const float lov = lo <= 4 ? 0.5f * static_cast<float>(lo) : (lo == 5 ? 3.0f : 4.0f);
    const float inv_step_2p24 = lo < 4 ? 33554432.0f : (lo < 6 ? 16777216.0f : 8388608.0f);
    const float thr = __fmul_rn(__fsub_rn(a, lov), inv_step_2p24);
    const uint32_t up = static_cast<float>(u24) < thr ? 1u : 0u;
    return sign | (lo + up);
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

__device__ __forceinline__ void st_global_16(void *p, uint4 v) {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Byte offset of scale (line, block) within a tile's 2-atom staging area:
// staging[a][g][8] holds, for k-atom a of the tile and line group g = line%32,
// the 8 bytes of this 64-line half: ((line%64)/32)*4 + block%4.
__device__ __forceinline__ uint32_t stage_offset(int line_in_tile, int block_in_tile) {
    return static_cast<uint32_t>((block_in_tile / 4) * 256 + (line_in_tile % 32) * 8 +
                                 (line_in_tile / 32) * 4 + (block_in_tile % 4));
}

// Write the staged scales of a 64-line x 8-block tile to the tiled layout.
__device__ __forceinline__ void flush_scales(const uint8_t *stage, const QuantArgs &p,
                                             int64_t line0, int64_t k0) {
    const int t = threadIdx.x;
    if (t < 64) {
        const int a = t / 32, g = t % 32;
        const uint64_t v = *reinterpret_cast<const uint64_t *>(stage + a * 256 + g * 8);
        const int64_t half = (line0 % 128) / 64;
        const int64_t atom = (line0 / 128) * p.katoms + k0 / 128 + a;
        *reinterpret_cast<uint64_t *>(p.scales + atom * 512 + g * 16 + half * 8) = v;
    }
}

// ---------------------------------------------------------------- colwise
template <int ROTN, bool RAND, bool SR>
__global__ void __launch_bounds__(kThreads) mxq_colwise_kernel(const __grid_constant__ CUtensorMap src_map,
                                                               const QuantArgs p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *tiles = smem;                                   // kStages x 32 KB
    uint8_t *sstage = smem + kStages * kTileBytes;           // 512 B
    uint64_t *full = reinterpret_cast<uint64_t *>(sstage + kScaleStage);
    float2 *xchg = reinterpret_cast<float2 *>(smem + kStages * kTileBytes + 1024);  // 64 KB
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&src_map);
    }
    __syncthreads();

    auto issue = [&](int tile, int s) {
        const int tt = tile / p.tiles_inner, ct = tile % p.tiles_inner;
        mbar_arrive_expect_tx(&full[s], kTileBytes);
        tma_load_2d(tiles + s * kTileBytes, &src_map, &full[s], ct * 64, tt * 256);
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            const int tile = blockIdx.x + s * gridDim.x;
            if (tile < p.num_tiles) issue(tile, s);
        }
    }

    for (int it = 0;; ++it) {
        const int tile = blockIdx.x + it * gridDim.x;
        if (tile >= p.num_tiles) break;
        const int s = it % kStages;
        const uint32_t parity = (it / kStages) & 1u;
        const int64_t t0 = static_cast<int64_t>(tile / p.tiles_inner) * 256;
        const int64_t c0 = static_cast<int64_t>(tile % p.tiles_inner) * 64;

        const bool ok = mbar_wait(&full[s], parity, p.status, &abort_flag);
        if (__syncthreads_or(!ok)) break;

        // Column pair (2*lane, 2*lane+1), tokens 32*warp .. 32*warp+31.
        float x0[32], x1[32];
        const uint32_t *tw = reinterpret_cast<const uint32_t *>(tiles + s * kTileBytes);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const uint32_t v = tw[(warp * 32 + i) * 32 + lane];
            x0[i] = __uint_as_float(v << 16);
            x1[i] = __uint_as_float(v & 0xFFFF0000u);
        }
        __syncthreads();  // stage s fully consumed
        if (threadIdx.x == 0) {
            const int nt = tile + kStages * gridDim.x;
            if (nt < p.num_tiles) issue(nt, s);
        }

        if (ROTN > 0) {
            if (RAND) {
                const uint32_t bits = sign_bits32(p.seed, static_cast<uint64_t>(t0 / 256), warp);
                apply_signs(x0, bits);
                apply_signs(x1, bits);
            }
            fwht_in_thread<ROTN>(x0);
            fwht_in_thread<ROTN>(x1);
            if (ROTN >= 64) {
#pragma unroll
                for (int h = 32; h < ROTN; h <<= 1) {
                    const int m = h / 32;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        xchg[(warp * 32 + i) * 32 + lane] = make_float2(x0[i], x1[i]);
                    __syncthreads();
                    const int pw = warp ^ m;
                    const bool lower = (warp & m) == 0;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float2 o = xchg[(pw * 32 + i) * 32 + lane];
                        x0[i] = lower ? __fadd_rn(x0[i], o.x) : __fsub_rn(o.x, x0[i]);
                        x1[i] = lower ? __fadd_rn(x1[i], o.y) : __fsub_rn(o.y, x1[i]);
                    }
                    __syncthreads();
                }
            }
            scale_by_norm<ROTN>(x0);
            scale_by_norm<ROTN>(x1);
        }

        const int64_t tb = t0 + 32 * warp;   // first token of this thread's block
        const int64_t c = c0 + 2 * lane;     // first of the thread's two channels
        uint32_t u[32];
        uint4 q0, q1;
        if (SR) sr_draws32(p.seed, p.sr_tag, static_cast<uint64_t>(c * p.L + tb), u);
        const uint32_t s0 = encode_block32<SR>(x0, q0, u);
        if (SR) sr_draws32(p.seed, p.sr_tag, static_cast<uint64_t>((c + 1) * p.L + tb), u);
        const uint32_t s1 = encode_block32<SR>(x1, q1, u);

        if (tb < p.L) {
            if (c < p.lines) st_global_16(p.codes + c * (p.L / 2) + tb / 2, q0);
            if (c + 1 < p.lines) st_global_16(p.codes + (c + 1) * (p.L / 2) + tb / 2, q1);
        }
        sstage[stage_offset(2 * lane, warp)] = static_cast<uint8_t>(s0);
        sstage[stage_offset(2 * lane + 1, warp)] = static_cast<uint8_t>(s1);
        __syncthreads();
        flush_scales(sstage, p, c0, t0);
    }
}

// ---------------------------------------------------------------- rowwise
template <int ROTN, bool RAND, bool SR>
__global__ void __launch_bounds__(kThreads) mxq_rowwise_kernel(const __grid_constant__ CUtensorMap src_map,
                                                               const QuantArgs p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *tiles = smem;
    uint8_t *sstage = smem + kStages * kTileBytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(sstage + kScaleStage);
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = 8 * warp + (lane & 7);     // row within the 64-row tile
    const int blk_a = lane >> 3;             // blocks blk_a and blk_a + 4 of the 256 columns
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&src_map);
    }
    __syncthreads();

    auto issue = [&](int tile, int s) {
        const int rt = tile / p.tiles_inner, ct = tile % p.tiles_inner;
        mbar_arrive_expect_tx(&full[s], kTileBytes);
#pragma unroll
        for (int b = 0; b < 4; ++b)
            tma_load_2d(tiles + s * kTileBytes + b * 8192, &src_map, &full[s], ct * 256 + b * 64,
                        rt * 64);
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            const int tile = blockIdx.x + s * gridDim.x;
            if (tile < p.num_tiles) issue(tile, s);
        }
    }

    for (int it = 0;; ++it) {
        const int tile = blockIdx.x + it * gridDim.x;
        if (tile >= p.num_tiles) break;
        const int s = it % kStages;
        const uint32_t parity = (it / kStages) & 1u;
        const int64_t row0 = static_cast<int64_t>(tile / p.tiles_inner) * 64;
        const int64_t col0 = static_cast<int64_t>(tile % p.tiles_inner) * 256;

        const bool ok = mbar_wait(&full[s], parity, p.status, &abort_flag);
        if (__syncthreads_or(!ok)) break;

        float xa[32], xb[32];
        const uint8_t *stile = tiles + s * kTileBytes;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int blk = blk_a + 4 * half;
            const uint8_t *box = stile + (blk / 2) * 8192 + r * 128;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int phys = ((blk % 2) * 4 + j) ^ (r & 7);  // 128-byte swizzle
                const uint4 v = *reinterpret_cast<const uint4 *>(box + phys * 16);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float lo = __uint_as_float(w[k] << 16);
                    const float hi = __uint_as_float(w[k] & 0xFFFF0000u);
                    if (half == 0) {
                        xa[8 * j + 2 * k] = lo;
                        xa[8 * j + 2 * k + 1] = hi;
                    } else {
                        xb[8 * j + 2 * k] = lo;
                        xb[8 * j + 2 * k + 1] = hi;
                    }
                }
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            const int nt = tile + kStages * gridDim.x;
            if (nt < p.num_tiles) issue(nt, s);
        }

        if (ROTN > 0) {
            if (RAND) {
                uint64_t o[4];
                philox4x64_10(static_cast<uint64_t>(col0 / 256), p.seed, 0, o);
                const int ba = blk_a, bb = blk_a + 4;
                apply_signs(xa, static_cast<uint32_t>(o[ba / 2] >> (32 * (ba % 2))));
                apply_signs(xb, static_cast<uint32_t>(o[bb / 2] >> (32 * (bb % 2))));
            }
            fwht_in_thread<ROTN>(xa);
            fwht_in_thread<ROTN>(xb);
            if (ROTN >= 64) {  // stride 32: partner block blk^1 lives in lane^8
                const bool lower = (blk_a & 1) == 0;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float oa = __shfl_xor_sync(0xFFFFFFFFu, xa[i], 8);
                    const float ob = __shfl_xor_sync(0xFFFFFFFFu, xb[i], 8);
                    xa[i] = lower ? __fadd_rn(xa[i], oa) : __fsub_rn(oa, xa[i]);
                    xb[i] = lower ? __fadd_rn(xb[i], ob) : __fsub_rn(ob, xb[i]);
                }
            }
            if (ROTN >= 128) {  // stride 64: partner block blk^2 lives in lane^16
                const bool lower = (blk_a & 2) == 0;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float oa = __shfl_xor_sync(0xFFFFFFFFu, xa[i], 16);
                    const float ob = __shfl_xor_sync(0xFFFFFFFFu, xb[i], 16);
                    xa[i] = lower ? __fadd_rn(xa[i], oa) : __fsub_rn(oa, xa[i]);
                    xb[i] = lower ? __fadd_rn(xb[i], ob) : __fsub_rn(ob, xb[i]);
                }
            }
            if (ROTN >= 256) {  // stride 128: blocks blk_a and blk_a + 4, both here
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float a = xa[i], b = xb[i];
                    xa[i] = __fadd_rn(a, b);
                    xb[i] = __fsub_rn(a, b);
                }
            }
            scale_by_norm<ROTN>(xa);
            scale_by_norm<ROTN>(xb);
        }

        const int64_t row = row0 + r;
        uint32_t u[32];
        uint4 qa, qb;
        const int64_t ca = col0 + 32 * blk_a, cb = ca + 128;
        if (SR) sr_draws32(p.seed, p.sr_tag, static_cast<uint64_t>(row * p.L + ca), u);
        const uint32_t sa = encode_block32<SR>(xa, qa, u);
        if (SR) sr_draws32(p.seed, p.sr_tag, static_cast<uint64_t>(row * p.L + cb), u);
        const uint32_t sb = encode_block32<SR>(xb, qb, u);
        if (row < p.lines) {
            if (ca < p.L) st_global_16(p.codes + row * (p.L / 2) + ca / 2, qa);
            if (cb < p.L) st_global_16(p.codes + row * (p.L / 2) + cb / 2, qb);
        }
        sstage[stage_offset(r, blk_a)] = static_cast<uint8_t>(sa);
        sstage[stage_offset(r, blk_a + 4)] = static_cast<uint8_t>(sb);
        __syncthreads();
        flush_scales(sstage, p, row0, col0);
    }
}

// ---------------------------------------------------------------- dispatch
template <typename Kern>
cudaError_t launch_persistent(Kern kernel, const CUtensorMap &map, const QuantArgs &a,
                              size_t smem, const DeviceInfo &dev, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int grid = a.num_tiles < dev.sm_count * per_sm ? a.num_tiles : dev.sm_count * per_sm;
    kernel<<<grid, kThreads, smem, stream>>>(map, a);
    return cudaGetLastError();
}

template <bool COLWISE, int ROTN, bool RAND>
cudaError_t launch_rot(bool sr, const CUtensorMap &map, const QuantArgs &a,
                       const DeviceInfo &dev, cudaStream_t stream) {
    const size_t smem = kStages * kTileBytes + 1024 + (COLWISE && ROTN >= 64 ? 65536 : 0) + 1024;
    if (COLWISE) {
        return sr ? launch_persistent(mxq_colwise_kernel<ROTN, RAND, true>, map, a, smem, dev, stream)
                  : launch_persistent(mxq_colwise_kernel<ROTN, RAND, false>, map, a, smem, dev, stream);
    }
    return sr ? launch_persistent(mxq_rowwise_kernel<ROTN, RAND, true>, map, a, smem, dev, stream)
              : launch_persistent(mxq_rowwise_kernel<ROTN, RAND, false>, map, a, smem, dev, stream);
}

template <bool COLWISE>
cudaError_t launch_dir(int rot, int rot_block, bool sr, const CUtensorMap &map,
                       const QuantArgs &a, const DeviceInfo &dev, cudaStream_t stream) {
    if (rot == 0) return launch_rot<COLWISE, 0, false>(sr, map, a, dev, stream);
    const bool rnd = rot == 2;
#define MX_ROT_CASE(N)                                                                      \
    case N:                                                                                 \
        return rnd ? launch_rot<COLWISE, N, true>(sr, map, a, dev, stream)                  \
                   : launch_rot<COLWISE, N, false>(sr, map, a, dev, stream);
    switch (rot_block) {
        MX_ROT_CASE(16)
        MX_ROT_CASE(32)
        MX_ROT_CASE(64)
        MX_ROT_CASE(128)
        MX_ROT_CASE(256)
        default:
            return cudaErrorInvalidValue;
    }
#undef MX_ROT_CASE
}

}  // namespace

cudaError_t launch_quantize(const void *src, int64_t rows, int64_t cols, int contract, int rot,
                            int rot_block, int rnd, uint64_t seed, uint64_t sr_tag,
                            void *codes, void *scales, const DeviceInfo &dev,
                            cudaStream_t stream) {
    const bool colwise = contract == 0;
    QuantArgs a{};
    a.L = colwise ? rows : cols;
    a.lines = colwise ? cols : rows;
    a.katoms = scale_katoms(a.L);
    a.codes = static_cast<uint8_t *>(codes);
    a.scales = static_cast<uint8_t *>(scales);
    a.seed = seed;
    a.sr_tag = sr_tag;
    a.status = dev.status;
    // Tiles cover the padded scale layout: lines to a multiple of 128 and the
    // contraction dim to a multiple of 256, so padding scale bytes get zeros.
    const int64_t line_tiles = scale_groups(a.lines) * 2;  // 64 lines per tile
    const int64_t k_tiles = (a.L + 255) / 256;
    if (line_tiles * k_tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
    CUtensorMap map;
    if (colwise) {
        a.tiles_inner = static_cast<int>(line_tiles);
        a.num_tiles = static_cast<int>(line_tiles * k_tiles);
        if (!encode_tmap_2d(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, src, cols, rows, cols * 2, 64,
                            256, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
        return launch_dir<true>(rot, rot_block, rnd == 1, map, a, dev, stream);
    }
    a.tiles_inner = static_cast<int>(k_tiles);
    a.num_tiles = static_cast<int>(line_tiles * k_tiles);
    if (!encode_tmap_2d(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, src, cols, rows, cols * 2, 64, 64,
                        CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    return launch_dir<false>(rot, rot_block, rnd == 1, map, a, dev, stream);
}

}  // namespace mx
