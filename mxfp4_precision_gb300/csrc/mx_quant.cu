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
// Three kernels, all persistent with a ring of 32 KB TMA tiles (3 deep for the
// wide kernel's Hadamard 64, 2 for the others; two resident CTAs per SM):
//   mxq_colwise       contraction down the rows of src[T][C] (Wgrad operands,
//                     Dgrad's W), no rotation or Hadamard 16/32: a 128-token
//                     x 128-channel tile; each thread owns 2 adjacent
//                     channels x 32 tokens as packed f32x2 pairs, so the
//                     transpose is free (it reads a column pair from shared
//                     memory) and the Hadamard and the block amax stay in
//                     registers.  A ninth warp refills the ring (thread 0
//                     in the dual variant).  Outputs
//                     leave through a shared-memory staging image (one TMA
//                     box of codes, one bulk copy of the scale atom per
//                     tile).  With DUAL it also encodes the staged tile
//                     along the channels (the Dgrad encoding of the same
//                     dY); with other element formats it writes MXFP8 or
//                     NVFP4 instead.
//   mxq_colwise_wide  the same direction for Hadamard 64/128/256 (128 x 128
//                     tiles, 256 x 64 for 256): each thread owns one
//                     channel x 64 tokens as pairs {t, t+32}; the
//                     stride-64 and stride-128 stages pair lanes by warp
//                     shuffles.
//   mxq_rowwise       contraction along the rows of src[R][C] (Fprop
//                     operands, Dgrad's dY): a 64-row x 256-column tile
//                     arrives as four 128-byte-swizzled TMA boxes; each
//                     thread owns 2 blocks of 32 of one row; Hadamard stages
//                     of stride 32/64 use warp shuffles, stride 128 is
//                     in-thread.
// Fp32 arithmetic uses explicit round-to-nearest intrinsics so that the
// rotated values are bit-identical to the canonical butterfly order.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "mx_encode.cuh"
#include "mx_internal.h"
#include "mx_ptx.cuh"

namespace mx {
namespace {
using namespace enc;

#ifndef MXQ_STAGES
#define MXQ_STAGES 2
#endif
constexpr int kStages = MXQ_STAGES;  // TMA ring depth per CTA (wide and row kernels)
// The column kernel: a 2-deep ring and two output staging buffers, so that a
// tile's staged outputs need not wait for the previous tile's store (down_proj
// operands: 68.3 us against 70.3 us for a 3-deep ring and one buffer, 66.2
// against 70.3 us without rotation; o_proj equal; three buffers no better).
#ifndef MXQ_COL_RING
#define MXQ_COL_RING 2
#endif
#ifndef MXQ_STAGE_BUFS
#define MXQ_STAGE_BUFS 2
#endif
constexpr int kColRing = MXQ_COL_RING;      // TMA ring depth of the column kernel
constexpr int kStageBufs = MXQ_STAGE_BUFS;  // its output staging buffers
// The dual variant stages two images per tile and keeps one buffer of each
// (39.6 us on o_proj's dY against 41.6 us with two).
// Two resident CTAs per SM (shared memory allows no more with two stages):
// the round-to-nearest colwise kernels are held to 128 registers so that the
// random-sign variants do not fall to one CTA per SM.
constexpr int kColMinBlocks = 2;
// The stochastic-rounding column kernel also runs two CTAs per SM: at the
// 96-register bound it spills a few words, and the second CTA's warps hide
// the Philox multiply chains (down_proj SR encode 448.8 -> 334.6 us).
#ifndef MXQ_SR_MINB
#define MXQ_SR_MINB 2
#endif
constexpr int kColSRMinBlocks = MXQ_SR_MINB;
constexpr int kThreads = 256;           // compute threads (8 warps)
constexpr int kColProducerThreads = kThreads + 32;  // + a TMA producer warp
constexpr uint32_t kTileBytes = 32768;  // one staged bf16 tile (128 x 128, 256 x 64 or 64 x 256)
constexpr uint32_t kScaleStage = 512;   // two half-atoms of scales per tile

struct QuantArgs {
    int64_t L;         // contraction length
    int64_t lines;     // number of encoded lines
    int64_t katoms;    // scale k-atoms per 128-line group
    uint8_t *codes;
    uint8_t *scales;
    size_t codes_bytes;   // extents of the two output buffers (store guards)
    size_t scales_bytes;
    uint64_t seed;
    uint64_t sr_tag;
    unsigned int *amax;  // NVFP4: the operand's tensor amax (fp32 bits; max-reduced)
    int *status;
    int tiles_inner;   // tiles along the fast tile axis
    int num_tiles;
};

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
        uint8_t *dst = p.scales + atom * 512 + g * 16 + half * 8;
        if (MX_STORE_OK(dst, 8, p.scales, p.scales_bytes, p.status))
            *reinterpret_cast<uint64_t *>(dst) = v;
    }
}

// ---------------------------------------------------------------- dual output
// Row-direction (channel-contiguous) encode of one 32-channel block of one
// token, straight from a staged column-wise tile: no rotation, blocks of 32
// along the row.  w holds the block's 16 words (two bf16 channels each,
// channel 2i in the low half).
template <bool SR>
__device__ __forceinline__ uint32_t encode_row_block(const uint32_t (&w)[16], uint4 &q,
                                                     uint64_t seed, uint64_t tag, uint64_t e0) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    if (SR) {
        uint32_t u[32];
        sr_draws32(seed, tag, e0, u);
        return encode_block32<true>(v, q, u);
    }
    float inv;
    const uint32_t sb = scale_of(block_amax32(v), inv);
    const uint64_t mult = pack2(inv, inv);
    float r[32];
#pragma unroll
    for (int i = 0; i < 16; ++i) unpack2(mul2(pack2(v[2 * i], v[2 * i + 1]), mult), r[2 * i], r[2 * i + 1]);
    uint32_t c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        c[j] = cvt_e2m1x8(r[8 * j], r[8 * j + 1], r[8 * j + 2], r[8 * j + 3], r[8 * j + 4],
                          r[8 * j + 5], r[8 * j + 6], r[8 * j + 7]);
    q = sb == 0xFFu ? make_uint4(0, 0, 0, 0) : make_uint4(c[0], c[1], c[2], c[3]);
    return sb;
}

// ---------------------------------------------------------------- colwise
// Row direction of a dual encode: each thread encodes two (token, 32-channel)
// blocks of a staged TT x TC column tile.  The four 16-byte reads of a block
// start at a row-dependent chunk so that a warp's reads spread over all banks.
template <int TC, bool SR>
__device__ __forceinline__ void dual_rows(const uint32_t *tw, int64_t t0, int64_t c0,
                                          const QuantArgs &a0, const QuantArgs &ar) {
    const int64_t row_lines_pad = (ar.lines + 127) / 128 * 128;
    const int64_t grid_end = (a0.lines + 127) / 128 * 128;  // channels the tiles cover
    const int64_t kb_pad = ar.katoms * 4;                    // padded blocks per row
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int b = threadIdx.x + kThreads * h;
        const int trow = b / (TC / 32), cb = b % (TC / 32);
        const int64_t t = t0 + trow;
        if (t >= row_lines_pad) continue;
        const int64_t c = c0 + 32 * cb;
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int jj = (j + trow) & 3;
            const uint4 v = *reinterpret_cast<const uint4 *>(tw + trow * (TC / 2) + 16 * cb + 4 * jj);
            w[4 * jj] = v.x, w[4 * jj + 1] = v.y, w[4 * jj + 2] = v.z, w[4 * jj + 3] = v.w;
        }
        uint4 q;
        const uint32_t sb =
            encode_row_block<SR>(w, q, a0.seed, ar.sr_tag, static_cast<uint64_t>(t * ar.L + c));
        uint8_t *cdst = ar.codes + t * (ar.L / 2) + c / 2;
        if (t < ar.lines && c < ar.L && MX_STORE_OK(cdst, 16, ar.codes, ar.codes_bytes, ar.status))
            st_global_16(cdst, q);
        uint8_t *sdst = ar.scales + scale_offset(t, c / 32, ar.katoms);
        if (MX_STORE_OK(sdst, 1, ar.scales, ar.scales_bytes, ar.status))
            *sdst = static_cast<uint8_t>(sb);
        // Padding blocks past the last channel tile: no tile covers them.
        if (c0 + TC == grid_end) {
#pragma unroll
            for (int e = 0; e < 128 / TC; ++e) {
                const int64_t pb = grid_end / 32 + cb + e * (TC / 32);
                uint8_t *pdst = ar.scales + scale_offset(t, pb, ar.katoms);
                if (pb < kb_pad && MX_STORE_OK(pdst, 1, ar.scales, ar.scales_bytes, ar.status))
                    *pdst = 0;
            }
        }
    }
}

// The same row-direction encode for the staged column kernel (TC = 128): the
// codes go to the row image's [128 tokens][64 B] box (64-byte swizzle) and the
// scale bytes to its 512-byte atom (tokens t0 .. t0+127, channel atom c0/128);
// only the padding blocks past the last channel tile, which no tile's atom
// covers, are stored directly.
template <bool SR>
__device__ __forceinline__ void dual_rows_staged(const uint32_t *tw, int64_t t0, int64_t c0,
                                                 const QuantArgs &a0, const QuantArgs &ar,
                                                 uint8_t *rc, uint8_t *rs) {
    constexpr int TC = 128;
    const int64_t row_lines_pad = (ar.lines + 127) / 128 * 128;
    const int64_t grid_end = (a0.lines + 127) / 128 * 128;  // channels the tiles cover
    const int64_t kb_pad = ar.katoms * 4;                    // padded blocks per row
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int b = threadIdx.x + kThreads * h;
        const int trow = b / (TC / 32), cb = b % (TC / 32);
        const int64_t t = t0 + trow;
        const int64_t c = c0 + 32 * cb;
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int jj = (j + trow) & 3;
            const uint4 v = *reinterpret_cast<const uint4 *>(tw + trow * (TC / 2) + 16 * cb + 4 * jj);
            w[4 * jj] = v.x, w[4 * jj + 1] = v.y, w[4 * jj + 2] = v.z, w[4 * jj + 3] = v.w;
        }
        uint4 q;
        const uint32_t sb =
            encode_row_block<SR>(w, q, a0.seed, ar.sr_tag, static_cast<uint64_t>(t * ar.L + c));
        *reinterpret_cast<uint4 *>(rc + trow * 64 + ((cb ^ ((trow >> 1) & 3)) * 16)) = q;
        rs[(trow % 32) * 16 + (trow / 32) * 4 + cb] = static_cast<uint8_t>(sb);
        if (c0 + TC == grid_end && t < row_lines_pad) {
            const int64_t pb = grid_end / 32 + cb;
            uint8_t *pdst = ar.scales + scale_offset(t, pb, ar.katoms);
            if (pb < kb_pad && MX_STORE_OK(pdst, 1, ar.scales, ar.scales_bytes, ar.status))
                *pdst = 0;
        }
    }
}

// Column-wise encode for no rotation and Hadamard sizes 16 and 32.  One
// launch encodes up to two operands (the two Wgrad operands): tiles
// [0, a0.num_tiles) belong to operand 0, the rest to operand 1.  Every warp
// works on its own 32-token slice of the tile and marks the stage consumed on
// an mbarrier as soon as it holds its values; the stage is refilled once all
// eight have.  Tile: 128 tokens x 128 channels of bf16 (32 KB, 256-byte
// contiguous row segments).
template <int ROTN>
struct ColTile {
    static_assert(ROTN <= 32, "larger Hadamard sizes use mxq_colwise_wide_kernel");
    static constexpr int TT = 128;
    static constexpr int TC = 128;
    static constexpr int TOKEN_BLOCKS = TT / 32;  // warps along tokens
};

// With DUAL, the launch has one source operand (a0) and also writes its
// row-direction encoding (blocks of 32 along the channels, no rotation) to
// `ar`, from the same staged tiles: one HBM read serves both encodings.
// Without DUAL, a ninth warp is the TMA producer: it refills each stage once
// all eight compute warps have released it.  (The dual variant keeps its
// registers for the row encode and refills from thread 0 instead.)
//
// Element formats of the column encoder: MXFP4; MXFP8 (the FP8 comparator:
// no rotation, round to nearest; each block becomes 32 E4M3 code bytes under
// the same E8M0 scale layout); and the two passes of NVFP4 (the tensor amax
// of the rotated operand, then the encode with its tensor scale: blocks of
// 16, UE4M3 scales in their own tiled layout).
constexpr int kFmtMX4 = 0, kFmtMX8 = 1, kFmtNVAmax = 2, kFmtNV4 = 3;
//
// Output path (every variant but DUAL and the amax pass): each warp writes
// its codes and scale bytes into a shared-memory staging buffer laid out as
// the tile's global image -- the codes as a [128 lines][64 B] box (128 B for
// MXFP8) in the TMA's swizzled layout, the scales as the tile's whole
// 512-byte scale atom (two atoms for NVFP4), which the tiled layout stores
// contiguously.  After a named barrier, one thread stores the box with a TMA
// tensor store and the atom with a bulk copy: whole lines reach L2 instead of
// 16-byte pieces of 64 lines and single bytes.  The staging buffers
// alternate; the barrier before a tile's first staging write also ANDs the
// warps' wait results, so an abort leaves every warp the same way and no
// warp waits at a barrier the others have left.
template <int FMT>
struct ColStage {
    static constexpr uint32_t kCodeBytes = FMT == kFmtMX8 ? 16384u : 8192u;  // 128 lines
    static constexpr uint32_t kScaleBytes = FMT == kFmtNV4 ? 1024u : 512u;
    // One buffer, a whole number of 1 KB (the swizzle patterns repeat every 512 B
    // or 1 KB, so every codes box starts on such a boundary).
    static constexpr uint32_t kBytes = (kCodeBytes + kScaleBytes + 1023u) / 1024u * 1024u;
    static constexpr int kRing = FMT == kFmtMX8 && kColRing > 2 ? 2 : kColRing;  // TMA ring depth
};
constexpr int kStageBarrier = 1;   // named barrier of the 8 compute warps
// L2 priorities of the column kernel's copies: the bf16 input (read once)
// is evicted first, the encoded codes and scales (read next by the GEMM)
// last.
#ifndef MXQ_L2_HINTS
#define MXQ_L2_HINTS 1
#endif
// The column kernel waits for its staging buffer (and votes on its tile's
// load) after the tile's arithmetic, not before it (o_proj operands, Hadamard
// 32: 37.5 -> 35.5 us; random-sign Hadamard 32 on down_proj: 78.5 -> 74.4 us).
#ifndef MXQ_LATE_STAGE_WAIT
#define MXQ_LATE_STAGE_WAIT 1
#endif

template <int ROTN, bool RAND, bool SR, bool DUAL, int FMT = kFmtMX4>
__global__ void __launch_bounds__(DUAL ? kThreads : kColProducerThreads,
                                  SR ? (DUAL ? 1 : kColSRMinBlocks) : kColMinBlocks)
    mxq_colwise_kernel(
    const __grid_constant__ CUtensorMap map0, const __grid_constant__ CUtensorMap map1,
    const __grid_constant__ CUtensorMap cmap0, const __grid_constant__ CUtensorMap cmap1,
    const QuantArgs a0, const QuantArgs a1, const QuantArgs ar) {
    constexpr bool kStaged = FMT != kFmtNVAmax;
    // (Hadamard 16 measured 70.3 us with the early wait against 72.4 us with
    // the late one on the down_proj operands; 32 and the random signs gain.)
    constexpr bool kLateStageWait = !DUAL && MXQ_LATE_STAGE_WAIT && ROTN != 16;
    using S = ColStage<FMT>;
    // The dual variant stages two images (column and row direction) and
    // keeps a 2-deep ring so that two CTAs still fit.
    constexpr int kColRing = DUAL ? 2 : S::kRing;
    constexpr int kImages = DUAL ? 2 : 1;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned base, kept as a shared-space pointer (offset arithmetic
    // only) so that the compiler emits shared-memory loads.
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *tiles = smem;                                   // kColRing x 32 KB
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kColRing * kTileBytes);
    uint64_t *empty = full + kColRing;
    // Random-sign words of each stage's tile (4 x 32 tokens), written by the
    // thread that issues the stage's load before it arms the stage barrier:
    // one Philox call per tile instead of one per warp.
    uint32_t *signw = reinterpret_cast<uint32_t *>(empty + kColRing);
    constexpr int kBufs = DUAL ? 1 : kStageBufs;
    uint8_t *staging = smem + kColRing * kTileBytes + 1024;  // kBufs x kImages x S::kBytes
    __shared__ int abort_flag;

    using G = ColTile<ROTN>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tbi = warp % G::TOKEN_BLOCKS;   // this warp's 32-token block in the tile
    const int chalf = warp / G::TOKEN_BLOCKS;  // this warp's 64-channel slice of the tile
    const int total = a0.num_tiles + a1.num_tiles;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kColRing; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kThreads / 32);
        }
        abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&map0);
        if (a1.num_tiles > 0) prefetch_tmap(&map1);
        if (kStaged) {
            prefetch_tmap(&cmap0);
            if (a1.num_tiles > 0) prefetch_tmap(&cmap1);
        }
    }
    __syncthreads();
    griddep_wait();
    griddep_launch_dependents();

    auto issue = [&](int tile, int s) {
        const bool second = tile >= a0.num_tiles;
        const int lt = second ? tile - a0.num_tiles : tile;
        const int inner = second ? a1.tiles_inner : a0.tiles_inner;
        if constexpr (RAND) {
            static_assert(G::TT == 128, "one 128-bit sign block per tile");
            const int64_t t0 = static_cast<int64_t>(lt / inner) * G::TT;
            uint32_t o[4];
            sign_block128(a0.seed, static_cast<uint64_t>(t0 / 128), o);
#pragma unroll
            for (int k = 0; k < G::TOKEN_BLOCKS; ++k) signw[s * G::TOKEN_BLOCKS + k] = o[k];
        }
        mbar_arrive_expect_tx(&full[s], kTileBytes);
#if MXQ_L2_HINTS
        // The bf16 input is read once: its lines are the first L2 evicts.
        tma_load_2d_hint(tiles + s * kTileBytes, second ? &map1 : &map0, &full[s],
                         (lt % inner) * G::TC, (lt / inner) * G::TT, l2_evict_first_policy());
#else
        tma_load_2d(tiles + s * kTileBytes, second ? &map1 : &map0, &full[s], (lt % inner) * G::TC,
                    (lt / inner) * G::TT);
#endif
    };
    if (DUAL) {
        if (threadIdx.x == 0) {
            for (int s = 0; s < kColRing; ++s) {
                const int tile = blockIdx.x + s * gridDim.x;
                if (tile < total) issue(tile, s);
            }
        }
    } else if (warp == kThreads / 32) {
        // ---- producer warp: stage s of iteration it is refilled once the
        // compute warps have released its previous use (iteration it - kColRing).
        if (lane == 0) {
            for (int it = 0;; ++it) {
                const int tile = blockIdx.x + it * gridDim.x;
                if (tile >= total) break;
                const int s = it % kColRing;
                if (it >= kColRing &&
                    !mbar_wait(&empty[s], ((it / kColRing) - 1) & 1u, a0.status, &abort_flag))
                    break;
                issue(tile, s);
            }
        }
        return;
    }

    float amax_run0 = 0.0f, amax_run1 = 0.0f;  // NVFP4 amax pass: running maxima per operand
    for (int it = 0;; ++it) {
        const int tile = blockIdx.x + it * gridDim.x;
        if (tile >= total) break;
        const int s = it % kColRing;
        const uint32_t parity = (it / kColRing) & 1u;
        const bool second = tile >= a0.num_tiles;
        const int lt = second ? tile - a0.num_tiles : tile;
        const int inner = second ? a1.tiles_inner : a0.tiles_inner;
        const int64_t L = second ? a1.L : a0.L;
        const int64_t lines = second ? a1.lines : a0.lines;
        const int64_t katoms = second ? a1.katoms : a0.katoms;
        uint8_t *const codes = second ? a1.codes : a0.codes;
        uint8_t *const scales = second ? a1.scales : a0.scales;
        const size_t codes_bytes = second ? a1.codes_bytes : a0.codes_bytes;
        const size_t scales_bytes = second ? a1.scales_bytes : a0.scales_bytes;
        (void)codes_bytes;
        (void)scales_bytes;
        (void)lines;
        (void)codes;
        const int64_t t0 = static_cast<int64_t>(lt / inner) * G::TT;
        const int64_t c0 = static_cast<int64_t>(lt % inner) * G::TC;

        int ok = 1;
        if (lane == 0) ok = mbar_wait(&full[s], parity, a0.status, &abort_flag) ? 1 : 0;
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        // The staging buffer of this tile was last stored kBufs tiles ago:
        // that store has read it once at most kBufs - 1 are pending.
        // The same CTA barrier ANDs the warps' wait results.  It sits right
        // before the first staging write, so that the tile's loads and
        // arithmetic overlap the previous store's read (the dual variant
        // writes its row image first and takes it here).
        auto staging_free = [&]() -> bool {
            if (threadIdx.x == 0) bulk_wait_group_read<kBufs - 1>();
            return bar_and(kStageBarrier, kThreads, ok != 0);
        };
        if constexpr (kStaged && kLateStageWait) {
        } else if constexpr (kStaged) {
            if (!staging_free()) break;
        } else if (!ok) {
            break;
        }

        // Column pair (64*chalf + 2*lane, +1), tokens 32*tbi .. 32*tbi+31, as
        // 32 register pairs {channel 2*lane, channel 2*lane+1}.
        uint64_t x[32];
        const uint32_t *tw = reinterpret_cast<const uint32_t *>(tiles + s * kTileBytes);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const uint32_t v = tw[(tbi * 32 + i) * (G::TC / 2) + chalf * 32 + lane];
            x[i] = pack2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
        }
        const uint32_t sbits = RAND ? signw[s * G::TOKEN_BLOCKS + tbi] : 0u;
        // This tile's staging buffer: the column image (codes box, scale
        // atoms), then with DUAL the row image.
        uint8_t *stc = staging + (it % kBufs) * kImages * S::kBytes;
        uint8_t *sts = stc + S::kCodeBytes;
        if constexpr (DUAL)
            dual_rows_staged<SR>(tw, t0, c0, a0, ar, stc + S::kBytes, stc + S::kBytes + S::kCodeBytes);
        __syncwarp();
        if (lane == 0 && ok) mbar_arrive(&empty[s]);
        if (DUAL && threadIdx.x == 0) {
            const int nt = tile + kColRing * gridDim.x;
            if (nt < total && mbar_wait(&empty[s], parity, a0.status, &abort_flag)) issue(nt, s);
        }

        if (ROTN > 0) {
            if (RAND) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    x[i] ^= ((sbits >> i) & 1u) ? 0x8000000080000000ull : 0ull;
            }
            fwht_pairs<ROTN>(x);
            if (SR || FMT >= kFmtNVAmax) {  // MXFP4 RNE folds the factor into its scale multiply
                const float cn = hadamard_norm<ROTN>();
                const uint64_t cc = pack2(cn, cn);
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] = mul2(x[i], cc);
            }
        }

        const int64_t tb = t0 + 32 * tbi;               // first token of this thread's block
        const int64_t c = c0 + 64 * chalf + 2 * lane;  // first of the thread's two channels
        if constexpr (FMT == kFmtNVAmax) {
            // Largest finite magnitude of the thread's 64 rotated values,
            // kept per operand across the warp's tiles; the warp's maxima
            // reach global memory once, at the end (one atomic per warp and
            // operand instead of one per tile on a single word).
            static_assert(!SR && !DUAL, "NVFP4: round to nearest, one direction");
            float m = second ? amax_run1 : amax_run0;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                float lo, hi;
                unpack2(x[i], lo, hi);
                lo = fabsf(lo);
                hi = fabsf(hi);
                m = fmaxf(m, lo <= 3.402823466e38f ? lo : 0.0f);
                m = fmaxf(m, hi <= 3.402823466e38f ? hi : 0.0f);
            }
            (second ? amax_run1 : amax_run0) = m;
            continue;
        }
        const int r0 = 64 * chalf + 2 * lane;                 // line of the tile (r0, r0 + 1)
        if constexpr (FMT == kFmtNV4) {
            static_assert(!SR && !DUAL, "NVFP4: round to nearest, one direction");
            if constexpr (kLateStageWait)
                if (!staging_free()) break;
            const float s_enc = nv_tensor_scale(__uint_as_float(*(second ? a1.amax : a0.amax)));
            float l[32], h[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) unpack2(x[i], l[i], h[i]);
            uint2 c00, c01, c10, c11;
            const uint32_t f00 = nv_encode_block16(l, s_enc, c00);
            const uint32_t f01 = nv_encode_block16(l + 16, s_enc, c01);
            const uint32_t f10 = nv_encode_block16(h, s_enc, c10);
            const uint32_t f11 = nv_encode_block16(h + 16, s_enc, c11);
            // 64-byte swizzle: 16-byte chunk j of line r at j ^ ((r >> 1) & 3).
            const int sw = tbi ^ ((r0 >> 1) & 3);
            *reinterpret_cast<uint4 *>(stc + r0 * 64 + sw * 16) = make_uint4(c00.x, c00.y, c01.x, c01.y);
            *reinterpret_cast<uint4 *>(stc + (r0 + 1) * 64 + sw * 16) =
                make_uint4(c10.x, c10.y, c11.x, c11.y);
            // Blocks 2*tbi and 2*tbi + 1 of 16: atom tbi / 2, bytes 2 * (tbi % 2) + {0, 1}.
            const int so = (tbi / 2) * 512 + 4 * (r0 / 32) + 2 * (tbi % 2);
            *reinterpret_cast<uint16_t *>(sts + so + (r0 % 32) * 16) =
                static_cast<uint16_t>(f00 | (f01 << 8));
            *reinterpret_cast<uint16_t *>(sts + so + ((r0 + 1) % 32) * 16) =
                static_cast<uint16_t>(f10 | (f11 << 8));
        } else {
        uint4 q0, q1;
        uint32_t s0, s1;
        if constexpr (FMT == kFmtMX8) {
            static_assert(ROTN == 0 && !RAND && !SR && !DUAL, "MXFP8: plain encode only");
            uint4 p0[2], p1[2];
            encode_pair_e4m3(x, p0, p1, s0, s1);
            if constexpr (kLateStageWait)
                if (!staging_free()) break;
            // 128-byte lines, 128-byte swizzle: chunk j of line r at j ^ (r & 7).
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                *reinterpret_cast<uint4 *>(stc + r0 * 128 + ((2 * tbi + k) ^ (r0 & 7)) * 16) = p0[k];
                *reinterpret_cast<uint4 *>(stc + (r0 + 1) * 128 + ((2 * tbi + k) ^ ((r0 + 1) & 7)) * 16) =
                    p1[k];
            }
        } else {
        if (SR) {
            const uint64_t tag = second ? a1.sr_tag : a0.sr_tag;
            float x0[32], x1[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) unpack2(x[i], x0[i], x1[i]);
            s0 = encode_block32_sr(x0, q0, a0.seed, tag, static_cast<uint64_t>(c * L + tb));
            s1 = encode_block32_sr(x1, q1, a0.seed, tag, static_cast<uint64_t>((c + 1) * L + tb));
        } else {
            encode_pair_rne<(ROTN > 0)>(x, ROTN > 0 ? hadamard_norm<ROTN>() : 1.0f, q0, q1, s0, s1);
        }
        if constexpr (kLateStageWait)
            if (!staging_free()) break;

        // 64-byte swizzle: 16-byte chunk j of line r at j ^ ((r >> 1) & 3).
        const int sw = tbi ^ ((r0 >> 1) & 3);
        *reinterpret_cast<uint4 *>(stc + r0 * 64 + sw * 16) = q0;
        *reinterpret_cast<uint4 *>(stc + (r0 + 1) * 64 + sw * 16) = q1;
        }
        // Scale atom: line r, block tbi at (r % 32) * 16 + (r / 32) * 4 + tbi.
        sts[(r0 % 32) * 16 + 4 * (r0 / 32) + tbi] = static_cast<uint8_t>(s0);
        sts[((r0 + 1) % 32) * 16 + 4 * (r0 / 32) + tbi] = static_cast<uint8_t>(s1);
        }
        (void)c;
        (void)tb;
        if constexpr (kStaged) {
            // Publish the staged tile to the async proxy, then one thread stores
            // it: the codes box at (token byte t0 / 2 or t0, line c0) -- the TMA
            // clips lines past `lines` and tokens past L -- and the scale
            // atom(s) of (line group c0 / 128, tokens t0 .. t0 + 127).
            fence_proxy_async_smem();
            asm volatile("bar.sync %0, %1;" ::"n"(kStageBarrier), "n"(kThreads) : "memory");
            if (threadIdx.x == 0) {
                const int64_t atom = (c0 / 128) * katoms + (FMT == kFmtNV4 ? t0 / 64 : t0 / 128);
                uint8_t *sdst = scales + atom * 512;
#if MXQ_L2_HINTS
                // The codes and scales are read next by the GEMM: keep them in L2.
                const uint64_t keep = l2_evict_last_policy();
                tma_store_2d_hint(second ? &cmap1 : &cmap0, stc,
                                  static_cast<int32_t>(FMT == kFmtMX8 ? t0 : t0 / 2),
                                  static_cast<int32_t>(c0), keep);
                if (MX_STORE_OK(sdst, S::kScaleBytes, scales, scales_bytes, a0.status))
                    bulk_store_hint(sdst, sts, S::kScaleBytes, keep);
#else
                tma_store_2d(second ? &cmap1 : &cmap0, stc,
                             static_cast<int32_t>(FMT == kFmtMX8 ? t0 : t0 / 2),
                             static_cast<int32_t>(c0));
                if (MX_STORE_OK(sdst, S::kScaleBytes, scales, scales_bytes, a0.status))
                    bulk_store(sdst, sts, S::kScaleBytes);
#endif
                if constexpr (DUAL) {
                    // The row image: tokens t0 .. t0+127 as lines, channels as
                    // the contraction (box at channel byte c0 / 2, line t0;
                    // cmap1 maps the row codes).  Tiles past the last 128-token
                    // scale group only hold padding rows.
                    if (t0 < (ar.lines + 127) / 128 * 128) {
                        tma_store_2d(&cmap1, stc + S::kBytes, static_cast<int32_t>(c0 / 2),
                                     static_cast<int32_t>(t0));
                        uint8_t *rdst = ar.scales + ((t0 / 128) * ar.katoms + c0 / 128) * 512;
                        if (MX_STORE_OK(rdst, 512, ar.scales, ar.scales_bytes, a0.status))
                            bulk_store(rdst, stc + S::kBytes + S::kCodeBytes, 512);
                    }
                }
                bulk_commit_group();
            }
        }
    }
    if constexpr (FMT == kFmtNVAmax) {
        const unsigned int w0 = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(amax_run0));
        const unsigned int w1 = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(amax_run1));
        if (lane == 0 && w0 != 0u) atomicMax(a0.amax, w0);
        if (lane == 0 && w1 != 0u && a1.num_tiles > 0) atomicMax(a1.amax, w1);
    }
    // Every store has completed (global writes included) before the CTA leaves.
    if (kStaged && threadIdx.x == 0) bulk_wait_group_0();
}

// Column-wise encode for Hadamard sizes 64, 128 and 256.  Each thread owns
// one channel x 64 consecutive tokens of the tile, held as 32 register pairs
// {token i, token i+32}: butterfly strides 1..16 run on the pairs, stride 32
// inside each pair, and strides 64 and 128 pair this thread with the lane that
// holds the same channel's neighbouring 64 tokens (one warp shuffle per
// element per stage).  The two MX blocks of the segment are the pairs' low and
// high halves.  No shared-memory exchange and no CTA barrier is needed.
template <int ROTN>
struct WideTile {
    // 128 x 128 tiles; a 256-token Hadamard block needs 256 tokens x 64 channels.
    static constexpr int TT = ROTN == 256 ? 256 : 128;  // tokens per tile
    static constexpr int TC = 32768 / (2 * TT);           // channels per tile
    static constexpr int LPC = ROTN / 64;                 // lanes per channel
    static constexpr int CPW = 32 / LPC;                  // channels per warp (ROTN > 64)
};

// Ring depth and output path of the wide kernel, per Hadamard size (measured
// on the down_proj operands): size 64 gains from a 3-deep ring and the staged
// output (84.6 -> ~79 us); sizes 128 and 256, whose cross-lane stages
// dominate, are fastest with a 2-deep ring and direct stores.
#ifndef MXQ_WIDE_STAGE_MAX
#define MXQ_WIDE_STAGE_MAX 64
#endif
template <bool DUAL, int ROTN>
struct WideRing {
    static constexpr int kRing = !DUAL && ROTN == 64 ? 3 : 2;
};

template <int ROTN, bool RAND, bool SR, bool DUAL>
__global__ void __launch_bounds__(kThreads, SR ? 1 : kColMinBlocks) mxq_colwise_wide_kernel(
    const __grid_constant__ CUtensorMap map0, const __grid_constant__ CUtensorMap map1,
    const __grid_constant__ CUtensorMap cmap0, const __grid_constant__ CUtensorMap cmap1,
    const QuantArgs a0, const QuantArgs a1, const QuantArgs ar) {
    static_assert(ROTN == 64 || ROTN == 128 || ROTN == 256, "sizes 64..256 only");
    using G = WideTile<ROTN>;
    // Hadamard 64 writes through the staging image of the column kernel (one
    // TMA box of codes, one scale atom per 128 x 128 tile); 128 and 256 store
    // directly (see WideRing).
    constexpr bool kStagedW = !DUAL && G::TT == 128 && ROTN <= MXQ_WIDE_STAGE_MAX;
    constexpr int kStages = WideRing<DUAL, ROTN>::kRing;
    using S = ColStage<kFmtMX4>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *tiles = smem;                                   // kStages x 32 KB
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kTileBytes);
    uint64_t *empty = full + kStages;
    // Random-sign words of each stage's tile (one 64-bit word per 64-token
    // segment), written by the issuing thread before it arms the stage.
    uint64_t *signw = empty + kStages;
    uint8_t *stc = smem + kStages * kTileBytes + 1024;       // staging image (kStagedW)
    uint8_t *sts = stc + S::kCodeBytes;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // This thread's channel of the tile and its 64-token segment.
    const int ch = ROTN == 64 ? (warp % 4) * 32 + lane : warp * G::CPW + lane % G::CPW;
    const int seg = ROTN == 64 ? warp / 4 : lane / G::CPW;
    const int total = a0.num_tiles + a1.num_tiles;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kThreads / 32);
        }
        abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&map0);
        if (a1.num_tiles > 0) prefetch_tmap(&map1);
        if (kStagedW) {
            prefetch_tmap(&cmap0);
            if (a1.num_tiles > 0) prefetch_tmap(&cmap1);
        }
    }
    __syncthreads();
    griddep_wait();
    griddep_launch_dependents();

    auto issue = [&](int tile, int s) {
        const bool second = tile >= a0.num_tiles;
        const int lt = second ? tile - a0.num_tiles : tile;
        const int inner = second ? a1.tiles_inner : a0.tiles_inner;
        if constexpr (RAND) {
            // Sign word of each 64-token segment: two 32-bit words of its 128-bit block.
            static_assert(G::TT % 128 == 0, "tiles start on a sign block");
            const int64_t t0 = static_cast<int64_t>(lt / inner) * G::TT;
#pragma unroll
            for (int h = 0; h < G::TT / 128; ++h) {
                uint32_t o[4];
                sign_block128(a0.seed, static_cast<uint64_t>(t0 / 128 + h), o);
                signw[s * 4 + 2 * h] = o[0] | (static_cast<uint64_t>(o[1]) << 32);
                signw[s * 4 + 2 * h + 1] = o[2] | (static_cast<uint64_t>(o[3]) << 32);
            }
        }
        mbar_arrive_expect_tx(&full[s], kTileBytes);
        tma_load_2d(tiles + s * kTileBytes, second ? &map1 : &map0, &full[s], (lt % inner) * G::TC,
                    (lt / inner) * G::TT);
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            const int tile = blockIdx.x + s * gridDim.x;
            if (tile < total) issue(tile, s);
        }
    }

    for (int it = 0;; ++it) {
        const int tile = blockIdx.x + it * gridDim.x;
        if (tile >= total) break;
        const int s = it % kStages;
        const uint32_t parity = (it / kStages) & 1u;
        const bool second = tile >= a0.num_tiles;
        const int lt = second ? tile - a0.num_tiles : tile;
        const int inner = second ? a1.tiles_inner : a0.tiles_inner;
        const int64_t L = second ? a1.L : a0.L;
        const int64_t lines = second ? a1.lines : a0.lines;
        const int64_t katoms = second ? a1.katoms : a0.katoms;
        uint8_t *const codes = second ? a1.codes : a0.codes;
        uint8_t *const scales = second ? a1.scales : a0.scales;
        const size_t codes_bytes = second ? a1.codes_bytes : a0.codes_bytes;
        const size_t scales_bytes = second ? a1.scales_bytes : a0.scales_bytes;
        (void)codes_bytes;
        (void)scales_bytes;
        const int64_t t0 = static_cast<int64_t>(lt / inner) * G::TT;
        const int64_t c0 = static_cast<int64_t>(lt % inner) * G::TC;

        int ok = 1;
        if (lane == 0) ok = mbar_wait(&full[s], parity, a0.status, &abort_flag) ? 1 : 0;
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if constexpr (kStagedW) {
            // The staging image was last stored one tile ago; the barrier also
            // ANDs the warps' wait results (see the column kernel).
            if (threadIdx.x == 0) bulk_wait_group_read<0>();
            if (!bar_and(kStageBarrier, kThreads, ok != 0)) break;
        } else if (!ok) {
            break;
        }

        uint64_t x[32];
        const uint16_t *th = reinterpret_cast<const uint16_t *>(tiles + s * kTileBytes);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const uint32_t lo = th[(seg * 64 + i) * G::TC + ch];
            const uint32_t hi = th[(seg * 64 + 32 + i) * G::TC + ch];
            x[i] = pack2(__uint_as_float(lo << 16), __uint_as_float(hi << 16));
        }
        const uint64_t sw = RAND ? signw[s * 4 + seg] : 0ull;
        if (DUAL)
            dual_rows<G::TC, SR>(reinterpret_cast<const uint32_t *>(th), t0, c0, a0, ar);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (threadIdx.x == 0) {
            const int nt = tile + kStages * gridDim.x;
            if (nt < total && mbar_wait(&empty[s], parity, a0.status, &abort_flag)) issue(nt, s);
        }

        const int64_t tb = t0 + 64 * seg;  // first token of this thread's segment
        if (RAND) {
            // The segment's two 32-bit sign words (tokens tb .. tb+31, tb+32 .. tb+63).
            const uint32_t blo = static_cast<uint32_t>(sw), bhi = static_cast<uint32_t>(sw >> 32);
#pragma unroll
            for (int i = 0; i < 32; ++i)
                x[i] ^= (((blo >> i) & 1u) ? 0x80000000ull : 0ull) |
                        (((bhi >> i) & 1u) ? 0x8000000000000000ull : 0ull);
        }
        fwht_pairs<64>(x);  // strides 1 .. 16
#pragma unroll
        for (int i = 0; i < 32; ++i) {  // stride 32: within each pair
            float a, b;
            unpack2(x[i], a, b);
            x[i] = pack2(__fadd_rn(a, b), __fsub_rn(a, b));
        }
#pragma unroll
        for (int m = 1; 64 * m < ROTN; m <<= 1) {  // strides 64, 128: across lanes
            // The lower segment takes o + x, the upper one o - x = o + (-x):
            // the same fp32 results as the canonical (a + b, a - b).
            // (Selecting between the two results measured faster for 128,
            // the sign flip for 256; both give identical values.)
            const bool lower = (seg & m) == 0;
            const uint64_t neg = lower ? 0ull : 0x8000000080000000ull;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, static_cast<unsigned long long>(x[i]),
                                                   m * G::CPW);
                if constexpr (ROTN == 128)
                    x[i] = lower ? add2(x[i], o) : sub2(o, x[i]);
                else
                    x[i] = add2(o, x[i] ^ neg);
            }
        }

        const int64_t c = c0 + ch;
        uint4 q0, q1;
        uint32_t s0, s1;
        if (SR) {
            const float cn = hadamard_norm<ROTN>();
            const uint64_t cc = pack2(cn, cn);
            float x0[32], x1[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) unpack2(mul2(x[i], cc), x0[i], x1[i]);
            const uint64_t tag = second ? a1.sr_tag : a0.sr_tag;
            uint32_t u[32];
            sr_draws32(a0.seed, tag, static_cast<uint64_t>(c * L + tb), u);
            s0 = encode_block32<true>(x0, q0, u);
            sr_draws32(a0.seed, tag, static_cast<uint64_t>(c * L + tb + 32), u);
            s1 = encode_block32<true>(x1, q1, u);
        } else {
            encode_pair_rne<true>(x, hadamard_norm<ROTN>(), q0, q1, s0, s1);
        }
        if constexpr (kStagedW) {
            // Line ch of the codes box: chunks 2*seg and 2*seg + 1 (64-byte
            // swizzle); scale atom bytes of blocks 2*seg, 2*seg + 1.
            const int sx = (ch >> 1) & 3;
            *reinterpret_cast<uint4 *>(stc + ch * 64 + ((2 * seg) ^ sx) * 16) = q0;
            *reinterpret_cast<uint4 *>(stc + ch * 64 + ((2 * seg + 1) ^ sx) * 16) = q1;
            *reinterpret_cast<uint16_t *>(sts + (ch % 32) * 16 + (ch / 32) * 4 + 2 * seg) =
                static_cast<uint16_t>(s0 | (s1 << 8));
            fence_proxy_async_smem();
            asm volatile("bar.sync %0, %1;" ::"n"(kStageBarrier), "n"(kThreads) : "memory");
            if (threadIdx.x == 0) {
                tma_store_2d(second ? &cmap1 : &cmap0, stc, static_cast<int32_t>(t0 / 2),
                             static_cast<int32_t>(c0));
                uint8_t *sdst = scales + ((c0 / 128) * katoms + t0 / 128) * 512;
                if (MX_STORE_OK(sdst, 512, scales, scales_bytes, a0.status))
                    bulk_store(sdst, sts, 512);
                bulk_commit_group();
            }
            continue;
        }
        if (tb < L && c < lines) {
            uint8_t *d = codes + c * (L / 2) + tb / 2;
            if (MX_STORE_OK(d, 32, codes, codes_bytes, a0.status)) {
                st_global_16(d, q0);
                st_global_16(d + 16, q1);
            }
        }
        const int64_t kb = tb / 32;
        uint8_t *e0 = scales + scale_offset(c, kb, katoms), *e1 = scales + scale_offset(c, kb + 1, katoms);
        if (MX_STORE_OK(e0, 1, scales, scales_bytes, a0.status)) *e0 = static_cast<uint8_t>(s0);
        if (MX_STORE_OK(e1, 1, scales, scales_bytes, a0.status)) *e1 = static_cast<uint8_t>(s1);
    }
    if (kStagedW && threadIdx.x == 0) bulk_wait_group_0();
}

// ---------------------------------------------------------------- rowwise
template <int ROTN, bool RAND, bool SR>
__global__ void __launch_bounds__(kThreads) mxq_rowwise_kernel(const __grid_constant__ CUtensorMap src_map,
                                                               const QuantArgs p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned base, kept as a shared-space pointer (offset arithmetic
    // only) so that the compiler emits shared-memory loads.
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
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
    griddep_wait();
    griddep_launch_dependents();

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
                // blocks blk_a and blk_a + 4: word blk_a of the tile's two 128-bit sign blocks
                uint32_t oa[4], ob[4];
                sign_block128(p.seed, static_cast<uint64_t>(col0 / 128), oa);
                sign_block128(p.seed, static_cast<uint64_t>(col0 / 128 + 1), ob);
                apply_signs(xa, blk_a == 0 ? oa[0] : blk_a == 1 ? oa[1] : blk_a == 2 ? oa[2] : oa[3]);
                apply_signs(xb, blk_a == 0 ? ob[0] : blk_a == 1 ? ob[1] : blk_a == 2 ? ob[2] : ob[3]);
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
            uint8_t *da = p.codes + row * (p.L / 2) + ca / 2, *db = p.codes + row * (p.L / 2) + cb / 2;
            if (ca < p.L && MX_STORE_OK(da, 16, p.codes, p.codes_bytes, p.status)) st_global_16(da, qa);
            if (cb < p.L && MX_STORE_OK(db, 16, p.codes, p.codes_bytes, p.status)) st_global_16(db, qb);
        }
        sstage[stage_offset(r, blk_a)] = static_cast<uint8_t>(sa);
        sstage[stage_offset(r, blk_a + 4)] = static_cast<uint8_t>(sb);
        __syncthreads();
        flush_scales(sstage, p, row0, col0);
    }
}

// ---------------------------------------------------------------- dispatch
template <typename Kern, typename... Args>
cudaError_t launch_persistent_n(Kern kernel, int threads, int num_tiles, size_t smem,
                                const DeviceInfo &dev, cudaStream_t stream, Args... args) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int grid = num_tiles < dev.sm_count * per_sm ? num_tiles : dev.sm_count * per_sm;
    // Programmatic dependent launch: the kernel may start while the stream's
    // previous kernel finishes; it waits for it (griddep_wait) before touching
    // global memory.
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, args...);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename Kern, typename... Args>
cudaError_t launch_persistent(Kern kernel, int num_tiles, size_t smem, const DeviceInfo &dev,
                              cudaStream_t stream, Args... args) {
    return launch_persistent_n(kernel, kThreads, num_tiles, smem, dev, stream, args...);
}

struct Operands {
    CUtensorMap map0, map1;
    CUtensorMap cmap0, cmap1;  // codes outputs (column encodes that stage their tiles)
    QuantArgs a0, a1;
    QuantArgs ar;  // row-direction output of a dual encode
    bool dual = false;
};

template <int FMT, bool DUAL = false>
constexpr size_t col_smem() {
    return (DUAL ? 2 : ColStage<FMT>::kRing) * kTileBytes + 1024 + 1024 +
           (DUAL ? 1 : kStageBufs) * (DUAL ? 2 : 1) * ColStage<FMT>::kBytes;
}

template <bool COLWISE, int ROTN, bool RAND>
cudaError_t launch_rot(bool sr, const Operands &o, const DeviceInfo &dev, cudaStream_t stream) {
    if constexpr (COLWISE && ROTN >= 64) {
        // Ring tiles, the barrier region and (128-token tiles) one staging image.
        const size_t smem = WideRing<false, ROTN>::kRing * kTileBytes + 1024 + 1024 +
                            (ROTN <= MXQ_WIDE_STAGE_MAX && ROTN < 256 ? ColStage<kFmtMX4>::kBytes
                                                                       : 0);
        const size_t dsmem = WideRing<true, ROTN>::kRing * kTileBytes + 1024 + 1024;
        const int n = o.a0.num_tiles + o.a1.num_tiles;
        if (o.dual)
            return sr ? launch_persistent(mxq_colwise_wide_kernel<ROTN, RAND, true, true>, n, dsmem,
                                          dev, stream, o.map0, o.map1, o.cmap0, o.cmap1, o.a0,
                                          o.a1, o.ar)
                      : launch_persistent(mxq_colwise_wide_kernel<ROTN, RAND, false, true>, n,
                                          dsmem, dev, stream, o.map0, o.map1, o.cmap0, o.cmap1,
                                          o.a0, o.a1, o.ar);
        return sr ? launch_persistent(mxq_colwise_wide_kernel<ROTN, RAND, true, false>, n, smem,
                                      dev, stream, o.map0, o.map1, o.cmap0, o.cmap1, o.a0, o.a1,
                                      o.ar)
                  : launch_persistent(mxq_colwise_wide_kernel<ROTN, RAND, false, false>, n, smem,
                                      dev, stream, o.map0, o.map1, o.cmap0, o.cmap1, o.a0, o.a1,
                                      o.ar);
    }
    else if constexpr (COLWISE) {
        const size_t smem = col_smem<kFmtMX4>();
        const size_t dsmem = col_smem<kFmtMX4, true>();
        const int n = o.a0.num_tiles + o.a1.num_tiles;
        if (o.dual)
            return sr ? launch_persistent(mxq_colwise_kernel<ROTN, RAND, true, true>, n, dsmem,
                                          dev, stream, o.map0, o.map1, o.cmap0, o.cmap1, o.a0,
                                          o.a1, o.ar)
                      : launch_persistent(mxq_colwise_kernel<ROTN, RAND, false, true>, n, dsmem,
                                          dev, stream, o.map0, o.map1, o.cmap0, o.cmap1, o.a0,
                                          o.a1, o.ar);
        return sr ? launch_persistent_n(mxq_colwise_kernel<ROTN, RAND, true, false>,
                                        kColProducerThreads, n, smem, dev, stream, o.map0, o.map1,
                                        o.cmap0, o.cmap1, o.a0, o.a1, o.ar)
                  : launch_persistent_n(mxq_colwise_kernel<ROTN, RAND, false, false>,
                                        kColProducerThreads, n, smem, dev, stream, o.map0, o.map1,
                                        o.cmap0, o.cmap1, o.a0, o.a1, o.ar);
    }
    const size_t smem = kStages * kTileBytes + 1024 + 1024;
    return sr ? launch_persistent(mxq_rowwise_kernel<ROTN, RAND, true>, o.a0.num_tiles, smem, dev,
                                  stream, o.map0, o.a0)
              : launch_persistent(mxq_rowwise_kernel<ROTN, RAND, false>, o.a0.num_tiles, smem,
                                  dev, stream, o.map0, o.a0);
}

template <bool COLWISE>
cudaError_t launch_dir(int rot, int rot_block, bool sr, const Operands &o, const DeviceInfo &dev,
                       cudaStream_t stream) {
    if (rot == 0) return launch_rot<COLWISE, 0, false>(sr, o, dev, stream);
    const bool rnd = rot == 2;
#define MX_ROT_CASE(N)                                                                      \
    case N:                                                                                 \
        return rnd ? launch_rot<COLWISE, N, true>(sr, o, dev, stream)                       \
                   : launch_rot<COLWISE, N, false>(sr, o, dev, stream);
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

// Fills the per-operand arguments (and tensor map) of one encode.
bool prepare_operand(const void *src, int64_t rows, int64_t cols, bool colwise, int col_tt,
                     uint64_t seed, uint64_t sr_tag, void *codes, void *scales,
                     const DeviceInfo &dev, CUtensorMap *map, QuantArgs *a, int fmt = kFmtMX4,
                     CUtensorMap *cmap = nullptr) {
    *a = QuantArgs{};
    a->L = colwise ? rows : cols;
    a->lines = colwise ? cols : rows;
    const bool nv = fmt == kFmtNV4 || fmt == kFmtNVAmax;
    a->katoms = nv ? nv_scale_katoms(a->L) : scale_katoms(a->L);
    a->codes = static_cast<uint8_t *>(codes);
    a->scales = static_cast<uint8_t *>(scales);
    a->codes_bytes =
        static_cast<size_t>(a->lines) * static_cast<size_t>(fmt == kFmtMX8 ? a->L : a->L / 2);
    a->scales_bytes = static_cast<size_t>(128 * scale_groups(a->lines)) *
                      static_cast<size_t>(4 * a->katoms);
    a->seed = seed;
    a->sr_tag = sr_tag;
    a->status = dev.status;
    // Tiles cover the padded scale layout: lines to a multiple of 128 and the
    // contraction dim to a multiple of 256, so padding scale bytes get zeros.
    if (colwise) {
        const int col_tc = 32768 / (2 * col_tt);
        const int64_t line_tiles = scale_groups(a->lines) * (128 / col_tc);
        const int64_t k_tiles = ((a->L + 255) / 256) * (256 / col_tt);
        if (line_tiles * k_tiles > 0x3FFFFFFF) return false;
        a->num_tiles = static_cast<int>(line_tiles * k_tiles);
        a->tiles_inner = static_cast<int>(line_tiles);
        if (cmap != nullptr) {
            // The staged codes box of a 128-token x 128-line tile: 64 B (128 B
            // for MXFP8) of each line, swizzled like the staging writes.
            const bool f8 = fmt == kFmtMX8;
            const uint64_t row = static_cast<uint64_t>(f8 ? a->L : a->L / 2);
            if (!encode_tmap_2d(cmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, row,
                                static_cast<uint64_t>(a->lines), row, f8 ? 128 : 64, 128,
                                f8 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
                return false;
        }
        return encode_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, src, cols, rows, cols * 2,
                              col_tc, col_tt, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    const int64_t line_tiles = scale_groups(a->lines) * 2;  // 64 lines per tile
    const int64_t k_tiles = (a->L + 255) / 256;
    if (line_tiles * k_tiles > 0x3FFFFFFF) return false;
    a->num_tiles = static_cast<int>(line_tiles * k_tiles);
    a->tiles_inner = static_cast<int>(k_tiles);
    return encode_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, src, cols, rows, cols * 2, 64, 64,
                          CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

cudaError_t launch_quantize(const void *src, int64_t rows, int64_t cols, int contract, int rot,
                            int rot_block, int rnd, uint64_t seed, uint64_t sr_tag,
                            void *codes, void *scales, const DeviceInfo &dev,
                            cudaStream_t stream) {
    const bool colwise = contract == 0;
    Operands o;
    const int tt = (rot != 0 && rot_block == 256) ? 256 : 128;
    if (!prepare_operand(src, rows, cols, colwise, tt, seed, sr_tag, codes, scales, dev, &o.map0,
                         &o.a0, kFmtMX4, colwise ? &o.cmap0 : nullptr))
        return cudaErrorInvalidValue;
    o.map1 = o.map0;
    o.cmap1 = o.cmap0;
    o.a1 = QuantArgs{};
    o.ar = QuantArgs{};
    if (colwise) return launch_dir<true>(rot, rot_block, rnd == 1, o, dev, stream);
    return launch_dir<false>(rot, rot_block, rnd == 1, o, dev, stream);
}

cudaError_t launch_quantize_pair_colwise(const void *src0, int64_t rows0, int64_t cols0,
                                         const void *src1, int64_t rows1, int64_t cols1, int rot,
                                         int rot_block, int rnd, uint64_t seed, void *codes0,
                                         void *scales0, void *codes1, void *scales1,
                                         const DeviceInfo &dev, cudaStream_t stream) {
    Operands o;
    const int tt = (rot != 0 && rot_block == 256) ? 256 : 128;
    if (!prepare_operand(src0, rows0, cols0, true, tt, seed, 1, codes0, scales0, dev, &o.map0,
                         &o.a0, kFmtMX4, &o.cmap0) ||
        !prepare_operand(src1, rows1, cols1, true, tt, seed, 2, codes1, scales1, dev, &o.map1,
                         &o.a1, kFmtMX4, &o.cmap1))
        return cudaErrorInvalidValue;
    o.ar = QuantArgs{};
    return launch_dir<true>(rot, rot_block, rnd == 1, o, dev, stream);
}

cudaError_t launch_quantize_dual(const void *src, int64_t rows, int64_t cols, int rot,
                                 int rot_block, int rnd, uint64_t seed, void *codes_t,
                                 void *scales_t, void *codes_n, void *scales_n,
                                 const DeviceInfo &dev, cudaStream_t stream) {
    Operands o;
    const int tt = (rot != 0 && rot_block == 256) ? 256 : 128;
    if (!prepare_operand(src, rows, cols, true, tt, seed, 1, codes_t, scales_t, dev, &o.map0,
                         &o.a0, kFmtMX4, &o.cmap0))
        return cudaErrorInvalidValue;
    o.map1 = o.map0;
    // The column kernel's dual variant has no second operand: cmap1 maps the
    // row-direction codes [rows][cols / 2] in 128-token x 64-byte boxes.
    if (!encode_tmap_2d(&o.cmap1, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes_n,
                        static_cast<uint64_t>(cols / 2), static_cast<uint64_t>(rows),
                        static_cast<uint64_t>(cols / 2), 64, 128, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    o.a1 = QuantArgs{};
    o.ar = QuantArgs{};
    o.ar.L = cols;
    o.ar.lines = rows;
    o.ar.katoms = scale_katoms(cols);
    o.ar.codes = static_cast<uint8_t *>(codes_n);
    o.ar.scales = static_cast<uint8_t *>(scales_n);
    o.ar.codes_bytes = static_cast<size_t>(rows) * static_cast<size_t>(cols / 2);
    o.ar.scales_bytes = static_cast<size_t>(128 * scale_groups(rows)) *
                        static_cast<size_t>(4 * scale_katoms(cols));
    o.ar.seed = seed;
    o.ar.sr_tag = 1;
    o.ar.status = dev.status;
    o.dual = true;
    return launch_dir<true>(rot, rot_block, rnd == 1, o, dev, stream);
}

cudaError_t launch_quantize_mxfp8_colwise(const void *src0, int64_t rows0, int64_t cols0,
                                          const void *src1, int64_t rows1, int64_t cols1,
                                          void *codes0, void *scales0, void *codes1,
                                          void *scales1, const DeviceInfo &dev,
                                          cudaStream_t stream) {
    Operands o;
    if (!prepare_operand(src0, rows0, cols0, true, 128, 0, 1, codes0, scales0, dev, &o.map0,
                         &o.a0, kFmtMX8, &o.cmap0))
        return cudaErrorInvalidValue;
    o.map1 = o.map0;
    o.cmap1 = o.cmap0;
    o.a1 = QuantArgs{};
    if (src1 != nullptr &&
        !prepare_operand(src1, rows1, cols1, true, 128, 0, 2, codes1, scales1, dev, &o.map1,
                         &o.a1, kFmtMX8, &o.cmap1))
        return cudaErrorInvalidValue;
    o.ar = QuantArgs{};
    return launch_persistent_n(mxq_colwise_kernel<0, false, false, false, kFmtMX8>,
                               kColProducerThreads, o.a0.num_tiles + o.a1.num_tiles,
                               col_smem<kFmtMX8>(), dev, stream, o.map0, o.map1, o.cmap0, o.cmap1,
                               o.a0, o.a1, o.ar);
}

namespace {
template <int ROTN, bool RAND>
cudaError_t launch_nv_passes(const Operands &o, const DeviceInfo &dev, cudaStream_t stream) {
    const int n = o.a0.num_tiles + o.a1.num_tiles;
    // The amax pass stores nothing: no staging buffers.
    cudaError_t e = launch_persistent_n(mxq_colwise_kernel<ROTN, RAND, false, false, kFmtNVAmax>,
                                        kColProducerThreads, n,
                                        ColStage<kFmtNVAmax>::kRing * kTileBytes + 1024 + 1024,
                                        dev, stream, o.map0, o.map1, o.cmap0, o.cmap1, o.a0, o.a1,
                                        o.ar);
    if (e != cudaSuccess) return e;
    return launch_persistent_n(mxq_colwise_kernel<ROTN, RAND, false, false, kFmtNV4>,
                               kColProducerThreads, n, col_smem<kFmtNV4>(), dev, stream, o.map0,
                               o.map1, o.cmap0, o.cmap1, o.a0, o.a1, o.ar);
}
}  // namespace

cudaError_t launch_quantize_nvfp4_colwise(const void *src0, int64_t rows0, int64_t cols0,
                                          const void *src1, int64_t rows1, int64_t cols1, int rot,
                                          int rot_block, uint64_t seed, void *codes0,
                                          void *scales0, void *codes1, void *scales1,
                                          float *amax, const DeviceInfo &dev,
                                          cudaStream_t stream) {
    Operands o;
    if (!prepare_operand(src0, rows0, cols0, true, 128, seed, 1, codes0, scales0, dev, &o.map0,
                         &o.a0, kFmtNV4, &o.cmap0))
        return cudaErrorInvalidValue;
    o.a0.amax = reinterpret_cast<unsigned int *>(amax);
    o.map1 = o.map0;
    o.cmap1 = o.cmap0;
    o.a1 = QuantArgs{};
    if (src1 != nullptr) {
        if (!prepare_operand(src1, rows1, cols1, true, 128, seed, 2, codes1, scales1, dev, &o.map1,
                             &o.a1, kFmtNV4, &o.cmap1))
            return cudaErrorInvalidValue;
        o.a1.amax = reinterpret_cast<unsigned int *>(amax + 1);
    }
    o.ar = QuantArgs{};
    cudaError_t e = cudaMemsetAsync(amax, 0, (src1 != nullptr ? 2 : 1) * sizeof(float), stream);
    if (e != cudaSuccess) return e;
    if (rot == 0) return launch_nv_passes<0, false>(o, dev, stream);
    if (rot_block == 16) return rot == 2 ? launch_nv_passes<16, true>(o, dev, stream)
                                         : launch_nv_passes<16, false>(o, dev, stream);
    if (rot_block == 32) return rot == 2 ? launch_nv_passes<32, true>(o, dev, stream)
                                         : launch_nv_passes<32, false>(o, dev, stream);
    return cudaErrorInvalidValue;
}

}  // namespace mx
