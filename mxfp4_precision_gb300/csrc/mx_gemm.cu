// mx_gemm.cu -- block-scaled MXFP4 GEMM on the sm_103a tensor cores.
//
// C[M][N] (fp32) = A . B^T with A, B MXFP4-encoded along the contraction
// dimension K: the Fprop, Dgrad and Wgrad GEMMs of "Neue Studie von AMD
// durchbricht die bestehende Erkenntnis" (eu.36kr.com), section
// "Fehlerdiagnoseexperiment", run on native FP4 tensor cores with fp32
// accumulation.
//
// Design (persistent; one 2-CTA cluster per SM pair; 256 x 256 output tiles):
//   A tile's 256 rows and B tile's 256 rows are split 128/128 between the two
//   CTAs of the pair; tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 64) is
//   issued by one thread of the even CTA and leaves rows 0..127 of the fp32
//   tile in the even CTA's tensor memory and rows 128..255 in the odd one's.
//   Each CTA thereby reads only half of B from its own shared memory.
//
//   warp 0       operand producer: this CTA's 128 rows of A and of B, two
//                256-wide K sub-tiles (128-byte swizzle) per stage, into a
//                3-stage shared-memory ring.  Both CTAs' operand loads
//                complete on the even CTA's stage barrier.
//   warp 2       scale producer: the stages' block scales (this CTA's A rows;
//                all 256 B rows) into a ring of their own, for the MX formats
//                two slots deeper than the operand ring, so that they already
//                wait in shared memory when a stage's tensor-memory scale
//                columns come free.
//   warp 1       tensor-memory allocation (pair); in the even CTA, the MMA
//                issuer: per stage, 8 MMAs and one commit that frees the
//                stage in both CTAs.
//   warps 4..7   scale writers: once the MMAs that last read the stage's
//                scale columns have finished, warp 4+q moves the block scales
//                from shared memory into lane quarter q of its CTA's tensor
//                memory with tcgen05.st (copy instructions would enter the MMA
//                pipe and serialise with the MMAs) and arrives on the stage's
//                full barrier, which thus covers operands and scales: the MMA
//                thread waits on one barrier per stage.
//   warps 8..15  epilogue: tcgen05.ld the CTA's 128 x 256 accumulator half
//                (each warp one 32-lane quarter x 128 columns) into registers,
//                release tensor memory to the MMA thread at once, then store
//                fp32 rows.  The stores are spread over the next tile's main
//                loop (one 32-byte store per thread per loaded stage), so that
//                the output of all SMs does not reach L2 in one burst that
//                would stall the operand loads.
//   The producer, MMA and scale-writer warpgroups give up registers
//   (setmaxnreg) so that the epilogue can hold 128 values per thread.
// Every wait is bounded (see mx_ptx.cuh); a timeout records an error and the
// CTA unwinds without faulting.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>
#include <vector>

#include "mx_encode.cuh"
#include "mx_internal.h"
#include "mx_ptx.cuh"

namespace mx {
namespace {

constexpr int kTile = 256;                        // output tile (rows and columns) per pair
constexpr int kHalf = 128;                        // rows of A / of B per CTA
constexpr int kBKBytes = 128;                     // 256 FP4 per row per K sub-tile
constexpr int kMaxStages = 5;
constexpr int kMaxSFRing = 7;
constexpr int kWriterWarp0 = 4;                   // warps 4..7: scale writers
constexpr int kEpiWarp0 = 8;                      // warps 8..15: epilogue
constexpr int kEpiWarps = 8;
constexpr int kEncWarp0 = 16;                     // fused launch: warps 16..23 encode
constexpr int kEncWarps = 8;
// Threads and register split (setmaxnreg) of the two variants.  GEMM alone:
// 512 threads x 128 launch registers = 256 x kRegsLow (producers, MMA, scale
// writers) + 256 x kRegsHigh (epilogue, whole accumulator half in registers).
// Fused Wgrad: 768 x 80 = 256 x 48 + 256 x 96 (epilogue, two passes of 64
// columns) + 256 x 96 (encoder warps).
template <bool FUSED>
struct Variant {
    static constexpr int kThreads = FUSED ? 768 : 512;
    static constexpr int kLaunchRegs = FUSED ? 80 : 128;
    static constexpr int kRegsLow = FUSED ? 48 : 56;
    static constexpr int kRegsHigh = FUSED ? 96 : 200;
    static_assert(256 * kRegsLow + (kThreads - 256) * kRegsHigh <= kThreads * kLaunchRegs,
                  "register split fits the launch");
    static_assert(kThreads * kLaunchRegs <= 65536, "launch registers fit the SM");
};
constexpr uint32_t kSubBytes = kHalf * kBKBytes;  // 16 KB: 128 rows x one K sub-tile
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;                    // accumulator: columns [0, 256)
constexpr uint32_t kSFCol = 256;                   // scale slots from column 256
// Element formats and the stage geometry each needs.  A 128-byte K sub-tile
// row holds 256 E2M1 (MXFP4, NVFP4) or 128 E4M3 (MXFP8).  Scales arrive as
// 512-byte atoms of 128 rows: two per sub-tile for MXFP4 (E8M0 per 32), one
// for MXFP8, four for NVFP4 (UE4M3 per 16).  In tensor memory a sub-tile's
// scales take 24 columns (MX: A 8, B 16) or 48 (NVFP4: 4 per MMA for A, 8
// for B), so NVFP4 stages hold one sub-tile and five stages fit beside the
// accumulator; the MX formats run three stages of two sub-tiles.
constexpr int kFmtMX4 = 0, kFmtMX8 = 1, kFmtNV4 = 2;
template <int FMT>
struct Elem {
    static constexpr bool kNV = FMT == kFmtNV4;
    static constexpr int kSubK = FMT == kFmtMX8 ? 128 : 256;   // elements per sub-tile row
    static_assert(kSubK == 128 || kSubK == 256, "128-byte sub-tile rows");
    static constexpr int kAtoms = FMT == kFmtMX8 ? 1 : kNV ? 4 : 2;
    static constexpr uint32_t kSFBytes = 512u * kAtoms;         // scale bytes per 128 rows
    static constexpr int kKSub = kNV ? 1 : 2;                   // sub-tiles per stage
    static constexpr int kStages = kNV ? 5 : 3;
    static constexpr uint32_t kSFSub = kNV ? 2048 : 1024;       // scale room per sub-tile
    static constexpr uint32_t kOffA = 0;
    static constexpr uint32_t kOffB = kKSub * kSubBytes;
    static constexpr uint32_t kStageBytes = 2 * kKSub * kSubBytes;         // 64 KB / 32 KB
    // Scales travel in a ring of their own (A's row group, then B's two).
    // MX: two slots deeper than the operand ring, so that they are in
    // shared memory before the stage's tensor-memory scale columns come
    // free.  NVFP4 (four MMAs per stage, twice the scale columns per MMA):
    // as deep as the operand ring and loaded once the stage is free, so
    // that the writers wait on one barrier per stage (a second wait made
    // them slower than its MMAs).
    static constexpr int kSFRing = kNV ? kStages : kStages + 2;
    static constexpr bool kSFAhead = kSFRing > kStages;
    static constexpr uint32_t kOffSFB = kKSub * kSFSub;
    static constexpr uint32_t kSFSlotBytes = 3 * kKSub * kSFSub;          // 6 KB
    static constexpr uint32_t kSFCols = kNV ? 48 : 24;          // tensor-memory columns per sub-tile
    static constexpr uint32_t kSFSlot = kSFCols * kKSub;
    static_assert(kStages <= kMaxStages && kSFRing <= kMaxSFRing, "barrier arrays");
    static_assert(kSFCol + kStages * kSFSlot <= kTmemCols, "scale slots fit in tensor memory");
};

// Fused Wgrad: the encoder warps of every CTA encode both operands (dY
// [T][N], X [T][K], contraction T) into the workspace while the GEMM runs.
// Units of work: (panel of 256 lines, chunk of 512 tokens, quarter of 64
// lines, slice of 64 tokens).  Units run in the order the GEMM first needs
// them: the panels a round of tiles touches for the first time form a group,
// encoded chunk by chunk, and consecutive units go to warps of different
// CTAs, so a chunk is spread over the whole GPU and done early.  A (panel,
// chunk) counter in the workspace (zeroed before the launch) reaches
// kUnitsPerChunk when all its units are stored; the GEMM's producers wait
// for it before loading that stage.
constexpr int kMaxPanels = 512;
constexpr int kMaxGroups = 128;
constexpr int kSlices = 8;                        // 64-token slices of a 512-token chunk
constexpr int kUnitsPerChunk = 4 * kSlices;       // quarters x slices
struct FusedArgs {
    const uint32_t *src[2];     // dY, X as 32-bit words (two bf16 channels each)
    uint8_t *codes[2];          // [lines][T/2]
    uint8_t *scales[2];         // tiled layout
    int64_t words_per_row[2];   // N / 2, K / 2
    int64_t T;
    int64_t katoms;             // scale k-atoms per 128-line group (contraction T)
    unsigned int *counters;     // [panel][chunk], zero at launch
    int rot_block;              // 0 (no rotation), 16 or 32
    int chunks;                 // T / 512
    int panels_a;               // A panels come first in the global panel index
    int groups;
    int units;                  // kUnitsPerChunk * chunks * panels
    uint16_t group_start[kMaxGroups + 1];
    uint16_t panel[kMaxPanels]; // global panel indices in first-use order
};

struct GemmArgs {
    const uint8_t *As;
    const uint8_t *Bs;
    float *C;
    int64_t M, N, K;
    int64_t katoms;      // scale k-atoms per 128-row group
    int64_t a_groups;    // 128-row scale groups that exist for A
    int64_t b_groups;    // ... and for B
    int k_tiles;         // 256-wide K sub-tiles
    int k_stages;        // stages per tile (ceil(k_tiles / sub-tiles per stage))
    int m_tiles;
    int n_tiles;
    int num_tiles;
    int num_items;       // one item per tile
    int c_v8;            // C rows allow 32-byte stores (N % 8 == 0, C 32-byte aligned)
    size_t c_bytes;      // extent of C (store guards)
    const float *amax_a; // NVFP4: tensor amaxes of A and B (the result is divided by
    const float *amax_b; //   the product of their encode scales)
    int *status;
};

struct SharedCtl {
    uint64_t full[kMaxStages];      // even CTA: both CTAs' operand bytes of the stage have landed
                                    //   and both CTAs' scales are in tensor memory
    uint64_t empty[kMaxStages];     // the pair's MMAs have finished reading the stage
    uint64_t sf_full[kMaxSFRing];   // this CTA's scale bytes of a scale slot have landed
    uint64_t sf_free[kMaxSFRing];   // this CTA's scale writers have read the slot
    uint64_t acc_full;           // the tile's accumulator is complete
    uint64_t acc_empty;          // even CTA: both CTAs' epilogues have read the accumulator
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    int issued;                  // stages whose operand loads this CTA has issued (monotonic)
};

// The output is written once and not read here: its stores bypass L1 and
// are the first lines L2 evicts, so that they do not push the operand panels
// (read by every tile of a band) out of L2 (o_proj GEMM 56.1 -> 54.0 us).
// 1: streaming stores instead; 0: plain stores.
#ifndef MXG_ST_KIND
#define MXG_ST_KIND 2
#endif
#if MXG_ST_KIND == 1
#define MXG_ST_OP "st.global.cs.v8.b32"
#elif MXG_ST_KIND == 2
#define MXG_ST_OP "st.global.L1::no_allocate.L2::evict_first.v8.b32"
#else
#define MXG_ST_OP "st.global.v8.b32"
#endif
// L2 prefetch of the B panel of each pair's next tile when it starts a new
// column (down_proj GEMM 144.5 -> 142.9 us in the lab).
#ifndef MXG_PFB
#define MXG_PFB 1
#endif
// Pairs per launch: as many as fit, or (MXG_BALANCE) just enough for the
// same number of rounds, so that every pair holds a tile in the last round
// (o_proj: 64 pairs x 4 tiles instead of 76 pairs with 28 in the last round;
// the same makespan with less contention).
#ifndef MXG_BALANCE
#define MXG_BALANCE 1
#endif
// Tile order: bands of kBand tile rows, column by column within a band, so
// that the tiles in flight at once share few A and B panels (L2 reuse).
#ifndef MXG_BAND
#define MXG_BAND 16
#endif
constexpr int kBand = MXG_BAND;
__device__ __forceinline__ void tile_coords(const GemmArgs &g, int t, int &mb, int &nb) {
    const int per_band = kBand * g.n_tiles;
    const int band = t / per_band, r = t % per_band;
    const int first = band * kBand;
    const int rows = g.m_tiles - first < kBand ? g.m_tiles - first : kBand;
    mb = first + r % rows;
    nb = r / rows;
}

// Work item w: tile t over K stages [ks0, ks1).
struct Item {
    int tile, ks0, ks1;
};
__device__ __forceinline__ Item item_of(const GemmArgs &g, int w) {
    return Item{w, 0, g.k_stages};
}

__device__ __forceinline__ void st_global_v4f(float *p, uint32_t a, uint32_t b, uint32_t c,
                                              uint32_t d) {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// One full 32-byte sector per store (the address must be 32-byte aligned).
__device__ __forceinline__ void st_global_v8(float *p, const uint32_t *v) {
    asm volatile(MXG_ST_OP " [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

// Arrive on the barrier `bar` of the even CTA of this pair (a local arrive in
// the even CTA, a remote one in the odd CTA).  The arrivals here only order
// tensor-memory work, which the tcgen05 fences around them cover.
__device__ __forceinline__ void arrive_even(uint64_t *bar) {
    mbar_arrive_remote(mapa_shared(smem_u32(bar), 0u));
}

// Stores 32 fp32 values of one C row starting at column cc (columns past N
// are skipped).
__device__ __forceinline__ void store_row32(const GemmArgs &g, float *crow, int64_t cc,
                                            const uint32_t (&v)[32]) {
    if (g.c_v8 && cc + 31 < g.N) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (MX_STORE_OK(crow + cc + 8 * j, 32, g.C, g.c_bytes, g.status))
                st_global_v8(crow + cc + 8 * j, &v[8 * j]);
        return;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int64_t col = cc + 4 * j;
        if (col + 3 < g.N) {
            if (MX_STORE_OK(crow + col, 16, g.C, g.c_bytes, g.status))
                st_global_v4f(crow + col, v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (col + e < g.N && MX_STORE_OK(crow + col + e, 4, g.C, g.c_bytes, g.status))
                    crow[col + e] = __uint_as_float(v[4 * j + e]);
        }
    }
}

// Bounded wait until this CTA's producer has issued at least `target` stages
// (a monotonic counter, so no phase can be mistaken for another).  Lane 0
// polls; the warp follows.  Returns false on timeout or abort.
__device__ __forceinline__ bool wait_issued(const SharedCtl *ctl, int target, int *status,
                                            volatile int *abort) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) {
        const volatile int *issued = &ctl->issued;
        if (*issued < target) {
            const uint64_t t0 = global_timer_ns();
            while (*issued < target) {
                if (*abort || global_timer_ns() - t0 > kWaitLimitNs) {
                    if (!*abort) atomicExch(status, kDevTimeout);
                    *abort = 1;
                    ok = 0;
                    break;
                }
                __nanosleep(64);
            }
        }
    }
    return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

// Bounded wait until (panel, chunk) counter `ctr` reaches `want` (acquire
// at GPU scope), then a proxy fence so that the TMA reads see what the
// encoder warps (generic stores on other SMs) wrote.
__device__ __forceinline__ bool wait_encoded(const unsigned int *ctr, unsigned int want,
                                             int *status, volatile int *abort) {
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        unsigned int v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v >= want) break;
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            atomicExch(status, kDevTimeout);
            *abort = 1;
            return false;
        }
        __nanosleep(64);
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

// Encoder warp of the fused Wgrad launch: units gw, gw + W, ... .  Each lane
// owns two adjacent lines (channels) and 32 tokens per step: 32 coalesced
// 128-byte warp loads straight from global memory (the transpose is the
// lane's own column read), then the same rotation and encode as the
// stand-alone column encoder (enc::fwht_pairs, enc::encode_pair_rne).
template <int ROTN>
__device__ __forceinline__ void encode_units(const FusedArgs &f, int gw, int W, int *status,
                                             volatile int *abort) {
    const int lane = threadIdx.x & 31;
    const float cn = ROTN > 0 ? enc::hadamard_norm<ROTN>() : 1.0f;
    for (int u = gw; u < f.units; u += W) {
        if (__shfl_sync(0xFFFFFFFFu, *abort, 0)) return;
        int gi = 0;
        while (gi + 1 < f.groups && kUnitsPerChunk * f.chunks * f.group_start[gi + 1] <= u) ++gi;
        const int gp = f.group_start[gi + 1] - f.group_start[gi];
        const int r = u - kUnitsPerChunk * f.chunks * f.group_start[gi];
        const int chunk = r / (kUnitsPerChunk * gp);
        const int rem = r % (kUnitsPerChunk * gp);
        const int gpanel = f.panel[f.group_start[gi] + rem / kUnitsPerChunk];
        const int quarter = (rem % kUnitsPerChunk) / kSlices;
        const int slice = rem % kSlices;
        const int o = gpanel >= f.panels_a ? 1 : 0;
        const int64_t pn = gpanel - (o ? f.panels_a : 0);
        const int64_t c = pn * 256 + quarter * 64 + 2 * lane;   // first of the lane's two lines
        const int64_t wpr = f.words_per_row[o];
        const uint32_t *src = f.src[o] + c / 2;
        uint8_t *codes = f.codes[o];
        uint8_t *scales = f.scales[o];
#pragma unroll 1
        for (int step = 0; step < 2; ++step) {
            const int64_t t0 = static_cast<int64_t>(chunk) * 512 + 64 * slice + 32 * step;
            uint64_t x[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const uint32_t v = __ldg(src + (t0 + i) * wpr);
                x[i] = enc::pack2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
            }
            if (ROTN > 0) enc::fwht_pairs<ROTN>(x);
            uint4 q0, q1;
            uint32_t s0, s1;
            enc::encode_pair_rne<(ROTN > 0)>(x, cn, q0, q1, s0, s1);
            enc::st_global_16(codes + c * (f.T / 2) + t0 / 2, q0);
            enc::st_global_16(codes + (c + 1) * (f.T / 2) + t0 / 2, q1);
            scales[enc::scale_offset(c, t0 / 32, f.katoms)] = static_cast<uint8_t>(s0);
            scales[enc::scale_offset(c + 1, t0 / 32, f.katoms)] = static_cast<uint8_t>(s1);
        }
        // Every lane makes its stores visible at GPU scope, then lane 0
        // counts the unit once all lanes are past their fence (a shuffle as
        // the convergence point: bar.warp.sync here defeats ptxas's register
        // split).
        __threadfence();
        if (__shfl_sync(0xFFFFFFFFu, lane, 0) == 0 && lane == 0)
            atomicAdd(f.counters + static_cast<int64_t>(gpanel) * f.chunks + chunk, 1u);
    }
}

template <bool FUSED, int FMT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Variant<FUSED>::kThreads, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                   const __grid_constant__ CUtensorMap map_b, const GemmArgs g,
                   const __grid_constant__ FusedArgs f) {
    using V = Variant<FUSED>;
    using E = Elem<FMT>;
    static_assert(!(FUSED && FMT != kFmtMX4), "the fused launch encodes MXFP4 only");
    constexpr int kStages = E::kStages, kKSub = E::kKSub;
    constexpr int kSFRing = E::kSFRing;
    constexpr uint32_t kStageBytes = E::kStageBytes, kSFSlot = E::kSFSlot, kSFSub = E::kSFSub;
    constexpr uint32_t kOffA = E::kOffA, kOffB = E::kOffB, kOffSFB = E::kOffSFB,
                       kSFSlotBytes = E::kSFSlotBytes;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned base, kept as a shared-space pointer (offset arithmetic
    // only) so that the compiler emits shared-memory loads.  The offset is the
    // same in both CTAs of the pair (same kernel, same static layout).
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sf_ring = smem + kStages * kStageBytes;
    SharedCtl *ctl = reinterpret_cast<SharedCtl *>(sf_ring + kSFRing * kSFSlotBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            // The even CTA's producer (arming the operand bytes) and the four
            // scale writers of each CTA.
            mbar_init(&ctl->full[s], 1 + 2 * 4);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int j = 0; j < kSFRing; ++j) {
            mbar_init(&ctl->sf_full[j], 1);
            mbar_init(&ctl->sf_free[j], 4);
        }
        mbar_init(&ctl->acc_full, 1);
        mbar_init(&ctl->acc_empty, 2 * kEpiWarps);
        mbar_init(&ctl->drain, 1);
        ctl->abort_flag = 0;
        ctl->issued = 0;
        fence_barrier_init();
        prefetch_tmap(&map_a);
        prefetch_tmap(&map_b);
    }
    if (warp == 1) {
        tmem_alloc_pair(&ctl->tmem_base, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    // Both CTAs of the pair have initialised their barriers (and allocated
    // tensor memory) before either signals the other.
    __syncwarp();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    volatile int *abort = &ctl->abort_flag;
    // Barriers and tensor memory are set up; global memory is touched only
    // once the stream's previous kernel (the encoder) has completed.
    griddep_wait();
    griddep_launch_dependents();

    if (warp < kWriterWarp0) {
        // Warpgroup 0: producers and the MMA issuer need few registers.
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(V::kRegsLow) : "memory");
        if ((warp == 0 || warp == 2) && lane == 0) {
            // ------------------------------------------------------------ producers
            // Warp 0 fills the operand ring, warp 2 the scale ring.
            const bool scales = warp == 2;
            const int ring = scales ? kSFRing : kStages;
            const bool on_free = scales && E::kSFAhead;
            int stage = 0, n_issued = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int w = pair; ok && w < g.num_items; w += npairs) {
                const Item it = item_of(g, w);
                int mb, nb;
                tile_coords(g, it.tile, mb, nb);
                const int64_t ga = 2 * static_cast<int64_t>(mb) + rank;  // this CTA's A scale group
#if MXG_PFB
                if (!FUSED && !scales && w + npairs < g.num_items) {
                    // The B panel of this pair's next tile, when it is a new
                    // column: read from DRAM by all the column's pairs at once
                    // otherwise.  Each pair of this band brings its share of
                    // the panel's K range into L2 a tile ahead.  (Not in the
                    // fused launch, whose panels may not be encoded yet.)
                    int mb2, nb2;
                    tile_coords(g, item_of(g, w + npairs).tile, mb2, nb2);
                    if (nb2 != nb) {
                        const int nseg = g.m_tiles < kBand ? g.m_tiles : kBand;
                        const int seg = mb % nseg;
                        const int per = (g.k_tiles + nseg - 1) / nseg;
                        const int k_end = (seg + 1) * per < g.k_tiles ? (seg + 1) * per : g.k_tiles;
                        for (int kt = seg * per; kt < k_end; ++kt)
                            tma_prefetch_2d(&map_b, kt * kBKBytes, nb2 * kTile + kHalf * rank);
                    }
                }
#endif
                for (int ks = it.ks0; ks < it.ks1; ++ks) {
                    if (!mbar_wait_inl(on_free ? &ctl->sf_free[stage] : &ctl->empty[stage],
                                       phase ^ 1u, g.status, abort)) {
                        ok = false;
                        break;
                    }
                    const int kt0 = ks * kKSub;
                    const int nsub = g.k_tiles - kt0 < kKSub ? g.k_tiles - kt0 : kKSub;
                    uint8_t *st = smem + stage * kStageBytes;
                    uint8_t *sfs = sf_ring + stage * kSFSlotBytes;
                    if constexpr (FUSED) {
                        // This stage's 512 tokens of both panels are encoded.
                        const unsigned int want = kUnitsPerChunk;
                        if (!wait_encoded(f.counters + static_cast<int64_t>(mb) * f.chunks + ks,
                                          want, g.status, abort) ||
                            !wait_encoded(f.counters +
                                              static_cast<int64_t>(f.panels_a + nb) * f.chunks + ks,
                                          want, g.status, abort)) {
                            ok = false;
                            break;
                        }
                    }
                    if (scales) {
                        const uint32_t sub_bytes = static_cast<uint32_t>(nsub) * E::kSFBytes;
                        uint32_t bytes = 0;
                        if (ga < g.a_groups) bytes += sub_bytes;
                        for (int rb = 0; rb < 2; ++rb)
                            if (2 * static_cast<int64_t>(nb) + rb < g.b_groups) bytes += sub_bytes;
                        mbar_arrive_expect_tx(&ctl->sf_full[stage], bytes);
                        if (ga < g.a_groups)
                            bulk_load(sfs, g.As + (ga * g.katoms + E::kAtoms * kt0) * 512,
                                      sub_bytes, &ctl->sf_full[stage]);
                        for (int rb = 0; rb < 2; ++rb) {
                            const int64_t gb = 2 * static_cast<int64_t>(nb) + rb;
                            if (gb < g.b_groups)
                                bulk_load(sfs + kOffSFB + rb * kKSub * kSFSub,
                                          g.Bs + (gb * g.katoms + E::kAtoms * kt0) * 512,
                                          sub_bytes, &ctl->sf_full[stage]);
                        }
                    } else {
                        // Both CTAs' operand loads complete on the even CTA's
                        // barrier, which the even CTA arms with the pair's bytes
                        // (boxes partly or wholly outside the operand still count
                        // in full; the TMA fills them with zeros).
                        if (rank == 0)
                            mbar_arrive_expect_tx(&ctl->full[stage],
                                                  static_cast<uint32_t>(nsub) * 4u * kSubBytes);
                        const uint32_t full_even = mapa_shared(smem_u32(&ctl->full[stage]), 0u);
                        for (int u = 0; u < nsub; ++u) {
                            tma_load_2d_pair(st + kOffA + u * kSubBytes, &map_a, full_even,
                                             (kt0 + u) * kBKBytes, mb * kTile + kHalf * rank);
                            tma_load_2d_pair(st + kOffB + u * kSubBytes, &map_b, full_even,
                                             (kt0 + u) * kBKBytes, nb * kTile + kHalf * rank);
                        }
                        *reinterpret_cast<volatile int *>(&ctl->issued) = ++n_issued;
                    }
                    if (++stage == ring) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        } else if (warp == 1 && lane == 0 && rank == 0) {
            // ------------------------------------------------------------ MMA issuer
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            const uint32_t idesc0 = idesc_mxf4(2 * kHalf, kTile, 0, 0);
            const uint32_t idesc2 = idesc_mxf4(2 * kHalf, kTile, 2, 2);
            uint32_t idesc8[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) idesc8[j] = idesc_mxf8(2 * kHalf, kTile, j, j);
            const uint32_t idesc_nv = idesc_nvf4(2 * kHalf, kTile);
            for (int w = pair; ok && w < g.num_items; w += npairs) {
                const Item it = item_of(g, w);
                if (!mbar_wait_inl(&ctl->acc_empty, acc_phase ^ 1u, g.status, abort)) break;
                tc_fence_after();
                for (int ks = it.ks0; ks < it.ks1; ++ks) {
                    if (!mbar_wait_inl(&ctl->full[stage], phase, g.status, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int kt0 = ks * kKSub;
                    const int nsub = g.k_tiles - kt0 < kKSub ? g.k_tiles - kt0 : kKSub;
                    const uint32_t sbase = smem_u32(smem + stage * kStageBytes);
                    const uint32_t slot = tmem + kSFCol + kSFSlot * static_cast<uint32_t>(stage);
                    for (int u = 0; u < nsub; ++u) {
                        const uint32_t sa = sbase + kOffA + u * kSubBytes;
                        const uint32_t sb = sbase + kOffB + u * kSubBytes;
                        const uint32_t sf = slot + E::kSFCols * static_cast<uint32_t>(u);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t acc = (ks > it.ks0 || u > 0 || j > 0) ? 1u : 0u;
                            if constexpr (FMT == kFmtMX8) {
                                // K = 32 per MMA: block j of the sub-tile's
                                // single scale atom (byte j of its columns).
                                mma_mxf8_pair(tmem + kAccCol, sdesc_sw128(sa + 32u * j),
                                              sdesc_sw128(sb + 32u * j), idesc8[j], sf, sf + 8u,
                                              acc);
                            } else if constexpr (FMT == kFmtNV4) {
                                // K = 64 per MMA: four UE4M3 scales per row,
                                // one whole column per row group.
                                mma_nvf4_pair(tmem + kAccCol, sdesc_sw128(sa + 32u * j),
                                              sdesc_sw128(sb + 32u * j), idesc_nv, sf + 4u * j,
                                              sf + 16u + 8u * j, acc);
                            } else {
                                const uint32_t ka = static_cast<uint32_t>(j / 2);
                                mma_mxf4_pair(tmem + kAccCol, sdesc_sw128(sa + 32u * j),
                                              sdesc_sw128(sb + 32u * j), (j & 1) ? idesc2 : idesc0,
                                              sf + 4u * ka, sf + 8u + 8u * ka, acc);
                            }
                        }
                    }
                    tc_commit_pair(&ctl->empty[stage], 0x3);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                tc_commit_pair(&ctl->acc_full, 0x3);
                acc_phase ^= 1u;
            }
            // Every tensor-core operation issued here has finished before
            // either CTA releases its tensor memory.
            tc_commit_pair(&ctl->drain, 0x1);
            mbar_wait_inl(&ctl->drain, 0, g.status, nullptr, 100ull * 1000ull * 1000ull);
        }
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------------------ scale writers
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(V::kRegsLow) : "memory");
        // Tensor-memory scale layout of one K sub-tile (24 columns, as the
        // tcgen05.mma block-scale path reads it), the same in every lane
        // quarter q: for k-atom ka (4 blocks of 32), A row 32*c + r of this
        // CTA at lane 32q + r, column 4*ka + c (the quarter's own rows are at
        // c = q); B row 128*rb + 32*c + r (all 256 rows) at lane 32q + r,
        // column 8 + 8*ka + 4*rb + c; byte b of a column is block 4*ka + b.
        // A lane reads its 16-byte row of each 512-byte scale atom, which
        // holds exactly those four rows.
        const int q = warp & 3;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16);
        // Per stage: the scales are in this CTA's scale slot (sf_full) and
        // the stage's tensor-memory columns are free (empty: the MMAs that
        // last read them have finished); then write, release the scale slot
        // and arrive on the even CTA's full barrier.
        int stage = 0, sj = 0;
        uint32_t phase = 0, sphase = 0;
        for (int w = pair; w < g.num_items; w += npairs) {
            const Item it = item_of(g, w);
            bool ok = true;
            for (int ks = it.ks0; ks < it.ks1; ++ks) {
                int okw = 1;
                if (lane == 0) {
                    // Without the deeper ring the scales were loaded after
                    // the stage came free: sf_full implies empty.
                    okw = mbar_wait_inl(&ctl->sf_full[sj], sphase, g.status, abort) ? 1 : 0;
                    if (E::kSFAhead && okw)
                        okw = mbar_wait_inl(&ctl->empty[stage], phase ^ 1u, g.status, abort) ? 1 : 0;
                }
                okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
                if (!okw) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int kt0 = ks * kKSub;
                const int nsub = g.k_tiles - kt0 < kKSub ? g.k_tiles - kt0 : kKSub;
                const uint8_t *sfs = sf_ring + sj * kSFSlotBytes;
                const uint32_t slot =
                    lane_base + kSFCol + kSFSlot * static_cast<uint32_t>(stage);
                for (int u = 0; u < nsub; ++u) {
                    const uint8_t *sfa = sfs + u * E::kSFBytes;
                    const uint8_t *sfb = sfs + kOffSFB + u * E::kSFBytes;
                    const uint32_t col = slot + E::kSFCols * static_cast<uint32_t>(u);
                    if constexpr (FMT == kFmtNV4) {
                        // Atom j holds MMA j's scales: A at columns 4j..4j+3,
                        // B at 16 + 8j + 4rb + c.
                        uint32_t a16[16], b16[16];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(sfa + j * 512 + lane * 16);
                            a16[4 * j + 0] = v.x;
                            a16[4 * j + 1] = v.y;
                            a16[4 * j + 2] = v.z;
                            a16[4 * j + 3] = v.w;
                        }
                        tmem_st_32x32b_x16(col, a16);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
#pragma unroll
                            for (int jj = 0; jj < 2; ++jj)
#pragma unroll
                                for (int rb = 0; rb < 2; ++rb) {
                                    const uint4 v = *reinterpret_cast<const uint4 *>(
                                        sfb + rb * kKSub * kSFSub + (2 * h + jj) * 512 + lane * 16);
                                    b16[8 * jj + 4 * rb + 0] = v.x;
                                    b16[8 * jj + 4 * rb + 1] = v.y;
                                    b16[8 * jj + 4 * rb + 2] = v.z;
                                    b16[8 * jj + 4 * rb + 3] = v.w;
                                }
                            tmem_st_32x32b_x16(col + 16u + 16u * h, b16);
                        }
                    } else if constexpr (FMT == kFmtMX8) {
                        // One atom: A at columns 0..3, B at 8..15 (ka = 0).
                        uint32_t a4[4], b8[8];
                        const uint4 va = *reinterpret_cast<const uint4 *>(sfa + lane * 16);
                        a4[0] = va.x;
                        a4[1] = va.y;
                        a4[2] = va.z;
                        a4[3] = va.w;
#pragma unroll
                        for (int rb = 0; rb < 2; ++rb) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(
                                sfb + rb * kKSub * kSFSub + lane * 16);
                            b8[4 * rb + 0] = v.x;
                            b8[4 * rb + 1] = v.y;
                            b8[4 * rb + 2] = v.z;
                            b8[4 * rb + 3] = v.w;
                        }
                        tmem_st_32x32b_x4(col, a4);
                        tmem_st_32x32b_x8(col + 8u, b8);
                    } else {
                    uint32_t a[8], b[16];
#pragma unroll
                    for (int ka = 0; ka < 2; ++ka) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(sfa + ka * 512 + lane * 16);
                        a[4 * ka + 0] = v.x;
                        a[4 * ka + 1] = v.y;
                        a[4 * ka + 2] = v.z;
                        a[4 * ka + 3] = v.w;
                    }
#pragma unroll
                    for (int ka = 0; ka < 2; ++ka)
#pragma unroll
                        for (int rb = 0; rb < 2; ++rb) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(
                                sfb + rb * kKSub * kSFSub + ka * 512 + lane * 16);
                            b[8 * ka + 4 * rb + 0] = v.x;
                            b[8 * ka + 4 * rb + 1] = v.y;
                            b[8 * ka + 4 * rb + 2] = v.z;
                            b[8 * ka + 4 * rb + 3] = v.w;
                        }
                    tmem_st_32x32b_x8(col, a);
                    tmem_st_32x32b_x16(col + 8u, b);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (E::kSFAhead) mbar_arrive(&ctl->sf_free[sj]);
                    arrive_even(&ctl->full[stage]);
                }
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (++sj == kSFRing) {
                    sj = 0;
                    sphase ^= 1u;
                }
            }
            if (!ok) break;
        }
    } else if (!FUSED || warp < kEncWarp0) {
        // ------------------------------------------------------------ epilogue
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(V::kRegsHigh) : "memory");
        const int q = warp & 3;                   // TMEM lane quarter this warp may access
        const int half = (warp - kEpiWarp0) / 4;  // column half of the 256-wide tile
        float alpha = 1.0f;
        if constexpr (FMT == kFmtNV4)
            alpha = __frcp_rn(__fmul_rn(enc::nv_tensor_scale(*g.amax_a),
                                        enc::nv_tensor_scale(*g.amax_b)));
        (void)alpha;
        uint32_t acc_phase = 0;
        int staged = 0;                           // stages of this pair's items so far
        for (int w = pair; w < g.num_items; w += npairs) {
            const Item it = item_of(g, w);
            int mb, nb;
            tile_coords(g, it.tile, mb, nb);
            staged += it.ks1 - it.ks0;
            // One lane waits; its result is broadcast so the warp stays
            // converged for the .sync.aligned tensor-memory loads.
            int ok = 1;
            if (lane == 0) ok = mbar_wait_inl(&ctl->acc_full, acc_phase, g.status, abort) ? 1 : 0;
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            acc_phase ^= 1u;
            const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16) + kAccCol +
                                   128u * static_cast<uint32_t>(half);
            if constexpr (FUSED) {
                // Two passes of 64 columns (the encoder warps need the
                // registers): the first pass is stored at once, the second
                // after tensor memory is released, paced like below.
                const int64_t row =
                    static_cast<int64_t>(mb) * kTile + kHalf * rank + 32 * q + lane;
                float *crow = g.C + row * g.N;
                const int64_t col0 = static_cast<int64_t>(nb) * kTile + 128 * half;
                const int next = w + npairs;
                uint32_t v0[32], v1[32];
                tmem_ld_32x32b_x32(tbase, v0);
                tmem_ld_32x32b_x32(tbase + 32u, v1);
                tmem_ld_wait();
                if (row < g.M) {
                    store_row32(g, crow, col0, v0);
                    store_row32(g, crow, col0 + 32, v1);
                }
                tmem_ld_32x32b_x32(tbase + 64u, v0);
                tmem_ld_32x32b_x32(tbase + 96u, v1);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) arrive_even(&ctl->acc_empty);
                if (next < g.num_items && g.c_v8 && col0 + 127 < g.N) {
                    const Item nx = item_of(g, next);
                    const int ns = nx.ks1 - nx.ks0;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int need = 1 + (j * ns) / 8;
                        if (j == 0 || need != 1 + ((j - 1) * ns) / 8)
                            if (!wait_issued(ctl, staged + need, g.status, abort)) break;
                        const uint32_t *src = j < 4 ? &v0[8 * j] : &v1[8 * (j - 4)];
                        if (row < g.M &&
                            MX_STORE_OK(crow + col0 + 64 + 8 * j, 32, g.C, g.c_bytes, g.status))
                            st_global_v8(crow + col0 + 64 + 8 * j, src);
                    }
                } else if (row < g.M) {
                    store_row32(g, crow, col0 + 64, v0);
                    store_row32(g, crow, col0 + 96, v1);
                }
                continue;
            }
            uint32_t v0[32], v1[32], v2[32], v3[32];
            tmem_ld_32x32b_x32(tbase, v0);
            tmem_ld_32x32b_x32(tbase + 32u, v1);
            tmem_ld_32x32b_x32(tbase + 64u, v2);
            tmem_ld_32x32b_x32(tbase + 96u, v3);
            tmem_ld_wait();
            if constexpr (FMT == kFmtNV4) {
                // C = (sum of e2m1 * sf products) / (s_enc(A) * s_enc(B)).
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    v0[i] = __float_as_uint(__fmul_rn(__uint_as_float(v0[i]), alpha));
                    v1[i] = __float_as_uint(__fmul_rn(__uint_as_float(v1[i]), alpha));
                    v2[i] = __float_as_uint(__fmul_rn(__uint_as_float(v2[i]), alpha));
                    v3[i] = __float_as_uint(__fmul_rn(__uint_as_float(v3[i]), alpha));
                }
            }
            // The accumulator is in registers: the next item may start.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_even(&ctl->acc_empty);

            const int64_t row =
                static_cast<int64_t>(mb) * kTile + kHalf * rank + 32 * q + lane;
            float *crow = g.C + row * g.N;
            const int64_t col0 = static_cast<int64_t>(nb) * kTile + 128 * half;
            const int next = w + npairs;
            if (next < g.num_items && g.c_v8 && col0 + 127 < g.N) {
                // Store chunk j (8 values) once the producer has issued stage
                // 1 + j * s / 16 of the next item (s stages).
                const Item nx = item_of(g, next);
                const int ns = nx.ks1 - nx.ks0;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int need = 1 + (j * ns) / 16;
                    if (j == 0 || need != 1 + ((j - 1) * ns) / 16)
                        if (!wait_issued(ctl, staged + need, g.status, abort)) break;
                    const uint32_t *src = j < 4    ? &v0[8 * j]
                                          : j < 8  ? &v1[8 * (j - 4)]
                                          : j < 12 ? &v2[8 * (j - 8)]
                                                   : &v3[8 * (j - 12)];
                    if (row < g.M && MX_STORE_OK(crow + col0 + 8 * j, 32, g.C, g.c_bytes, g.status))
                        st_global_v8(crow + col0 + 8 * j, src);
                }
            } else if (row < g.M) {
                store_row32(g, crow, col0, v0);
                store_row32(g, crow, col0 + 32, v1);
                store_row32(g, crow, col0 + 64, v2);
                store_row32(g, crow, col0 + 96, v3);
            }
        }
    } else if constexpr (FUSED) {
        // ------------------------------------------------------------ encoder
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(V::kRegsHigh) : "memory");
        const int gw = (warp - kEncWarp0) * gridDim.x + blockIdx.x;
        const int W = gridDim.x * kEncWarps;
        if (f.rot_block == 32)
            encode_units<32>(f, gw, W, g.status, abort);
        else if (f.rot_block == 16)
            encode_units<16>(f, gw, W, g.status, abort);
        else
            encode_units<0>(f, gw, W, g.status, abort);
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    // Neither CTA of the pair releases tensor memory (or leaves) while the
    // other's operations may still touch it.
    __syncwarp();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

template <int FMT>
constexpr size_t gemm_smem() {
    return Elem<FMT>::kStages * Elem<FMT>::kStageBytes +
           Elem<FMT>::kSFRing * Elem<FMT>::kSFSlotBytes + sizeof(SharedCtl) + 1024;
}

// Co-resident 2-CTA clusters of a mx_gemm_kernel variant on a device,
// measured once.
template <bool FUSED, int FMT>
int gemm_clusters(const DeviceInfo &dev) {
    static std::atomic<int> cache[64];
    const int idx = dev.ordinal >= 0 && dev.ordinal < 64 ? dev.ordinal : 0;
    int n = cache[idx].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaFuncSetAttribute(mx_gemm_kernel<FUSED, FMT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(gemm_smem<FMT>())) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(Variant<FUSED>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = gemm_smem<FMT>();
    if (cudaOccupancyMaxActiveClusters(&n, mx_gemm_kernel<FUSED, FMT>, &cfg) != cudaSuccess ||
        n < 1)
        return 0;
    cache[idx].store(n, std::memory_order_relaxed);
    return n;
}

// Common set-up of both variants: tensor maps and the GEMM arguments.
bool gemm_setup(int fmt, const void *Aq, const void *As, const void *Bq, const void *Bs,
                float *C, int64_t M, int64_t N, int64_t K, const DeviceInfo &dev,
                CUtensorMap *map_a, CUtensorMap *map_b, GemmArgs *g) {
    const bool f8 = fmt == kFmtMX8, nv = fmt == kFmtNV4;
    const int64_t row_bytes = f8 ? K : K / 2;
    if (!encode_tmap_2d(map_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, Aq, row_bytes, M, row_bytes,
                        kBKBytes, kHalf, CU_TENSOR_MAP_SWIZZLE_128B))
        return false;
    if (!encode_tmap_2d(map_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, Bq, row_bytes, N, row_bytes,
                        kBKBytes, kHalf, CU_TENSOR_MAP_SWIZZLE_128B))
        return false;
    *g = GemmArgs{};
    g->As = static_cast<const uint8_t *>(As);
    g->Bs = static_cast<const uint8_t *>(Bs);
    g->C = C;
    g->M = M;
    g->N = N;
    g->K = K;
    g->katoms = nv ? nv_scale_katoms(K) : scale_katoms(K);
    g->a_groups = scale_groups(M);
    g->b_groups = scale_groups(N);
    const int64_t sub_k = f8 ? Elem<kFmtMX8>::kSubK : Elem<kFmtMX4>::kSubK;
    const int ksub = nv ? Elem<kFmtNV4>::kKSub : Elem<kFmtMX4>::kKSub;
    g->k_tiles = static_cast<int>((K + sub_k - 1) / sub_k);
    g->k_stages = (g->k_tiles + ksub - 1) / ksub;
    const int64_t m_tiles = (M + kTile - 1) / kTile;
    const int64_t n_tiles = (N + kTile - 1) / kTile;
    if (m_tiles * n_tiles > 0x3FFFFFFF) return false;
    g->m_tiles = static_cast<int>(m_tiles);
    g->n_tiles = static_cast<int>(n_tiles);
    g->num_tiles = static_cast<int>(m_tiles * n_tiles);
    g->num_items = g->num_tiles;
    g->c_v8 = (N % 8 == 0 && (reinterpret_cast<uintptr_t>(C) & 31) == 0) ? 1 : 0;
    g->c_bytes = static_cast<size_t>(M) * static_cast<size_t>(N) * sizeof(float);
    g->status = dev.status;
    return true;
}

template <bool FUSED, int FMT>
cudaError_t gemm_launch(const CUtensorMap &map_a, const CUtensorMap &map_b, const GemmArgs &g,
                        const FusedArgs &f, int pairs, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(mx_gemm_kernel<FUSED, FMT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(gemm_smem<FMT>()));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.blockDim = dim3(Variant<FUSED>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = gemm_smem<FMT>();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, mx_gemm_kernel<FUSED, FMT>, map_a, map_b, g, f);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

namespace {
template <int FMT>
cudaError_t launch_gemm_elem(const void *Aq, const void *As, const void *Bq, const void *Bs,
                             float *C, int64_t M, int64_t N, int64_t K, const float *amax_a,
                             const float *amax_b, const DeviceInfo &dev, cudaStream_t stream) {
    CUtensorMap map_a, map_b;
    GemmArgs g;
    if (!gemm_setup(FMT, Aq, As, Bq, Bs, C, M, N, K, dev, &map_a, &map_b, &g))
        return cudaErrorInvalidValue;
    g.amax_a = amax_a;
    g.amax_b = amax_b;
    // Resident CTAs: as many 2-CTA clusters as fit at once, one tile per pair.
    const int pairs_max = gemm_clusters<false, FMT>(dev);
    if (pairs_max < 1) return cudaErrorLaunchOutOfResources;
    int pairs = g.num_items < pairs_max ? g.num_items : pairs_max;
#if MXG_BALANCE
    // As many rounds of tiles as all pairs need, spread evenly over fewer
    // pairs (the last round then keeps every pair busy).
    {
        const int rounds = (g.num_items + pairs - 1) / pairs;
        pairs = (g.num_items + rounds - 1) / rounds;
    }
#endif
    FusedArgs f;
    std::memset(&f, 0, sizeof(f));
    return gemm_launch<false, FMT>(map_a, map_b, g, f, pairs, stream);
}
}  // namespace

cudaError_t launch_gemm(const void *Aq, const void *As, const void *Bq, const void *Bs, float *C,
                        int64_t M, int64_t N, int64_t K, const DeviceInfo &dev,
                        cudaStream_t stream) {
    return launch_gemm_elem<kFmtMX4>(Aq, As, Bq, Bs, C, M, N, K, nullptr, nullptr, dev, stream);
}

cudaError_t launch_gemm_fmt(int fmt, const void *Aq, const void *As, const void *Bq,
                            const void *Bs, float *C, int64_t M, int64_t N, int64_t K,
                            const float *amax_a, const float *amax_b, const DeviceInfo &dev,
                            cudaStream_t stream) {
    switch (fmt) {
        case kGemmMXFP4:
            return launch_gemm_elem<kFmtMX4>(Aq, As, Bq, Bs, C, M, N, K, nullptr, nullptr, dev,
                                             stream);
        case kGemmMXFP8:
            return launch_gemm_elem<kFmtMX8>(Aq, As, Bq, Bs, C, M, N, K, nullptr, nullptr, dev,
                                             stream);
        case kGemmNVFP4:
            if (amax_a == nullptr || amax_b == nullptr) return cudaErrorInvalidValue;
            return launch_gemm_elem<kFmtNV4>(Aq, As, Bq, Bs, C, M, N, K, amax_a, amax_b, dev,
                                             stream);
        default:
            return cudaErrorInvalidValue;
    }
}

size_t wgrad_fused_counter_bytes(int64_t T, int64_t N, int64_t K) {
    return static_cast<size_t>(4) * static_cast<size_t>((N + 255) / 256 + (K + 255) / 256) *
           static_cast<size_t>((T + 511) / 512);
}

bool wgrad_fusable(int64_t T, int64_t N, int64_t K, int rot, int rot_block, int rnd) {
    if (rnd != 0) return false;                               // round to nearest only
    if (rot == 2) return false;                               // no random signs
    if (rot == 1 && rot_block != 16 && rot_block != 32) return false;
    if (T < 512 || T % 512 != 0 || N < 256 || N % 256 != 0 || K < 256 || K % 256 != 0)
        return false;
    if (N / 256 + K / 256 > kMaxPanels) return false;
    return true;
}

cudaError_t launch_wgrad_fused(const void *dY, const void *X, float *dW, int64_t T, int64_t N,
                               int64_t K, int rot, int rot_block, void *Aq, void *As, void *Bq,
                               void *Bs, void *counters, const DeviceInfo &dev,
                               cudaStream_t stream) {
    CUtensorMap map_a, map_b;
    GemmArgs g;
    // dW[N][K] = A . B^T with A = dY^T (N lines), B = X^T (K lines), contraction T.
    if (!gemm_setup(kFmtMX4, Aq, As, Bq, Bs, dW, N, K, T, dev, &map_a, &map_b, &g))
        return cudaErrorInvalidValue;
    const int pairs_max = gemm_clusters<true, kFmtMX4>(dev);
    if (pairs_max < 1) return cudaErrorLaunchOutOfResources;
    const int pairs = g.num_items < pairs_max ? g.num_items : pairs_max;

    FusedArgs f;
    std::memset(&f, 0, sizeof(f));
    f.src[0] = static_cast<const uint32_t *>(dY);
    f.src[1] = static_cast<const uint32_t *>(X);
    f.codes[0] = static_cast<uint8_t *>(Aq);
    f.codes[1] = static_cast<uint8_t *>(Bq);
    f.scales[0] = static_cast<uint8_t *>(As);
    f.scales[1] = static_cast<uint8_t *>(Bs);
    f.words_per_row[0] = N / 2;
    f.words_per_row[1] = K / 2;
    f.T = T;
    f.katoms = scale_katoms(T);
    f.counters = static_cast<unsigned int *>(counters);
    f.rot_block = rot == 0 ? 0 : rot_block;
    f.chunks = static_cast<int>(T / 512);
    f.panels_a = g.m_tiles;
    // First-use order of the panels: walk the tiles round by round (one tile
    // per pair per round, in the kernel's banded order).
    std::vector<char> seen(static_cast<size_t>(g.m_tiles + g.n_tiles), 0);
    int np = 0, ng = 0;
    for (int r0 = 0; r0 < g.num_tiles; r0 += pairs) {
        const int start = np;
        for (int pass = 0; pass < 2; ++pass)
            for (int t = r0; t < g.num_tiles && t < r0 + pairs; ++t) {
                const int per_band = kBand * g.n_tiles;
                const int band = t / per_band, rr = t % per_band;
                const int first = band * kBand;
                const int rows = g.m_tiles - first < kBand ? g.m_tiles - first : kBand;
                const int p = pass == 0 ? first + rr % rows : g.m_tiles + rr / rows;
                if (!seen[p]) {
                    seen[p] = 1;
                    if (np >= kMaxPanels) return cudaErrorNotSupported;
                    f.panel[np++] = static_cast<uint16_t>(p);
                }
            }
        if (np > start) {
            if (ng >= kMaxGroups) return cudaErrorNotSupported;
            f.group_start[ng++] = static_cast<uint16_t>(start);
        }
    }
    f.group_start[ng] = static_cast<uint16_t>(np);
    f.groups = ng;
    f.units = kUnitsPerChunk * f.chunks * np;
    cudaError_t e = cudaMemsetAsync(counters, 0, wgrad_fused_counter_bytes(T, N, K), stream);
    if (e != cudaSuccess) return e;
    return gemm_launch<true, kFmtMX4>(map_a, map_b, g, f, pairs, stream);
}

}  // namespace mx
