// mx_gemm.cu -- block-scaled MXFP4 GEMM on the sm_103a tensor cores.
//
// C[M][N] (fp32) = A . B^T with A, B MXFP4-encoded along the contraction
// dimension K: the Fprop, Dgrad and Wgrad GEMMs of "Neue Studie von AMD
// durchbricht die bestehende Erkenntnis" (eu.36kr.com), section
// "Fehlerdiagnoseexperiment", run on native FP4 tensor cores with fp32
// accumulation.
//
// Design (one CTA per SM, persistent over 128 x 256 output tiles):
//   schedule     CTA b takes work items b, b + G, b + 2G, ... (G CTAs, in
//                clusters of two).  An item is a whole tile, except in a last
//                round that would leave at least half of the CTAs idle (tiles
//                mod G <= G/2): there each remaining tile becomes two items,
//                the two halves of its K range, run by the two CTAs of one
//                cluster.  Each CTA then stores one column half of the tile:
//                it leaves its fp32 partial of the other column half in its
//                own shared memory (its stage ring is idle by then), reads
//                the partner's partial of its own half through distributed
//                shared memory, adds the two (fp32 addition of the two K
//                halves is commutative, so both CTAs' sums are the same bits)
//                and stores.  The last round then takes about half a tile
//                time instead of a whole one.
//   warp 0       TMA producer: 128B-swizzled A/B code tiles (K-tile of 256
//                FP4 = 128 bytes per row) and the two matching 1 KB scale
//                slabs per 128 rows, into a 4-stage shared-memory ring.
//   warp 1       tensor-memory allocator and single-thread MMA issuer: per
//                stage, tcgen05.cp moves the scale slabs into tensor memory,
//                then four tcgen05.mma kind::mxf4 (K = 64 each, two E8M0
//                scales per row per MMA) accumulate into a 128 x 256 fp32
//                tile held in tensor memory; tcgen05.commit frees the stage.
//   warps 2..9   epilogue: tcgen05.ld the accumulator (each warp one 32-lane
//                quarter x 128 columns) into registers, release tensor
//                memory to the MMA warp at once, then store fp32 rows while
//                the next tile's main loop runs.  A CTA's last item, whose
//                stores nothing overlaps, is staged in the idle stage ring
//                (128-byte swizzled 32 x 32 boxes) and written by TMA stores
//                of whole lines.
// Every wait is bounded (see mx_ptx.cuh); a timeout records an error and the
// CTA unwinds without faulting.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>

#include "mx_internal.h"
#include "mx_ptx.cuh"

namespace mx {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBKBytes = 128;                 // 256 FP4 values per row per K-tile
constexpr int kStages = 4;
constexpr int kThreads = 320;                 // 10 warps
constexpr int kEpiWarps = 8;
constexpr uint32_t kABytes = kBM * kBKBytes;  // 16 KB
constexpr uint32_t kBBytes = kBN * kBKBytes;  // 32 KB
constexpr uint32_t kSFABytes = 1024;          // 128 rows x 8 blocks
constexpr uint32_t kSFBBytes = 2048;          // 256 rows x 8 blocks
constexpr uint32_t kStageBytes = kABytes + kBBytes + kSFABytes + kSFBBytes;  // 52 KB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;               // accumulator: columns [0, 256)
constexpr uint32_t kSFCol = 256;              // per-stage scale columns: 32 per stage

struct GemmArgs {
    const uint8_t *As;
    const uint8_t *Bs;
    float *C;
    int64_t M, N, K;
    int64_t katoms;      // scale k-atoms per 128-row group
    int64_t b_groups;    // 128-row scale groups that exist for B
    int k_tiles;
    int n_tiles;
    int num_tiles;
    int num_items;       // whole tiles [0, dp_tiles), then two K halves per remaining tile
    int dp_tiles;
    int k_split;         // first K-tile of a second half
    int c_v8;            // C rows allow 32-byte stores (N % 8 == 0, C 32-byte aligned)
    int c_tma;           // C allows TMA stores (N % 4 == 0, C 16-byte aligned)
    size_t c_bytes;      // extent of C (store guards)
    int *status;
};

struct SharedCtl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t acc_full;
    uint64_t acc_empty;
    uint64_t drain;
    uint64_t part_ready;  // split tile: the partner's partial of this CTA's column half is in place
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ void st_global_v4f(float *p, uint32_t a, uint32_t b, uint32_t c,
                                              uint32_t d) {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// One full 32-byte sector per store (the address must be 32-byte aligned).
__device__ __forceinline__ void st_global_v8(float *p, const uint32_t *v) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

// Work item w: output tile, K-tile range [k0, k1), and which K half it is
// (-1: the whole range).
struct Item {
    int tile, k0, k1, khalf;
};
__device__ __forceinline__ Item item_of(const GemmArgs &g, int w) {
    if (w < g.dp_tiles) return Item{w, 0, g.k_tiles, -1};
    const int j = w - g.dp_tiles, h = j % 2;
    return Item{g.dp_tiles + j / 2, h == 0 ? 0 : g.k_split, h == 0 ? g.k_split : g.k_tiles, h};
}

// A split tile's partial of one column half: the 128 epilogue threads that
// hold that half (4 warps) keep 128 fp32 values each, as 32 chunks of 16
// bytes; chunk i of thread t of the half sits at (i * 128 + t) * 16, so a
// warp's 16-byte accesses to one chunk are contiguous.
constexpr int kHalfThreads = 16 * kEpiWarps;
constexpr uint32_t kPartialBytes = 32u * kHalfThreads * 16u;  // 64 KB
static_assert(kPartialBytes <= kStages * kStageBytes, "the partial lives in the stage ring");
// TMA-store staging of a last item: per epilogue warp, four 32 x 32 fp32
// boxes (4 KB each, 128-byte swizzle), after the partial.
constexpr uint32_t kStageOutBytes = 4u * 4096u;
static_assert(kPartialBytes + kEpiWarps * kStageOutBytes <= kStages * kStageBytes,
              "the output staging lives in the stage ring");

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                   const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ CUtensorMap map_c, const GemmArgs g) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned base, kept as a shared-space pointer (offset arithmetic
    // only) so that the compiler emits shared-memory loads.
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    SharedCtl *ctl = reinterpret_cast<SharedCtl *>(smem + kStages * kStageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        mbar_init(&ctl->acc_full, 1);
        mbar_init(&ctl->acc_empty, kEpiWarps);
        mbar_init(&ctl->drain, 1);
        mbar_init(&ctl->part_ready, kEpiWarps / 2);
        ctl->abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&map_a);
        prefetch_tmap(&map_b);
        if (g.c_tma) prefetch_tmap(&map_c);
    }
    if (warp == 1) {
        tmem_alloc(&ctl->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    // Both CTAs of the cluster have initialised their barriers before either
    // signals the other.
    __syncwarp();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    volatile int *abort = &ctl->abort_flag;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int w = blockIdx.x; ok && w < g.num_items; w += gridDim.x) {
                const Item it = item_of(g, w);
                const int mb = it.tile / g.n_tiles, nb = it.tile % g.n_tiles;
                for (int kt = it.k0; kt < it.k1; ++kt) {
                    if (!mbar_wait(&ctl->empty[stage], phase ^ 1u, g.status, abort)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sa = smem + stage * kStageBytes;
                    uint8_t *sb = sa + kABytes;
                    uint8_t *sfa = sb + kBBytes;
                    uint8_t *sfb = sfa + kSFABytes;
                    const int64_t g0 = 2 * static_cast<int64_t>(nb);
                    const uint32_t nsfb = (g0 + 1 < g.b_groups) ? 2u : 1u;
                    mbar_arrive_expect_tx(&ctl->full[stage],
                                          kABytes + kBBytes + kSFABytes + nsfb * 1024u);
                    tma_load_2d(sa, &map_a, &ctl->full[stage], kt * kBKBytes, mb * kBM);
                    tma_load_2d(sb, &map_b, &ctl->full[stage], kt * kBKBytes, nb * kBN);
                    bulk_load(sfa, g.As + (static_cast<int64_t>(mb) * g.katoms + 2 * kt) * 512,
                              1024u, &ctl->full[stage]);
                    for (uint32_t rb = 0; rb < nsfb; ++rb)
                        bulk_load(sfb + rb * 1024u,
                                  g.Bs + ((g0 + rb) * g.katoms + 2 * kt) * 512, 1024u,
                                  &ctl->full[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int w = blockIdx.x; ok && w < g.num_items; w += gridDim.x) {
                const Item it = item_of(g, w);
                if (!mbar_wait(&ctl->acc_empty, acc_phase ^ 1u, g.status, abort)) break;
                tc_fence_after();
                for (int kt = it.k0; kt < it.k1; ++kt) {
                    if (!mbar_wait(&ctl->full[stage], phase, g.status, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * kStageBytes);
                    const uint32_t sb = sa + kABytes;
                    const uint32_t sfa = sb + kBBytes;
                    const uint32_t sfb = sfa + kSFABytes;
                    const uint32_t sf_col = tmem + kSFCol + 32u * stage;
                    // Scale slabs -> tensor memory.  A: 4 columns per k-atom.
                    // B: per k-atom, 4 columns per 128-row group (rows 128..255
                    // of the 256-row tile follow rows 0..127).
#pragma unroll
                    for (int ka = 0; ka < 2; ++ka) {
                        tmem_cp_32x128b_x4(sf_col + 4u * ka, sdesc_sf(sfa + 512u * ka));
#pragma unroll
                        for (int rb = 0; rb < 2; ++rb)
                            tmem_cp_32x128b_x4(sf_col + 8u + 8u * ka + 4u * rb,
                                               sdesc_sf(sfb + 1024u * rb + 512u * ka));
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int ka = j / 2, sf_id = (j % 2) * 2;
                        mma_mxf4(tmem + kAccCol, sdesc_sw128(sa + 32u * j),
                                 sdesc_sw128(sb + 32u * j), idesc_mxf4(kBM, kBN, sf_id, sf_id),
                                 sf_col + 4u * ka, sf_col + 8u + 8u * ka,
                                 (kt > it.k0 || j > 0) ? 1u : 0u);
                    }
                    tc_commit(&ctl->empty[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                tc_commit(&ctl->acc_full);
                acc_phase ^= 1u;
            }
            // Make sure every tensor-core operation issued here has finished
            // before tensor memory is released.
            tc_commit(&ctl->drain);
            mbar_wait(&ctl->drain, 0, g.status, nullptr, 100ull * 1000ull * 1000ull);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;           // TMEM lane quarter this warp may access
        const int half = (warp - 2) / 4;  // column half of the 256-wide tile
        uint32_t acc_phase = 0;
        const int ht = ((warp - 2) & 3) * 32 + lane;  // thread index within its column half
        for (int w = blockIdx.x; w < g.num_items; w += gridDim.x) {
            const Item it = item_of(g, w);
            const int mb = it.tile / g.n_tiles, nb = it.tile % g.n_tiles;
            // One lane waits; the verdict is broadcast so the warp stays
            // converged for the .sync.aligned tensor-memory loads.
            int ok = 1;
            if (lane == 0) ok = mbar_wait(&ctl->acc_full, acc_phase, g.status, abort) ? 1 : 0;
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            uint32_t v[4][32];
            const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16) + kAccCol +
                                   128u * half;
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(tbase + 32u * c, v[c]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->acc_empty);
            acc_phase ^= 1u;

            if (it.khalf >= 0) {
                // Split tile: CTA rank r (= it.khalf) stores column half r.
                if (half != it.khalf) {
                    // Leave this half's partial for the partner and signal it.
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            uint4 *dst = reinterpret_cast<uint4 *>(
                                smem + (static_cast<uint32_t>((8 * c + j) * kHalfThreads + ht) << 4));
                            *dst = make_uint4(v[c][4 * j], v[c][4 * j + 1], v[c][4 * j + 2],
                                              v[c][4 * j + 3]);
                        }
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->part_ready), 1u - it.khalf));
                    continue;
                }
                int okp = 1;
                if (lane == 0) okp = mbar_wait_cluster(&ctl->part_ready, 0, g.status, abort) ? 1 : 0;
                okp = __shfl_sync(0xFFFFFFFFu, okp, 0);
                if (!okp) break;
                // Every lane takes the acquire itself (the phase is complete).
                mbar_wait_cluster(&ctl->part_ready, 0, g.status, abort);
                const uint32_t peer = mapa_shared(smem_u32(smem), 1u - it.khalf);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 p[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        p[j] = ld_shared_cluster_v4(
                            peer + (static_cast<uint32_t>((8 * c + j) * kHalfThreads + ht) << 4));
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        v[c][4 * j] = __float_as_uint(__uint_as_float(v[c][4 * j]) + __uint_as_float(p[j].x));
                        v[c][4 * j + 1] =
                            __float_as_uint(__uint_as_float(v[c][4 * j + 1]) + __uint_as_float(p[j].y));
                        v[c][4 * j + 2] =
                            __float_as_uint(__uint_as_float(v[c][4 * j + 2]) + __uint_as_float(p[j].z));
                        v[c][4 * j + 3] =
                            __float_as_uint(__uint_as_float(v[c][4 * j + 3]) + __uint_as_float(p[j].w));
                    }
                }
            }

            if (g.c_tma && w + static_cast<int>(gridDim.x) >= g.num_items) {
                // Last item: stage this warp's 32 rows x 128 columns as four
                // swizzled boxes and store them with TMA (rows and columns
                // outside C are not written).
                uint8_t *stg = smem + kPartialBytes + static_cast<uint32_t>(warp - 2) * kStageOutBytes;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint4 *dst = reinterpret_cast<uint4 *>(
                            stg + c * 4096 + lane * 128 + (((j ^ (lane & 7)) & 7) << 4));
                        *dst = make_uint4(v[c][4 * j], v[c][4 * j + 1], v[c][4 * j + 2],
                                          v[c][4 * j + 3]);
                    }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const int32_t r0 = mb * kBM + 32 * q;
                    const int32_t cb = nb * kBN + 128 * half;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        if (cb + 32 * c < g.N && r0 < g.M)  // boxes that start inside C only
                            tma_store_2d(&map_c, stg + c * 4096, cb + 32 * c, r0);
                    bulk_commit_group();
                    bulk_wait_group_0();
                }
                __syncwarp();
                continue;
            }
            const int64_t row = static_cast<int64_t>(mb) * kBM + 32 * q + lane;
            if (row < g.M) {
                float *crow = g.C + row * g.N;
                const int64_t col0 = static_cast<int64_t>(nb) * kBN + 128 * half;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (g.c_v8 && col0 + 32 * c + 31 < g.N) {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (MX_STORE_OK(crow + col0 + 32 * c + 8 * j, 32, g.C, g.c_bytes, g.status))
                                st_global_v8(crow + col0 + 32 * c + 8 * j, &v[c][8 * j]);
                        continue;
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int64_t col = col0 + 32 * c + 4 * j;
                        if (col + 3 < g.N) {
                            if (MX_STORE_OK(crow + col, 16, g.C, g.c_bytes, g.status))
                                st_global_v4f(crow + col, v[c][4 * j], v[c][4 * j + 1],
                                              v[c][4 * j + 2], v[c][4 * j + 3]);
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (col + e < g.N &&
                                    MX_STORE_OK(crow + col + e, 4, g.C, g.c_bytes, g.status))
                                    crow[col + e] = __uint_as_float(v[c][4 * j + e]);
                        }
                    }
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    // Neither CTA of a cluster leaves while the other may still read its
    // shared memory.
    __syncwarp();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

constexpr size_t kGemmSmem = kStages * kStageBytes + sizeof(SharedCtl) + 1024;

// Co-resident 2-CTA clusters of mx_gemm_kernel on a device, measured once.
int gemm_clusters(const DeviceInfo &dev) {
    static std::atomic<int> cache[64];
    const int idx = dev.ordinal >= 0 && dev.ordinal < 64 ? dev.ordinal : 0;
    int n = cache[idx].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaFuncSetAttribute(mx_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kGemmSmem)) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kGemmSmem;
    if (cudaOccupancyMaxActiveClusters(&n, mx_gemm_kernel, &cfg) != cudaSuccess || n < 1) return 0;
    cache[idx].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace

cudaError_t launch_gemm(const void *Aq, const void *As, const void *Bq, const void *Bs, float *C,
                        int64_t M, int64_t N, int64_t K, const DeviceInfo &dev,
                        cudaStream_t stream) {
    CUtensorMap map_a, map_b, map_c;
    if (!encode_tmap_2d(&map_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, Aq, K / 2, M, K / 2, kBKBytes, kBM,
                        CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (!encode_tmap_2d(&map_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, Bq, K / 2, N, K / 2, kBKBytes, kBN,
                        CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    GemmArgs g{};
    g.As = static_cast<const uint8_t *>(As);
    g.Bs = static_cast<const uint8_t *>(Bs);
    g.C = C;
    g.M = M;
    g.N = N;
    g.K = K;
    g.katoms = scale_katoms(K);
    g.b_groups = scale_groups(N);
    g.k_tiles = static_cast<int>((K + 255) / 256);
    const int64_t m_tiles = (M + kBM - 1) / kBM;
    const int64_t n_tiles = (N + kBN - 1) / kBN;
    if (m_tiles * n_tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
    g.n_tiles = static_cast<int>(n_tiles);
    g.num_tiles = static_cast<int>(m_tiles * n_tiles);
    g.c_v8 = (N % 8 == 0 && (reinterpret_cast<uintptr_t>(C) & 31) == 0) ? 1 : 0;
    std::memset(&map_c, 0, sizeof(map_c));
    g.c_tma = (N % 4 == 0 && (reinterpret_cast<uintptr_t>(C) & 15) == 0 &&
               encode_tmap_2d(&map_c, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, N, M,
                              static_cast<uint64_t>(N) * sizeof(float), 32, 32,
                              CU_TENSOR_MAP_SWIZZLE_128B))
                  ? 1
                  : 0;
    g.c_bytes = static_cast<size_t>(M) * static_cast<size_t>(N) * sizeof(float);
    g.status = dev.status;
    cudaError_t e = cudaFuncSetAttribute(mx_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kGemmSmem));
    if (e != cudaSuccess) return e;
    // Resident CTAs: as many 2-CTA clusters as fit at once.
    const int slots = 2 * gemm_clusters(dev);
    if (slots < 2) return cudaErrorLaunchOutOfResources;
    const int rem = g.num_tiles % slots;
    g.dp_tiles = g.num_tiles;
    g.num_items = g.num_tiles;
    g.k_split = g.k_tiles;
    if (rem > 0 && 2 * rem <= slots && g.k_tiles >= 2) {
        g.dp_tiles = g.num_tiles - rem;
        g.num_items = g.dp_tiles + 2 * rem;
        g.k_split = g.k_tiles / 2;
    }
    int grid = g.num_items < slots ? g.num_items : slots;
    grid += grid & 1;
    mx_gemm_kernel<<<grid, kThreads, kGemmSmem, stream>>>(map_a, map_b, map_c, g);
    return cudaGetLastError();
}

}  // namespace mx
