// mx_peak.cu -- tensor-core issue-rate microbenchmark (measurement only).
//
// The roofline of the block-scaled GEMM needs the rate at which one SM
// retires tcgen05.mma instructions of the shapes the GEMM uses, and the cost
// of the tcgen05.cp copies that move block scales into tensor memory.  This
// kernel issues a stream of MMAs on operands that sit in shared memory (no
// TMA, no global traffic), optionally interleaved with scale copies and with
// a per-iteration commit handshake, and reports per-CTA elapsed time.  It is
// not on the compute path of any GEMM.
//
// Kinds timed (one MMA instruction, K per MMA = 32 bytes of each operand row):
//   0  kind::mxf4        E2M1 x E2M1, UE8M0 scales per 32, scale_vec::2X, K=64
//   1  kind::mxf4nvf4    the same operands and scales (scale_vec::2X),      K=64
//   2  kind::mxf4nvf4    UE4M3 scales per 16 (scale_vec::4X),               K=64
//   3  kind::f8f6f4      E4M3 x E4M3, no block scales,                      K=32
//   4  kind::f16         bf16 x bf16,                                       K=16
//   5  kind::mxf8f6f4    E4M3 x E4M3, UE8M0 scales per 32 (scale_vec::1X),  K=32
// All accumulate in fp32 in tensor memory.  cta_group::2 runs the M=256 form
// on a 2-CTA cluster (each CTA holds 128 rows of A and N/2 rows of B).
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/mx.h"
#include "mx_internal.h"
#include "mx_ptx.cuh"

namespace mx {
namespace {

constexpr int kPeakThreads = 256;
// Variants: copies fill the next iteration's scale slot instead of this one's;
// a commit every iteration with no wait; four more warps keep writing tensor
// memory with tcgen05.st while the MMAs run.
constexpr int kPeakCopyAhead = 1, kPeakCommitOnly = 2, kPeakStoreWarps = 4;
constexpr uint32_t kPeakA = 0;            // A tile: 128 rows x 128 B (16 KB)
constexpr uint32_t kPeakB = 16384;        // B tile: 256 rows x 128 B (32 KB)
constexpr uint32_t kPeakSF = 49152;       // scale source: 8 KB
constexpr uint32_t kPeakBars = 57344;     // 9 mbarriers: a ring of 8, one for set-up and drain
// Requested so that only one CTA fits on an SM (tensor memory stays free).
constexpr size_t kPeakSmem = 160 * 1024;

__host__ __device__ constexpr uint32_t peak_idesc(int kind, int M, int N, int sf_id) {
    // Block-scaled layout: B sf id [4,6), A fmt [7,10), B fmt [10,13), N>>3
    // [17,23), scale type [23], M>>4 [24,29), A sf id [29,31).  Plain layout:
    // accumulator format [4,6) (1 = fp32), formats and dims as above.
    return kind == 0 || kind == 1
               ? ((uint32_t(sf_id & 3) << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) |
                  (1u << 23) | (uint32_t(M >> 4) << 24) | (uint32_t(sf_id & 3) << 29))
           : kind == 2
               ? ((1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24))
           : kind == 3 ? ((1u << 4) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24))
           : kind == 4 ? ((1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) |
                          (uint32_t(M >> 4) << 24))
                       : ((uint32_t(sf_id & 3) << 4) | (uint32_t(N >> 3) << 17) | (1u << 23) |
                          (uint32_t(M >> 4) << 24) | (uint32_t(sf_id & 3) << 29));
}

#define MX_PEAK_MMA_BS(CG, KINDSTR)                                                          \
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"                          \
                 "tcgen05.mma.cta_group::" #CG "." KINDSTR                                   \
                 " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),                           \
                 "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)                     \
                 : "memory")
#define MX_PEAK_MMA(CG, KINDSTR)                                                             \
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"                          \
                 "tcgen05.mma.cta_group::" #CG "." KINDSTR " [%0], %1, %2, %3, p;\n\t}" ::"r"(d), \
                 "l"(a), "l"(b), "r"(idesc), "r"(acc)                                         \
                 : "memory")

template <int KIND, int CG>
__device__ __forceinline__ void peak_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t sfa, uint32_t sfb, uint32_t acc) {
    if constexpr (CG == 1) {
        if constexpr (KIND == 0) MX_PEAK_MMA_BS(1, "kind::mxf4.block_scale.scale_vec::2X");
        if constexpr (KIND == 1) MX_PEAK_MMA_BS(1, "kind::mxf4nvf4.block_scale.scale_vec::2X");
        if constexpr (KIND == 2) MX_PEAK_MMA_BS(1, "kind::mxf4nvf4.block_scale.scale_vec::4X");
        if constexpr (KIND == 3) MX_PEAK_MMA(1, "kind::f8f6f4");
        if constexpr (KIND == 4) MX_PEAK_MMA(1, "kind::f16");
        if constexpr (KIND == 5) MX_PEAK_MMA_BS(1, "kind::mxf8f6f4.block_scale.scale_vec::1X");
    } else {
        if constexpr (KIND == 0) MX_PEAK_MMA_BS(2, "kind::mxf4.block_scale.scale_vec::2X");
        if constexpr (KIND == 1) MX_PEAK_MMA_BS(2, "kind::mxf4nvf4.block_scale.scale_vec::2X");
        if constexpr (KIND == 2) MX_PEAK_MMA_BS(2, "kind::mxf4nvf4.block_scale.scale_vec::4X");
        if constexpr (KIND == 3) MX_PEAK_MMA(2, "kind::f8f6f4");
        if constexpr (KIND == 4) MX_PEAK_MMA(2, "kind::f16");
        if constexpr (KIND == 5) MX_PEAK_MMA_BS(2, "kind::mxf8f6f4.block_scale.scale_vec::1X");
    }
}
#undef MX_PEAK_MMA_BS
#undef MX_PEAK_MMA

// Scale copies (shared -> tensor memory) of the three shapes timed.
template <int CG>
__device__ __forceinline__ void peak_copy(int shape, uint32_t taddr, uint64_t sdesc) {
    if constexpr (CG == 1) {
        if (shape == 0)
            asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                         : "memory");
        else if (shape == 1)
            asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc)
                         : "memory");
        else
            asm volatile("tcgen05.cp.cta_group::1.128x128b [%0], %1;" ::"r"(taddr), "l"(sdesc)
                         : "memory");
    } else {
        if (shape == 0)
            asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                         : "memory");
        else if (shape == 1)
            asm volatile("tcgen05.cp.cta_group::2.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc)
                         : "memory");
        else
            asm volatile("tcgen05.cp.cta_group::2.128x128b [%0], %1;" ::"r"(taddr), "l"(sdesc)
                         : "memory");
    }
}

// Shared-memory descriptor of a non-swizzled copy source: 8-row x 16-byte
// core matrices of 128 contiguous bytes, 8-row groups 128 bytes apart and
// 16-byte column chunks 2048 bytes apart.
__device__ __forceinline__ uint64_t peak_cp_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(2048 >> 4) << 16) |
           (static_cast<uint64_t>(128 >> 4) << 32) | (static_cast<uint64_t>(1) << 46);
}

template <int CG>
__device__ __forceinline__ void peak_commit(uint64_t *bar) {
    if constexpr (CG == 1) {
        tc_commit(bar);
    } else {
        // Signals the barrier at the same offset in both CTAs of the pair.
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
            " [%0], %1;" ::"r"(smem_u32(bar)),
            "h"(static_cast<uint16_t>(3))
            : "memory");
    }
}

struct PeakArgs {
    int n;               // MMA N (128 or 256)
    int mmas_per_iter;   // MMAs issued per iteration
    int copies_per_iter; // scale copies issued before them
    int copy_shape;      // 0: 32x128b.warpx4, 1: 128x256b, 2: 128x128b
    int depth;           // 0: no handshake; d: commit per iteration, wait for iteration it-d
    int flags;           // kPeakCopyAhead | kPeakCommitOnly | kPeakStoreWarps
    int64_t iters;
    int64_t *ns_out;     // per CTA: elapsed ns of the issuing thread (0 for pair peers)
    int *status;
};

template <int KIND, int CG>
__global__ void __launch_bounds__(kPeakThreads, 1) mx_peak_mma_kernel(const PeakArgs g) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ int store_done;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kPeakBars);
    const int warp = threadIdx.x >> 5;
    uint32_t rank = 0;
    if constexpr (CG == 2) asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));

    // Operand and scale bytes: small finite values of every element type.
    for (uint32_t i = threadIdx.x; i < kPeakBars / 4; i += blockDim.x) {
        uint32_t h = i * 0x9E3779B1u + 0x7F4A7C15u;
        h ^= h >> 15;
        h *= 0x2C1B3C6Du;
        h ^= h >> 12;
        uint32_t w = h & 0x3F3F3F3Fu;
        if (i * 4 >= kPeakSF) w = KIND == 2 ? 0x38383838u : 0x7F7F7F7Fu;  // scale 1.0
        reinterpret_cast<uint32_t *>(smem)[i] = w;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < 9; ++s) mbar_init(&bars[s], 1);
        abort_flag = 0;
        store_done = (g.flags & kPeakStoreWarps) ? 0 : 1;
        fence_barrier_init();
    }
    fence_proxy_async_smem();
    if (warp == 0) {
        if constexpr (CG == 1) {
            tmem_alloc(&tmem_slot, 512);
            tmem_relinquish();
        } else {
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                             smem_u32(&tmem_slot))
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (CG == 2) cluster_sync();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (threadIdx.x == 0 && rank == 0) {
        const int M = 128 * CG;
        const uint32_t sa = smem_u32(smem + kPeakA), sb = smem_u32(smem + kPeakB);
        const uint32_t sf = smem_u32(smem + kPeakSF);
        // Valid scales in every scale column before the timed loop.
        for (uint32_t c = 256; c < 512; c += 4) peak_copy<CG>(0, tmem + c, sdesc_sf(sf));
        peak_commit<CG>(&bars[8]);
        bool ok = mbar_wait(&bars[8], 0, g.status, &abort_flag);
        const uint64_t t0 = global_timer_ns();
        for (int64_t it = 0; ok && it < g.iters; ++it) {
            const uint32_t slot = 256u + 48u * static_cast<uint32_t>(it & 3);
            const uint32_t cslot = (g.flags & kPeakCopyAhead)
                                       ? 256u + 48u * static_cast<uint32_t>((it + 1) & 3)
                                       : slot;
            for (int c = 0; c < g.copies_per_iter; ++c)
                peak_copy<CG>(g.copy_shape, tmem + cslot + 8u * static_cast<uint32_t>(c % 6),
                              g.copy_shape == 0 ? sdesc_sf(sf + 512u * (c & 7))
                                                : peak_cp_desc(sf + 16u * (c & 1)));
            for (int j = 0; j < g.mmas_per_iter; ++j) {
                const uint32_t ka = (j >> 1) & 1;
                const uint32_t idesc = peak_idesc(KIND, M, g.n, KIND == 5 ? (j & 3) : (j & 1) * 2);
                peak_mma<KIND, CG>(tmem, sdesc_sw128(sa + 32u * (j & 3)),
                                   sdesc_sw128(sb + 32u * (j & 3)), idesc, tmem + slot + 4u * ka,
                                   tmem + slot + 8u + 8u * ka, (it > 0 || j > 0) ? 1u : 0u);
            }
            if (g.depth > 0) {
                // Iteration it commits to ring barrier it % 8 (its (it / 8)-th
                // phase), then waits for the commit of iteration it - depth.
                // depth < 8, so that barrier's next commit is not issued yet
                // and its parity is unambiguous.
                peak_commit<CG>(&bars[it & 7]);
                if (!(g.flags & kPeakCommitOnly) && it >= g.depth) {
                    const int64_t w = it - g.depth;
                    ok = mbar_wait(&bars[w & 7], static_cast<uint32_t>(w >> 3) & 1u, g.status,
                                   &abort_flag);
                }
            }
        }
        // Drain: the set-up barrier's second phase completes once every
        // operation issued above has.
        if (ok) {
            peak_commit<CG>(&bars[8]);
            ok = mbar_wait(&bars[8], 1, g.status, &abort_flag);
        }
        const uint64_t t1 = global_timer_ns();
        g.ns_out[blockIdx.x] = ok ? static_cast<int64_t>(t1 - t0) : -1;
        store_done = 1;
    } else if (threadIdx.x == 0) {
        g.ns_out[blockIdx.x] = 0;
    } else if (rank == 0 && warp >= 4 && (g.flags & kPeakStoreWarps)) {
        // Warp w writes eight columns of its lane quarter over and over
        // (columns 448.., which no MMA reads) until the MMAs are done.
        const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + 448u;
        uint32_t v[8];
        for (int i = 0; i < 8; ++i) v[i] = 0x7F7F7F7Fu;
        volatile int *done = &store_done;
        for (int64_t k = 0; k < 100000000; ++k) {
            // One lane reads the flag for the whole warp: the stores below are
            // .sync.aligned, so the warp must leave the loop together.
            int stop = (threadIdx.x & 31) == 0 ? *done : 0;
            if (__shfl_sync(0xFFFFFFFFu, stop, 0)) break;
            asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                             taddr + 8u * static_cast<uint32_t>(k & 7)),
                         "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
                         "r"(v[6]), "r"(v[7])
                         : "memory");
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            __syncwarp();
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (CG == 2) cluster_sync();
    if (warp == 0) {
        tc_fence_after();
        if constexpr (CG == 1)
            tmem_dealloc(tmem, 512);
        else
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, 512;" ::"r"(tmem)
                         : "memory");
    }
}

template <int KIND, int CG>
cudaError_t launch_peak(const PeakArgs &g, const DeviceInfo &dev, cudaStream_t stream,
                        int *ctas) {
    auto kern = mx_peak_mma_kernel<KIND, CG>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kPeakSmem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.blockDim = dim3(kPeakThreads, 1, 1);
    cfg.dynamicSmemBytes = kPeakSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    cfg.gridDim = dim3(CG, 1, 1);
    e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters < 1) return cudaErrorLaunchOutOfResources;
    int n = clusters * CG;
    if (n > dev.sm_count) n = dev.sm_count - dev.sm_count % CG;
    if (n > 256) n = 256;
    cfg.gridDim = dim3(n, 1, 1);
    *ctas = n;
    e = cudaLaunchKernelEx(&cfg, kern, g);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace
}  // namespace mx

extern "C" mx_status mx_bench_mma(int kind, int cta_group, int n, int mmas_per_iter,
                                  int copies_per_iter, int copy_shape, int depth, int flags,
                                  int64_t iters, int64_t *d_ns, int *h_ctas, void *stream) {
    using namespace mx;
    if (kind < 0 || kind > 5 || (cta_group != 1 && cta_group != 2) || (n != 128 && n != 256) ||
        mmas_per_iter < 1 || mmas_per_iter > 64 || copies_per_iter < 0 || copies_per_iter > 32 ||
        copy_shape < 0 || copy_shape > 2 || depth < 0 || depth > 7 || flags < 0 || flags > 7 ||
        iters < 1 ||
        iters > 10000000 || d_ns == nullptr || h_ctas == nullptr)
        return MX_ERR_INVALID_ARG;
    cudaError_t err = cudaSuccess;
    const DeviceInfo *dev = current_device(&err);
    if (dev == nullptr) return MX_ERR_CUDA;
    if (!(dev->cc_major == 10 && dev->cc_minor == 3)) return MX_ERR_UNSUPPORTED;
    PeakArgs g{n, mmas_per_iter, copies_per_iter, copy_shape, depth, flags, iters, d_ns,
               dev->status};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaErrorInvalidValue;
#define MX_PEAK_CASE(K)                                                                 \
    case K:                                                                             \
        e = cta_group == 1 ? launch_peak<K, 1>(g, *dev, s, h_ctas)                      \
                           : launch_peak<K, 2>(g, *dev, s, h_ctas);                     \
        break;
    switch (kind) {
        MX_PEAK_CASE(0)
        MX_PEAK_CASE(1)
        MX_PEAK_CASE(2)
        MX_PEAK_CASE(3)
        MX_PEAK_CASE(4)
        MX_PEAK_CASE(5)
        default: break;
    }
#undef MX_PEAK_CASE
    return e == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}
