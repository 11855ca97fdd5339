// mx_ptx.cuh -- inline-PTX building blocks for sm_103a kernels: mbarriers
// with bounded waits, TMA (tensor and bulk) copies, and the tcgen05 tensor-core
// / tensor-memory instructions.  Written against the public PTX ISA.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace mx {

// Device status codes written into the per-device status word.
enum : int { kDevOk = 0, kDevTimeout = 6, kDevBounds = 8 };

// Store guard.  In a build with MX_CHECKED=1 every global store of the
// kernels first checks that [p, p + n) lies inside [base, base + size); a
// store that would not is skipped and recorded as kDevBounds in the status
// word (no trap).  Normal builds compile the guard away.
#if defined(MX_CHECKED) && MX_CHECKED
__device__ __forceinline__ bool mx_store_ok(const void *p, size_t n, const void *base, size_t size,
                                            int *status) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(base);
    if (a >= b && a + n <= b + size) return true;
    if (status != nullptr) atomicExch(status, kDevBounds);
    return false;
}
#define MX_STORE_OK(p, n, base, size, status) mx_store_ok((p), (n), (base), (size), (status))
#else
#define MX_STORE_OK(p, n, base, size, status) true
#endif

// Every spin-wait in this library gives up after this long (or after
// kWaitMaxPolls polls, whichever comes first) and records kDevTimeout.
constexpr uint64_t kWaitLimitNs = 2000ull * 1000ull * 1000ull;  // 2 s
constexpr uint32_t kWaitMaxPolls = 1u << 30;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- launch order
// Programmatic dependent launch.  The library's kernels are launched so that
// each may start while the previous kernel of its stream is still finishing:
// every thread first waits here until that kernel has completed and its
// memory is visible (a no-op for a kernel launched without the attribute),
// touching no global memory before.  Then it allows its own successor to
// launch early under the same rule.
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for phase `parity` of `bar`.  Returns false (and records a
// timeout in *status, if given) when the limit expires or when *abort is set
// by another thread of the CTA that already gave up.
static __device__ __noinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *status,
                                       volatile int *abort, uint64_t limit_ns = kWaitLimitNs) {
    const uint32_t addr = smem_u32(bar);
    if (mbar_try_wait(addr, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t poll = 0; poll < kWaitMaxPolls; ++poll) {
        if (mbar_try_wait(addr, parity)) return true;
        if ((poll & 63u) == 63u) {
            if (abort != nullptr && *abort) return false;
            if (global_timer_ns() - t0 > limit_ns) break;
        }
    }
    if (status != nullptr) atomicExch(status, kDevTimeout);
    if (abort != nullptr) *abort = 1;
    return false;
}

// The same bounded wait, inlined: kernels that split registers between
// warpgroups (setmaxnreg) cannot call out of line.
static __device__ __forceinline__ bool mbar_wait_inl(uint64_t *bar, uint32_t parity, int *status,
                                                     volatile int *abort,
                                                     uint64_t limit_ns = kWaitLimitNs) {
    const uint32_t addr = smem_u32(bar);
    if (mbar_try_wait(addr, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t poll = 0; poll < kWaitMaxPolls; ++poll) {
        if (mbar_try_wait(addr, parity)) return true;
        if ((poll & 63u) == 63u) {
            if (abort != nullptr && *abort) return false;
            if (global_timer_ns() - t0 > limit_ns) break;
        }
    }
    if (status != nullptr) atomicExch(status, kDevTimeout);
    if (abort != nullptr) *abort = 1;
    return false;
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load: box at (c0 = innermost coordinate, c1) into shared `dst`,
// completion signalled on `bar` (transaction bytes).
// Brings a 2-D box of a tensor into L2 ahead of its load (no shared memory,
// no barrier; coordinates outside the tensor are ignored like a load's).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int32_t c0, int32_t c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// L2 eviction policies for the cache-hinted copies below (the whole access
// range at one priority).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void tma_load_2d_hint(void *dst, const CUtensorMap *map, uint64_t *bar,
                                                 int32_t c0, int32_t c1, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap *map, const void *src,
                                                  int32_t c0, int32_t c1, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void bulk_store_hint(void *dst, const void *src, uint32_t bytes,
                                                uint64_t policy) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(
                     reinterpret_cast<uint64_t>(dst)),
                 "r"(smem_u32(src)), "r"(bytes), "l"(policy)
                 : "memory");
}

// 2-D tiled store of a shared-memory box at (c0 = innermost coordinate, c1);
// the part of the box outside the tensor is not written.  Completion is
// tracked by bulk groups (bulk_commit_group / bulk_wait_group_0).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int32_t c0,
                                             int32_t c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until every committed bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_group_0() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Waits until at most N committed bulk groups of this thread are still
// reading their shared-memory sources (the writes to global may still be in
// flight).
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Contiguous bulk store from shared to global memory (16-byte aligned
// addresses, size a multiple of 16), tracked by bulk groups.
__device__ __forceinline__ void bulk_store(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                     reinterpret_cast<uint64_t>(dst)),
                 "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
}
// Named barrier over `nthreads` threads (whole warps) that also ANDs a
// predicate across them: every participant gets the same result.
__device__ __forceinline__ bool bar_and(int id, int nthreads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}
// Orders this thread's prior shared-memory writes before later async-proxy
// (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Contiguous bulk load (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------- clusters
// All threads of every CTA in the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Shared::cluster address of the object at shared address `saddr` in the
// CTA of rank `rank` within this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
// 2-D tiled load into this CTA's shared memory whose completion (bytes) is
// signalled on an mbarrier in either CTA of the pair, given by its
// shared::cluster address.
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *map, uint32_t bar,
                                                 int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}
// Arrive on an mbarrier given by its shared::cluster address with the
// default semantics (release at CTA scope).  Enough where the arrive only
// orders tensor-core work (tcgen05 fences) or nothing at all; much cheaper
// than a cluster-scope release, which waits for this thread's outstanding
// memory traffic.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Arrive on an mbarrier given by its shared::cluster address, releasing this
// thread's prior writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}
// Bounded wait on an mbarrier of this CTA with acquire at cluster scope, for
// phases completed by arrivals from other CTAs of the cluster.  Same limits
// and error reporting as mbar_wait.
static __device__ __noinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity, int *status,
                                                      volatile int *abort) {
    const uint32_t addr = smem_u32(bar);
    const uint64_t t0 = global_timer_ns();
    for (uint32_t poll = 0; poll < kWaitMaxPolls; ++poll) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(addr), "r"(parity)
            : "memory");
        if (ok) return true;
        if ((poll & 63u) == 63u) {
            if (abort != nullptr && *abort) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) break;
        }
    }
    if (status != nullptr) atomicExch(status, kDevTimeout);
    if (abort != nullptr) *abort = 1;
    return false;
}
// 16-byte load from the shared memory of a CTA of this cluster.
__device__ __forceinline__ uint4 ld_shared_cluster_v4(uint32_t cluster_addr) {
    uint4 v;
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(cluster_addr)
                 : "memory");
    return v;
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t *slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, K-major operand tile stored with the
// 128-byte swizzle (rows of 128 bytes, 8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
    d |= static_cast<uint64_t>(1) << 16;                  // leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;          // stride byte offset: 8 rows
    d |= static_cast<uint64_t>(1) << 46;                  // descriptor version (sm_100 family)
    d |= static_cast<uint64_t>(2) << 61;                  // 128-byte swizzle
    return d;
}

// Shared-memory descriptor for a 32-row x 16-byte scale-factor slab
// (no swizzle; 8-row core matrices of 128 contiguous bytes).
__device__ __forceinline__ uint64_t sdesc_sf(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(128 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    return d;
}

// Instruction descriptor for kind::mxf4 (E2M1 x E2M1, E8M0 scales, fp32
// accumulate, both operands K-major), tile M x N, scale-factor byte ids.
__host__ __device__ constexpr uint32_t idesc_mxf4(int M, int N, int a_sf_id, int b_sf_id) {
    return (static_cast<uint32_t>(b_sf_id & 3) << 4)      // B scale-factor id
           | (1u << 7)                                    // A format: E2M1
           | (1u << 10)                                   // B format: E2M1
           | (static_cast<uint32_t>(N >> 3) << 17)        // N / 8
           | (1u << 23)                                   // scale format: UE8M0
           | (static_cast<uint32_t>(M >> 4) << 24)        // M / 16
           | (static_cast<uint32_t>(a_sf_id & 3) << 29);  // A scale-factor id
}

// D[tmem] (+)= A[smem] . B[smem]^T with per-32 block scales from tensor memory.
__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X"
        " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Copy a 32-row x 128-bit slab from shared memory into tensor memory,
// replicated into all four 32-lane sub-partitions.
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Each thread of the warp reads 32 consecutive fp32 columns of its lane.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32"
        " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- CTA pairs
// This CTA's rank within its cluster.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Tensor-memory allocation for a CTA pair: one warp of EACH CTA of the pair
// executes these together; both CTAs get the same column range.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D[tmem] (+)= A . B^T on a CTA pair (M = 256: each CTA holds 128 rows of A
// and half of B's rows at the same shared offsets; each CTA's tensor memory
// holds its own 128 rows of D).  Issued by one thread of the even CTA.
__device__ __forceinline__ void mma_mxf4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X"
        " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Instruction descriptor for kind::mxf8f6f4 with E4M3 x E4M3 operands, E8M0
// scales (scale_vec::1X: one scale byte per row per MMA, selected by the
// scale-factor ids), fp32 accumulate, K-major, tile M x N.
__host__ __device__ constexpr uint32_t idesc_mxf8(int M, int N, int a_sf_id, int b_sf_id) {
    return (static_cast<uint32_t>(b_sf_id & 3) << 4)      // B scale-factor id
           | (0u << 7)                                    // A format: E4M3
           | (0u << 10)                                   // B format: E4M3
           | (static_cast<uint32_t>(N >> 3) << 17)        // N / 8
           | (1u << 23)                                   // scale format: UE8M0
           | (static_cast<uint32_t>(M >> 4) << 24)        // M / 16
           | (static_cast<uint32_t>(a_sf_id & 3) << 29);  // A scale-factor id
}

// The MXFP8 form of mma_mxf4_pair (K = 32 per instruction).
__device__ __forceinline__ void mma_mxf8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X"
        " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Instruction descriptor for kind::mxf4nvf4 with scale_vec::4X (NVFP4: E2M1
// x E2M1, one UE4M3 scale per 16 elements, four per row per MMA), fp32
// accumulate, K-major, tile M x N.
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
    return (1u << 7)                                      // A format: E2M1
           | (1u << 10)                                   // B format: E2M1
           | (static_cast<uint32_t>(N >> 3) << 17)        // N / 8
           | (0u << 23)                                   // scale format: UE4M3
           | (static_cast<uint32_t>(M >> 4) << 24);       // M / 16
}

// The NVFP4 form of mma_mxf4_pair (K = 64 per instruction).
__device__ __forceinline__ void mma_nvf4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X"
        " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Arrive on the barrier at shared offset `bar` of every CTA in `cta_mask`
// once every pair operation issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit_pair(uint64_t *bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// Each thread of the warp writes its registers into consecutive 32-bit
// columns of its own tensor-memory lane.
__device__ __forceinline__ void tmem_st_32x32b_x4(uint32_t taddr, const uint32_t (&v)[4]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
                 : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                     taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
                 "r"(v[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0],"
        " {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15])
        : "memory");
}
// Waits until this thread's tensor-memory stores have completed.
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace mx
