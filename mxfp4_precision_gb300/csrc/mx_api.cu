// mx_api.cu -- the library's C ABI (include/mx.h): argument checks, workspace
// carving, tensor-map encoding, per-device status word, and the launches.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/mx.h"
#include <nvtx3/nvToolsExt.h>
#include "mx_internal.h"
#include "mx_ptx.cuh"

// One status word per device (lives as long as the module is loaded).
static __device__ int g_mx_status;

namespace mx {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool load_encode_fn() {
    if (g_encode != nullptr) return true;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return false;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return true;
}

__global__ void timeout_probe_kernel(int *status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    // Nothing ever arrives on `bar`: the bounded wait must give up.
    if (threadIdx.x == 0) mbar_wait(&bar, 0, status, nullptr, limit_ns);
    __syncthreads();
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool valid_rot(int rot, int rot_block) {
    if (rot == MX_ROT_NONE) return true;
    if (rot != MX_ROT_HADAMARD_DET && rot != MX_ROT_HADAMARD_RAND) return false;
    return rot_block == 16 || rot_block == 32 || rot_block == 64 || rot_block == 128 ||
           rot_block == 256;
}
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

mx_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MX_OK : MX_ERR_CUDA; }

// Checks shared by every encode: enums, shape (contraction length multiple of
// 32 and of rot_block), pointer alignment.
mx_status check_encode(const void *src, int64_t rows, int64_t cols, int contract, int rot,
                       int rot_block, int rnd, const void *codes, const void *scales) {
    if (contract != MX_CONTRACT_ROWS && contract != MX_CONTRACT_COLS) return MX_ERR_INVALID_ARG;
    if (!valid_rot(rot, rot_block)) return MX_ERR_INVALID_ARG;
    if (rnd != MX_ROUND_RNE && rnd != MX_ROUND_SR) return MX_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0) return MX_ERR_SHAPE;
    if (rows > 0x7FFFFFFF || cols > 0x7FFFFFFF) return MX_ERR_SHAPE;
    if (rows == 0 || cols == 0) return MX_OK;
    if (src == nullptr || codes == nullptr || scales == nullptr) return MX_ERR_INVALID_ARG;
    const int64_t L = contract == MX_CONTRACT_ROWS ? rows : cols;
    if (L % 32 != 0) return MX_ERR_SHAPE;
    if (rot != MX_ROT_NONE && L % rot_block != 0) return MX_ERR_SHAPE;
    if (!aligned16(src) || !aligned16(codes) || !aligned16(scales)) return MX_ERR_ALIGN;
    if (cols % 8 != 0) return MX_ERR_ALIGN;  // 16-byte rows for the TMA
    return MX_OK;
}

mx_status check_gemm(const void *Aq, const void *As, const void *Bq, const void *Bs,
                     const float *C, int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0) return MX_ERR_SHAPE;
    if (M > 0x7FFFFFFF || N > 0x7FFFFFFF || K > 0x7FFFFFFF) return MX_ERR_SHAPE;
    if (M == 0 || N == 0) return MX_OK;
    if (C == nullptr) return MX_ERR_INVALID_ARG;
    if (K % 32 != 0) return MX_ERR_SHAPE;
    if (N % 4 != 0 || !aligned16(C)) return MX_ERR_ALIGN;
    if (K == 0) return MX_OK;
    if (!Aq || !As || !Bq || !Bs) return MX_ERR_INVALID_ARG;
    if (!aligned16(Aq) || !aligned16(As) || !aligned16(Bq) || !aligned16(Bs)) return MX_ERR_ALIGN;
    return MX_OK;
}

// Lines and contraction length of both operands of a linear op.
struct OpShape {
    int64_t a_lines, b_lines, k;
};
bool op_shape(int op, int64_t T, int64_t N, int64_t K, OpShape *s) {
    switch (op) {
        case MX_OP_FPROP: *s = {T, N, K}; return true;
        case MX_OP_DGRAD: *s = {T, K, N}; return true;
        case MX_OP_WGRAD: *s = {N, K, T}; return true;
        default: return false;
    }
}

}  // namespace

const DeviceInfo *current_device(cudaError_t *err) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *err = e != cudaSuccess ? e : cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo &d = g_devices[dev];
    if (d.ordinal == dev) return &d;
    cudaDeviceProp prop;
    if ((e = cudaGetDeviceProperties(&prop, dev)) != cudaSuccess) {
        *err = e;
        return nullptr;
    }
    void *status = nullptr;
    if ((e = cudaGetSymbolAddress(&status, g_mx_status)) != cudaSuccess) {
        *err = e;
        return nullptr;
    }
    if (!load_encode_fn()) {
        *err = cudaErrorSymbolNotFound;
        return nullptr;
    }
    d.sm_count = prop.multiProcessorCount;
    d.cc_major = prop.major;
    d.cc_minor = prop.minor;
    d.status = static_cast<int *>(status);
    d.ordinal = dev;
    return &d;
}

bool encode_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                    uint64_t inner_elems, uint64_t outer_elems, uint64_t row_bytes,
                    uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
    if (g_encode == nullptr) return false;
    cuuint64_t dims[2] = {inner_elems, outer_elems};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace mx

using namespace mx;

namespace {
mx_status device_or_error(const DeviceInfo **out) {
    cudaError_t e = cudaSuccess;
    const DeviceInfo *d = current_device(&e);
    if (d == nullptr) return MX_ERR_CUDA;
    if (!(d->cc_major == 10 && d->cc_minor == 3)) return MX_ERR_UNSUPPORTED;
    *out = d;
    return MX_OK;
}

mx_status quantize_impl(const void *src, int64_t rows, int64_t cols, int contract, int rot,
                        int rot_block, int rnd, uint64_t seed, uint64_t sr_tag, void *codes,
                        void *scales, cudaStream_t stream) {
    mx_status st = check_encode(src, rows, cols, contract, rot, rot_block, rnd, codes, scales);
    if (st != MX_OK || rows == 0 || cols == 0) return st;
    const DeviceInfo *dev = nullptr;
    if ((st = device_or_error(&dev)) != MX_OK) return st;
    return from_cuda(launch_quantize(src, rows, cols, contract, rot, rot_block, rnd, seed, sr_tag,
                                     codes, scales, *dev, stream));
}

mx_status quantize_pair_impl(const void *src0, int64_t rows0, int64_t cols0, const void *src1,
                             int64_t rows1, int64_t cols1, int rot, int rot_block, int rnd,
                             uint64_t seed, void *codes0, void *scales0, void *codes1,
                             void *scales1, cudaStream_t stream) {
    if (rows0 != rows1) return MX_ERR_SHAPE;
    mx_status st = check_encode(src0, rows0, cols0, MX_CONTRACT_ROWS, rot, rot_block, rnd, codes0,
                                scales0);
    if (st != MX_OK) return st;
    st = check_encode(src1, rows1, cols1, MX_CONTRACT_ROWS, rot, rot_block, rnd, codes1, scales1);
    if (st != MX_OK) return st;
    const bool e0 = rows0 == 0 || cols0 == 0, e1 = rows1 == 0 || cols1 == 0;
    if (e0 && e1) return MX_OK;
    if (e0 || e1)  // one side empty: plain single-operand encode of the other
        return e0 ? quantize_impl(src1, rows1, cols1, MX_CONTRACT_ROWS, rot, rot_block, rnd, seed,
                                  2, codes1, scales1, stream)
                  : quantize_impl(src0, rows0, cols0, MX_CONTRACT_ROWS, rot, rot_block, rnd, seed,
                                  1, codes0, scales0, stream);
    const DeviceInfo *dev = nullptr;
    if ((st = device_or_error(&dev)) != MX_OK) return st;
    return from_cuda(launch_quantize_pair_colwise(src0, rows0, cols0, src1, rows1, cols1, rot,
                                                  rot_block, rnd, seed, codes0, scales0, codes1,
                                                  scales1, *dev, stream));
}

mx_status quantize_dual_impl(const void *src, int64_t T, int64_t N, int rot, int rot_block,
                             int rnd, uint64_t seed, void *codes_t, void *scales_t, void *codes_n,
                             void *scales_n, cudaStream_t stream) {
    mx_status st = check_encode(src, T, N, MX_CONTRACT_ROWS, rot, rot_block, rnd, codes_t,
                                scales_t);
    if (st != MX_OK) return st;
    st = check_encode(src, T, N, MX_CONTRACT_COLS, MX_ROT_NONE, 32, rnd, codes_n, scales_n);
    if (st != MX_OK || T == 0 || N == 0) return st;
    const DeviceInfo *dev = nullptr;
    if ((st = device_or_error(&dev)) != MX_OK) return st;
    return from_cuda(launch_quantize_dual(src, T, N, rot, rot_block, rnd, seed, codes_t, scales_t,
                                          codes_n, scales_n, *dev, stream));
}

mx_status gemm_impl(const void *Aq, const void *As, const void *Bq, const void *Bs, float *C,
                    int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    mx_status st = check_gemm(Aq, As, Bq, Bs, C, M, N, K);
    if (st != MX_OK || M == 0 || N == 0) return st;
    if (K == 0)
        return from_cuda(cudaMemsetAsync(C, 0, static_cast<size_t>(M) * N * sizeof(float), stream));
    const DeviceInfo *dev = nullptr;
    if ((st = device_or_error(&dev)) != MX_OK) return st;
    return from_cuda(launch_gemm(Aq, As, Bq, Bs, C, M, N, K, *dev, stream));
}

// MXFP8 comparator: encode down the rows of one or two operands, contract.
mx_status quantize_mxfp8_impl(const void *src0, int64_t rows0, int64_t cols0, const void *src1,
                              int64_t rows1, int64_t cols1, void *codes0, void *scales0,
                              void *codes1, void *scales1, cudaStream_t stream) {
    mx_status st = check_encode(src0, rows0, cols0, MX_CONTRACT_ROWS, MX_ROT_NONE, 32,
                                MX_ROUND_RNE, codes0, scales0);
    if (st != MX_OK) return st;
    if (src1 != nullptr) {
        st = check_encode(src1, rows1, cols1, MX_CONTRACT_ROWS, MX_ROT_NONE, 32, MX_ROUND_RNE,
                          codes1, scales1);
        if (st != MX_OK) return st;
        if (rows1 == 0 || cols1 == 0) src1 = nullptr;
    }
    if (rows0 == 0 || cols0 == 0) {
        if (src1 == nullptr) return MX_OK;
        src0 = src1, rows0 = rows1, cols0 = cols1, codes0 = codes1, scales0 = scales1;
        src1 = nullptr;
    }
    const DeviceInfo *dev = nullptr;
    if ((st = device_or_error(&dev)) != MX_OK) return st;
    return from_cuda(launch_quantize_mxfp8_colwise(src0, rows0, cols0, src1, rows1, cols1, codes0,
                                                   scales0, codes1, scales1, *dev, stream));
}

mx_status gemm_mxfp8_impl(const void *Aq, const void *As, const void *Bq, const void *Bs,
                          float *C, int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    mx_status st = check_gemm(Aq, As, Bq, Bs, C, M, N, K);
    if (st != MX_OK || M == 0 || N == 0) return st;
    if (K == 0)
        return from_cuda(cudaMemsetAsync(C, 0, static_cast<size_t>(M) * N * sizeof(float), stream));
    const DeviceInfo *dev = nullptr;
    if ((st = device_or_error(&dev)) != MX_OK) return st;
    return from_cuda(launch_gemm_fmt(kGemmMXFP8, Aq, As, Bq, Bs, C, M, N, K, nullptr, nullptr,
                                     *dev, stream));
}

// NVFP4 variant: encode down the rows of one or two operands (two launches:
// tensor amax, then the encode), contract with the tensor scales.
mx_status quantize_nvfp4_impl(const void *src0, int64_t rows0, int64_t cols0, const void *src1,
                              int64_t rows1, int64_t cols1, int rot, int rot_block, uint64_t seed,
                              void *codes0, void *scales0, void *codes1, void *scales1,
                              float *amax, cudaStream_t stream) {
    mx_status st = check_encode(src0, rows0, cols0, MX_CONTRACT_ROWS, rot, rot_block,
                                MX_ROUND_RNE, codes0, scales0);
    if (st != MX_OK) return st;
    if (rot != MX_ROT_NONE && rot_block != 16 && rot_block != 32) return MX_ERR_UNSUPPORTED;
    if (src1 != nullptr) {
        st = check_encode(src1, rows1, cols1, MX_CONTRACT_ROWS, rot, rot_block, MX_ROUND_RNE,
                          codes1, scales1);
        if (st != MX_OK) return st;
        if (rows1 == 0 || cols1 == 0) return MX_ERR_SHAPE;
    }
    if (rows0 == 0 || cols0 == 0) return src1 == nullptr ? MX_OK : MX_ERR_SHAPE;
    if (amax == nullptr) return MX_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(amax) & 7u) != 0) return MX_ERR_ALIGN;
    const DeviceInfo *dev = nullptr;
    if ((st = device_or_error(&dev)) != MX_OK) return st;
    return from_cuda(launch_quantize_nvfp4_colwise(src0, rows0, cols0, src1, rows1, cols1, rot,
                                                   rot_block, seed, codes0, scales0, codes1,
                                                   scales1, amax, *dev, stream));
}

mx_status gemm_nvfp4_impl(const void *Aq, const void *As, const float *amax_a, const void *Bq,
                          const void *Bs, const float *amax_b, float *C, int64_t M, int64_t N,
                          int64_t K, cudaStream_t stream) {
    mx_status st = check_gemm(Aq, As, Bq, Bs, C, M, N, K);
    if (st != MX_OK || M == 0 || N == 0) return st;
    if (K == 0)
        return from_cuda(cudaMemsetAsync(C, 0, static_cast<size_t>(M) * N * sizeof(float), stream));
    if (amax_a == nullptr || amax_b == nullptr) return MX_ERR_INVALID_ARG;
    const DeviceInfo *dev = nullptr;
    if ((st = device_or_error(&dev)) != MX_OK) return st;
    return from_cuda(launch_gemm_fmt(kGemmNVFP4, Aq, As, Bq, Bs, C, M, N, K, amax_a, amax_b,
                                     *dev, stream));
}

// Quantise both operands of a linear op into the workspace, then contract.
mx_status linear_impl(int op, const void *a_src, int64_t a_rows, int64_t a_cols, int a_contract,
                      const void *b_src, int64_t b_rows, int64_t b_cols, int b_contract, float *out,
                      int64_t T, int64_t N, int64_t K, int rot, int rot_block, int rnd,
                      uint64_t seed, void *ws, size_t ws_bytes, cudaStream_t stream,
                      bool fused = false) {
    OpShape s;
    if (!op_shape(op, T, N, K, &s)) return MX_ERR_INVALID_ARG;
    if (T < 0 || N < 0 || K < 0) return MX_ERR_SHAPE;
    if (s.a_lines == 0 || s.b_lines == 0) return MX_OK;
    if (out == nullptr) return MX_ERR_INVALID_ARG;
    if (s.k == 0) return gemm_impl(nullptr, nullptr, nullptr, nullptr, out, s.a_lines, s.b_lines, 0, stream);
    // Operand checks (the workspace is checked separately below).
    mx_status st = check_encode(a_src, a_rows, a_cols, a_contract, rot, rot_block, rnd, a_src,
                                a_src);
    if (st != MX_OK) return st;
    st = check_encode(b_src, b_rows, b_cols, b_contract, rot, rot_block, rnd, b_src, b_src);
    if (st != MX_OK) return st;
    if (s.b_lines % 4 != 0 || !aligned16(out)) return MX_ERR_ALIGN;
    const size_t need = mx_linear_workspace_bytes(op, T, N, K);
    if (ws == nullptr || ws_bytes < need) return MX_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MX_ERR_ALIGN;
    uint8_t *p = static_cast<uint8_t *>(ws);
    uint8_t *aq = p;
    p += align256(mx_codes_bytes(s.a_lines, s.k));
    uint8_t *as = p;
    p += align256(mx_scales_bytes(s.a_lines, s.k));
    uint8_t *bq = p;
    p += align256(mx_codes_bytes(s.b_lines, s.k));
    uint8_t *bs = p;
    if (fused) {
        // One launch: the GEMM's own encoder warps encode both operands while
        // it runs (its chunk counters, after the operands in the workspace,
        // are zeroed first).
        if (op != MX_OP_WGRAD || !wgrad_fusable(T, N, K, rot, rot_block, rnd))
            return MX_ERR_UNSUPPORTED;
        const DeviceInfo *dev = nullptr;
        if ((st = device_or_error(&dev)) != MX_OK) return st;
        uint8_t *counters = bs + align256(mx_scales_bytes(s.b_lines, s.k));
        return from_cuda(launch_wgrad_fused(a_src, b_src, out, T, N, K, rot, rot_block, aq, as, bq,
                                            bs, counters, *dev, stream));
    }
    if (a_contract == MX_CONTRACT_ROWS && b_contract == MX_CONTRACT_ROWS) {
        // Wgrad: both operands encoded down their rows in a single launch.
        st = quantize_pair_impl(a_src, a_rows, a_cols, b_src, b_rows, b_cols, rot, rot_block, rnd,
                                seed, aq, as, bq, bs, stream);
    } else {
        st = quantize_impl(a_src, a_rows, a_cols, a_contract, rot, rot_block, rnd, seed, 1, aq, as,
                           stream);
        if (st == MX_OK)
            st = quantize_impl(b_src, b_rows, b_cols, b_contract, rot, rot_block, rnd, seed, 2,
                               bq, bs, stream);
    }
    if (st != MX_OK) return st;
    return gemm_impl(aq, as, bq, bs, out, s.a_lines, s.b_lines, s.k, stream);
}
}  // namespace

namespace {
// Names each exported call in profiler timelines (NVTX; free without a tool attached).
struct TraceRange {
    explicit TraceRange(const char *name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange &) = delete;
    TraceRange &operator=(const TraceRange &) = delete;
};
}  // namespace

extern "C" {

size_t mx_codes_bytes(int64_t mn, int64_t k) {
    if (mn <= 0 || k <= 0) return 0;
    return static_cast<size_t>(mn) * static_cast<size_t>(k / 2);
}

size_t mx_scales_bytes(int64_t mn, int64_t k) {
    if (mn <= 0 || k <= 0) return 0;
    return static_cast<size_t>(scale_groups(mn)) * 128u * static_cast<size_t>(8 * ((k + 255) / 256));
}

mx_status mx_quantize(const void *d_src, int64_t rows, int64_t cols, int contract, int rot,
                      int rot_block, int rnd, uint64_t seed, void *d_codes, void *d_scales,
                      void *stream) {
    TraceRange trace("mx_quantize");
    return quantize_impl(d_src, rows, cols, contract, rot, rot_block, rnd, seed, 1, d_codes,
                         d_scales, static_cast<cudaStream_t>(stream));
}

mx_status mx_quantize_pair(const void *d_src0, int64_t rows0, int64_t cols0, const void *d_src1,
                           int64_t rows1, int64_t cols1, int rot, int rot_block, int rnd,
                           uint64_t seed, void *d_codes0, void *d_scales0, void *d_codes1,
                           void *d_scales1, void *stream) {
    TraceRange trace("mx_quantize_pair");
    return quantize_pair_impl(d_src0, rows0, cols0, d_src1, rows1, cols1, rot, rot_block, rnd, seed,
                              d_codes0, d_scales0, d_codes1, d_scales1,
                              static_cast<cudaStream_t>(stream));
}

mx_status mx_quantize_dual(const void *d_src, int64_t T, int64_t N, int rot, int rot_block,
                           int rnd, uint64_t seed, void *d_codes_t, void *d_scales_t,
                           void *d_codes_n, void *d_scales_n, void *stream) {
    TraceRange trace("mx_quantize_dual");
    return quantize_dual_impl(d_src, T, N, rot, rot_block, rnd, seed, d_codes_t, d_scales_t,
                              d_codes_n, d_scales_n, static_cast<cudaStream_t>(stream));
}

mx_status mx_scales_to_canonical(const void *d_scales, int64_t lines, int64_t k, void *d_canon,
                                 void *stream) {
    TraceRange trace("mx_scales_to_canonical");
    if (lines < 0 || k < 0) return MX_ERR_SHAPE;
    if (k % 32 != 0) return MX_ERR_SHAPE;
    if (lines == 0 || k == 0) return MX_OK;
    if (d_scales == nullptr || d_canon == nullptr) return MX_ERR_INVALID_ARG;
    const DeviceInfo *dev = nullptr;
    mx_status st = device_or_error(&dev);
    if (st != MX_OK) return st;
    return from_cuda(launch_scales_to_canonical(d_scales, lines, k, d_canon, *dev,
                                                static_cast<cudaStream_t>(stream)));
}

mx_status mx_gemm(const void *d_Aq, const void *d_As, const void *d_Bq, const void *d_Bs,
                  float *d_C, int64_t M, int64_t N, int64_t K, void *stream) {
    TraceRange trace("mx_gemm");
    return gemm_impl(d_Aq, d_As, d_Bq, d_Bs, d_C, M, N, K, static_cast<cudaStream_t>(stream));
}

size_t mx_linear_workspace_bytes(int op, int64_t T, int64_t N, int64_t K) {
    OpShape s;
    if (!op_shape(op, T, N, K, &s)) return 0;
    size_t bytes = align256(mx_codes_bytes(s.a_lines, s.k)) + align256(mx_scales_bytes(s.a_lines, s.k)) +
                   align256(mx_codes_bytes(s.b_lines, s.k)) + align256(mx_scales_bytes(s.b_lines, s.k));
    // Wgrad: room for the fused launch's (panel, chunk) counters.
    if (op == MX_OP_WGRAD && T > 0 && N > 0 && K > 0) bytes += align256(wgrad_fused_counter_bytes(T, N, K));
    return bytes;
}

mx_status mx_linear_wgrad(const void *d_dY, const void *d_X, float *d_dW, int64_t T, int64_t N,
                          int64_t K, int rot, int rot_block, int rnd, uint64_t seed, void *d_ws,
                          size_t ws_bytes, void *stream) {
    TraceRange trace("mx_linear_wgrad");
    // dW[N][K] = dY^T X: both operands encoded down their rows (contraction T).
    return linear_impl(MX_OP_WGRAD, d_dY, T, N, MX_CONTRACT_ROWS, d_X, T, K, MX_CONTRACT_ROWS,
                       d_dW, T, N, K, rot, rot_block, rnd, seed, d_ws, ws_bytes,
                       static_cast<cudaStream_t>(stream));
}

mx_status mx_linear_fprop(const void *d_X, const void *d_W, float *d_Y, int64_t T, int64_t N,
                          int64_t K, int rot, int rot_block, int rnd, uint64_t seed, void *d_ws,
                          size_t ws_bytes, void *stream) {
    TraceRange trace("mx_linear_fprop");
    // Y[T][N] = X W^T: X[T][K] and W[N][K] encoded along their rows (contraction K).
    return linear_impl(MX_OP_FPROP, d_X, T, K, MX_CONTRACT_COLS, d_W, N, K, MX_CONTRACT_COLS, d_Y,
                       T, N, K, rot, rot_block, rnd, seed, d_ws, ws_bytes,
                       static_cast<cudaStream_t>(stream));
}

mx_status mx_linear_dgrad(const void *d_dY, const void *d_W, float *d_dX, int64_t T, int64_t N,
                          int64_t K, int rot, int rot_block, int rnd, uint64_t seed, void *d_ws,
                          size_t ws_bytes, void *stream) {
    TraceRange trace("mx_linear_dgrad");
    // dX[T][K] = dY W: dY[T][N] along its rows, W[N][K] down its rows (contraction N).
    return linear_impl(MX_OP_DGRAD, d_dY, T, N, MX_CONTRACT_COLS, d_W, N, K, MX_CONTRACT_ROWS,
                       d_dX, T, N, K, rot, rot_block, rnd, seed, d_ws, ws_bytes,
                       static_cast<cudaStream_t>(stream));
}

size_t mx_mxfp8_codes_bytes(int64_t mn, int64_t k) {
    if (mn <= 0 || k <= 0) return 0;
    return static_cast<size_t>(mn) * static_cast<size_t>(k);
}

mx_status mx_quantize_mxfp8(const void *d_src, int64_t rows, int64_t cols, void *d_codes,
                            void *d_scales, void *stream) {
    TraceRange trace("mx_quantize_mxfp8");
    return quantize_mxfp8_impl(d_src, rows, cols, nullptr, 0, 0, d_codes, d_scales, nullptr,
                               nullptr, static_cast<cudaStream_t>(stream));
}

mx_status mx_gemm_mxfp8(const void *d_Aq, const void *d_As, const void *d_Bq, const void *d_Bs,
                        float *d_C, int64_t M, int64_t N, int64_t K, void *stream) {
    TraceRange trace("mx_gemm_mxfp8");
    return gemm_mxfp8_impl(d_Aq, d_As, d_Bq, d_Bs, d_C, M, N, K,
                           static_cast<cudaStream_t>(stream));
}

size_t mx_linear_wgrad_mxfp8_workspace_bytes(int64_t T, int64_t N, int64_t K) {
    if (T <= 0 || N <= 0 || K <= 0) return 0;
    return align256(mx_mxfp8_codes_bytes(N, T)) + align256(mx_scales_bytes(N, T)) +
           align256(mx_mxfp8_codes_bytes(K, T)) + align256(mx_scales_bytes(K, T));
}

mx_status mx_linear_wgrad_mxfp8(const void *d_dY, const void *d_X, float *d_dW, int64_t T,
                                int64_t N, int64_t K, void *d_ws, size_t ws_bytes, void *stream) {
    TraceRange trace("mx_linear_wgrad_mxfp8");
    const cudaStream_t st_ = static_cast<cudaStream_t>(stream);
    if (T < 0 || N < 0 || K < 0) return MX_ERR_SHAPE;
    if (N == 0 || K == 0) return MX_OK;
    if (d_dW == nullptr) return MX_ERR_INVALID_ARG;
    if (T == 0) return gemm_mxfp8_impl(nullptr, nullptr, nullptr, nullptr, d_dW, N, K, 0, st_);
    mx_status st = check_encode(d_dY, T, N, MX_CONTRACT_ROWS, MX_ROT_NONE, 32, MX_ROUND_RNE,
                                d_dY, d_dY);
    if (st != MX_OK) return st;
    st = check_encode(d_X, T, K, MX_CONTRACT_ROWS, MX_ROT_NONE, 32, MX_ROUND_RNE, d_X, d_X);
    if (st != MX_OK) return st;
    if (K % 4 != 0 || !aligned16(d_dW)) return MX_ERR_ALIGN;
    if (d_ws == nullptr || ws_bytes < mx_linear_wgrad_mxfp8_workspace_bytes(T, N, K))
        return MX_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(d_ws) & 255u) != 0) return MX_ERR_ALIGN;
    uint8_t *aq = static_cast<uint8_t *>(d_ws);
    uint8_t *as = aq + align256(mx_mxfp8_codes_bytes(N, T));
    uint8_t *bq = as + align256(mx_scales_bytes(N, T));
    uint8_t *bs = bq + align256(mx_mxfp8_codes_bytes(K, T));
    st = quantize_mxfp8_impl(d_dY, T, N, d_X, T, K, aq, as, bq, bs, st_);
    if (st != MX_OK) return st;
    return gemm_mxfp8_impl(aq, as, bq, bs, d_dW, N, K, T, st_);
}

size_t mx_nvfp4_scales_bytes(int64_t mn, int64_t k) {
    if (mn <= 0 || k <= 0) return 0;
    return static_cast<size_t>(scale_groups(mn)) * 128u * static_cast<size_t>(16 * ((k + 255) / 256));
}

mx_status mx_quantize_nvfp4(const void *d_src, int64_t rows, int64_t cols, int rot, int rot_block,
                            uint64_t seed, void *d_codes, void *d_scales, float *d_amax,
                            void *stream) {
    TraceRange trace("mx_quantize_nvfp4");
    return quantize_nvfp4_impl(d_src, rows, cols, nullptr, 0, 0, rot, rot_block, seed, d_codes,
                               d_scales, nullptr, nullptr, d_amax,
                               static_cast<cudaStream_t>(stream));
}

mx_status mx_gemm_nvfp4(const void *d_Aq, const void *d_As, const float *d_amax_a,
                        const void *d_Bq, const void *d_Bs, const float *d_amax_b, float *d_C,
                        int64_t M, int64_t N, int64_t K, void *stream) {
    TraceRange trace("mx_gemm_nvfp4");
    return gemm_nvfp4_impl(d_Aq, d_As, d_amax_a, d_Bq, d_Bs, d_amax_b, d_C, M, N, K,
                           static_cast<cudaStream_t>(stream));
}

size_t mx_linear_wgrad_nvfp4_workspace_bytes(int64_t T, int64_t N, int64_t K) {
    if (T <= 0 || N <= 0 || K <= 0) return 0;
    return align256(mx_codes_bytes(N, T)) + align256(mx_nvfp4_scales_bytes(N, T)) +
           align256(mx_codes_bytes(K, T)) + align256(mx_nvfp4_scales_bytes(K, T)) + 256;
}

mx_status mx_linear_wgrad_nvfp4(const void *d_dY, const void *d_X, float *d_dW, int64_t T,
                                int64_t N, int64_t K, int rot, int rot_block, uint64_t seed,
                                void *d_ws, size_t ws_bytes, void *stream) {
    TraceRange trace("mx_linear_wgrad_nvfp4");
    const cudaStream_t st_ = static_cast<cudaStream_t>(stream);
    if (T < 0 || N < 0 || K < 0) return MX_ERR_SHAPE;
    if (N == 0 || K == 0) return MX_OK;
    if (d_dW == nullptr) return MX_ERR_INVALID_ARG;
    if (T == 0) {
        mx_status st = check_gemm(nullptr, nullptr, nullptr, nullptr, d_dW, N, K, 0);
        if (st != MX_OK) return st;
        return from_cuda(cudaMemsetAsync(d_dW, 0, static_cast<size_t>(N) * K * sizeof(float), st_));
    }
    mx_status st = check_encode(d_dY, T, N, MX_CONTRACT_ROWS, rot, rot_block, MX_ROUND_RNE, d_dY,
                                d_dY);
    if (st != MX_OK) return st;
    st = check_encode(d_X, T, K, MX_CONTRACT_ROWS, rot, rot_block, MX_ROUND_RNE, d_X, d_X);
    if (st != MX_OK) return st;
    if (rot != MX_ROT_NONE && rot_block != 16 && rot_block != 32) return MX_ERR_UNSUPPORTED;
    if (K % 4 != 0 || !aligned16(d_dW)) return MX_ERR_ALIGN;
    if (d_ws == nullptr || ws_bytes < mx_linear_wgrad_nvfp4_workspace_bytes(T, N, K))
        return MX_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(d_ws) & 255u) != 0) return MX_ERR_ALIGN;
    uint8_t *aq = static_cast<uint8_t *>(d_ws);
    uint8_t *as = aq + align256(mx_codes_bytes(N, T));
    uint8_t *bq = as + align256(mx_nvfp4_scales_bytes(N, T));
    uint8_t *bs = bq + align256(mx_codes_bytes(K, T));
    float *amax = reinterpret_cast<float *>(bs + align256(mx_nvfp4_scales_bytes(K, T)));
    st = quantize_nvfp4_impl(d_dY, T, N, d_X, T, K, rot, rot_block, seed, aq, as, bq, bs, amax,
                             st_);
    if (st != MX_OK) return st;
    return gemm_nvfp4_impl(aq, as, amax, bq, bs, amax + 1, d_dW, N, K, T, st_);
}

int mx_linear_wgrad_fused_supported(int64_t T, int64_t N, int64_t K, int rot, int rot_block,
                                    int rnd) {
    return wgrad_fusable(T, N, K, rot, rot_block, rnd) ? 1 : 0;
}

mx_status mx_linear_wgrad_fused(const void *d_dY, const void *d_X, float *d_dW, int64_t T,
                                int64_t N, int64_t K, int rot, int rot_block, int rnd,
                                uint64_t seed, void *d_ws, size_t ws_bytes, void *stream) {
    TraceRange trace("mx_linear_wgrad_fused");
    return linear_impl(MX_OP_WGRAD, d_dY, T, N, MX_CONTRACT_ROWS, d_X, T, K, MX_CONTRACT_ROWS,
                       d_dW, T, N, K, rot, rot_block, rnd, seed, d_ws, ws_bytes,
                       static_cast<cudaStream_t>(stream), true);
}

mx_status mx_check_status(void *stream) {
    TraceRange trace("mx_check_status");
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return MX_ERR_CUDA;
    const DeviceInfo *dev = nullptr;
    cudaError_t de = cudaSuccess;
    if ((dev = current_device(&de)) == nullptr) return MX_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, dev->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MX_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return MX_ERR_CUDA;
        return v == kDevTimeout ? MX_ERR_TIMEOUT : v == kDevBounds ? MX_ERR_BOUNDS : MX_ERR_CUDA;
    }
    return MX_OK;
}

mx_status mx_debug_timeout_probe(int64_t limit_us, void *stream) {
    TraceRange trace("mx_debug_timeout_probe");
    if (limit_us <= 0 || limit_us > 10 * 1000 * 1000) return MX_ERR_INVALID_ARG;
    const DeviceInfo *dev = nullptr;
    mx_status st = device_or_error(&dev);
    if (st != MX_OK) return st;
    timeout_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        dev->status, static_cast<uint64_t>(limit_us) * 1000ull);
    return from_cuda(cudaGetLastError());
}

const char *mx_status_string(int status) {
    switch (status) {
        case MX_OK: return "MX_OK";
        case MX_ERR_INVALID_ARG: return "MX_ERR_INVALID_ARG";
        case MX_ERR_SHAPE: return "MX_ERR_SHAPE";
        case MX_ERR_ALIGN: return "MX_ERR_ALIGN";
        case MX_ERR_WORKSPACE: return "MX_ERR_WORKSPACE";
        case MX_ERR_CUDA: return "MX_ERR_CUDA";
        case MX_ERR_TIMEOUT: return "MX_ERR_TIMEOUT";
        case MX_ERR_UNSUPPORTED: return "MX_ERR_UNSUPPORTED";
        case MX_ERR_BOUNDS: return "MX_ERR_BOUNDS";
        default: return "MX_ERR_UNKNOWN";
    }
}

int mx_version(void) { return 100; }

}  // extern "C"
