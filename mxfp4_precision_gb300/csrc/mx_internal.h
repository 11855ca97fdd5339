// mx_internal.h -- host-side glue shared by the library's translation units.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mx {

struct DeviceInfo {
    int ordinal = -1;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    int *status = nullptr;  // device address of the per-device status word
};

// Lazily-filled info for the current device; nullptr (and *err set) on failure.
const DeviceInfo *current_device(cudaError_t *err);

// Host wrapper of cuTensorMapEncodeTiled for a 2-D row-major tensor.
bool encode_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                    uint64_t inner_elems, uint64_t outer_elems, uint64_t row_bytes,
                    uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);

// Scale-layout geometry (see mx.h): k-atoms (4 blocks of 32) per 128-line group.
inline int64_t scale_katoms(int64_t k) { return 2 * ((k + 255) / 256); }
inline int64_t scale_groups(int64_t mn) { return (mn + 127) / 128; }
// NVFP4 scale layout: 512-byte atoms of 128 lines x 4 blocks of 16.
inline int64_t nv_scale_katoms(int64_t k) { return 4 * ((k + 255) / 256); }

// Kernel launchers (argument validation happens before these are called).
cudaError_t launch_quantize(const void *src, int64_t rows, int64_t cols, int contract, int rot,
                            int rot_block, int rnd, uint64_t seed, uint64_t sr_tag,
                            void *codes, void *scales, const DeviceInfo &dev,
                            cudaStream_t stream);

// Both operands encoded down their rows (contraction = rows) in one launch;
// SR tags 1 and 2.
cudaError_t launch_quantize_pair_colwise(const void *src0, int64_t rows0, int64_t cols0,
                                         const void *src1, int64_t rows1, int64_t cols1, int rot,
                                         int rot_block, int rnd, uint64_t seed, void *codes0,
                                         void *scales0, void *codes1, void *scales1,
                                         const DeviceInfo &dev, cudaStream_t stream);
// One read of src [rows, cols] writes its column-direction encoding (blocks
// along rows, rotated) and its row-direction encoding (blocks along cols,
// no rotation).
// tiled scales [mx_scales_bytes(lines, k)] -> canonical [lines][k/32].
cudaError_t launch_scales_to_canonical(const void *tiled, int64_t lines, int64_t k, void *canon,
                                       const DeviceInfo &dev, cudaStream_t stream);
cudaError_t launch_quantize_dual(const void *src, int64_t rows, int64_t cols, int rot,
                                 int rot_block, int rnd, uint64_t seed, void *codes_t,
                                 void *scales_t, void *codes_n, void *scales_n,
                                 const DeviceInfo &dev, cudaStream_t stream);

// MXFP8 (E4M3 elements, the FP8 comparator) encode down the rows of one or
// two operands (src1 == nullptr: one) in one launch; no rotation, round to
// nearest.  Codes [cols][rows] bytes, scales in the tiled layout.
cudaError_t launch_quantize_mxfp8_colwise(const void *src0, int64_t rows0, int64_t cols0,
                                          const void *src1, int64_t rows1, int64_t cols1,
                                          void *codes0, void *scales0, void *codes1,
                                          void *scales1, const DeviceInfo &dev,
                                          cudaStream_t stream);

// NVFP4 encode down the rows of one or two operands (src1 == nullptr: one):
// zeroes amax[0..1], a first launch max-reduces each rotated operand's
// largest finite magnitude into it, a second encodes with the tensor scale
// 2688 / amax.  Rotation none, or Hadamard 16 / 32 (rot 1 deterministic, 2
// with random signs); round to nearest.  Codes [cols][rows/2], scales in the
// NVFP4 tiled layout.
cudaError_t launch_quantize_nvfp4_colwise(const void *src0, int64_t rows0, int64_t cols0,
                                          const void *src1, int64_t rows1, int64_t cols1, int rot,
                                          int rot_block, uint64_t seed, void *codes0,
                                          void *scales0, void *codes1, void *scales1,
                                          float *amax, const DeviceInfo &dev,
                                          cudaStream_t stream);

// Block-scaled GEMM over MXFP4 (fmt 0), MXFP8 (fmt 1) or NVFP4 (fmt 2)
// operands; NVFP4 reads the two tensor amaxes (device floats) and scales the
// result by 1 / (s_enc(a) * s_enc(b)).
enum { kGemmMXFP4 = 0, kGemmMXFP8 = 1, kGemmNVFP4 = 2 };
cudaError_t launch_gemm_fmt(int fmt, const void *Aq, const void *As, const void *Bq,
                            const void *Bs, float *C, int64_t M, int64_t N, int64_t K,
                            const float *amax_a, const float *amax_b, const DeviceInfo &dev,
                            cudaStream_t stream);

cudaError_t launch_gemm(const void *Aq, const void *As, const void *Bq, const void *Bs, float *C,
                        int64_t M, int64_t N, int64_t K, const DeviceInfo &dev,
                        cudaStream_t stream);

// Fused Wgrad: one launch whose encoder warps encode dY and X (contraction
// T) into Aq/As/Bq/Bs while the GEMM consumes them; `counters` is
// wgrad_fused_counter_bytes(T, N, K) of workspace (any contents).  Only for
// the shapes and modes wgrad_fusable() accepts.
bool wgrad_fusable(int64_t T, int64_t N, int64_t K, int rot, int rot_block, int rnd);
size_t wgrad_fused_counter_bytes(int64_t T, int64_t N, int64_t K);
cudaError_t launch_wgrad_fused(const void *dY, const void *X, float *dW, int64_t T, int64_t N,
                               int64_t K, int rot, int rot_block, void *Aq, void *As, void *Bq,
                               void *Bs, void *counters, const DeviceInfo &dev,
                               cudaStream_t stream);

}  // namespace mx
