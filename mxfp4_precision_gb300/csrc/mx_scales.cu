// mx_scales.cu -- canonical view of the tiled E8M0 scale layout.
//
// The encoders write the scales of an MXFP4 operand (one E8M0 byte per block
// of 32 elements, [36kr] "Was ist MXFP4?") in the layout the tcgen05 block-
// scaled MMA consumes; this kernel gathers them back into plain row-major
// [lines][k/32] bytes for tests and for code that expects that order.
#include <cstdint>
#include <cuda_runtime.h>

#include "mx_internal.h"

namespace mx {
namespace {

// Byte offset of the scale of (line, block) in the tiled layout: 512-byte
// atoms of 128 lines x 4 blocks, stored as 32 rows of (4 line quarters x 4
// blocks); the atoms of one 128-line group are contiguous along k.
__device__ __forceinline__ int64_t tiled_offset(int64_t line, int64_t block, int64_t katoms) {
    return ((line / 128) * katoms + block / 4) * 512 + (line % 32) * 16 + ((line % 128) / 32) * 4 +
           (block % 4);
}

__global__ void mx_scales_canon_kernel(const uint8_t *__restrict__ tiled, uint8_t *__restrict__ canon,
                                       int64_t lines, int64_t blocks, int64_t katoms) {
    const int64_t n = lines * blocks;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        canon[i] = tiled[tiled_offset(i / blocks, i % blocks, katoms)];
}

}  // namespace

cudaError_t launch_scales_to_canonical(const void *tiled, int64_t lines, int64_t k, void *canon,
                                       const DeviceInfo &dev, cudaStream_t stream) {
    const int64_t blocks = k / 32, n = lines * blocks;
    const int64_t want = (n + 255) / 256;
    const int grid = static_cast<int>(want < 4 * dev.sm_count ? want : 4 * dev.sm_count);
    mx_scales_canon_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint8_t *>(tiled),
                                                     static_cast<uint8_t *>(canon), lines, blocks,
                                                     scale_katoms(k));
    return cudaGetLastError();
}

}  // namespace mx
