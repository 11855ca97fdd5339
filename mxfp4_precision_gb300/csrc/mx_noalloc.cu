// mx_noalloc.cu -- mx_linear_wgrad_noalloc: the Wgrad entry point for callers
// that cannot hand the library a workspace.
//
// mx_linear_wgrad needs scratch memory for the two encoded operands and takes
// it from the caller.  Some callers have no way to provide it: a plugin or
// custom op running inside a host framework whose device memory is owned by
// that framework's pool (a cudaMalloc behind the pool's back breaks its
// accounting or fails under a hard memory cap), a bare C or Fortran host
// without a device allocator, or a hot loop that cannot pay for the implicit
// device-wide synchronisation of cudaMalloc/cudaFree.  For them this file
// keeps a fixed scratch area in a file-scope __device__ array that the CUDA
// module carries; the entry point allocates nothing and calls no allocator.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/mx.h"

namespace {

constexpr size_t kScratchBytes = MX_NOALLOC_SCRATCH_BYTES;

// The scratch area: every GPU that loads this library holds it until the
// process exits.  In host code `g_noalloc_scratch` is only a host-side stand-in
// for the symbol, never a device address; the device address is obtained with
// cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Once per device, with that device current: resolve the scratch array's
// device address (this also loads the module on that device).
mx_status scratch_for_current_device(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MX_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return MX_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return MX_OK;
}

}  // namespace

extern "C" mx_status mx_linear_wgrad_noalloc(const void *d_dY, const void *d_X, float *d_dW,
                                             int64_t T, int64_t N, int64_t K, int rot,
                                             int rot_block, int rnd, uint64_t seed,
                                             void *stream) {
    // Argument checks first, with mx_linear_wgrad's own rules and status
    // codes: without a workspace it either rejects the arguments, finishes a
    // call that needs no scratch (empty shapes), or reports MX_ERR_WORKSPACE
    // -- all before launching anything that needs one.
    mx_status st = mx_linear_wgrad(d_dY, d_X, d_dW, T, N, K, rot, rot_block, rnd, seed, nullptr,
                                   0, stream);
    if (st != MX_ERR_WORKSPACE) return st;
    const size_t need = mx_linear_workspace_bytes(MX_OP_WGRAD, T, N, K);
    if (need > kScratchBytes) return MX_ERR_WORKSPACE;  // beyond the fixed scratch area
    void *scratch = nullptr;
    st = scratch_for_current_device(&scratch);
    if (st != MX_OK) return st;
    // The encoded operands are fully rewritten on every call (padding
    // included), so nothing in the shared area needs clearing first.
    return mx_linear_wgrad(d_dY, d_X, d_dW, T, N, K, rot, rot_block, rnd, seed, scratch,
                           kScratchBytes, stream);
}
