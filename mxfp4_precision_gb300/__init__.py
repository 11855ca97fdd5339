"""GB300 (sm_103a) MXFP4 linear-layer GEMMs behind a C ABI (include/mx.h).

This package is a thin ctypes binding over the in-tree library
``_build/libmx.so``: it marshals torch tensors (device memory and the current
CUDA stream) into the C calls and nothing else.  Every step of the path runs
in the library's CUDA kernels; there is no CPU fallback -- if the library is
missing or fails to load, every call raises.
"""
from ._binding import (CONTRACT_COLS, CONTRACT_ROWS, OP_DGRAD, OP_FPROP, OP_WGRAD, ROT_HADAMARD_DET,
                       ROT_HADAMARD_RAND, ROT_NONE, ROUND_RNE, ROUND_SR, MMA_KINDS, MXError, bench_mma,
                       check_status,
                       codes_bytes, debug_timeout_probe, gemm, gemm_into, lib, library_path,
                       linear_dgrad, linear_fprop, linear_wgrad, linear_wgrad_fused, linear_wgrad_noalloc,
                       linear_workspace_bytes, NOALLOC_SCRATCH_BYTES, quantize, quantize_dual,
                       quantize_pair, quantize_into, scales_bytes, scales_to_canonical,
                       status_string, mxfp8_codes_bytes, quantize_mxfp8, gemm_mxfp8,
                       gemm_mxfp8_into, linear_wgrad_mxfp8, linear_wgrad_mxfp8_workspace_bytes,
                       nvfp4_scales_bytes, quantize_nvfp4, gemm_nvfp4, linear_wgrad_nvfp4,
                       linear_wgrad_nvfp4_workspace_bytes)

__all__ = [
    "CONTRACT_COLS", "CONTRACT_ROWS", "OP_DGRAD", "OP_FPROP", "OP_WGRAD", "ROT_HADAMARD_DET",
    "ROT_HADAMARD_RAND", "ROT_NONE", "ROUND_RNE", "ROUND_SR", "MMA_KINDS", "MXError", "bench_mma",
    "check_status",
    "codes_bytes", "debug_timeout_probe", "gemm", "gemm_into", "lib", "library_path",
    "linear_dgrad", "linear_fprop", "linear_wgrad", "linear_wgrad_fused", "linear_wgrad_noalloc", "linear_workspace_bytes",
    "NOALLOC_SCRATCH_BYTES", "quantize", "quantize_dual", "quantize_pair",
    "quantize_into", "scales_bytes", "scales_to_canonical", "status_string",
    "mxfp8_codes_bytes", "quantize_mxfp8", "gemm_mxfp8", "gemm_mxfp8_into", "linear_wgrad_mxfp8",
    "linear_wgrad_mxfp8_workspace_bytes", "nvfp4_scales_bytes", "quantize_nvfp4", "gemm_nvfp4",
    "linear_wgrad_nvfp4", "linear_wgrad_nvfp4_workspace_bytes",
]
