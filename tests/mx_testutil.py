"""Helpers shared by the GPU parity tests (layout conversion, tolerance).

The tiled scale layout is the one documented in include/mx.h:
  byte(line r, block b) at ((r/128)*(KB/4) + b/4)*512 + (r%32)*16 + ((r%128)/32)*4 + b%4
with lines padded to MP = 128*ceil(mn/128) and blocks to KB = 8*ceil(k/256).
"""
import numpy as np

# Per-element GEMM tolerance: |C_gpu - C_ref| <= TOL * sum_t |a_t| |b_t|.
GEMM_TOL = 1e-5


def padded_dims(mn: int, k: int):
    return 128 * ((mn + 127) // 128), 8 * ((k + 255) // 256)


def tile_scales(canon: np.ndarray, mn: int, k: int) -> np.ndarray:
    """canonical scales [mn, k/32] -> flat tiled layout (padding zero)."""
    MP, KB = padded_dims(mn, k)
    full = np.zeros((MP, KB), dtype=np.uint8)
    full[:mn, :k // 32] = canon
    arr = full.reshape(MP // 128, 4, 32, KB // 4, 4)          # [g, sub, r32, ka, b4]
    return np.ascontiguousarray(arr.transpose(0, 3, 2, 1, 4)).reshape(-1)


def tile_scales_nv(canon: np.ndarray, mn: int, k: int) -> np.ndarray:
    """NVFP4 canonical scales [mn, k/16] -> flat tiled layout: the same atom
    geometry (128 lines x 4 blocks per 512 bytes) over KB = 16*ceil(k/256)
    blocks of 16 per line (padding zero)."""
    MP, KB = 128 * ((mn + 127) // 128), 16 * ((k + 255) // 256)
    full = np.zeros((MP, KB), dtype=np.uint8)
    full[:mn, :k // 16] = canon
    arr = full.reshape(MP // 128, 4, 32, KB // 4, 4)
    return np.ascontiguousarray(arr.transpose(0, 3, 2, 1, 4)).reshape(-1)


def untile_scales(flat: np.ndarray, mn: int, k: int) -> np.ndarray:
    MP, KB = padded_dims(mn, k)
    arr = np.asarray(flat, dtype=np.uint8)[:MP * KB].reshape(MP // 128, KB // 4, 32, 4, 4)
    full = arr.transpose(0, 3, 2, 1, 4).reshape(MP, KB)       # [g, sub, r32, ka, b4]
    return full[:mn, :k // 32]


def assert_gemm_close(C_gpu: np.ndarray, C_ref: np.ndarray, C_abs: np.ndarray, what: str = ""):
    C_gpu = np.asarray(C_gpu, dtype=np.float64)
    err = np.abs(C_gpu - C_ref)
    bound = GEMM_TOL * C_abs
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} entries outside tolerance; first "
            f"{[(tuple(i), float(C_gpu[tuple(i)]), float(C_ref[tuple(i)]), float(C_abs[tuple(i)])) for i in idx]}")
    ratio = np.where(C_abs > 0, err / np.where(C_abs > 0, C_abs, 1), 0.0)
    return float(ratio.max())
