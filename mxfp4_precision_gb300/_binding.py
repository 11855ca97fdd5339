"""ctypes declarations of include/mx.h and torch-tensor marshalling.

Functions here only check that tensors have the dtype/device/contiguity the C
ABI documents, pass raw data pointers and the current CUDA stream, and turn
a non-zero mx_status into an exception.  Output buffers are allocated with
torch (device memory plumbing); all compute happens in the library.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB

ROT_NONE, ROT_HADAMARD_DET, ROT_HADAMARD_RAND = 0, 1, 2
ROUND_RNE, ROUND_SR = 0, 1
CONTRACT_ROWS, CONTRACT_COLS = 0, 1
OP_FPROP, OP_DGRAD, OP_WGRAD = 0, 1, 2

EXPORTED = [
    "mx_codes_bytes", "mx_scales_bytes", "mx_scales_to_canonical", "mx_quantize", "mx_quantize_pair", "mx_quantize_dual",
    "mx_gemm", "mx_linear_workspace_bytes",
    "mx_linear_wgrad", "mx_linear_fprop", "mx_linear_dgrad", "mx_linear_wgrad_noalloc",
    "mx_linear_wgrad_fused", "mx_linear_wgrad_fused_supported",
    "mx_mxfp8_codes_bytes", "mx_quantize_mxfp8", "mx_gemm_mxfp8",
    "mx_linear_wgrad_mxfp8_workspace_bytes", "mx_linear_wgrad_mxfp8",
    "mx_nvfp4_scales_bytes", "mx_quantize_nvfp4", "mx_gemm_nvfp4",
    "mx_linear_wgrad_nvfp4_workspace_bytes", "mx_linear_wgrad_nvfp4",
    "mx_check_status",
    "mx_debug_timeout_probe", "mx_bench_mma", "mx_status_string", "mx_version",
]

_lock = threading.Lock()
_lib = None


class MXError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def library_path() -> str:
    return LIB


def lib() -> ctypes.CDLL:
    """Load the in-tree C-ABI library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB):
                raise RuntimeError(
                    f"MXFP4 CUDA library not found at {LIB}; build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(LIB)
            P, i64, u64, i32, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                    ctypes.c_int, ctypes.c_size_t)
            L.mx_codes_bytes.argtypes = [i64, i64]
            L.mx_codes_bytes.restype = sz
            L.mx_scales_bytes.argtypes = [i64, i64]
            L.mx_scales_bytes.restype = sz
            L.mx_quantize.argtypes = [P, i64, i64, i32, i32, i32, i32, u64, P, P, P]
            L.mx_quantize.restype = i32
            L.mx_quantize_pair.argtypes = [P, i64, i64, P, i64, i64, i32, i32, i32, u64, P, P, P,
                                           P, P]
            L.mx_quantize_pair.restype = i32
            L.mx_quantize_dual.argtypes = [P, i64, i64, i32, i32, i32, u64, P, P, P, P, P]
            L.mx_quantize_dual.restype = i32
            L.mx_scales_to_canonical.argtypes = [P, i64, i64, P, P]
            L.mx_scales_to_canonical.restype = i32
            L.mx_gemm.argtypes = [P, P, P, P, P, i64, i64, i64, P]
            L.mx_gemm.restype = i32
            L.mx_linear_workspace_bytes.argtypes = [i32, i64, i64, i64]
            L.mx_linear_workspace_bytes.restype = sz
            for name in ("mx_linear_wgrad", "mx_linear_fprop", "mx_linear_dgrad"):
                fn = getattr(L, name)
                fn.argtypes = [P, P, P, i64, i64, i64, i32, i32, i32, u64, P, sz, P]
                fn.restype = i32
            L.mx_linear_wgrad_noalloc.argtypes = [P, P, P, i64, i64, i64, i32, i32, i32, u64, P]
            L.mx_linear_wgrad_noalloc.restype = i32
            L.mx_linear_wgrad_fused.argtypes = [P, P, P, i64, i64, i64, i32, i32, i32, u64, P, sz, P]
            L.mx_linear_wgrad_fused.restype = i32
            L.mx_linear_wgrad_fused_supported.argtypes = [i64, i64, i64, i32, i32, i32]
            L.mx_linear_wgrad_fused_supported.restype = i32
            L.mx_mxfp8_codes_bytes.argtypes = [i64, i64]
            L.mx_mxfp8_codes_bytes.restype = sz
            L.mx_quantize_mxfp8.argtypes = [P, i64, i64, P, P, P]
            L.mx_quantize_mxfp8.restype = i32
            L.mx_gemm_mxfp8.argtypes = [P, P, P, P, P, i64, i64, i64, P]
            L.mx_gemm_mxfp8.restype = i32
            L.mx_linear_wgrad_mxfp8_workspace_bytes.argtypes = [i64, i64, i64]
            L.mx_linear_wgrad_mxfp8_workspace_bytes.restype = sz
            L.mx_linear_wgrad_mxfp8.argtypes = [P, P, P, i64, i64, i64, P, sz, P]
            L.mx_linear_wgrad_mxfp8.restype = i32
            L.mx_nvfp4_scales_bytes.argtypes = [i64, i64]
            L.mx_nvfp4_scales_bytes.restype = sz
            L.mx_quantize_nvfp4.argtypes = [P, i64, i64, i32, i32, u64, P, P, P, P]
            L.mx_quantize_nvfp4.restype = i32
            L.mx_gemm_nvfp4.argtypes = [P, P, P, P, P, P, P, i64, i64, i64, P]
            L.mx_gemm_nvfp4.restype = i32
            L.mx_linear_wgrad_nvfp4_workspace_bytes.argtypes = [i64, i64, i64]
            L.mx_linear_wgrad_nvfp4_workspace_bytes.restype = sz
            L.mx_linear_wgrad_nvfp4.argtypes = [P, P, P, i64, i64, i64, i32, i32, u64, P, sz, P]
            L.mx_linear_wgrad_nvfp4.restype = i32
            L.mx_check_status.argtypes = [P]
            L.mx_check_status.restype = i32
            L.mx_debug_timeout_probe.argtypes = [i64, P]
            L.mx_debug_timeout_probe.restype = i32
            L.mx_bench_mma.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i64, P, P, P]
            L.mx_bench_mma.restype = i32
            L.mx_status_string.argtypes = [i32]
            L.mx_status_string.restype = ctypes.c_char_p
            L.mx_version.argtypes = []
            L.mx_version.restype = i32
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().mx_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != 0:
        raise MXError(status, what)


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _dev_ptr(t: torch.Tensor, name: str) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return int(t.data_ptr())


def codes_bytes(mn: int, k: int) -> int:
    return int(lib().mx_codes_bytes(mn, k))


def scales_bytes(mn: int, k: int) -> int:
    return int(lib().mx_scales_bytes(mn, k))


def linear_workspace_bytes(op: int, T: int, N: int, K: int) -> int:
    return int(lib().mx_linear_workspace_bytes(op, T, N, K))


def _as_bf16_bits(x: torch.Tensor) -> torch.Tensor:
    if x.dtype == torch.bfloat16:
        return x
    if x.dtype in (torch.int16, torch.uint16):
        return x
    raise ValueError("bf16 input expected (torch.bfloat16 or raw 16-bit patterns)")


# ---------------------------------------------------------------------------
def quantize_into(src: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, contract: int,
                  rot: int = ROT_NONE, rot_block: int = 32, rnd: int = ROUND_RNE, seed: int = 0,
                  stream=None) -> None:
    src = _as_bf16_bits(src)
    rows, cols = src.shape
    st = lib().mx_quantize(_dev_ptr(src, "src"), rows, cols, contract, rot, rot_block, rnd,
                           seed, _dev_ptr(codes, "codes"), _dev_ptr(scales, "scales"),
                           _stream(stream))
    _check(st, "mx_quantize")


def quantize(src: torch.Tensor, contract: int, rot: int = ROT_NONE, rot_block: int = 32,
             rnd: int = ROUND_RNE, seed: int = 0, stream=None):
    """Returns (codes uint8 [lines, k/2], scales uint8 [mx_scales_bytes] in the tiled layout)."""
    rows, cols = src.shape
    L, lines = (rows, cols) if contract == CONTRACT_ROWS else (cols, rows)
    codes = torch.empty((lines, L // 2), dtype=torch.uint8, device=src.device)
    scales = torch.empty((max(1, scales_bytes(lines, L)),), dtype=torch.uint8, device=src.device)
    quantize_into(src, codes, scales, contract, rot, rot_block, rnd, seed, stream)
    return codes, scales


def quantize_pair(src0: torch.Tensor, src1: torch.Tensor, rot: int = ROT_HADAMARD_DET,
                  rot_block: int = 32, rnd: int = ROUND_RNE, seed: int = 0, stream=None):
    """Both Wgrad operands (encoded down their rows) in one launch; returns
    ((codes0, scales0), (codes1, scales1))."""
    src0, src1 = _as_bf16_bits(src0), _as_bf16_bits(src1)
    (r0, c0), (r1, c1) = src0.shape, src1.shape
    out = []
    for r, c, d in ((r0, c0, src0.device), (r1, c1, src1.device)):
        out.append((torch.empty((c, r // 2), dtype=torch.uint8, device=d),
                    torch.empty((max(1, scales_bytes(c, r)),), dtype=torch.uint8, device=d)))
    st = lib().mx_quantize_pair(_dev_ptr(src0, "src0"), r0, c0, _dev_ptr(src1, "src1"), r1, c1, rot,
                                rot_block, rnd, seed, _dev_ptr(out[0][0], "codes0"),
                                _dev_ptr(out[0][1], "scales0"), _dev_ptr(out[1][0], "codes1"),
                                _dev_ptr(out[1][1], "scales1"), _stream(stream))
    _check(st, "mx_quantize_pair")
    return out[0], out[1]


def quantize_dual(src: torch.Tensor, rot: int = ROT_HADAMARD_DET, rot_block: int = 32,
                  rnd: int = ROUND_RNE, seed: int = 0, stream=None):
    """Both encodings of an output gradient dY [T, N] from one read: returns
    ((codes_t, scales_t), (codes_n, scales_n)) -- the Wgrad operand (contraction
    T, rotated) and the Dgrad operand (contraction N, no rotation)."""
    src = _as_bf16_bits(src)
    T, N = src.shape
    d = src.device
    codes_t = torch.empty((N, T // 2), dtype=torch.uint8, device=d)
    scales_t = torch.empty((max(1, scales_bytes(N, T)),), dtype=torch.uint8, device=d)
    codes_n = torch.empty((T, N // 2), dtype=torch.uint8, device=d)
    scales_n = torch.empty((max(1, scales_bytes(T, N)),), dtype=torch.uint8, device=d)
    st = lib().mx_quantize_dual(_dev_ptr(src, "src"), T, N, rot, rot_block, rnd, seed,
                                _dev_ptr(codes_t, "codes_t"), _dev_ptr(scales_t, "scales_t"),
                                _dev_ptr(codes_n, "codes_n"), _dev_ptr(scales_n, "scales_n"),
                                _stream(stream))
    _check(st, "mx_quantize_dual")
    return (codes_t, scales_t), (codes_n, scales_n)


def scales_to_canonical(scales: torch.Tensor, lines: int, k: int, stream=None) -> torch.Tensor:
    """Tiled scales -> canonical uint8 [lines, k/32] on the same device."""
    out = torch.empty((lines, k // 32), dtype=torch.uint8, device=scales.device)
    st = lib().mx_scales_to_canonical(_dev_ptr(scales, "scales"), lines, k, _dev_ptr(out, "canon"),
                                      _stream(stream))
    _check(st, "mx_scales_to_canonical")
    return out


def gemm_into(Aq, As, Bq, Bs, C: torch.Tensor, M: int, N: int, K: int, stream=None) -> None:
    st = lib().mx_gemm(_dev_ptr(Aq, "Aq"), _dev_ptr(As, "As"), _dev_ptr(Bq, "Bq"),
                       _dev_ptr(Bs, "Bs"), _dev_ptr(C, "C"), M, N, K, _stream(stream))
    _check(st, "mx_gemm")


def gemm(Aq, As, Bq, Bs, M: int, N: int, K: int, stream=None) -> torch.Tensor:
    C = torch.empty((M, N), dtype=torch.float32, device=Aq.device)
    gemm_into(Aq, As, Bq, Bs, C, M, N, K, stream)
    return C


def _linear(fn_name, op, a, b, out_shape, T, N, K, rot, rot_block, rnd, seed, ws, out, stream):
    a, b = _as_bf16_bits(a), _as_bf16_bits(b)
    need = linear_workspace_bytes(op, T, N, K)
    if ws is None:
        ws = torch.empty((max(need, 256),), dtype=torch.uint8, device=a.device)
    if out is None:
        out = torch.empty(out_shape, dtype=torch.float32, device=a.device)
    fn = getattr(lib(), fn_name)
    st = fn(_dev_ptr(a, "a"), _dev_ptr(b, "b"), _dev_ptr(out, "out"), T, N, K, rot, rot_block,
            rnd, seed, _dev_ptr(ws, "workspace"), ws.numel() * ws.element_size(), _stream(stream))
    _check(st, fn_name)
    return out


def linear_wgrad(dY, X, rot=ROT_HADAMARD_DET, rot_block=32, rnd=ROUND_RNE, seed=0, ws=None,
                 out=None, stream=None) -> torch.Tensor:
    """dW[N, K] = dY^T X with dY [T, N], X [T, K] (bf16); fp32 output."""
    T, N = dY.shape
    K = X.shape[1]
    return _linear("mx_linear_wgrad", OP_WGRAD, dY, X, (N, K), T, N, K, rot, rot_block, rnd,
                   seed, ws, out, stream)


NOALLOC_SCRATCH_BYTES = 64 << 20


# --------------------------------------------------------------------------- MXFP8 comparator
def mxfp8_codes_bytes(mn: int, k: int) -> int:
    return int(lib().mx_mxfp8_codes_bytes(mn, k))


def quantize_mxfp8(src: torch.Tensor, stream=None):
    """MXFP8 encode down the rows of src [rows, cols] (bf16): returns (codes
    uint8 [cols, rows], scales uint8 [mx_scales_bytes(cols, rows)], tiled)."""
    src = _as_bf16_bits(src)
    rows, cols = src.shape
    codes = torch.empty((cols, rows), dtype=torch.uint8, device=src.device)
    scales = torch.empty((max(1, scales_bytes(cols, rows)),), dtype=torch.uint8, device=src.device)
    st = lib().mx_quantize_mxfp8(_dev_ptr(src, "src"), rows, cols, _dev_ptr(codes, "codes"),
                                 _dev_ptr(scales, "scales"), _stream(stream))
    _check(st, "mx_quantize_mxfp8")
    return codes, scales


def gemm_mxfp8_into(Aq, As, Bq, Bs, C: torch.Tensor, M: int, N: int, K: int, stream=None) -> None:
    st = lib().mx_gemm_mxfp8(_dev_ptr(Aq, "Aq"), _dev_ptr(As, "As"), _dev_ptr(Bq, "Bq"),
                             _dev_ptr(Bs, "Bs"), _dev_ptr(C, "C"), M, N, K, _stream(stream))
    _check(st, "mx_gemm_mxfp8")


def gemm_mxfp8(Aq, As, Bq, Bs, M: int, N: int, K: int, stream=None) -> torch.Tensor:
    C = torch.empty((M, N), dtype=torch.float32, device=Aq.device)
    gemm_mxfp8_into(Aq, As, Bq, Bs, C, M, N, K, stream)
    return C


def linear_wgrad_mxfp8_workspace_bytes(T: int, N: int, K: int) -> int:
    return int(lib().mx_linear_wgrad_mxfp8_workspace_bytes(T, N, K))


# --------------------------------------------------------------------------- NVFP4 variant
def nvfp4_scales_bytes(mn: int, k: int) -> int:
    return int(lib().mx_nvfp4_scales_bytes(mn, k))


def quantize_nvfp4(src: torch.Tensor, rot: int = ROT_NONE, rot_block: int = 16, seed: int = 0,
                   stream=None):
    """NVFP4 encode down the rows of src [rows, cols] (bf16): returns (codes
    uint8 [cols, rows/2], scales uint8 [mx_nvfp4_scales_bytes], tiled, tensor
    amax as a one-element float32 device tensor)."""
    src = _as_bf16_bits(src)
    rows, cols = src.shape
    d = src.device
    codes = torch.empty((cols, rows // 2), dtype=torch.uint8, device=d)
    scales = torch.empty((max(1, nvfp4_scales_bytes(cols, rows)),), dtype=torch.uint8, device=d)
    amax = torch.empty((2,), dtype=torch.float32, device=d)
    st = lib().mx_quantize_nvfp4(_dev_ptr(src, "src"), rows, cols, rot, rot_block, seed,
                                 _dev_ptr(codes, "codes"), _dev_ptr(scales, "scales"),
                                 _dev_ptr(amax, "amax"), _stream(stream))
    _check(st, "mx_quantize_nvfp4")
    return codes, scales, amax[:1]


def gemm_nvfp4(Aq, As, amax_a, Bq, Bs, amax_b, M: int, N: int, K: int, stream=None):
    C = torch.empty((M, N), dtype=torch.float32, device=Aq.device)
    st = lib().mx_gemm_nvfp4(_dev_ptr(Aq, "Aq"), _dev_ptr(As, "As"), _dev_ptr(amax_a, "amax_a"),
                             _dev_ptr(Bq, "Bq"), _dev_ptr(Bs, "Bs"), _dev_ptr(amax_b, "amax_b"),
                             _dev_ptr(C, "C"), M, N, K, _stream(stream))
    _check(st, "mx_gemm_nvfp4")
    return C


def linear_wgrad_nvfp4_workspace_bytes(T: int, N: int, K: int) -> int:
    return int(lib().mx_linear_wgrad_nvfp4_workspace_bytes(T, N, K))


def linear_wgrad_nvfp4(dY, X, rot=ROT_NONE, rot_block=16, seed=0, ws=None, out=None,
                       stream=None) -> torch.Tensor:
    """dW[N, K] = dY^T X with both operands NVFP4-encoded along T; fp32 output."""
    dY, X = _as_bf16_bits(dY), _as_bf16_bits(X)
    T, N = dY.shape
    K = X.shape[1]
    if ws is None:
        need = linear_wgrad_nvfp4_workspace_bytes(T, N, K)
        ws = torch.empty((max(need, 256),), dtype=torch.uint8, device=dY.device)
    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=dY.device)
    st = lib().mx_linear_wgrad_nvfp4(_dev_ptr(dY, "dY"), _dev_ptr(X, "X"), _dev_ptr(out, "out"),
                                     T, N, K, rot, rot_block, seed, _dev_ptr(ws, "workspace"),
                                     ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "mx_linear_wgrad_nvfp4")
    return out


def linear_wgrad_mxfp8(dY, X, ws=None, out=None, stream=None) -> torch.Tensor:
    """dW[N, K] = dY^T X with both operands MXFP8-encoded along T; fp32 output."""
    dY, X = _as_bf16_bits(dY), _as_bf16_bits(X)
    T, N = dY.shape
    K = X.shape[1]
    if ws is None:
        need = linear_wgrad_mxfp8_workspace_bytes(T, N, K)
        ws = torch.empty((max(need, 256),), dtype=torch.uint8, device=dY.device)
    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=dY.device)
    st = lib().mx_linear_wgrad_mxfp8(_dev_ptr(dY, "dY"), _dev_ptr(X, "X"), _dev_ptr(out, "out"),
                                     T, N, K, _dev_ptr(ws, "workspace"),
                                     ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "mx_linear_wgrad_mxfp8")
    return out


def linear_wgrad_fused(dY, X, rot=ROT_HADAMARD_DET, rot_block=32, rnd=ROUND_RNE, seed=0, ws=None,
                       out=None, stream=None) -> torch.Tensor:
    """mx_linear_wgrad as one launch (encoder warps inside the GEMM); same
    result bits.  Raises MXError(MX_ERR_UNSUPPORTED) outside its modes."""
    T, N = dY.shape
    K = X.shape[1]
    return _linear("mx_linear_wgrad_fused", OP_WGRAD, dY, X, (N, K), T, N, K, rot, rot_block, rnd,
                   seed, ws, out, stream)


def linear_wgrad_noalloc(dY, X, rot=ROT_HADAMARD_DET, rot_block=32, rnd=ROUND_RNE, seed=0,
                         out=None, stream=None) -> torch.Tensor:
    """dW = dY^T X through mx_linear_wgrad_noalloc: the library's fixed scratch
    area instead of a workspace (for callers that cannot allocate; see mx.h)."""
    dY, X = _as_bf16_bits(dY), _as_bf16_bits(X)
    T, N = dY.shape
    K = X.shape[1]
    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=dY.device)
    st = lib().mx_linear_wgrad_noalloc(_dev_ptr(dY, "dY"), _dev_ptr(X, "X"), _dev_ptr(out, "out"),
                                       T, N, K, rot, rot_block, rnd, seed, _stream(stream))
    _check(st, "mx_linear_wgrad_noalloc")
    return out


def linear_fprop(X, W, rot=ROT_NONE, rot_block=32, rnd=ROUND_RNE, seed=0, ws=None, out=None,
                 stream=None) -> torch.Tensor:
    """Y[T, N] = X W^T with X [T, K], W [N, K] (bf16); fp32 output."""
    T, K = X.shape
    N = W.shape[0]
    return _linear("mx_linear_fprop", OP_FPROP, X, W, (T, N), T, N, K, rot, rot_block, rnd, seed,
                   ws, out, stream)


def linear_dgrad(dY, W, rot=ROT_NONE, rot_block=32, rnd=ROUND_RNE, seed=0, ws=None, out=None,
                 stream=None) -> torch.Tensor:
    """dX[T, K] = dY W with dY [T, N], W [N, K] (bf16); fp32 output."""
    T, N = dY.shape
    K = W.shape[1]
    return _linear("mx_linear_dgrad", OP_DGRAD, dY, W, (T, K), T, N, K, rot, rot_block, rnd,
                   seed, ws, out, stream)


def check_status(stream=None) -> None:
    _check(lib().mx_check_status(_stream(stream)), "mx_check_status")


def debug_timeout_probe(limit_us: int, stream=None) -> int:
    """Launch the never-completed-barrier probe; returns mx_check_status's code."""
    _check(lib().mx_debug_timeout_probe(limit_us, _stream(stream)), "mx_debug_timeout_probe")
    return int(lib().mx_check_status(_stream(stream)))


# Kinds of mx_bench_mma and the K one MMA instruction covers.
MMA_KINDS = {0: ("mxf4", 64), 1: ("mxf4nvf4.2X", 64), 2: ("mxf4nvf4.4X", 64), 3: ("f8f6f4.e4m3", 32),
             4: ("f16.bf16", 16), 5: ("mxf8f6f4.e4m3", 32)}


def bench_mma(kind: int, cta_group: int = 1, n: int = 256, mmas_per_iter: int = 4,
              copies_per_iter: int = 0, copy_shape: int = 0, depth: int = 0, flags: int = 0,
              iters: int = 20000, stream=None) -> dict:
    """Runs the tensor-core issue-rate microbenchmark once and returns the
    per-MMA time and the implied whole-GPU rate (the slowest CTA sets it)."""
    ns = torch.zeros(256, dtype=torch.int64, device="cuda")
    ctas = ctypes.c_int(0)
    _check(lib().mx_bench_mma(kind, cta_group, n, mmas_per_iter, copies_per_iter, copy_shape,
                              depth, flags, iters, _dev_ptr(ns, "ns"), ctypes.byref(ctas), _stream(stream)),
           "mx_bench_mma")
    check_status(stream)
    t = ns[:ctas.value].cpu().numpy()
    issuing = t[::cta_group] if cta_group == 2 else t
    if (issuing <= 0).any():
        raise MXError(6, "mx_bench_mma: a bounded wait expired")
    k = MMA_KINDS[kind][1]
    mmas = mmas_per_iter * iters
    flop_per_mma_sm = 2.0 * 128 * n * k
    ns_per_mma = float(issuing.max()) / mmas
    return {"kind": MMA_KINDS[kind][0], "cta_group": cta_group, "n": n, "ctas": ctas.value,
            "mmas_per_iter": mmas_per_iter, "copies_per_iter": copies_per_iter,
            "copy_shape": copy_shape, "depth": depth, "flags": flags, "iters": iters,
            "ns_per_mma": ns_per_mma, "ns_per_mma_median": float(sorted(issuing)[len(issuing) // 2]) / mmas,
            "tflops": flop_per_mma_sm * ctas.value / ns_per_mma / 1e3}
