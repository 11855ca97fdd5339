"""CPU oracle for the MXFP4 path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
reference arm may import this package.  The product package
(``mxfp4_precision_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``mx_oracle.c`` (plain single-threaded C, fp32
operations rounded once each, double for the contraction); this module only
compiles it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mx_oracle.c")
_HDR = os.path.join(_HERE, "mx_oracle.h")
_BUILD_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD_DIR, "liboracle.so")

FMT_MXFP4, FMT_MXFP8, FMT_NVFP4 = 0, 1, 2
ROT_NONE, ROT_HADAMARD_DET, ROT_HADAMARD_RAND = 0, 1, 2
ROUND_RNE, ROUND_SR = 0, 1
CONTRACT_ROWS, CONTRACT_COLS = 0, 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FP contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_SO)
             or os.path.getmtime(_SO) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-Wall", "-Wextra", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            P = ctypes.c_void_p
            i64, u64, i32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_int
            L.oracle_philox4x32_10.argtypes = [P, P, P]
            L.oracle_sign.argtypes = [u64, i64]
            L.oracle_sign.restype = i32
            L.oracle_sr_u24.argtypes = [u64, u64, u64]
            L.oracle_sr_u24.restype = ctypes.c_uint32
            L.oracle_fwht_f32.argtypes = [P, i32]
            L.oracle_hadamard_f64.argtypes = [P, i32, P]
            L.oracle_scale_byte.argtypes = [ctypes.c_float]
            L.oracle_scale_byte.restype = ctypes.c_uint8
            L.oracle_e2m1_rne.argtypes = [ctypes.c_float]
            L.oracle_e2m1_rne.restype = ctypes.c_uint8
            L.oracle_e2m1_sr.argtypes = [ctypes.c_float, ctypes.c_uint32]
            L.oracle_e2m1_sr.restype = ctypes.c_uint8
            L.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
            L.oracle_e2m1_value.restype = ctypes.c_double
            L.oracle_scale_bytes.argtypes = [P, i64, P]
            L.oracle_e2m1_rne_vec.argtypes = [P, i64, P]
            L.oracle_e2m1_sr_vec.argtypes = [P, P, i64, P]
            L.oracle_rotate_line.argtypes = [P, i64, i64, i64, i32, i32, u64, i32, P]
            L.oracle_rotate_line.restype = i32
            L.oracle_quantize.argtypes = [P, i64, i64, i32, i32, i32, i32, u64, u64, P, i64,
                                          i32, P, P]
            L.oracle_quantize.restype = i32
            L.oracle_dequantize.argtypes = [P, P, i64, i64, P]
            L.oracle_gemm_entries.argtypes = [P, P, P, P, i64, P, P, i64, P, P]
            L.oracle_gemm_rows.argtypes = [P, P, P, P, i64, i64, i64, i64, i64, P, P]
            L.oracle_scale_byte_e4m3.argtypes = [ctypes.c_float]
            L.oracle_scale_byte_e4m3.restype = ctypes.c_uint8
            L.oracle_e4m3_rne.argtypes = [ctypes.c_float]
            L.oracle_e4m3_rne.restype = ctypes.c_uint8
            L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_value.restype = ctypes.c_double
            L.oracle_scale_bytes_e4m3.argtypes = [P, i64, P]
            L.oracle_e4m3_rne_vec.argtypes = [P, i64, P]
            L.oracle_quantize_mxfp8.argtypes = [P, i64, i64, i32, i32, i32, u64, P, i64, i32,
                                                P, P]
            L.oracle_quantize_mxfp8.restype = i32
            d = ctypes.c_double
            L.oracle_dequantize_fmt.argtypes = [i32, P, P, i64, i64, d, P]
            L.oracle_gemm_entries_fmt.argtypes = [i32, P, P, d, P, P, d, i64, P, P, i64, P, P]
            L.oracle_gemm_rows_fmt.argtypes = [i32, P, P, d, P, P, d, i64, i64, i64, i64, i64,
                                               P, P]
            L.oracle_nvfp4_tensor_scale.argtypes = [ctypes.c_float]
            L.oracle_nvfp4_tensor_scale.restype = ctypes.c_float
            L.oracle_nvfp4_block_scale.argtypes = [ctypes.c_float, ctypes.c_float]
            L.oracle_nvfp4_block_scale.restype = ctypes.c_uint8
            L.oracle_quantize_nvfp4.argtypes = [P, i64, i64, i32, i32, i32, u64, P, i64, i32,
                                                P, P, P, P]
            L.oracle_quantize_nvfp4.restype = i32
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# --------------------------------------------------------------------------
# scalar / vector element routines
# --------------------------------------------------------------------------
def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32).reshape(4))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32).reshape(2))
    out = np.zeros(4, dtype=np.uint32)
    lib().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def sign(seed: int, t: int) -> int:
    return int(lib().oracle_sign(seed, t))


def sr_u24(seed: int, tag: int, e: int) -> int:
    return int(lib().oracle_sr_u24(seed, tag, e))


def fwht_f32(x) -> np.ndarray:
    y = np.ascontiguousarray(np.array(x, dtype=np.float32))
    lib().oracle_fwht_f32(_ptr(y), int(y.size))
    return y


def hadamard_f64(x) -> np.ndarray:
    xd = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    y = np.zeros_like(xd)
    lib().oracle_hadamard_f64(_ptr(xd), int(xd.size), _ptr(y))
    return y


def scale_bytes(amax) -> np.ndarray:
    shape = np.shape(amax)
    a = np.ascontiguousarray(np.asarray(amax, dtype=np.float32).reshape(-1))
    out = np.zeros(a.shape, dtype=np.uint8)
    lib().oracle_scale_bytes(_ptr(a), int(a.size), _ptr(out))
    return out.reshape(shape)


def e2m1_rne(v) -> np.ndarray:
    shape = np.shape(v)
    a = np.ascontiguousarray(np.asarray(v, dtype=np.float32).reshape(-1))
    out = np.zeros(a.shape, dtype=np.uint8)
    lib().oracle_e2m1_rne_vec(_ptr(a), int(a.size), _ptr(out))
    return out.reshape(shape)


def e2m1_sr(v, u24) -> np.ndarray:
    shape = np.broadcast_shapes(np.shape(v), np.shape(u24))
    a = np.ascontiguousarray(np.broadcast_to(np.asarray(v, dtype=np.float32), shape).reshape(-1))
    u = np.ascontiguousarray(np.broadcast_to(np.asarray(u24, dtype=np.uint32), shape).reshape(-1))
    out = np.zeros(a.shape, dtype=np.uint8)
    lib().oracle_e2m1_sr_vec(_ptr(a), _ptr(u), int(a.size), _ptr(out))
    return out.reshape(shape)


def e2m1_value(code: int) -> float:
    return float(lib().oracle_e2m1_value(code))


def scale_bytes_e4m3(amax) -> np.ndarray:
    shape = np.shape(amax)
    a = np.ascontiguousarray(np.asarray(amax, dtype=np.float32).reshape(-1))
    out = np.zeros(a.shape, dtype=np.uint8)
    lib().oracle_scale_bytes_e4m3(_ptr(a), int(a.size), _ptr(out))
    return out.reshape(shape)


def e4m3_rne(v) -> np.ndarray:
    shape = np.shape(v)
    a = np.ascontiguousarray(np.asarray(v, dtype=np.float32).reshape(-1))
    out = np.zeros(a.shape, dtype=np.uint8)
    lib().oracle_e4m3_rne_vec(_ptr(a), int(a.size), _ptr(out))
    return out.reshape(shape)


def e4m3_value(code: int) -> float:
    return float(lib().oracle_e4m3_value(code))


# --------------------------------------------------------------------------
# operand encoding / decoding / contraction
# --------------------------------------------------------------------------
def rotate_line(line_bf16, rot: int, rot_block: int, seed: int = 0, precise: bool = False,
                t0: int = 0) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(line_bf16, dtype=np.uint16))
    out = np.zeros(x.size, dtype=np.float32)
    rc = lib().oracle_rotate_line(_ptr(x), 1, int(x.size), t0, rot, rot_block, seed,
                                  int(precise), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_rotate_line rejected its arguments")
    return out


def quantize(src_bf16: np.ndarray, contract: int, rot: int = ROT_NONE, rot_block: int = 32,
             rnd: int = ROUND_RNE, seed: int = 0, sr_tag: int = 1, lines=None,
             precise: bool = False):
    """Encode bf16 bits src[rows, cols]; returns (codes, canonical scales).

    contract=CONTRACT_ROWS -> codes [cols, rows/2], scales [cols, rows/32]
    contract=CONTRACT_COLS -> codes [rows, cols/2], scales [rows, cols/32]
    """
    src = np.ascontiguousarray(src_bf16, dtype=np.uint16)
    rows, cols = src.shape
    L = rows if contract == CONTRACT_ROWS else cols
    nl = cols if contract == CONTRACT_ROWS else rows
    if lines is not None:
        ln = np.ascontiguousarray(np.asarray(lines, dtype=np.int64))
        count, lp = ln.size, _ptr(ln)
    else:
        ln, count, lp = None, nl, None
    codes = np.zeros((count, L // 2), dtype=np.uint8)
    scales = np.zeros((count, L // 32), dtype=np.uint8)
    rc = lib().oracle_quantize(_ptr(src), rows, cols, contract, rot, rot_block, rnd, seed,
                               sr_tag, lp, count if ln is not None else 0, int(precise),
                               _ptr(codes), _ptr(scales))
    if rc != 0:
        raise ValueError("oracle_quantize rejected its arguments")
    return codes, scales


def quantize_mxfp8(src_bf16: np.ndarray, contract: int, rot: int = ROT_NONE,
                   rot_block: int = 32, seed: int = 0, lines=None, precise: bool = False):
    """MXFP8-encode bf16 bits src[rows, cols]; returns (codes, canonical scales).

    contract=CONTRACT_ROWS -> codes [cols, rows], scales [cols, rows/32]
    contract=CONTRACT_COLS -> codes [rows, cols], scales [rows, cols/32]
    """
    src = np.ascontiguousarray(src_bf16, dtype=np.uint16)
    rows, cols = src.shape
    L = rows if contract == CONTRACT_ROWS else cols
    nl = cols if contract == CONTRACT_ROWS else rows
    if lines is not None:
        ln = np.ascontiguousarray(np.asarray(lines, dtype=np.int64))
        count, lp = ln.size, _ptr(ln)
    else:
        ln, count, lp = None, nl, None
    codes = np.zeros((count, L), dtype=np.uint8)
    scales = np.zeros((count, L // 32), dtype=np.uint8)
    rc = lib().oracle_quantize_mxfp8(_ptr(src), rows, cols, contract, rot, rot_block, seed, lp,
                                     count if ln is not None else 0, int(precise), _ptr(codes),
                                     _ptr(scales))
    if rc != 0:
        raise ValueError("oracle_quantize_mxfp8 rejected its arguments")
    return codes, scales


def nvfp4_tensor_scale(amax: float) -> float:
    return float(lib().oracle_nvfp4_tensor_scale(amax))


def nvfp4_block_scale(block_amax: float, s_enc: float) -> int:
    return int(lib().oracle_nvfp4_block_scale(block_amax, s_enc))


def quantize_nvfp4(src_bf16: np.ndarray, contract: int, rot: int = ROT_NONE,
                   rot_block: int = 16, seed: int = 0, lines=None, precise: bool = False):
    """NVFP4-encode bf16 bits src[rows, cols]: returns (codes [lines, L/2],
    canonical scales [lines, L/16], tensor amax, s_enc)."""
    src = np.ascontiguousarray(src_bf16, dtype=np.uint16)
    rows, cols = src.shape
    L = rows if contract == CONTRACT_ROWS else cols
    nl = cols if contract == CONTRACT_ROWS else rows
    if lines is not None:
        ln = np.ascontiguousarray(np.asarray(lines, dtype=np.int64))
        count, lp = ln.size, _ptr(ln)
    else:
        ln, count, lp = None, nl, None
    codes = np.zeros((count, L // 2), dtype=np.uint8)
    scales = np.zeros((count, L // 16), dtype=np.uint8)
    amax, senc = ctypes.c_float(0), ctypes.c_float(0)
    rc = lib().oracle_quantize_nvfp4(_ptr(src), rows, cols, contract, rot, rot_block, seed, lp,
                                     count if ln is not None else 0, int(precise), _ptr(codes),
                                     _ptr(scales), ctypes.addressof(amax), ctypes.addressof(senc))
    if rc != 0:
        raise ValueError("oracle_quantize_nvfp4 rejected its arguments")
    return codes, scales, float(amax.value), float(senc.value)


def _k_of(codes: np.ndarray, fmt: int) -> int:
    return codes.shape[1] * (1 if fmt == FMT_MXFP8 else 2)


def dequantize(codes: np.ndarray, scales: np.ndarray, fmt: int = FMT_MXFP4,
               s_enc: float = 1.0) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    mn, k = c.shape[0], _k_of(c, fmt)
    out = np.zeros((mn, k), dtype=np.float64)
    lib().oracle_dequantize_fmt(fmt, _ptr(c), _ptr(s), mn, k, float(s_enc), _ptr(out))
    return out


def gemm_entries(Aq, As, Bq, Bs, ii, jj, fmt: int = FMT_MXFP4, a_senc: float = 1.0,
                 b_senc: float = 1.0):
    """C[i, j] and sum |a||b| for listed pairs (i, j); A, B contraction-major."""
    Aq, As, Bq, Bs = (np.ascontiguousarray(a, dtype=np.uint8) for a in (Aq, As, Bq, Bs))
    K = _k_of(Aq, fmt)
    ii = np.ascontiguousarray(np.asarray(ii, dtype=np.int64))
    jj = np.ascontiguousarray(np.asarray(jj, dtype=np.int64))
    C = np.zeros(ii.size, dtype=np.float64)
    Ca = np.zeros(ii.size, dtype=np.float64)
    lib().oracle_gemm_entries_fmt(fmt, _ptr(Aq), _ptr(As), float(a_senc), _ptr(Bq), _ptr(Bs),
                                  float(b_senc), K, _ptr(ii), _ptr(jj), int(ii.size), _ptr(C),
                                  _ptr(Ca))
    return C, Ca


def gemm_rows(Aq, As, Bq, Bs, m0: int = 0, m1: int | None = None, fmt: int = FMT_MXFP4,
              a_senc: float = 1.0, b_senc: float = 1.0):
    """Rows [m0, m1) of C = A B^T (double) and of sum |a||b|."""
    Aq, As, Bq, Bs = (np.ascontiguousarray(a, dtype=np.uint8) for a in (Aq, As, Bq, Bs))
    M, N, K = Aq.shape[0], Bq.shape[0], _k_of(Aq, fmt)
    m1 = M if m1 is None else m1
    C = np.zeros((m1 - m0, N), dtype=np.float64)
    Ca = np.zeros((m1 - m0, N), dtype=np.float64)
    lib().oracle_gemm_rows_fmt(fmt, _ptr(Aq), _ptr(As), float(a_senc), _ptr(Bq), _ptr(Bs),
                               float(b_senc), M, N, K, m0, m1, _ptr(C), _ptr(Ca))
    return C, Ca


def gemm(Aq, As, Bq, Bs, fmt: int = FMT_MXFP4, a_senc: float = 1.0, b_senc: float = 1.0):
    return gemm_rows(Aq, As, Bq, Bs, 0, None, fmt, a_senc, b_senc)
