"""The bounds-checked build (MX_CHECKED=1: every kernel store is guarded
against its buffer's extent and a violation is recorded as MX_ERR_BOUNDS
instead of being written) runs the ragged and edge shapes of the other
tests: no store may fall outside its buffer, and the results must equal
the normal build's byte for byte.  This stands in for compute-sanitizer,
which is not available here."""
import ctypes

import numpy as np
import pytest
import torch

import mxfp4_precision_gb300 as mx
from mxfp4_precision_gb300 import build
from workloads import bf16_bits

pytestmark = pytest.mark.gpu

P, i64, u64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int, ctypes.c_size_t


@pytest.fixture(scope="module")
def libs():
    build.build()
    normal = mx.lib()
    checked = ctypes.CDLL(build.build(checked=True))
    for L in (normal, checked):
        L.mx_quantize.argtypes = [P, i64, i64, i32, i32, i32, i32, u64, P, P, P]
        L.mx_quantize_pair.argtypes = [P, i64, i64, P, i64, i64, i32, i32, i32, u64, P, P, P, P, P]
        L.mx_quantize_dual.argtypes = [P, i64, i64, i32, i32, i32, u64, P, P, P, P, P]
        L.mx_gemm.argtypes = [P, P, P, P, P, i64, i64, i64, P]
        L.mx_check_status.argtypes = [P]
        L.mx_scales_bytes.argtypes = [i64, i64]
        L.mx_scales_bytes.restype = sz
        L.mx_quantize_mxfp8.argtypes = [P, i64, i64, P, P, P]
        L.mx_gemm_mxfp8.argtypes = [P, P, P, P, P, i64, i64, i64, P]
        L.mx_quantize_nvfp4.argtypes = [P, i64, i64, i32, i32, u64, P, P, P, P]
        L.mx_gemm_nvfp4.argtypes = [P, P, P, P, P, P, P, i64, i64, i64, P]
        L.mx_nvfp4_scales_bytes.argtypes = [i64, i64]
        L.mx_nvfp4_scales_bytes.restype = sz
        L.mx_linear_workspace_bytes.argtypes = [i32, i64, i64, i64]
        L.mx_linear_workspace_bytes.restype = sz
        L.mx_linear_wgrad_fused.argtypes = [P, P, P, i64, i64, i64, i32, i32, i32, u64, P, sz, P]
    return normal, checked


def _bits(shape, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape).astype(np.float32)
    x[:, rng.choice(shape[1], 2, replace=False)] *= 30
    return torch.from_numpy(bf16_bits(x).view(np.int16)).cuda()


def _buf(n):
    # exact-size buffers, so that any overrun leaves the allocation
    return torch.full((max(1, n),), 0xA5, dtype=torch.uint8, device="cuda")


def _quantize(L, src, contract, rot, nb, rnd):
    rows, cols = src.shape
    k, lines = (rows, cols) if contract == 0 else (cols, rows)
    codes, scales = _buf(lines * k // 2), _buf(L.mx_scales_bytes(lines, k))
    st = L.mx_quantize(src.data_ptr(), rows, cols, contract, rot, nb, rnd, 3, codes.data_ptr(),
                       scales.data_ptr(), None)
    assert st == 0
    assert L.mx_check_status(None) == 0
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("shape,contract", [((800, 136), 0), ((136, 800), 1), ((1280, 200), 0),
                                            ((256, 64), 0), ((96, 32), 0), ((200, 1280), 1)])
@pytest.mark.parametrize("rot,nb,rnd", [(0, 32, 0), (1, 32, 0), (1, 16, 1), (2, 32, 0)])
def test_checked_quantize_stays_in_bounds(libs, shape, contract, rot, nb, rnd):
    src = _bits(shape, 1)
    k = shape[0] if contract == 0 else shape[1]
    if k % nb:
        pytest.skip("contraction length not a multiple of the Hadamard size")
    normal, checked = libs
    a, b = _quantize(normal, src, contract, rot, nb, rnd), _quantize(checked, src, contract, rot, nb, rnd)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("nb", [64, 128, 256])
def test_checked_wide_hadamard_stays_in_bounds(libs, nb):
    src = _bits((1024, 200), 2)
    normal, checked = libs
    a, b = _quantize(normal, src, 0, 1, nb, 0), _quantize(checked, src, 0, 1, nb, 0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_checked_dual_and_pair_stay_in_bounds(libs):
    T, N, K = 800, 352, 96
    dy, x = _bits((T, N), 3), _bits((T, K), 4)
    outs = []
    for L in libs:
        ct, st_ = _buf(N * T // 2), _buf(L.mx_scales_bytes(N, T))
        cn, sn = _buf(T * N // 2), _buf(L.mx_scales_bytes(T, N))
        assert L.mx_quantize_dual(dy.data_ptr(), T, N, 1, 32, 0, 0, ct.data_ptr(), st_.data_ptr(),
                                  cn.data_ptr(), sn.data_ptr(), None) == 0
        c0, s0 = _buf(N * T // 2), _buf(L.mx_scales_bytes(N, T))
        c1, s1 = _buf(K * T // 2), _buf(L.mx_scales_bytes(K, T))
        assert L.mx_quantize_pair(dy.data_ptr(), T, N, x.data_ptr(), T, K, 1, 32, 0, 0,
                                  c0.data_ptr(), s0.data_ptr(), c1.data_ptr(), s1.data_ptr(),
                                  None) == 0
        assert L.mx_check_status(None) == 0
        outs.append([t.cpu().numpy() for t in (ct, st_, cn, sn, c0, s0, c1, s1)])
    for u, v in zip(*outs):
        assert np.array_equal(u, v)


@pytest.mark.parametrize("M,N,K", [(200, 328, 800), (136, 120, 96), (384, 1024, 1024)])
def test_checked_gemm_stays_in_bounds(libs, M, N, K):
    a, b = _bits((K, M), 5), _bits((K, N), 6)
    normal, _ = libs
    aq, as_ = _quantize(normal, a, 0, 0, 32, 0)
    bq, bs = _quantize(normal, b, 0, 0, 32, 0)
    d = [torch.from_numpy(v).cuda() for v in (aq, as_, bq, bs)]
    outs = []
    for L in libs:
        C = torch.empty((M, N), dtype=torch.float32, device="cuda")
        assert L.mx_gemm(*(t.data_ptr() for t in d), C.data_ptr(), M, N, K, None) == 0
        assert L.mx_check_status(None) == 0
        outs.append(C.cpu().numpy())
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("M,N,K", [(200, 136, 800), (136, 392, 288), (384, 256, 1056)])
def test_checked_mxfp8_and_nvfp4_stay_in_bounds(libs, M, N, K):
    """The FP8 comparator's and the NVFP4 variant's encoders (staged tile
    stores, the NVFP4 amax pass) and GEMMs, with exact-size buffers."""
    a, b = _bits((K, M), 7), _bits((K, N), 8)
    outs = []
    for L in libs:
        got = []
        # MXFP8: one code byte per element
        a8 = [_buf(M * K), _buf(L.mx_scales_bytes(M, K))]
        b8 = [_buf(N * K), _buf(L.mx_scales_bytes(N, K))]
        assert L.mx_quantize_mxfp8(a.data_ptr(), K, M, a8[0].data_ptr(), a8[1].data_ptr(), None) == 0
        assert L.mx_quantize_mxfp8(b.data_ptr(), K, N, b8[0].data_ptr(), b8[1].data_ptr(), None) == 0
        C8 = torch.empty((M, N), dtype=torch.float32, device="cuda")
        assert L.mx_gemm_mxfp8(a8[0].data_ptr(), a8[1].data_ptr(), b8[0].data_ptr(),
                               b8[1].data_ptr(), C8.data_ptr(), M, N, K, None) == 0
        # NVFP4 with a deterministic Hadamard 16
        amax = torch.zeros(4, dtype=torch.float32, device="cuda")
        a4 = [_buf(M * K // 2), _buf(L.mx_nvfp4_scales_bytes(M, K))]
        b4 = [_buf(N * K // 2), _buf(L.mx_nvfp4_scales_bytes(N, K))]
        assert L.mx_quantize_nvfp4(a.data_ptr(), K, M, 1, 16, 0, a4[0].data_ptr(),
                                   a4[1].data_ptr(), amax.data_ptr(), None) == 0
        assert L.mx_quantize_nvfp4(b.data_ptr(), K, N, 1, 16, 0, b4[0].data_ptr(),
                                   b4[1].data_ptr(), amax.data_ptr() + 8, None) == 0
        C4 = torch.empty((M, N), dtype=torch.float32, device="cuda")
        assert L.mx_gemm_nvfp4(a4[0].data_ptr(), a4[1].data_ptr(), amax.data_ptr(),
                               b4[0].data_ptr(), b4[1].data_ptr(), amax.data_ptr() + 8,
                               C4.data_ptr(), M, N, K, None) == 0
        assert L.mx_check_status(None) == 0
        outs.append([t.cpu().numpy() for t in (*a8, *b8, C8, *a4, *b4, C4, amax)])
    for u, v in zip(*outs):
        assert np.array_equal(u, v)


def test_checked_fused_wgrad_stays_in_bounds(libs):
    """The one-launch Wgrad (encoder warps inside the GEMM) on several panel groups."""
    T, N, K = 1024, 768, 512
    dy, x = _bits((T, N), 9), _bits((T, K), 10)
    outs = []
    for L in libs:
        need = L.mx_linear_workspace_bytes(2, T, N, K)       # MX_OP_WGRAD
        ws = _buf(need)
        dW = torch.empty((N, K), dtype=torch.float32, device="cuda")
        assert L.mx_linear_wgrad_fused(dy.data_ptr(), x.data_ptr(), dW.data_ptr(), T, N, K, 1, 32,
                                       0, 0, ws.data_ptr(), need, None) == 0
        assert L.mx_check_status(None) == 0
        outs.append(dW.cpu().numpy())
    assert np.array_equal(outs[0].view(np.int32), outs[1].view(np.int32))
