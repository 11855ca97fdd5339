"""mx_linear_wgrad_noalloc: the Wgrad entry point for callers that cannot
allocate device memory (framework plugins whose device memory belongs to the
host framework's pool, bare C/Fortran hosts, hot loops that cannot afford
cudaMalloc's implicit synchronisation).  It keeps its scratch in a fixed
area inside the library instead of a caller workspace.

Checked here through the C ABI:
  - a large call and then a smaller one with another rotation and rounding
    mode (so the smaller call runs on scratch the larger one filled) each give
    exactly the bits of mx_linear_wgrad, the workspace entry point, which runs
    the same kernels;
  - the large deterministic call also matches the oracle within the GEMM
    tolerance used by every parity test (1e-5 * sum |a||b|);
  - a warmed-up call changes neither torch's allocated bytes nor the device's
    free memory;
  - oversize requests are rejected before anything is launched.
This file is collected last on purpose so that a run stopping at the first
failure has run everything else; it passes alone as well.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import mxfp4_precision_gb300 as mx
from tests.mx_testutil import GEMM_TOL
from workloads import bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mxfp4_precision_gb300 import build
    build.build()
    mx.lib()


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def _noalloc_c_call(dY, X, out, rot, nb, rnd, seed):
    T, N = dY.shape
    K = X.shape[1]
    return mx.lib().mx_linear_wgrad_noalloc(
        ctypes.c_void_p(dY.data_ptr()), ctypes.c_void_p(X.data_ptr()),
        ctypes.c_void_p(out.data_ptr()), T, N, K, rot, nb, rnd, seed,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _inputs(T, N, K, seed):
    rng = np.random.default_rng(seed)
    dY = bf16_bits(rng.standard_normal((T, N)).astype(np.float32) * np.float32(1e-3))
    X = bf16_bits(rng.standard_normal((T, K)).astype(np.float32))
    return dY, X


def test_noalloc_large_then_small_call_bitwise_equal_to_workspace_entry_point():
    cases = [((8192, 4096, 4096), 31, mx.ROT_HADAMARD_DET, 32, mx.ROUND_RNE, 0),  # 35.7 MB
             ((1280, 200, 328), 32, mx.ROT_HADAMARD_RAND, 64, mx.ROUND_SR, 3)]
    for (T, N, K), s, rot, nb, rnd, seed in cases:
        dY_bits, X_bits = _inputs(T, N, K, s)
        dY, X = _dev(dY_bits), _dev(X_bits)
        out = torch.full((N, K), float("nan"), device="cuda")
        assert _noalloc_c_call(dY, X, out, rot, nb, rnd, seed) == 0
        mx.check_status()
        ref = mx.linear_wgrad(dY, X, rot=rot, rot_block=nb, rnd=rnd, seed=seed)
        mx.check_status()
        assert torch.equal(out.view(torch.int32), ref.view(torch.int32)), (T, N, K)
        if rnd == mx.ROUND_RNE:
            # and the oracle, on 4,096 random entries from every encoded line
            Aq, As = oracle.quantize(dY_bits, oracle.CONTRACT_ROWS, rot, nb, rnd, seed, 1)
            Bq, Bs = oracle.quantize(X_bits, oracle.CONTRACT_ROWS, rot, nb, rnd, seed, 2)
            rng = np.random.default_rng(5)
            ii, jj = rng.integers(0, N, 4096), rng.integers(0, K, 4096)
            C, Ca = oracle.gemm_entries(Aq, As, Bq, Bs, ii, jj)
            got = out.cpu().numpy()[ii, jj].astype(np.float64)
            assert np.all(np.abs(got - C) <= GEMM_TOL * Ca)


def test_noalloc_call_allocates_nothing():
    dY_bits, X_bits = _inputs(1024, 256, 512, 41)
    dY, X = _dev(dY_bits), _dev(X_bits)
    out = torch.empty((256, 512), device="cuda")
    for _ in range(2):                            # warm up: scratch address, modules
        assert _noalloc_c_call(dY, X, out, mx.ROT_HADAMARD_DET, 32, mx.ROUND_RNE, 0) == 0
    torch.cuda.synchronize()
    alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    assert _noalloc_c_call(dY, X, out, mx.ROT_HADAMARD_DET, 32, mx.ROUND_RNE, 0) == 0
    torch.cuda.synchronize()
    mx.check_status()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0


def test_noalloc_rejects_requests_beyond_the_scratch_area():
    T, N, K = 16384, 4096, 4096                 # needs 71.3 MB > 64 MiB
    assert mx.linear_workspace_bytes(mx.OP_WGRAD, T, N, K) > mx.NOALLOC_SCRATCH_BYTES
    dummy = torch.empty(16, dtype=torch.int16, device="cuda")
    out = torch.empty(4, dtype=torch.float32, device="cuda")
    st = mx.lib().mx_linear_wgrad_noalloc(
        ctypes.c_void_p(dummy.data_ptr()), ctypes.c_void_p(dummy.data_ptr()),
        ctypes.c_void_p(out.data_ptr()), T, N, K, mx.ROT_HADAMARD_DET, 32, mx.ROUND_RNE, 0,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 4                              # MX_ERR_WORKSPACE, nothing launched
    mx.check_status()
