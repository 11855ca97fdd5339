"""mx_linear_wgrad_noalloc: the Wgrad entry point for callers that cannot
allocate device memory (framework plugins whose device memory belongs to the
host framework's pool, bare C/Fortran hosts, hot loops that cannot afford
cudaMalloc's implicit synchronisation).  It keeps its scratch in a fixed
area inside the library instead of a caller workspace.

Checked here through the C ABI: two calls in a row (the second reuses the
scratch the first left behind) agree with mx_linear_wgrad, the workspace entry
point, within the GEMM tolerance used by every parity test
(1e-5 * sum |a||b|, sum taken from the oracle); oversize requests are
rejected before anything is launched.  This file is collected last on
purpose so that a run stopping at the first failure has run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import mxfp4_precision_gb300 as mx
from tests.mx_testutil import GEMM_TOL
from workloads import bf16_bits, config_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mxfp4_precision_gb300 import build
    build.build()
    mx.lib()


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def _sum_abs(dY, X, rot, nb, rnd, seed):
    Aq, As = oracle.quantize(dY, oracle.CONTRACT_ROWS, rot, nb, rnd, seed, 1)
    Bq, Bs = oracle.quantize(X, oracle.CONTRACT_ROWS, rot, nb, rnd, seed, 2)
    return oracle.gemm(Aq, As, Bq, Bs)[1]


def _noalloc_c_call(dY, X, out, rot, nb, rnd, seed):
    T, N = dY.shape
    K = X.shape[1]
    st = mx.lib().mx_linear_wgrad_noalloc(
        ctypes.c_void_p(dY.data_ptr()), ctypes.c_void_p(X.data_ptr()),
        ctypes.c_void_p(out.data_ptr()), T, N, K, rot, nb, rnd, seed,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def test_noalloc_matches_workspace_entry_point_two_calls():
    rng = np.random.default_rng(21)
    tiny = config_inputs("tiny", seed=0)
    cases = [
        (tiny["dY"], tiny["X"], mx.ROT_HADAMARD_DET, 32, mx.ROUND_RNE, 0),
        (bf16_bits(rng.standard_normal((1280, 200)).astype(np.float32) * np.float32(1e-3)),
         bf16_bits(rng.standard_normal((1280, 328)).astype(np.float32)),
         mx.ROT_HADAMARD_RAND, 64, mx.ROUND_SR, 3),
    ]
    for dY_bits, X_bits, rot, nb, rnd, seed in cases:      # two calls in a row
        dY, X = _dev(dY_bits), _dev(X_bits)
        out = torch.full((dY.shape[1], X.shape[1]), float("nan"), device="cuda")
        assert _noalloc_c_call(dY, X, out, rot, nb, rnd, seed) == 0
        mx.check_status()
        ref = mx.linear_wgrad(dY, X, rot=rot, rot_block=nb, rnd=rnd, seed=seed)
        mx.check_status()
        got = out.cpu().numpy().astype(np.float64)
        want = ref.cpu().numpy().astype(np.float64)
        bound = GEMM_TOL * _sum_abs(dY_bits, X_bits, rot, nb, rnd, seed)
        assert np.all(np.abs(got - want) <= bound)


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
