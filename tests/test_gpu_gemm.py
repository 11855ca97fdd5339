"""GPU parity: mx_gemm on oracle-encoded operands is within 1e-5 * sum|a||b|
of the oracle's double-precision contraction, element by element."""
import numpy as np
import pytest
import torch

import oracle
import mxfp4_precision_gb300 as mx
from tests.mx_testutil import assert_gemm_close, tile_scales
from workloads import bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mxfp4_precision_gb300 import build
    build.build()
    mx.lib()


def _operand(lines, k, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((lines, k)).astype(np.float32) * np.float32(scale)
    x[:, rng.choice(k, max(1, k // 100), replace=False)] *= 20
    bits = bf16_bits(x)
    q, s = oracle.quantize(bits, oracle.CONTRACT_COLS, oracle.ROT_HADAMARD_DET, 32)
    return q, s


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_gemm(Aq, As, Bq, Bs, M, N, K):
    C = mx.gemm(_dev(Aq), _dev(tile_scales(As, M, K)), _dev(Bq), _dev(tile_scales(Bs, N, K)),
                M, N, K)
    mx.check_status()
    return C.cpu().numpy()


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (200, 328, 800), (512, 768, 2048),
                                   (384, 1024, 1024), (136, 120, 96), (256, 512, 8192),
                                   (130, 252, 512), (300, 1028, 1024)])
def test_gemm_parity(M, N, K):
    Aq, As = _operand(M, K, 1, 1e-3)
    Bq, Bs = _operand(N, K, 2)
    C = run_gemm(Aq, As, Bq, Bs, M, N, K)
    Cref, Cabs = oracle.gemm(Aq, As, Bq, Bs)
    worst = assert_gemm_close(C, Cref, Cabs, f"gemm {M}x{N}x{K}")
    assert worst < 1e-5


def _pairs():
    # the GEMM runs one 256 x 256 tile per 2-CTA pair at a time
    return torch.cuda.get_device_properties(0).multi_processor_count // 2


@pytest.mark.parametrize("N", [2048, 2048 - 100, 1792 + 100])
def test_gemm_small_last_round(N):
    """A few more 256 x 256 tiles than pairs: two rounds (the launcher spreads
    them over fewer pairs).  N = 1948 and N = 1892 leave the last column tile
    156 and 100 wide; M is ragged too."""
    n_tiles = (N + 255) // 256
    m_tiles = (_pairs() + 4 + n_tiles - 1) // n_tiles
    M, K = 256 * m_tiles - 37, 1024
    Aq, As = _operand(M, K, 11, 1e-3)
    Bq, Bs = _operand(N, K, 12)
    C = run_gemm(Aq, As, Bq, Bs, M, N, K)
    Cref, Cabs = oracle.gemm(Aq, As, Bq, Bs)
    assert assert_gemm_close(C, Cref, Cabs, f"small last round {M}x{N}x{K}") < 1e-5


@pytest.mark.parametrize("K", [1536, 1312, 1280, 1056])
def test_gemm_odd_stage_count(K):
    """Three 512-wide K stages per tile, over several tiles per pair (so the
    operand and scale rings wrap).  1312: the last 256-wide sub-tile is ragged;
    1280 and 1056: the last stage holds one sub-tile (1056: ragged too)."""
    n_tiles = 8
    m_tiles = (_pairs() + 6 + n_tiles - 1) // n_tiles
    M, N = 256 * m_tiles, 256 * n_tiles
    Aq, As = _operand(M, K, 15, 1e-3)
    Bq, Bs = _operand(N, K, 16)
    C = run_gemm(Aq, As, Bq, Bs, M, N, K)
    Cref, Cabs = oracle.gemm(Aq, As, Bq, Bs)
    assert assert_gemm_close(C, Cref, Cabs, f"odd split {M}x{N}x{K}") < 1e-5


def test_gemm_last_round_across_bands():
    """Tiles run in bands of 16 tile rows; here the last round spans the end of
    one band and a whole later band of one row (17 x 5 tiles)."""
    M, N, K = 17 * 256, 5 * 256, 1024
    Aq, As = _operand(M, K, 17, 1e-3)
    Bq, Bs = _operand(N, K, 18)
    C = run_gemm(Aq, As, Bq, Bs, M, N, K)
    Cref, Cabs = oracle.gemm(Aq, As, Bq, Bs)
    assert assert_gemm_close(C, Cref, Cabs, f"tail across bands {M}x{N}x{K}") < 1e-5


def test_gemm_large_last_round():
    """More tiles than pairs, by more than half the pairs (two rounds)."""
    n_tiles = 8
    m_tiles = (_pairs() + _pairs() // 2 + 10 + n_tiles - 1) // n_tiles
    M, N, K = 256 * m_tiles, 256 * n_tiles, 512
    Aq, As = _operand(M, K, 13, 1e-3)
    Bq, Bs = _operand(N, K, 14)
    C = run_gemm(Aq, As, Bq, Bs, M, N, K)
    Cref, Cabs = oracle.gemm(Aq, As, Bq, Bs)
    assert assert_gemm_close(C, Cref, Cabs, f"large last round {M}x{N}x{K}") < 1e-5


def test_gemm_deterministic():
    """Repeated runs give the same bits: every output element is accumulated
    in one fixed order."""
    n_tiles = 8
    m_tiles = (_pairs() + 4 + n_tiles - 1) // n_tiles
    M, N, K = 256 * m_tiles, 256 * n_tiles, 1024
    Aq, As = _operand(M, K, 21, 1e-3)
    Bq, Bs = _operand(N, K, 22)
    args = (_dev(Aq), _dev(tile_scales(As, M, K)), _dev(Bq), _dev(tile_scales(Bs, N, K)), M, N, K)
    first = mx.gemm(*args)
    for _ in range(3):
        again = mx.gemm(*args)
        assert torch.equal(first, again)
    mx.check_status()


def test_gemm_zero_and_nan_scales():
    # a block whose scale byte is 0 (all-zero block) contributes nothing
    M, N, K = 128, 256, 512
    Aq, As = _operand(M, K, 3)
    Bq, Bs = _operand(N, K, 4)
    Aq[:, :16] = 0
    As[:, 0] = 0
    C = run_gemm(Aq, As, Bq, Bs, M, N, K)
    Cref, Cabs = oracle.gemm(Aq, As, Bq, Bs)
    assert_gemm_close(C, Cref, Cabs, "zero block")


def test_gemm_k_zero_and_empty():
    C = torch.full((4, 8), 5.0, device="cuda")
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    mx.gemm_into(z, z, z, z, C, 4, 8, 0)
    mx.check_status()
    assert float(C.abs().sum()) == 0.0
    C2 = torch.full((4, 8), 5.0, device="cuda")
    mx.gemm_into(z, z, z, z, C2, 0, 8, 64)
    mx.check_status()
    assert float(C2.sum()) == 5.0 * 32


def test_gemm_representable_matches_plain_matmul():
    # inputs already on the MXFP4 grid: the result is the plain GEMM of the inputs
    rng = np.random.default_rng(5)
    M, N, K = 256, 256, 1024
    grid = np.array([0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -1.5, -2, -3, -4, -6])
    A = rng.choice(grid, (M, K)) * np.exp2(rng.integers(-4, 4, (M, 1)))
    B = rng.choice(grid, (N, K)) * np.exp2(rng.integers(-4, 4, (N, 1)))
    Aq, As = oracle.quantize(bf16_bits(A.astype(np.float32)), oracle.CONTRACT_COLS)
    Bq, Bs = oracle.quantize(bf16_bits(B.astype(np.float32)), oracle.CONTRACT_COLS)
    C = run_gemm(Aq, As, Bq, Bs, M, N, K)
    deqA, deqB = oracle.dequantize(Aq, As), oracle.dequantize(Bq, Bs)
    exact = deqA @ deqB.T
    assert_gemm_close(C, exact, np.abs(deqA) @ np.abs(deqB).T, "representable")
