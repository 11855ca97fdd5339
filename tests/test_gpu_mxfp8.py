"""GPU parity of the MXFP8 comparator path (E4M3 elements under the MX block
scale: the FP8 baseline of "Ende-zu-Ende-Effizienz", [36kr]) against the
oracle, through the C ABI:
  - the encoder bit-exact (codes, canonical scales and the zero padding of the
    tiled layout) on ragged shapes and on blocks with subnormal, saturating,
    zero and non-finite values, and on every line of an o_proj-sized operand;
  - the GEMM within the GEMM tolerance on ragged shapes (partial tiles, a
    ragged last K sub-tile, more tiles than resident CTA pairs), bitwise
    deterministic;
  - the Wgrad entry point at the o_proj and down_proj shapes on sampled
    output entries, each computed by the oracle from its own encodes.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import mxfp4_precision_gb300 as mx
from tests.mx_testutil import assert_gemm_close, tile_scales
from workloads import bf16_bits, bf16_bits_to_f32, config_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mxfp4_precision_gb300 import build
    build.build()
    mx.lib()


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def _random_bits(rows, cols, seed, spread=12):
    """bf16 [rows, cols]: normal values with a per-column magnitude spread."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols)) * np.exp2(rng.integers(-spread, spread, size=(1, cols)))
    return bf16_bits(x.astype(np.float32))


def _check_encode(bits):
    rows, cols = bits.shape
    codes, scales = mx.quantize_mxfp8(_dev(bits))
    mx.check_status()
    ref_c, ref_s = oracle.quantize_mxfp8(bits, oracle.CONTRACT_ROWS)
    got_c = codes.cpu().numpy()
    assert got_c.shape == ref_c.shape
    bad = np.argwhere(got_c != ref_c)
    assert bad.size == 0, f"{len(bad)} code bytes differ, first {bad[:4].tolist()}"
    tiled = scales.cpu().numpy()[:mx.scales_bytes(cols, rows)]
    assert np.array_equal(tiled, tile_scales(ref_s, cols, rows))   # padding bytes zero too
    return codes, scales


@pytest.mark.parametrize("rows,cols", [(32, 8), (320, 200), (1024, 136), (288, 392),
                                       (2048, 1032)])
def test_encode_bit_exact_ragged(rows, cols):
    _check_encode(_random_bits(rows, cols, rows + cols))


def test_encode_edge_values_bit_exact():
    rows, cols = 256, 64
    x = np.random.default_rng(3).standard_normal((rows, cols)).astype(np.float32)
    x[:, 0] = 0.0                                        # all-zero blocks
    x[:, 1] *= 2.0 ** -128                               # bf16 subnormals: scale clamps at 2^-127
    x[:, 2] *= 2.0 ** 120                                # near the top of the bf16 range
    x[32:64, 3] = 0.0
    x[40, 3] = 3.3895313892515355e38                     # bf16 max in a zero block
    x[64, 4] = np.inf                                    # Inf block: NaN scale, zero codes
    x[100, 5] = np.nan
    x[128:160, 6] = np.linspace(-1.99, 1.99, 32)         # 1.99 * 256 > 448: saturates
    x[160:192, 7] = 2.0 ** -10 * np.arange(32)           # values far below the block's amax
    x[0:32, 8] = -0.0
    x[:, 9] = np.where(np.arange(rows) % 2 == 0, 1.0, -1.0) * (1 + 1 / 16)   # E4M3 ties
    x[:, 10] = np.float32(2.0 ** -133)                   # smallest bf16 subnormal
    _check_encode(bf16_bits(x))


def _par_quantize_mxfp8(bits, n_lines, parts=None):
    parts = parts or max(1, min(os.cpu_count() or 1, 32))
    edges = np.linspace(0, n_lines, parts + 1).astype(int)

    def one(i):
        return oracle.quantize_mxfp8(bits, oracle.CONTRACT_ROWS,
                                     lines=np.arange(edges[i], edges[i + 1]))
    with ThreadPoolExecutor(parts) as ex:
        res = list(ex.map(one, range(parts)))
    return np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res])


@pytest.mark.slow
def test_encode_every_line_o_proj_operand():
    dY = config_inputs("o_proj", only=("dY",))["dY"]                 # [8192, 4096]
    codes, scales = mx.quantize_mxfp8(_dev(dY))
    mx.check_status()
    ref_c, ref_s = _par_quantize_mxfp8(dY, dY.shape[1])
    assert np.array_equal(codes.cpu().numpy(), ref_c)
    canon = mx.scales_to_canonical(scales, dY.shape[1], dY.shape[0]).cpu().numpy()
    assert np.array_equal(canon, ref_s)


@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (200, 136, 288), (520, 392, 1056),
                                   (2304, 2560, 160), (128, 4096, 2080)])
def test_gemm_parity_ragged(M, N, K):
    a = _random_bits(K, M, 11 + M)
    b = _random_bits(K, N, 12 + N)
    Aq, As = _check_encode(a)
    Bq, Bs = _check_encode(b)
    C = mx.gemm_mxfp8(Aq, As, Bq, Bs, M, N, K)
    mx.check_status()
    ra = oracle.quantize_mxfp8(a, oracle.CONTRACT_ROWS)
    rb = oracle.quantize_mxfp8(b, oracle.CONTRACT_ROWS)
    Cref, Cabs = oracle.gemm(*ra, *rb, fmt=oracle.FMT_MXFP8)
    assert_gemm_close(C.cpu().numpy(), Cref, Cabs, f"mxfp8 gemm {M}x{N}x{K}")
    C2 = mx.gemm_mxfp8(Aq, As, Bq, Bs, M, N, K)
    mx.check_status()
    assert torch.equal(C.view(torch.int32), C2.view(torch.int32))


def test_gemm_zero_contraction_and_empty():
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    C = torch.full((64, 64), float("nan"), device="cuda")
    mx.gemm_mxfp8_into(z, z, z, z, C, 64, 64, 0)
    mx.check_status()
    assert torch.count_nonzero(C).item() == 0
    assert mx.lib().mx_gemm_mxfp8(None, None, None, None, None, 0, 64, 64, None) == 0
    assert mx.lib().mx_quantize_mxfp8(None, 0, 64, None, None, None) == 0
    # the contraction length must be a multiple of 32
    st = mx.lib().mx_gemm_mxfp8(z.data_ptr(), z.data_ptr(), z.data_ptr(), z.data_ptr(),
                                C.data_ptr(), 64, 64, 48, None)
    assert st == 2                                                    # MX_ERR_SHAPE


@pytest.mark.slow
@pytest.mark.parametrize("name", ["o_proj", "down_proj"])
def test_wgrad_full_size_sampled(name):
    d = config_inputs(name, only=("dY", "X"))
    dY, X = d["dY"], d["X"]
    T, N = dY.shape
    K = X.shape[1]
    out = mx.linear_wgrad_mxfp8(_dev(dY), _dev(X))
    mx.check_status()
    rng = np.random.default_rng(7)
    ia = np.unique(np.concatenate([[0, 127, 128, N - 1], rng.choice(N, 60, replace=False)]))
    jb = np.unique(np.concatenate([[0, 255, 256, K - 1], rng.choice(K, 60, replace=False)]))
    Aq, As = oracle.quantize_mxfp8(dY, oracle.CONTRACT_ROWS, lines=ia)
    Bq, Bs = oracle.quantize_mxfp8(X, oracle.CONTRACT_ROWS, lines=jb)
    Cref, Cabs = oracle.gemm(Aq, As, Bq, Bs, fmt=oracle.FMT_MXFP8)
    got = out.cpu().numpy()[np.ix_(ia, jb)]
    assert_gemm_close(got, Cref, Cabs, f"{name} mxfp8 wgrad")
    # the MXFP8 result is closer to the exact product than the MXFP4 one
    exact = bf16_bits_to_f32(dY[:, ia]).astype(np.float64).T @ \
        bf16_bits_to_f32(X[:, jb]).astype(np.float64)
    out4 = mx.linear_wgrad(_dev(dY), _dev(X), rot=mx.ROT_HADAMARD_DET, rot_block=32)
    mx.check_status()
    e8 = np.linalg.norm(got - exact) / np.linalg.norm(exact)
    e4 = np.linalg.norm(out4.cpu().numpy()[np.ix_(ia, jb)] - exact) / np.linalg.norm(exact)
    assert e8 < e4
