"""GPU parity of the NVFP4 variant (E2M1 in blocks of 16, UE4M3 block scale,
fp32 tensor scale; the prior-work format of [36kr]'s introduction) against
the oracle, through the C ABI:
  - the two-launch encoder bit-exact: the tensor amax, every code byte and
    the tiled scale bytes (padding included), with no rotation and with
    Hadamard 16 / 32 (deterministic and with random signs), on ragged shapes
    and on blocks with zeros, subnormals, Inf/NaN and saturating values;
  - the GEMM (kind::mxf4nvf4 scale_vec::4X, result divided by the two tensor
    scales) within the GEMM tolerance on ragged shapes, deterministic;
  - the Wgrad entry point at the o_proj and down_proj shapes on sampled
    output entries.
"""
import numpy as np
import pytest
import torch

import oracle
import mxfp4_precision_gb300 as mx
from tests.mx_testutil import assert_gemm_close, tile_scales_nv
from workloads import bf16_bits, config_inputs

pytestmark = pytest.mark.gpu

OROT = {mx.ROT_NONE: oracle.ROT_NONE, mx.ROT_HADAMARD_DET: oracle.ROT_HADAMARD_DET,
        mx.ROT_HADAMARD_RAND: oracle.ROT_HADAMARD_RAND}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mxfp4_precision_gb300 import build
    build.build()
    mx.lib()


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def _random_bits(rows, cols, seed, spread=10):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols)) * np.exp2(rng.integers(-spread, spread, size=(1, cols)))
    return bf16_bits(x.astype(np.float32))


def _check_encode(bits, rot=mx.ROT_NONE, nb=16, seed=0):
    rows, cols = bits.shape
    codes, scales, amax = mx.quantize_nvfp4(_dev(bits), rot, nb, seed)
    mx.check_status()
    ref_c, ref_s, ref_amax, _ = oracle.quantize_nvfp4(bits, oracle.CONTRACT_ROWS, OROT[rot], nb,
                                                      seed)
    assert float(amax.item()) == ref_amax
    got_c = codes.cpu().numpy()
    bad = np.argwhere(got_c != ref_c)
    assert bad.size == 0, f"{len(bad)} code bytes differ, first {bad[:4].tolist()}"
    tiled = scales.cpu().numpy()[:mx.nvfp4_scales_bytes(cols, rows)]
    exp = tile_scales_nv(ref_s, cols, rows)
    bad = np.flatnonzero(tiled != exp)
    assert bad.size == 0, f"{len(bad)} scale bytes differ, first {bad[:4].tolist()}"
    return codes, scales, amax


@pytest.mark.parametrize("rows,cols", [(32, 8), (320, 200), (1024, 136), (288, 392)])
@pytest.mark.parametrize("rot,nb", [(mx.ROT_NONE, 16), (mx.ROT_HADAMARD_DET, 16),
                                    (mx.ROT_HADAMARD_DET, 32), (mx.ROT_HADAMARD_RAND, 16),
                                    (mx.ROT_HADAMARD_RAND, 32)])
def test_encode_bit_exact_ragged(rows, cols, rot, nb):
    if rows % nb:
        pytest.skip("rotation block does not divide the contraction length")
    _check_encode(_random_bits(rows, cols, rows * 7 + cols), rot, nb, seed=5)


def test_encode_edge_values_bit_exact():
    rows, cols = 256, 64
    x = np.random.default_rng(3).standard_normal((rows, cols)).astype(np.float32)
    x[:, 0] = 0.0
    x[:, 1] *= 2.0 ** -128                          # subnormal blocks: scales round to small codes
    x[:, 2] *= 2.0 ** 100
    x[16:32, 3] = 0.0
    x[20, 3] = 3.3895313892515355e38                # bf16 max: the tensor amax
    x[64, 4] = np.inf
    x[100, 5] = np.nan
    x[0:16, 6] = -0.0
    x[:, 7] = 2.0 ** -133
    _check_encode(bf16_bits(x))
    # a tiny tensor: the tensor scale saturates at FLT_MAX
    y = (np.random.default_rng(4).standard_normal((64, 16)) * 1e-37).astype(np.float32)
    _check_encode(bf16_bits(y))
    _check_encode(bf16_bits(np.zeros((64, 16), np.float32)))


@pytest.mark.parametrize("M,N,K,rot", [(256, 256, 256, mx.ROT_NONE), (200, 136, 288, mx.ROT_NONE),
                                       (520, 392, 1056, mx.ROT_HADAMARD_DET),
                                       (2304, 2560, 160, mx.ROT_HADAMARD_RAND),
                                       (128, 4096, 2080, mx.ROT_NONE)])
def test_gemm_parity_ragged(M, N, K, rot):
    a = _random_bits(K, M, 21 + M)
    b = _random_bits(K, N, 22 + N)
    Aq, As, am = _check_encode(a, rot, 16, 1)
    Bq, Bs, bm = _check_encode(b, rot, 16, 1)
    C = mx.gemm_nvfp4(Aq, As, am, Bq, Bs, bm, M, N, K)
    mx.check_status()
    ra = oracle.quantize_nvfp4(a, oracle.CONTRACT_ROWS, OROT[rot], 16, 1)
    rb = oracle.quantize_nvfp4(b, oracle.CONTRACT_ROWS, OROT[rot], 16, 1)
    Cref, Cabs = oracle.gemm(ra[0], ra[1], rb[0], rb[1], oracle.FMT_NVFP4, ra[3], rb[3])
    assert_gemm_close(C.cpu().numpy(), Cref, Cabs, f"nvfp4 gemm {M}x{N}x{K}")
    C2 = mx.gemm_nvfp4(Aq, As, am, Bq, Bs, bm, M, N, K)
    mx.check_status()
    assert torch.equal(C.view(torch.int32), C2.view(torch.int32))


def test_unsupported_rotation_sizes_rejected():
    x = torch.zeros((256, 64), dtype=torch.int16, device="cuda")
    c = torch.empty(64 * 128, dtype=torch.uint8, device="cuda")
    s = torch.empty(mx.nvfp4_scales_bytes(64, 256), dtype=torch.uint8, device="cuda")
    a = torch.empty(2, dtype=torch.float32, device="cuda")
    st = mx.lib().mx_quantize_nvfp4(x.data_ptr(), 256, 64, mx.ROT_HADAMARD_DET, 64, 0,
                                    c.data_ptr(), s.data_ptr(), a.data_ptr(), None)
    assert st == 7                                              # MX_ERR_UNSUPPORTED
    mx.check_status()


@pytest.mark.slow
@pytest.mark.parametrize("name", ["o_proj", "down_proj"])
def test_wgrad_full_size_sampled(name):
    d = config_inputs(name, only=("dY", "X"))
    dY, X = d["dY"], d["X"]
    N, K = dY.shape[1], X.shape[1]
    out = mx.linear_wgrad_nvfp4(_dev(dY), _dev(X), rot=mx.ROT_HADAMARD_DET, rot_block=16)
    mx.check_status()
    rng = np.random.default_rng(9)
    ia = np.unique(np.concatenate([[0, 127, 128, N - 1], rng.choice(N, 60, replace=False)]))
    jb = np.unique(np.concatenate([[0, 255, 256, K - 1], rng.choice(K, 60, replace=False)]))
    A = oracle.quantize_nvfp4(dY, oracle.CONTRACT_ROWS, oracle.ROT_HADAMARD_DET, 16, lines=ia)
    B = oracle.quantize_nvfp4(X, oracle.CONTRACT_ROWS, oracle.ROT_HADAMARD_DET, 16, lines=jb)
    Cref, Cabs = oracle.gemm(A[0], A[1], B[0], B[1], oracle.FMT_NVFP4, A[3], B[3])
    assert_gemm_close(out.cpu().numpy()[np.ix_(ia, jb)], Cref, Cabs, f"{name} nvfp4 wgrad")


@pytest.mark.slow
def test_encode_every_line_o_proj_operand():
    """Every code and scale byte of the o_proj dY operand (8192 x 4096,
    Hadamard 16), the oracle partitioned by lines over the host cores (each
    call takes the tensor amax over every line, then encodes its share)."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    dY = config_inputs("o_proj", only=("dY",))["dY"]
    T, N = dY.shape
    codes, scales, amax = mx.quantize_nvfp4(_dev(dY), mx.ROT_HADAMARD_DET, 16, 0)
    mx.check_status()
    parts = max(1, min(os.cpu_count() or 1, 32))
    edges = np.linspace(0, N, parts + 1).astype(int)

    def one(i):
        return oracle.quantize_nvfp4(dY, oracle.CONTRACT_ROWS, oracle.ROT_HADAMARD_DET, 16,
                                     lines=np.arange(edges[i], edges[i + 1]))
    with ThreadPoolExecutor(parts) as ex:
        res = list(ex.map(one, range(parts)))
    assert float(amax.item()) == res[0][2]
    ref_c = np.concatenate([r[0] for r in res])
    ref_s = np.concatenate([r[1] for r in res])
    assert np.array_equal(codes.cpu().numpy(), ref_c)
    tiled = scales.cpu().numpy()[:mx.nvfp4_scales_bytes(N, T)]
    assert np.array_equal(tiled, tile_scales_nv(ref_s, N, T))
