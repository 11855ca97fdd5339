"""GPU parity: mx_quantize codes and scales are bit-exact with the oracle.

Shapes span several tiles with ragged tails (200 lines: not a multiple of the
64/128-line tiles; contraction 800: not a multiple of the 256 tile) and every
rotation size, random-sign mode and stochastic rounding."""
import numpy as np
import pytest
import torch

import oracle
import mxfp4_precision_gb300 as mx
from tests.mx_testutil import tile_scales, untile_scales
from workloads import bf16_bits, config_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mxfp4_precision_gb300 import build
    build.build()
    mx.lib()


def gpu_quantize(bits: np.ndarray, contract, rot, nb, rnd, seed):
    src = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    codes, scales = mx.quantize(src, contract, rot, nb, rnd, seed)
    mx.check_status()
    return codes.cpu().numpy(), scales.cpu().numpy()


def check_against_oracle(bits, contract, rot, nb, rnd, seed=0):
    rows, cols = bits.shape
    L, lines = (rows, cols) if contract == mx.CONTRACT_ROWS else (cols, rows)
    codes, scales = gpu_quantize(bits, contract, rot, nb, rnd, seed)
    oc, os_ = oracle.quantize(bits, contract, rot, nb, rnd, seed, 1)
    assert codes.shape == oc.shape
    diff = np.argwhere(codes != oc)
    assert diff.size == 0, f"{len(diff)} code bytes differ; first {diff[:4].tolist()}"
    assert np.array_equal(untile_scales(scales, lines, L), os_)
    assert np.array_equal(scales, tile_scales(os_, lines, L))   # padding bytes are zero


def _rand_bits(shape, seed, scale=1.0, outliers=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape).astype(np.float32) * np.float32(scale)
    if outliers:
        x[:, rng.choice(shape[1], 3, replace=False)] *= 20
    return bf16_bits(x)


ROTS = [(mx.ROT_NONE, 32), (mx.ROT_HADAMARD_DET, 16), (mx.ROT_HADAMARD_DET, 32),
        (mx.ROT_HADAMARD_DET, 64), (mx.ROT_HADAMARD_DET, 128), (mx.ROT_HADAMARD_DET, 256),
        (mx.ROT_HADAMARD_RAND, 32), (mx.ROT_HADAMARD_RAND, 256)]


@pytest.mark.parametrize("rot,nb", ROTS)
@pytest.mark.parametrize("rnd", [mx.ROUND_RNE, mx.ROUND_SR])
def test_colwise_parity(rot, nb, rnd):
    check_against_oracle(_rand_bits((1280, 200), 1), mx.CONTRACT_ROWS, rot, nb, rnd, seed=5)


@pytest.mark.parametrize("rot,nb", ROTS)
@pytest.mark.parametrize("rnd", [mx.ROUND_RNE, mx.ROUND_SR])
def test_rowwise_parity(rot, nb, rnd):
    check_against_oracle(_rand_bits((200, 1280), 2), mx.CONTRACT_COLS, rot, nb, rnd, seed=5)


@pytest.mark.parametrize("seed", [2**40 + 12345, 2**64 - 3])
@pytest.mark.parametrize("contract", [mx.CONTRACT_ROWS, mx.CONTRACT_COLS])
@pytest.mark.parametrize("rot,nb,rnd", [(mx.ROT_NONE, 32, mx.ROUND_SR),
                                        (mx.ROT_HADAMARD_RAND, 32, mx.ROUND_RNE),
                                        (mx.ROT_HADAMARD_RAND, 128, mx.ROUND_SR)])
def test_random_streams_use_the_whole_seed(seed, contract, rot, nb, rnd):
    """Seeds of more than 32 bits: the seed's high half is the second Philox key word of the
    random-sign and SR streams, in the column, wide and row kernels alike."""
    shape = (1280, 200) if contract == mx.CONTRACT_ROWS else (200, 1280)
    check_against_oracle(_rand_bits(shape, 3), contract, rot, nb, rnd, seed=seed)


@pytest.mark.parametrize("contract", [mx.CONTRACT_ROWS, mx.CONTRACT_COLS])
@pytest.mark.parametrize("rot,nb", [(mx.ROT_NONE, 32), (mx.ROT_HADAMARD_DET, 16),
                                    (mx.ROT_HADAMARD_DET, 32)])
def test_ragged_contraction_tail(contract, rot, nb):
    shape = (800, 136) if contract == mx.CONTRACT_ROWS else (136, 800)
    check_against_oracle(_rand_bits(shape, 3), contract, rot, nb, mx.ROUND_RNE)


def _edge_matrix():
    """256 x 64 bf16 (T x C) where each column exercises one edge case."""
    x = np.zeros((256, 64), dtype=np.float32)
    x[7, 1] = 3.0                                          # single non-zero
    x[:, 2] = np.exp2(np.arange(256) % 40 - 20)            # exact powers of two
    x[:, 3] = 1.75 * np.exp2(np.arange(256) % 7)           # amax mantissa > 1.5: saturation
    x[:, 4] = np.exp2(-133.0) * (np.arange(256) % 100 + 1)  # bf16 subnormals
    x[:, 5] = -0.0                                         # negative zeros
    ties = np.array([4, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.25, -0.75, -1.25, -1.75,
                     -2.5, -3.5, -5, 6, 0.5, 1, 1.5, 2, 3, -4, -6, 0.1, -0.1, 7, -7.5,
                     0.3, 1.1, 2.9, 4.4, -5.5], dtype=np.float32)
    x[:, 6] = np.tile(ties, 8) * np.float32(2.0 ** 3)      # exact ties at scale 2^3
    x[:, 7] = np.tile(ties, 8) * np.float32(2.0 ** -120)
    x[100, 8] = np.inf
    x[40, 9] = np.nan
    x[:, 10] = 3.0e38 * np.sign(np.arange(256) - 127.5)    # near the bf16 maximum
    x[:, 11] = 1.2e-38 * (np.arange(256) % 5 - 2)          # smallest normals
    x[5, 12] = -np.inf
    rng = np.random.default_rng(9)
    x[:, 13:] = rng.standard_normal((256, 51)) * np.exp2(rng.integers(-30, 30, (1, 51)))
    return bf16_bits(x)


@pytest.mark.parametrize("rot,nb", [(mx.ROT_NONE, 32), (mx.ROT_HADAMARD_DET, 32),
                                    (mx.ROT_HADAMARD_DET, 256), (mx.ROT_HADAMARD_RAND, 64)])
@pytest.mark.parametrize("rnd", [mx.ROUND_RNE, mx.ROUND_SR])
def test_edge_cases(rot, nb, rnd):
    x = _edge_matrix()
    check_against_oracle(x, mx.CONTRACT_ROWS, rot, nb, rnd, seed=3)
    check_against_oracle(np.ascontiguousarray(x.T), mx.CONTRACT_COLS, rot, nb, rnd, seed=3)


def test_deterministic_and_seeded():
    x = _rand_bits((512, 128), 4)
    a = gpu_quantize(x, mx.CONTRACT_ROWS, mx.ROT_HADAMARD_DET, 32, mx.ROUND_RNE, 0)
    b = gpu_quantize(x, mx.CONTRACT_ROWS, mx.ROT_HADAMARD_DET, 32, mx.ROUND_RNE, 77)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    r1 = gpu_quantize(x, mx.CONTRACT_ROWS, mx.ROT_HADAMARD_RAND, 32, mx.ROUND_SR, 1)
    r2 = gpu_quantize(x, mx.CONTRACT_ROWS, mx.ROT_HADAMARD_RAND, 32, mx.ROUND_SR, 1)
    r3 = gpu_quantize(x, mx.CONTRACT_ROWS, mx.ROT_HADAMARD_RAND, 32, mx.ROUND_SR, 2)
    assert np.array_equal(r1[0], r2[0]) and not np.array_equal(r1[0], r3[0])


def test_empty_inputs_are_noops():
    src = torch.zeros((0, 64), dtype=torch.int16, device="cuda")
    codes = torch.zeros(16, dtype=torch.uint8, device="cuda")
    mx.quantize_into(src, codes, codes, mx.CONTRACT_ROWS)
    mx.check_status()
    assert int(codes.sum()) == 0


def test_tiny_config_both_operands():
    d = config_inputs("tiny", seed=0)
    for name in ("dY", "X"):
        check_against_oracle(d[name], mx.CONTRACT_ROWS, mx.ROT_HADAMARD_DET, 32, mx.ROUND_RNE)


def _pair_check(dy_bits, x_bits, rot, nb, rnd, seed):
    (c0, s0), (c1, s1) = mx.quantize_pair(
        torch.from_numpy(np.ascontiguousarray(dy_bits).view(np.int16)).cuda(),
        torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda(), rot, nb, rnd, seed)
    mx.check_status()
    T = dy_bits.shape[0]
    for bits, (c, sc), tag in ((dy_bits, (c0, s0), 1), (x_bits, (c1, s1), 2)):
        oc, os_ = oracle.quantize(bits, oracle.CONTRACT_ROWS, rot, nb, rnd, seed, tag)
        assert np.array_equal(c.cpu().numpy(), oc)
        assert np.array_equal(sc.cpu().numpy(), tile_scales(os_, bits.shape[1], T))


@pytest.mark.parametrize("rot,nb,rnd", [(mx.ROT_HADAMARD_DET, 32, mx.ROUND_RNE),
                                        (mx.ROT_NONE, 32, mx.ROUND_SR),
                                        (mx.ROT_HADAMARD_DET, 16, mx.ROUND_RNE),
                                        (mx.ROT_HADAMARD_RAND, 32, mx.ROUND_RNE),
                                        (mx.ROT_HADAMARD_DET, 128, mx.ROUND_SR)])
def test_pair_launch_matches_oracle(rot, nb, rnd):
    # two operands of different widths (ragged vs the 64/128-line tiles), one launch
    _pair_check(_rand_bits((1280, 200), 7, 1e-3), _rand_bits((1280, 328), 8), rot, nb, rnd, 11)


def test_pair_launch_tiny_config():
    d = config_inputs("tiny", seed=0)
    _pair_check(d["dY"], d["X"], mx.ROT_HADAMARD_DET, 32, mx.ROUND_RNE, 0)


def _dual_check(bits, rot, nb, rnd, seed):
    (ct, st), (cn, sn) = mx.quantize_dual(
        torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda(), rot, nb, rnd, seed)
    mx.check_status()
    T, N = bits.shape
    # column direction (Wgrad operand): N lines, contraction T, rotated
    oc, os_ = oracle.quantize(bits, oracle.CONTRACT_ROWS, rot, nb, rnd, seed, 1)
    assert np.array_equal(ct.cpu().numpy(), oc)
    assert np.array_equal(st.cpu().numpy(), tile_scales(os_, N, T))
    # row direction (Dgrad operand): T lines, contraction N, no rotation
    oc, os_ = oracle.quantize(bits, oracle.CONTRACT_COLS, oracle.ROT_NONE, 32, rnd, seed, 1)
    assert np.array_equal(cn.cpu().numpy(), oc)
    assert np.array_equal(sn.cpu().numpy(), tile_scales(os_, T, N))  # padding bytes are zero


@pytest.mark.parametrize("rot,nb", ROTS)
@pytest.mark.parametrize("rnd", [mx.ROUND_RNE, mx.ROUND_SR])
def test_dual_parity(rot, nb, rnd):
    # N = 352: ceil(N/128) is odd, so the row-direction scale padding reaches past
    # the last channel tile; T = 1280 spans several token tiles
    _dual_check(_rand_bits((1280, 352), 12), rot, nb, rnd, 5)


@pytest.mark.parametrize("T,N", [(800, 96), (256, 128), (512, 224), (96, 32)])
def test_dual_ragged_shapes(T, N):
    # T = 800 / 96: the token tiles run past the row-direction padding
    _dual_check(_rand_bits((T, N), 13), mx.ROT_HADAMARD_DET, 32, mx.ROUND_RNE, 0)


def test_dual_edge_cases():
    x = _edge_matrix()
    _dual_check(x, mx.ROT_HADAMARD_DET, 32, mx.ROUND_RNE, 3)
    _dual_check(x, mx.ROT_NONE, 32, mx.ROUND_SR, 3)


def test_dual_tiny_config_dy():
    d = config_inputs("tiny", seed=0, only=("dY",))
    _dual_check(d["dY"], mx.ROT_HADAMARD_DET, 32, mx.ROUND_RNE, 0)


@pytest.mark.parametrize("lines,k", [(128, 256), (200, 800), (4096, 8192), (7, 32)])
def test_scales_to_canonical_matches_the_documented_layout(lines, k):
    MP, KB = 128 * ((lines + 127) // 128), 8 * ((k + 255) // 256)
    tiled = np.random.default_rng(lines + k).integers(0, 256, MP * KB, dtype=np.uint8)
    got = mx.scales_to_canonical(torch.from_numpy(tiled).cuda(), lines, k)
    mx.check_status()
    assert np.array_equal(got.cpu().numpy(), untile_scales(tiled, lines, k))


def test_scales_to_canonical_of_an_encode_equals_the_oracle_scales():
    bits = _rand_bits((800, 136), 17)
    codes, scales = mx.quantize(torch.from_numpy(bits.view(np.int16)).cuda(), mx.CONTRACT_ROWS,
                                mx.ROT_HADAMARD_DET, 32)
    got = mx.scales_to_canonical(scales, 136, 800)
    mx.check_status()
    _, os_ = oracle.quantize(bits, oracle.CONTRACT_ROWS, oracle.ROT_HADAMARD_DET, 32)
    assert np.array_equal(got.cpu().numpy(), os_)


@pytest.mark.slow
@pytest.mark.parametrize("rot,nb,rnd", [(mx.ROT_HADAMARD_DET, 32, mx.ROUND_RNE),
                                        (mx.ROT_HADAMARD_DET, 128, mx.ROUND_RNE),
                                        (mx.ROT_NONE, 32, mx.ROUND_SR)])
def test_dual_o_proj_full_size(rot, nb, rnd):
    """Every byte of both encodings of the o_proj output gradient (8192 x 4096),
    padding included, against the oracle encodes (partitioned over the host
    cores by lines; the oracle's arithmetic is unchanged)."""
    from concurrent.futures import ThreadPoolExecutor
    import os
    bits = config_inputs("o_proj", seed=0, only=("dY",))["dY"]
    T, N = bits.shape
    (ct, st), (cn, sn) = mx.quantize_dual(
        torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda(), rot, nb, rnd, 0)
    mx.check_status()
    cores = os.cpu_count() or 1

    def par(contract, r, b, n):
        chunks = np.array_split(np.arange(n), cores)
        with ThreadPoolExecutor(cores) as ex:
            res = list(ex.map(lambda ln: oracle.quantize(bits, contract, r, b, rnd, 0, 1, lines=ln),
                              chunks))
        return np.concatenate([x[0] for x in res]), np.concatenate([x[1] for x in res])

    oc, os_ = par(oracle.CONTRACT_ROWS, rot, nb, N)
    assert np.array_equal(ct.cpu().numpy(), oc)
    assert np.array_equal(st.cpu().numpy(), tile_scales(os_, N, T))
    oc, os_ = par(oracle.CONTRACT_COLS, oracle.ROT_NONE, 32, T)
    assert np.array_equal(cn.cpu().numpy(), oc)
    assert np.array_equal(sn.cpu().numpy(), tile_scales(os_, T, N))
