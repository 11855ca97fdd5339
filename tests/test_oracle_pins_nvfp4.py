"""Pins for the oracle's NVFP4 path (E2M1 elements in blocks of 16, a UE4M3
scale per block, an fp32 scale per tensor; the prior-work format named in
[36kr]'s introduction, taken in NVIDIA's definition).

Independent anchors: PyTorch's float8_e4m3fn cast and decode table (library
routines) for the block scale, the E2M1 bit layout from the facts fixture,
exact round trips of inputs built on the NVFP4 grid, brute-force nearest
searches over every code, numpy matmul on representable inputs, and
invariants (a line subset encodes with the whole tensor's scale).
"""
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import bf16_bits, bf16_bits_to_f32, config_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
E4M3_MAX, E2M1_MAX = 448.0, 6.0


def _e2m1_table() -> np.ndarray:
    # E2M1 from its bit layout (1 sign, 2 exponent bits with bias 1, 1 mantissa bit)
    out = []
    for c in range(16):
        e, m = (c >> 1) & 3, c & 1
        mag = (m / 2) if e == 0 else (1 + m / 2) * 2.0 ** (e - 1)
        out.append(-mag if c & 8 else mag)
    return np.array(out)


def _e4m3_table() -> np.ndarray:
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_tensor_scale_maps_amax_onto_the_largest_block_value():
    # catches 448 or 6 alone instead of 448 * 6, an inverted ratio, no guard at 0
    for a in [1.0, 65.0, 3.0e-3, 1.7e38, 2688.0, 7.0]:
        s = oracle.nvfp4_tensor_scale(a)
        assert abs(s * a / (E4M3_MAX * E2M1_MAX) - 1) < 2 ** -23
    assert oracle.nvfp4_tensor_scale(0.0) == 1.0
    assert oracle.nvfp4_tensor_scale(float("inf")) == 1.0
    assert oracle.nvfp4_tensor_scale(1e-40) == np.finfo(np.float32).max   # would overflow


def test_block_scale_is_library_e4m3_cast_of_the_decode_scale():
    # every finite bf16 block amax, several tensor scales: the code is PyTorch's
    # round-to-nearest E4M3 cast of (amax / 6) * s_enc, saturating at 448
    bits = np.arange(0, 0x7F80, dtype=np.uint16)
    amax = bf16_bits_to_f32(bits)
    for s_enc in (1.0, 41.353847, 2688.0 / 3.5, 3.0e4, 0.002):
        with np.errstate(over="ignore"):
            u = (amax / np.float32(6.0)).astype(np.float32) * np.float32(s_enc)
        got = np.array([oracle.nvfp4_block_scale(float(a), s_enc) for a in amax[::7]],
                       dtype=np.uint8)
        uu = u[::7]
        lib = torch.from_numpy(np.minimum(uu, np.float32(E4M3_MAX))).to(
            torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(got, lib)
        assert got.max() <= 0x7E                      # positive, never NaN


def _grid_tensor(rng, lines, L, m):
    """Values e * sf * 2^-m (e E2M1, sf E4M3 per block of 16) with every block
    holding +-6*sf and one element at 6*448*2^-m: NVFP4 represents them exactly
    when s_enc = 2^m."""
    e2 = _e2m1_table()
    e4 = _e4m3_table()
    sf_choices = e4[(e4 >= 2.0 ** -6) & (e4 <= 448) & ~np.isnan(e4)]
    x = np.zeros((lines, L))
    for i in range(lines):
        for b in range(L // 16):
            sf = 448.0 if i == 0 and b == 0 else rng.choice(sf_choices)
            blk = rng.choice(e2, size=16)
            blk[rng.integers(16)] = rng.choice([-6.0, 6.0])
            x[i, 16 * b:16 * b + 16] = blk * sf
    x[0, 0] = 6.0 * 448.0                                  # the tensor amax
    return x * 2.0 ** -m


@pytest.mark.parametrize("m", [0, 7, -5])
def test_representable_inputs_round_trip_exactly(m):
    # catches a wrong block length, a wrong scale formula or a transposed operand
    rng = np.random.default_rng(11 + m)
    x = _grid_tensor(rng, 24, 128, m)                               # [lines, L]
    bits = bf16_bits(np.ascontiguousarray(x.T).astype(np.float32))  # [L, lines]
    assert np.array_equal(bf16_bits_to_f32(bits).T.astype(np.float64), x)
    codes, scales, amax, s_enc = oracle.quantize_nvfp4(bits, oracle.CONTRACT_ROWS)
    assert amax == 2688.0 * 2.0 ** -m and s_enc == 2.0 ** m
    assert codes.shape == (24, 64) and scales.shape == (24, 8)
    dec = oracle.dequantize(codes, scales, oracle.FMT_NVFP4, s_enc)
    assert np.array_equal(dec, x)


def _brute_force_nvfp4(xf: np.ndarray, s_enc: np.float32):
    """Per block of 16: the E4M3 code nearest to the fp32 decode scale (full
    table search, ties to the even code), then each element's nearest E2M1
    code (full search, ties even) for x * fl(s_enc / sf)."""
    e4 = _e4m3_table()
    e2 = _e2m1_table()
    fin4 = np.flatnonzero(~np.isnan(e4[:128]))
    blocks = xf.reshape(-1, 16)
    codes = np.zeros(blocks.shape, dtype=np.uint8)
    sfs = np.zeros(blocks.shape[0], dtype=np.uint8)
    for i, blk in enumerate(blocks):
        amax = np.float32(np.abs(blk).max())
        u = np.float32(np.float32(amax / np.float32(6)) * s_enc)
        d = np.abs(e4[fin4] - float(min(u, 448.0)))
        best = fin4[d == d.min()]
        sf = int(best[best % 2 == 0][0] if len(best) > 1 else best[0])
        sfs[i] = sf
        if sf == 0:
            continue
        q = np.float32(s_enc / np.float32(e4[sf]))
        v = (blk.astype(np.float32) * q).astype(np.float64)
        av = np.minimum(np.abs(v), 6.0)                           # saturate at the largest
        dd = np.abs(av[:, None] - e2[None, :8])
        mag = []
        for r in dd:
            near = np.flatnonzero(r == r.min())
            mag.append(near[near % 2 == 0][0] if len(near) > 1 else near[0])
        codes[i] = np.array(mag) | np.where(np.signbit(v), 8, 0)
    return codes, sfs


def test_tiny_config_brute_force():
    x = config_inputs("tiny", only=("X",))["X"]                     # [T=256, 256 lines]
    codes, scales, amax, s_enc = oracle.quantize_nvfp4(x, oracle.CONTRACT_ROWS)
    xf = bf16_bits_to_f32(x).T.copy()
    assert amax == np.abs(xf).max()
    exp_codes, exp_sf = _brute_force_nvfp4(xf, np.float32(s_enc))
    assert np.array_equal(scales.reshape(-1), exp_sf)
    got = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(-1, 16)
    assert np.array_equal(got, exp_codes)


def test_line_subset_uses_the_whole_tensor_scale_and_transpose_agrees():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((256, 96)).astype(np.float32)
    x[:, 50] *= 30.0                                               # the tensor amax lives here
    bits = bf16_bits(x)
    for rot, nb in ((oracle.ROT_NONE, 16), (oracle.ROT_HADAMARD_DET, 16),
                    (oracle.ROT_HADAMARD_RAND, 32)):
        full = oracle.quantize_nvfp4(bits, oracle.CONTRACT_ROWS, rot, nb, seed=3)
        part = oracle.quantize_nvfp4(bits, oracle.CONTRACT_ROWS, rot, nb, seed=3, lines=[7, 0])
        assert part[2] == full[2] and part[3] == full[3]
        assert np.array_equal(part[0], full[0][[7, 0]]) and np.array_equal(part[1], full[1][[7, 0]])
        tr = oracle.quantize_nvfp4(np.ascontiguousarray(bits.T), oracle.CONTRACT_COLS, rot, nb,
                                   seed=3)
        assert all(np.array_equal(a, b) for a, b in zip(full[:2], tr[:2]))


def test_zero_tensor_and_nonfinite_block():
    z = np.zeros((64, 8), dtype=np.float32)
    c, s, amax, se = oracle.quantize_nvfp4(bf16_bits(z), oracle.CONTRACT_ROWS)
    assert amax == 0.0 and se == 1.0 and not c.any() and not s.any()
    z[:, 1] = 1.0
    z[20, 2] = np.inf
    z[40, 3] = np.nan
    c, s, amax, se = oracle.quantize_nvfp4(bf16_bits(z), oracle.CONTRACT_ROWS)
    assert amax == 1.0 and se == np.float32(2688.0)
    assert np.all(s[1] == 0x7E) and np.all(c[1] == 0x77)            # 1.0 = 6 * 448 / 2688
    assert s[2, 1] == 0x7F and not c[2, 8:16].any()                 # rows 16..31: Inf block
    assert s[3, 2] == 0x7F and s[3, 0] == 0                         # NaN block; zero block


def test_gemm_matches_numpy_on_representable_inputs():
    rng = np.random.default_rng(6)
    a = _grid_tensor(rng, 40, 256, 3)                                # [N lines, T]
    b = _grid_tensor(rng, 24, 256, -2)
    A = oracle.quantize_nvfp4(bf16_bits(np.ascontiguousarray(a.T).astype(np.float32)),
                              oracle.CONTRACT_ROWS)
    B = oracle.quantize_nvfp4(bf16_bits(np.ascontiguousarray(b.T).astype(np.float32)),
                              oracle.CONTRACT_ROWS)
    C, Cabs = oracle.gemm(A[0], A[1], B[0], B[1], oracle.FMT_NVFP4, A[3], B[3])
    assert np.array_equal(C, a @ b.T) and np.array_equal(Cabs, np.abs(a) @ np.abs(b).T)
    ii, jj = np.array([0, 39, 5]), np.array([23, 0, 9])
    Ce, Cae = oracle.gemm_entries(A[0], A[1], B[0], B[1], ii, jj, oracle.FMT_NVFP4, A[3], B[3])
    assert np.array_equal(Ce, C[ii, jj]) and np.array_equal(Cae, Cabs[ii, jj])


def test_nvfp4_error_below_mxfp4_on_gaussian_data():
    # finer blocks and a 3-bit-mantissa scale: smaller error than MXFP4's
    rng = np.random.default_rng(9)
    x = bf16_bits(rng.standard_normal((512, 64)).astype(np.float32))
    xf = bf16_bits_to_f32(x).T.astype(np.float64)
    c, s, _, se = oracle.quantize_nvfp4(x, oracle.CONTRACT_ROWS)
    e_nv = np.linalg.norm(oracle.dequantize(c, s, oracle.FMT_NVFP4, se) - xf)
    c4, s4 = oracle.quantize(x, oracle.CONTRACT_ROWS)
    e_mx = np.linalg.norm(oracle.dequantize(c4, s4) - xf)
    assert e_nv < 0.9 * e_mx
