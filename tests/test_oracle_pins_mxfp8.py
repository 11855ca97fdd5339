"""Pins for the oracle's MXFP8 path (E4M3 elements under the MX block scale),
the FP8 comparator of the pages' MXFP4-vs-FP8 comparison ([36kr]
"Ende-zu-Ende-Effizienz"; E4M3 named in [show] section 2.2).

Each check ties the oracle to something other than itself: PyTorch's own
float8_e4m3fn conversion (a library routine), the bit layout read from the
golden facts fixture, a quantum-rounding formulation, closed forms and brute
force on tiny inputs.  Each test names the plausible mistake it would catch.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import bf16_bits, bf16_bits_to_f32, config_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _facts():
    out = {}
    with open(os.path.join(GOLDEN, "mxfp4_format_facts.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = (s.strip() for s in line.split("=", 1))
                out[k] = v
    return out


def _e4m3_from_bits(code: int) -> float:
    """Value of a 1/4/3 sign/exponent/mantissa float, bias 2^(4-1)-1 = 7,
    exponent field 0 subnormal, the all-ones pattern NaN (no infinity)."""
    f = _facts()
    eb, mb = int(f["fp8_exp_bits"]), int(f["fp8_man_bits"])
    assert f["fp8_element"] == "E4M3" and (eb, mb) == (4, 3)
    bias = (1 << (eb - 1)) - 1
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> mb) & ((1 << eb) - 1)
    m = code & ((1 << mb) - 1)
    if e == (1 << eb) - 1 and m == (1 << mb) - 1:
        return float("nan")
    if e == 0:
        return sign * (m / (1 << mb)) * 2.0 ** (1 - bias)
    return sign * (1 + m / (1 << mb)) * 2.0 ** (e - bias)


def _torch_e4m3_table() -> np.ndarray:
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


# ---------------------------------------------------------------------------
# E4M3 values and rounding
# ---------------------------------------------------------------------------
def test_e4m3_value_table_matches_bit_layout_and_torch():
    # catches a wrong bias, a missing subnormal branch or a NaN placed wrong
    got = np.array([oracle.e4m3_value(c) for c in range(256)])
    bits = np.array([_e4m3_from_bits(c) for c in range(256)])
    lib = _torch_e4m3_table()
    assert np.array_equal(np.isnan(got), np.isnan(lib))
    fin = ~np.isnan(got)
    assert np.array_equal(got[fin], bits[fin]) and np.array_equal(got[fin], lib[fin])
    assert np.isnan(got).sum() == 2 and got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def _rne_e4m3_by_quantum(v: np.ndarray) -> np.ndarray:
    """Round |v| to the E4M3 grid with numpy's half-to-even on the binade's
    quantum (2^(e-3), at least 2^-9), saturating at 448.  Signed result."""
    a = np.abs(v.astype(np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    q = np.exp2(np.maximum(e, -6) - 3)
    r = np.minimum(np.round(a / q) * q, 448.0)
    return np.copysign(r, v.astype(np.float64))


def test_e4m3_rne_exhaustive_bf16_two_formulations():
    # catches ties going the wrong way, a lost subnormal or a missing saturation
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = bf16_bits_to_f32(bits)
    v = v[np.isfinite(v)]
    codes = oracle.e4m3_rne(v)
    table = _torch_e4m3_table()
    assert np.array_equal(table[codes], _rne_e4m3_by_quantum(v))
    assert np.array_equal((codes >> 7).astype(bool), np.signbit(v))
    # the library cast agrees wherever it does not overflow (it has no saturation)
    inr = np.abs(v) <= 448.0
    lib = torch.from_numpy(v[inr]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes[inr], lib)


def test_e4m3_rne_ties_and_saturation():
    ties = {2.0 ** -10: 0.0, 3 * 2.0 ** -10: 2.0 ** -8, 17.0: 16.0, 19.0: 20.0,
            1.0625: 1.0, 1.1875: 1.25, 432.0: 448.0, 416.0: 416.0, 449.0: 448.0,
            500.0: 448.0, 1e30: 448.0}
    for x, e in ties.items():
        for s in (1.0, -1.0):
            c = int(oracle.e4m3_rne(np.array([s * x], np.float32))[0])
            assert oracle.e4m3_value(c) == s * e, (s * x, c)


# ---------------------------------------------------------------------------
# MXFP8 scale rule
# ---------------------------------------------------------------------------
def _scale_byte_e4m3_closed_form(bits: np.ndarray) -> np.ndarray:
    """floor(log2 |x|) - 8 clamped to [-127, 127], + 127, from the bf16 fields."""
    b = bits.astype(np.int64) & 0x7FFF
    e, m = b >> 7, b & 0x7F
    out = np.zeros(b.shape, dtype=np.int64)
    normal = (e > 0) & (e < 255)
    out[normal] = e[normal] - 127
    sub = (e == 0) & (m > 0)
    out[sub] = np.floor(np.log2(np.maximum(m[sub], 1))).astype(np.int64) - 133
    s = np.clip(out - 8, -127, 127) + 127
    s[(e == 0) & (m == 0)] = 0
    s[e == 255] = 0xFF
    return s.astype(np.uint8)


def test_scale_byte_e4m3_all_bf16_patterns():
    # catches the E2M1 offset (2) reused for E4M3 (8), or a wrong clamp
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    amax = np.abs(bf16_bits_to_f32(bits))
    got = oracle.scale_bytes_e4m3(amax)
    assert np.array_equal(got, _scale_byte_e4m3_closed_form(bits))
    fin = np.isfinite(amax) & (amax > 0) & (got > 0) & (got < 0xFF)
    ratio = amax[fin].astype(np.float64) / np.exp2(got[fin].astype(np.float64) - 127)
    assert ratio.min() >= 256.0 and ratio.max() < 512.0


# ---------------------------------------------------------------------------
# Whole-operand encoding
# ---------------------------------------------------------------------------
def _brute_force_mxfp8(xf: np.ndarray):
    """Independent encoder (rot none): per block of 32 the power of two that
    puts amax in [256, 512), then the nearest finite value of all 256 codes
    (PyTorch's decode table) times that power, ties to the even code."""
    blocks = xf.reshape(-1, 32).astype(np.float64)
    amax = np.abs(blocks).max(axis=1)
    s = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1))) - 8, -127)
    s = np.clip(s, -127, 127)
    vals = _torch_e4m3_table()
    fin = np.flatnonzero(~np.isnan(vals))
    cand = vals[fin][None, None, :] * np.exp2(s)[:, None, None]
    d = np.abs(blocks[:, :, None] - cand)
    dmin = d.min(axis=2, keepdims=True)
    tie = d == dmin
    even = (fin % 2 == 0)[None, None, :]
    best = np.where(tie.sum(axis=2) > 1, np.argmax(tie & even, axis=2), np.argmin(d, axis=2))
    mag = np.abs(vals[fin][best])
    return np.copysign(mag, blocks) * np.exp2(s)[:, None], (s + 127).astype(np.uint8)


def test_tiny_config_brute_force():
    x = config_inputs("tiny", only=("X",))["X"]                     # [T=256, 256]
    codes, scales = oracle.quantize_mxfp8(x, oracle.CONTRACT_ROWS)
    assert codes.shape == (256, 256) and scales.shape == (256, 8)
    deq = oracle.dequantize(codes, scales, oracle.FMT_MXFP8)
    exp_vals, exp_sc = _brute_force_mxfp8(bf16_bits_to_f32(x).T.copy())
    assert np.array_equal(scales.reshape(-1), exp_sc)
    assert np.array_equal(deq.reshape(-1, 32), exp_vals)


def test_wide_range_blocks_brute_force():
    # blocks spanning subnormal E4M3 values, and scales near both clamps
    rng = np.random.default_rng(8)
    x = rng.standard_normal((128, 16)) * np.exp2(rng.integers(-20, 20, size=(128, 16)))
    x[:, 3] *= 2.0 ** 100
    x[:, 4] *= 2.0 ** -110
    x = bf16_bits_to_f32(bf16_bits(x.astype(np.float32)))
    codes, scales = oracle.quantize_mxfp8(bf16_bits(x), oracle.CONTRACT_ROWS)
    deq = oracle.dequantize(codes, scales, oracle.FMT_MXFP8)
    exp_vals, exp_sc = _brute_force_mxfp8(x.T.copy())
    assert np.array_equal(scales.reshape(-1), exp_sc)
    assert np.array_equal(deq.reshape(-1, 32), exp_vals)


def test_contract_rows_equals_cols_of_transpose():
    # catches a transposed operand or a code row stride of L/2 (the MXFP4 one)
    rng = np.random.default_rng(3)
    x = bf16_bits(rng.standard_normal((256, 96)).astype(np.float32))
    for rot, nb in ((oracle.ROT_NONE, 32), (oracle.ROT_HADAMARD_DET, 64),
                    (oracle.ROT_HADAMARD_RAND, 128)):
        a = oracle.quantize_mxfp8(x, oracle.CONTRACT_ROWS, rot, nb, seed=4)
        b = oracle.quantize_mxfp8(np.ascontiguousarray(x.T), oracle.CONTRACT_COLS, rot, nb,
                                  seed=4)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    part = oracle.quantize_mxfp8(x, oracle.CONTRACT_ROWS, lines=[95, 0, 7])
    full = oracle.quantize_mxfp8(x, oracle.CONTRACT_ROWS)
    assert np.array_equal(part[0], full[0][[95, 0, 7]])


def test_representable_roundtrip_and_special_blocks():
    x = config_inputs("tiny", only=("dY",))["dY"]
    codes, scales = oracle.quantize_mxfp8(x, oracle.CONTRACT_COLS)
    deq = oracle.dequantize(codes, scales, oracle.FMT_MXFP8)
    xb = bf16_bits(deq.astype(np.float32))
    assert np.array_equal(bf16_bits_to_f32(xb).astype(np.float64), deq)  # exact in bf16
    codes2, scales2 = oracle.quantize_mxfp8(xb, oracle.CONTRACT_COLS)
    assert np.array_equal(codes, codes2) and np.array_equal(scales, scales2)
    z = np.zeros((64, 4), dtype=np.float32)
    z[:32, 1] = 1.0
    z[40, 2] = np.inf
    z[33, 3] = np.nan
    c, s = oracle.quantize_mxfp8(bf16_bits(z), oracle.CONTRACT_ROWS)
    assert s[0, 0] == 0 and not c[0].any()
    assert s[1, 0] == 127 - 8 and np.all(c[1, :32] == 0x78)   # 1.0 = 256 (0x78) * 2^-8
    assert s[2, 1] == 0xFF and s[3, 1] == 0xFF
    assert not c[2, 32:].any() and not c[3, 32:].any()


# ---------------------------------------------------------------------------
# Contraction
# ---------------------------------------------------------------------------
def test_gemm_matches_numpy_on_representable_inputs():
    # inputs already on the MXFP8 grid: the encoded GEMM is numpy's matmul
    rng = np.random.default_rng(5)
    T, N, K = 256, 40, 24
    vals = _torch_e4m3_table()
    grid = vals[~np.isnan(vals)]

    def rep(shape):
        v = rng.choice(grid, size=shape)
        v[::32, :] = 448.0                                  # every block holds the max
        return v * np.exp2(rng.integers(-12, 12, size=(1, shape[1])))
    dY, X = rep((T, N)), rep((T, K))
    Aq, As = oracle.quantize_mxfp8(bf16_bits(dY.astype(np.float32)), oracle.CONTRACT_ROWS)
    Bq, Bs = oracle.quantize_mxfp8(bf16_bits(X.astype(np.float32)), oracle.CONTRACT_ROWS)
    C, Cabs = oracle.gemm(Aq, As, Bq, Bs, oracle.FMT_MXFP8)
    assert np.array_equal(C, dY.T @ X)
    assert np.array_equal(Cabs, np.abs(dY).T @ np.abs(X))
    ii, jj = np.array([0, 39, 7]), np.array([23, 0, 11])
    Ce, Cae = oracle.gemm_entries(Aq, As, Bq, Bs, ii, jj, oracle.FMT_MXFP8)
    assert np.array_equal(Ce, C[ii, jj]) and np.array_equal(Cae, Cabs[ii, jj])


def test_mxfp8_error_small_and_below_mxfp4():
    # three more mantissa bits: the error is much smaller than MXFP4's
    d = config_inputs("tiny")
    exact = bf16_bits_to_f32(d["dY"]).astype(np.float64).T @ \
        bf16_bits_to_f32(d["X"]).astype(np.float64)
    A8 = oracle.quantize_mxfp8(d["dY"], oracle.CONTRACT_ROWS)
    B8 = oracle.quantize_mxfp8(d["X"], oracle.CONTRACT_ROWS)
    C8, _ = oracle.gemm(*A8, *B8, fmt=oracle.FMT_MXFP8)
    A4 = oracle.quantize(d["dY"], oracle.CONTRACT_ROWS)
    B4 = oracle.quantize(d["X"], oracle.CONTRACT_ROWS)
    C4, _ = oracle.gemm(*A4, *B4)
    e8 = np.linalg.norm(C8 - exact) / np.linalg.norm(exact)
    e4 = np.linalg.norm(C4 - exact) / np.linalg.norm(exact)
    assert 1e-5 < e8 < 0.06 and e8 < e4 / 3    # outlier channels make both larger
