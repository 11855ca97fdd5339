"""Pins for the CPU oracle: each check ties the oracle to something other than
itself -- a library routine (Triton's Philox, scipy's Hadamard matrix, numpy
matmul), a closed form, an invariant the pages state, or brute force on tiny
inputs.  Each test names the plausible oracle mistake it would catch.
"""
import os

import numpy as np
import pytest
import scipy.linalg

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


# ---------------------------------------------------------------------------
# Format facts from the pages (golden fixture) and the E2M1 value set
# ---------------------------------------------------------------------------
def _e2m1_from_bits(code: int) -> float:
    """Value of a 1/2/1 sign/exponent/mantissa float with bias 1 (OCP E2M1),
    derived from the bit layout alone: exponent field 0 is subnormal."""
    f = _facts()
    eb, mb = int(f["element_exp_bits"]), int(f["element_man_bits"])
    assert (eb, mb) == (2, 1)
    sign = -1.0 if code & 0b1000 else 1.0
    e = (code >> mb) & ((1 << eb) - 1)
    m = code & ((1 << mb) - 1)
    bias = 1
    if e == 0:
        return sign * (m / 2 ** mb) * 2.0 ** (1 - bias)
    return sign * (1 + m / 2 ** mb) * 2.0 ** (e - bias)


def test_e2m1_value_table_matches_bit_layout():
    # catches a wrong magnitude in the oracle's grid table
    for code in range(16):
        assert oracle.e2m1_value(code) == _e2m1_from_bits(code)
    mags = sorted({abs(_e2m1_from_bits(c)) for c in range(16)})
    assert mags == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_block_size_and_scale_granularity_from_pages():
    f = _facts()
    bs = int(f["block_size"])
    x = config_inputs("tiny", only=("X",))["X"]
    codes, scales = oracle.quantize(x, oracle.CONTRACT_ROWS)
    assert scales.shape == (x.shape[1], x.shape[0] // bs)
    assert codes.shape == (x.shape[1], x.shape[0] // 2)


def test_h16_block_size_supported():
    n = int(_facts()["hadamard_block_label"])
    y = oracle.fwht_f32(np.ones(n))
    assert y[0] == np.float32(n * (1.0 / np.sqrt(n))) and not y[1:].any()


# ---------------------------------------------------------------------------
# Philox4x32-10: the published known-answer vectors and a library implementation
# ---------------------------------------------------------------------------
# Known-answer vectors of Philox4x32-10 (Salmon et al., SC'11, as distributed with
# the authors' Random123 library): (counter, key) -> output.
PHILOX4X32_KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,want", PHILOX4X32_KAT)
def test_philox_known_answers(ctr, key, want):
    # catches a swapped multiplier, a wrong hi/lo half, a key bump in the wrong place
    assert [int(v) for v in oracle.philox4x32_10(ctr, key)] == list(want)


_TRITON_PHILOX = r"""
import os, sys, json
os.environ["TRITON_INTERPRET"] = "1"
import torch, triton, triton.language as tl

@triton.jit
def k(out_ptr, seed, c_ptr, N: tl.constexpr):
    i = tl.arange(0, N)
    c0 = tl.load(c_ptr + 4 * i)
    c1 = tl.load(c_ptr + 4 * i + 1)
    c2 = tl.load(c_ptr + 4 * i + 2)
    c3 = tl.load(c_ptr + 4 * i + 3)
    a, b, c, d = tl.philox(seed, c0, c1, c2, c3, 10)
    tl.store(out_ptr + 4 * i, a)
    tl.store(out_ptr + 4 * i + 1, b)
    tl.store(out_ptr + 4 * i + 2, c)
    tl.store(out_ptr + 4 * i + 3, d)

cases = json.loads(sys.stdin.read())
res = []
for seed, ctrs in cases:
    c = torch.tensor(ctrs, dtype=torch.int64).to(torch.int32).to(torch.uint32).reshape(-1)
    out = torch.zeros(c.numel(), dtype=torch.uint32)
    k[(1,)](out, seed, c, N=c.numel() // 4)
    res.append([int(v) & 0xFFFFFFFF for v in out.view(torch.int32).tolist()])
print(json.dumps(res))
"""


def test_philox_matches_triton():
    """Triton's own Philox4x32-10 (tl.philox, key = the seed's low and high halves), run by its
    CPU interpreter in a child process, on random counters and keys."""
    pytest.importorskip("triton")
    import json
    import subprocess
    import sys
    rng = np.random.default_rng(5)
    cases = []
    for _ in range(4):
        seed = int(rng.integers(0, 2**63)) * 2 + int(rng.integers(0, 2))
        ctrs = [[int(w) for w in rng.integers(0, 2**32, size=4)] for _ in range(8)]
        ctrs[0] = [0, 0, 0, 0]
        cases.append((seed, [w for c in ctrs for w in c]))
    r = subprocess.run([sys.executable, "-c", _TRITON_PHILOX], input=json.dumps(cases),
                       capture_output=True, text=True, timeout=300)
    if r.returncode != 0:
        pytest.skip("triton interpreter unavailable: " + r.stderr.strip().splitlines()[-1][:200])
    got_all = json.loads(r.stdout.strip().splitlines()[-1])
    for (seed, flat), ref in zip(cases, got_all):
        key = (seed & 0xFFFFFFFF, seed >> 32)
        for n in range(len(flat) // 4):
            out = oracle.philox4x32_10(flat[4 * n:4 * n + 4], key)
            assert [int(v) for v in out] == ref[4 * n:4 * n + 4]


def _philox_block(seed, tag, n):
    """Block n of the stream (seed, tag): key = seed halves, counter = (n, tag) halves."""
    return oracle.philox4x32_10([n & 0xFFFFFFFF, n >> 32, tag & 0xFFFFFFFF, tag >> 32],
                                [seed & 0xFFFFFFFF, seed >> 32])


def test_sign_vector_bits_follow_documented_mapping():
    # catches an off-by-one in word/bit selection of the random sign
    for seed in (0, 1, 99, 2**40 + 7):
        for t in (0, 1, 31, 32, 63, 64, 127, 128, 200, 255, 256, 1000, 4097, 2**33 + 5):
            words = _philox_block(seed, 0, t // 128)
            b = t % 128
            bit = (int(words[b // 32]) >> (b % 32)) & 1
            assert oracle.sign(seed, t) == (-1 if bit else 1)


def test_random_streams_depend_on_the_seed_high_half():
    # catches a seed truncated to 32 bits on its way into the Philox key
    lo = 12345
    for hi in (1, 2**31, 2**32 - 1):
        seed = (hi << 32) | lo
        assert [oracle.sr_u24(seed, 1, e) for e in range(8)] != [oracle.sr_u24(lo, 1, e) for e in range(8)]
        assert [oracle.sign(seed, t) for t in range(128)] != [oracle.sign(lo, t) for t in range(128)]


def test_sr_draw_follows_documented_mapping():
    for seed, tag in ((0, 1), (5, 2), (2**35 + 1, 1)):
        for e in (0, 1, 3, 4, 7, 8, 9, 1023, 123457, 2**34 + 6):
            w = int(_philox_block(seed, tag, e // 4)[e % 4])
            assert oracle.sr_u24(seed, tag, e) == w >> 8


# ---------------------------------------------------------------------------
# Hadamard rotation
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("n", [16, 32, 64, 128, 256])
def test_hadamard_f64_is_scipy_sylvester_normalised(n):
    # catches a transposed / mis-ordered / unnormalised Hadamard
    H = scipy.linalg.hadamard(n).astype(np.float64) / np.sqrt(n)
    I = np.eye(n)
    M = np.stack([oracle.hadamard_f64(I[:, j]) for j in range(n)], axis=1)
    assert np.abs(M - H).max() <= 4e-16
    assert np.abs(M @ M.T - I).max() <= n * 2.0 ** -52


@pytest.mark.parametrize("n", [16, 32, 64, 128, 256])
def test_fwht_f32_close_to_dense_and_exact_on_integers(n):
    rng = np.random.default_rng(n)
    x = rng.standard_normal(n).astype(np.float32)
    y32 = oracle.fwht_f32(x)
    y64 = oracle.hadamard_f64(x.astype(np.float64))
    c = 1.0 / np.sqrt(n)
    bound = (np.log2(n) + 1) * 2.0 ** -24 * np.abs(x).sum() * c + 2.0 ** -24 * np.abs(y64)
    assert np.all(np.abs(y32 - y64) <= bound)
    # small integers: every fp32 sum is exact, so only the final scaling rounds
    xi = rng.integers(-100, 100, n).astype(np.float32)
    H = scipy.linalg.hadamard(n).astype(np.float64)
    expect = (H @ xi.astype(np.float64)).astype(np.float32) * np.float32(c)
    assert np.array_equal(oracle.fwht_f32(xi), expect)


def test_constant_vector_closed_form():
    for n in (16, 32, 64, 128, 256):
        y = oracle.hadamard_f64(np.full(n, 3.0))
        assert abs(y[0] - 3.0 * np.sqrt(n)) < 1e-12 and np.abs(y[1:]).max() < 1e-12


def _rotate_f64_line(x, n, signs=None):
    x = np.asarray(x, dtype=np.float64).copy()
    if signs is not None:
        x *= signs
    out = np.empty_like(x)
    for b in range(0, x.size, n):
        out[b:b + n] = oracle.hadamard_f64(x[b:b + n])
    return out


@pytest.mark.parametrize("n", [16, 32, 64, 128, 256])
def test_wgrad_invariance_under_shared_rotation(n):
    # [36kr] "Fehlerdiagnoseexperiment": both rotations are orthogonal, so rotating
    # dY and X along T by the same Q leaves dY^T X unchanged.
    rng = np.random.default_rng(7)
    T = 512
    dY = rng.standard_normal((T, 6))
    X = rng.standard_normal((T, 5))
    signs = np.array([oracle.sign(3, t) for t in range(T)], dtype=np.float64)
    for s in (None, signs):
        QdY = np.stack([_rotate_f64_line(dY[:, i], n, s) for i in range(6)], axis=1)
        QX = np.stack([_rotate_f64_line(X[:, i], n, s) for i in range(5)], axis=1)
        ref = dY.T @ X
        assert np.abs(QdY.T @ QX - ref).max() <= 1e-12 * (np.abs(dY).T @ np.abs(X)).max()


@pytest.mark.parametrize("n", [16, 64, 256])
def test_integer_invariance_exact(n):
    # c_n is a power of two here, so the fp32 FWHT of small integers is exact and
    # (Q a) . (Q b) == a . b holds exactly.
    rng = np.random.default_rng(n + 1)
    a = rng.integers(-8, 8, n).astype(np.float32)
    b = rng.integers(-8, 8, n).astype(np.float32)
    qa = oracle.fwht_f32(a).astype(np.float64)
    qb = oracle.fwht_f32(b).astype(np.float64)
    assert qa @ qb == a.astype(np.float64) @ b.astype(np.float64)


def test_rotate_line_rand_is_sign_then_fwht():
    rng = np.random.default_rng(11)
    x = bf16_bits(rng.standard_normal(512).astype(np.float32))
    xf = bf16_bits_to_f32(x)
    for seed in (0, 17):
        d = np.array([oracle.sign(seed, t) for t in range(512)], dtype=np.float32)
        got = oracle.rotate_line(x, oracle.ROT_HADAMARD_RAND, 64, seed)
        exp = np.concatenate([oracle.fwht_f32(xf[b:b + 64] * d[b:b + 64])
                              for b in range(0, 512, 64)])
        assert np.array_equal(got, exp)
    det = oracle.rotate_line(x, oracle.ROT_HADAMARD_DET, 64)
    assert np.array_equal(det, np.concatenate([oracle.fwht_f32(xf[b:b + 64])
                                               for b in range(0, 512, 64)]))


# ---------------------------------------------------------------------------
# Shared scale: exhaustive over all bf16 bit patterns
# ---------------------------------------------------------------------------
def _scale_byte_closed_form(bits: np.ndarray) -> np.ndarray:
    """floor(log2 |x|) - 2 clamped to [-127, 127], + 127, from the bf16 fields."""
    b = bits.astype(np.int64) & 0x7FFF
    e = b >> 7
    m = b & 0x7F
    out = np.zeros(b.shape, dtype=np.int64)
    normal = (e > 0) & (e < 255)
    out[normal] = e[normal] - 127
    sub = (e == 0) & (m > 0)
    msb = np.floor(np.log2(np.maximum(m[sub], 1))).astype(np.int64)
    out[sub] = msb - 133                       # value = m * 2^-133
    s = np.clip(out - 2, -127, 127) + 127
    s[(e == 0) & (m == 0)] = 0
    s[e == 255] = 0xFF
    return s.astype(np.uint8)


def test_scale_byte_all_bf16_patterns():
    # catches an off-by-one in the exponent offset or the clamp
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    amax = np.abs(bf16_bits_to_f32(bits))
    got = oracle.scale_bytes(amax)
    assert np.array_equal(got, _scale_byte_closed_form(bits))
    # the scale places every unclamped amax in [4, 8) ("largest exponent" rule)
    fin = np.isfinite(amax) & (amax > 0) & (got > 0) & (got < 0xFF)
    ratio = amax[fin].astype(np.float64) / np.exp2(got[fin].astype(np.float64) - 127)
    assert ratio.min() >= 4.0 and ratio.max() < 8.0


# ---------------------------------------------------------------------------
# Element rounding: exhaustive over bf16 values, independent formulation
# ---------------------------------------------------------------------------
def _rne_e2m1_by_quantum(v: np.ndarray) -> np.ndarray:
    """Round |v| to the E2M1 grid by rounding to the binade's quantum with
    numpy's half-to-even, then saturating at 6 (a different method from the
    oracle's scan).  Returns the signed value."""
    a = np.abs(v.astype(np.float64))
    q = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    r = np.round(a / q) * q
    r = np.minimum(r, 6.0)
    return np.copysign(r, v.astype(np.float64))


def test_e2m1_rne_exhaustive_bf16():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = bf16_bits_to_f32(bits)
    v = v[np.isfinite(v)]
    codes = oracle.e2m1_rne(v)
    vals = np.array([oracle.e2m1_value(int(c)) for c in range(16)])[codes]
    exp = _rne_e2m1_by_quantum(v)
    assert np.array_equal(vals, exp)
    # sign bit is the sign of v (including -0 and negatives that round to 0)
    assert np.array_equal((codes >> 3).astype(bool), np.signbit(v))


def test_e2m1_rne_ties_and_saturation():
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0,
            6.0: 6.0, 7.0: 6.0, 7.99: 6.0, 100.0: 6.0}
    for x, e in ties.items():
        for s in (1, -1):
            c = int(oracle.e2m1_rne(np.float32(s * x)))
            assert oracle.e2m1_value(c) == s * e
    assert int(oracle.e2m1_rne(np.float32(-0.0))) == 0b1000
    assert int(oracle.e2m1_rne(np.float32(-0.1))) == 0b1000


# ---------------------------------------------------------------------------
# Stochastic rounding ([36kr] "Fehlerdiagnoseexperiment": zero-mean error)
# ---------------------------------------------------------------------------
def test_sr_outputs_neighbours_and_is_unbiased():
    vs = np.array([0.1, 0.3, 0.7, 1.2, 1.6, 2.2, 2.9, 3.3, 4.5, 5.9, -0.3, -4.7],
                  dtype=np.float32)
    u = (np.arange(0, 2 ** 24, 2 ** 4, dtype=np.uint32))     # 2^20 evenly spread draws
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    for v in vs:
        codes = oracle.e2m1_sr(np.full(u.shape, v, dtype=np.float32), u)
        vals = np.array([oracle.e2m1_value(int(c)) for c in range(16)])[codes]
        a = abs(float(v))
        lo = grid[grid <= a].max()
        hi = grid[grid > a].min()
        assert set(np.unique(np.abs(vals))) <= {lo, hi}
        # exact expectation over the even sweep is within one step of the sweep's grain
        assert abs(vals.mean() - float(v)) <= (hi - lo) * 2.0 ** -20 + 1e-12
        # variance: a draw that lands on lo or hi with probability 1 - p, p
        # (p = (|v| - lo) / (hi - lo)) has E[(SR - v)^2] = p (1 - p) (hi - lo)^2,
        # never below the squared error of rounding to the nearest neighbour
        p = (a - lo) / (hi - lo)
        mse_sr = float(((np.abs(vals) - a) ** 2).mean())
        assert abs(mse_sr - p * (1 - p) * (hi - lo) ** 2) <= (hi - lo) ** 2 * 2.0 ** -19
        rne = oracle.e2m1_value(int(oracle.e2m1_rne(np.array([a], dtype=np.float32))[0]))
        assert mse_sr >= (rne - a) ** 2 - 1e-12


def test_sr_representable_unchanged_and_saturates():
    u = np.array([0, 1, 2 ** 23, 2 ** 24 - 1], dtype=np.uint32)
    for g in (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0):
        for s in (1, -1):
            c = oracle.e2m1_sr(np.full(4, s * g, dtype=np.float32), u)
            assert all(oracle.e2m1_value(int(k)) == s * g for k in c)
    c = oracle.e2m1_sr(np.full(4, 7.5, dtype=np.float32), u)
    assert all(oracle.e2m1_value(int(k)) == 6.0 for k in c)



def test_sr_decision_exact_at_thresholds():
    """The SR rule as exact rational arithmetic: round |v| up to the next E2M1 grid point iff
    u24 < (|v| - lo) / (hi - lo) * 2^24, with v's fp32 value taken exactly.  Draws on both sides
    of each threshold catch a <= for <, a wrong step in one binade or a lost low mantissa bit."""
    from fractions import Fraction
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 0x40E00000, size=6000, dtype=np.uint32)     # |v| from 0 to 7
    bits = np.concatenate([bits, np.array([0x00000001, 0x3EFFFFFF, 0x3F000001, 0x3F7FFFFF,
                                           0x3FBFFFFF, 0x3FC00001, 0x40BFFFFF], np.uint32)])
    grid = [Fraction(g) for g in ("0", "0.5", "1", "1.5", "2", "3", "4", "6")]
    vs, us, want = [], [], []
    for b in bits:
        v = np.uint32(b).view(np.float32)
        a = Fraction(float(v))
        if a >= 6:
            vs.append(v); us.append(12345); want.append(6.0)
            continue
        lo = max(g for g in grid if g <= a)
        hi = min(g for g in grid if g > a)
        t = (a - lo) / (hi - lo) * 2 ** 24
        f = int(t)                                   # floor (t >= 0)
        for u in {max(f - 1, 0), f, min(f + 1, 2 ** 24 - 1)}:
            vs.append(v); us.append(u)
            want.append(float(hi if u < t else lo))
    sign = np.where(rng.integers(0, 2, size=len(vs)) == 1, -1.0, 1.0)
    v_arr = (np.array(vs, dtype=np.float32) * sign).astype(np.float32)
    codes = oracle.e2m1_sr(v_arr, np.array(us, dtype=np.uint32))
    got = np.array([oracle.e2m1_value(int(c)) for c in codes])
    assert np.array_equal(got, np.array(want) * sign)


# ---------------------------------------------------------------------------
# Whole-operand encoding
# ---------------------------------------------------------------------------
def _brute_force_encode(xf: np.ndarray):
    """Independent numpy encoder for rot=none, RNE: for each block of 32 along
    the last axis, the scale is the power of two placing amax in [4, 8) and
    each element takes the nearest of all 16 codes' values (ties to even)."""
    blocks = xf.reshape(-1, 32).astype(np.float64)
    amax = np.abs(blocks).max(axis=1)
    s = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1))) - 2, -127)
    s = np.clip(s, -127, 127)
    vals = np.array([_e2m1_from_bits(c) for c in range(16)])
    cand = vals[None, None, :] * np.exp2(s)[:, None, None]          # [B,1,16]
    d = np.abs(blocks[:, :, None] - cand)
    even = (np.arange(16) % 2 == 0)
    best = np.argmin(d + np.where(even, 0.0, 1e-300 * 0.0), axis=2)
    # resolve exact ties to the even code explicitly
    dmin = d.min(axis=2, keepdims=True)
    tie = (d == dmin)
    pick_even = np.argmax(tie & even[None, None, :], axis=2)
    n_ties = tie.sum(axis=2)
    best = np.where(n_ties > 1, pick_even, best)
    # sign of zero follows the input
    mag = np.abs(vals[best])
    return np.copysign(mag, blocks) * np.exp2(s)[:, None], (s + 127).astype(np.uint8)


def test_tiny_config_brute_force_rot_none():
    x = config_inputs("tiny", only=("X",))["X"]                     # [T=256, 256]
    codes, scales = oracle.quantize(x, oracle.CONTRACT_ROWS)
    deq = oracle.dequantize(codes, scales)                          # [256 ch, 256 T]
    xf = bf16_bits_to_f32(x).T.copy()
    exp_vals, exp_sc = _brute_force_encode(xf)
    assert np.array_equal(scales.reshape(-1), exp_sc)
    assert np.array_equal(deq.reshape(-1, 32), exp_vals)


def test_contract_rows_equals_cols_of_transpose():
    # catches a transposed operand in either contraction direction
    rng = np.random.default_rng(3)
    x = bf16_bits(rng.standard_normal((256, 96)).astype(np.float32))
    for rot, nb in ((oracle.ROT_NONE, 32), (oracle.ROT_HADAMARD_DET, 64),
                    (oracle.ROT_HADAMARD_RAND, 128)):
        for rnd in (oracle.ROUND_RNE, oracle.ROUND_SR):
            a = oracle.quantize(x, oracle.CONTRACT_ROWS, rot, nb, rnd, seed=4)
            b = oracle.quantize(np.ascontiguousarray(x.T), oracle.CONTRACT_COLS, rot, nb, rnd,
                                seed=4)
            assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_idempotent_and_representable_roundtrip():
    x = config_inputs("tiny", only=("dY",))["dY"]
    codes, scales = oracle.quantize(x, oracle.CONTRACT_COLS)
    deq = oracle.dequantize(codes, scales)
    xb = bf16_bits(deq.astype(np.float32))
    assert np.array_equal(bf16_bits_to_f32(xb).astype(np.float64), deq)  # exact in bf16
    codes2, scales2 = oracle.quantize(xb, oracle.CONTRACT_COLS)
    assert np.array_equal(codes, codes2) and np.array_equal(scales, scales2)
    # representable inputs round-trip exactly
    assert np.array_equal(oracle.dequantize(codes2, scales2), deq)


def test_zero_block_and_nonfinite_block():
    x = np.zeros((64, 4), dtype=np.float32)
    x[:32, 1] = 1.0
    x[40, 2] = np.inf
    x[33, 3] = np.nan
    codes, scales = oracle.quantize(bf16_bits(x), oracle.CONTRACT_ROWS)
    assert scales[0, 0] == 0 and scales[0, 1] == 0 and not codes[0].any()
    assert scales[1, 0] == 127 - 2 and scales[2, 1] == 0xFF and scales[3, 1] == 0xFF
    assert not codes[2, 16:].any() and not codes[3, 16:].any()


def test_rand_modes_depend_on_seed_det_does_not():
    x = config_inputs("tiny", only=("X",))["X"]
    det0 = oracle.quantize(x, oracle.CONTRACT_ROWS, oracle.ROT_HADAMARD_DET, 32, seed=0)
    det1 = oracle.quantize(x, oracle.CONTRACT_ROWS, oracle.ROT_HADAMARD_DET, 32, seed=9)
    assert np.array_equal(det0[0], det1[0])
    r0 = oracle.quantize(x, oracle.CONTRACT_ROWS, oracle.ROT_HADAMARD_RAND, 32, seed=0)
    r1 = oracle.quantize(x, oracle.CONTRACT_ROWS, oracle.ROT_HADAMARD_RAND, 32, seed=9)
    assert not np.array_equal(r0[0], r1[0])
    s0 = oracle.quantize(x, oracle.CONTRACT_ROWS, rnd=oracle.ROUND_SR, seed=0)
    s1 = oracle.quantize(x, oracle.CONTRACT_ROWS, rnd=oracle.ROUND_SR, seed=9)
    assert not np.array_equal(s0[0], s1[0])


# ---------------------------------------------------------------------------
# Contraction
# ---------------------------------------------------------------------------
def test_gemm_matches_numpy_on_representable_inputs():
    # with rot=none and inputs already on the MXFP4 grid the encoded GEMM is the
    # plain GEMM of the raw inputs (reduces to numpy matmul)
    rng = np.random.default_rng(5)
    T, N, K = 256, 48, 40
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -1.5, -2, -3, -4, -6])

    def rep(shape):
        v = rng.choice(grid, size=shape)
        v[::32, :] = 6.0                                    # every block holds a 6
        return v * np.exp2(rng.integers(-6, 6, size=(1, shape[1])))
    dY, X = rep((T, N)), rep((T, K))
    Aq, As = oracle.quantize(bf16_bits(dY.astype(np.float32)), oracle.CONTRACT_ROWS)
    Bq, Bs = oracle.quantize(bf16_bits(X.astype(np.float32)), oracle.CONTRACT_ROWS)
    C, Cabs = oracle.gemm(Aq, As, Bq, Bs)
    assert np.array_equal(C, dY.T @ X)
    assert np.array_equal(Cabs, np.abs(dY).T @ np.abs(X))


def test_gemm_entries_agree_with_rows_and_error_is_small():
    d = config_inputs("tiny")
    dY, X = d["dY"], d["X"]
    Aq, As = oracle.quantize(dY, oracle.CONTRACT_ROWS, oracle.ROT_HADAMARD_DET, 32)
    Bq, Bs = oracle.quantize(X, oracle.CONTRACT_ROWS, oracle.ROT_HADAMARD_DET, 32)
    C, Cabs = oracle.gemm(Aq, As, Bq, Bs)
    ii = np.array([0, 5, 127, 64])
    jj = np.array([0, 200, 255, 3])
    Ce, Cae = oracle.gemm_entries(Aq, As, Bq, Bs, ii, jj)
    assert np.array_equal(Ce, C[ii, jj]) and np.array_equal(Cae, Cabs[ii, jj])
    exact = bf16_bits_to_f32(dY).astype(np.float64).T @ bf16_bits_to_f32(X).astype(np.float64)
    rel = np.linalg.norm(C - exact) / np.linalg.norm(exact)
    assert 1e-4 < rel < 0.2            # MXFP4 error: present, but bounded


def test_sampled_lines_equal_full():
    d = config_inputs("tiny")
    full = oracle.quantize(d["X"], oracle.CONTRACT_ROWS, oracle.ROT_HADAMARD_RAND, 64,
                           oracle.ROUND_SR, seed=2, sr_tag=2)
    lines = [255, 0, 17]
    part = oracle.quantize(d["X"], oracle.CONTRACT_ROWS, oracle.ROT_HADAMARD_RAND, 64,
                           oracle.ROUND_SR, seed=2, sr_tag=2, lines=lines)
    assert np.array_equal(part[0], full[0][lines]) and np.array_equal(part[1], full[1][lines])


def test_tiny_digests_stable():
    # the stored digests were written by tests/golden/make_golden.py (oracle only)
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden",
                                                  os.path.join(GOLDEN, "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    stored = {}
    with open(os.path.join(GOLDEN, "tiny_oracle_digests.txt")) as f:
        for line in f:
            if not line.startswith("#"):
                k, v = line.split()
                stored[k] = v
    assert dict(mg.digests()) == stored
