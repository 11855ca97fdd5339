"""GPU parity of the linear-layer entry points (Wgrad / Fprop / Dgrad) against
the oracle, on small ragged shapes (full outputs) and on the full-size
Llama-3.1-8B-shaped workloads (every code byte where affordable, otherwise
sampled lines; sampled output entries computed one by one by the oracle)."""
import os

import numpy as np
import pytest
import torch

import oracle
import mxfp4_precision_gb300 as mx
from tests.mx_testutil import assert_gemm_close, untile_scales
from workloads import bf16_bits, config_inputs

pytestmark = pytest.mark.gpu

OC = {mx.CONTRACT_ROWS: oracle.CONTRACT_ROWS, mx.CONTRACT_COLS: oracle.CONTRACT_COLS}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mxfp4_precision_gb300 import build
    build.build()
    mx.lib()


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def _operands(op, a, b):
    """(contract, lines) of operands A and B for an op, from the input shapes."""
    if op == mx.OP_WGRAD:          # dY [T,N] -> lines N; X [T,K] -> lines K
        return (mx.CONTRACT_ROWS, a.shape[1]), (mx.CONTRACT_ROWS, b.shape[1])
    if op == mx.OP_FPROP:          # X [T,K] -> lines T; W [N,K] -> lines N
        return (mx.CONTRACT_COLS, a.shape[0]), (mx.CONTRACT_COLS, b.shape[0])
    return (mx.CONTRACT_COLS, a.shape[0]), (mx.CONTRACT_ROWS, b.shape[1])  # DGRAD


def run_op(op, a, b, rot, nb, rnd, seed):
    fn = {mx.OP_WGRAD: mx.linear_wgrad, mx.OP_FPROP: mx.linear_fprop,
          mx.OP_DGRAD: mx.linear_dgrad}[op]
    out = fn(_dev(a), _dev(b), rot=rot, rot_block=nb, rnd=rnd, seed=seed)
    mx.check_status()
    return out


def sample_lines(n, count, seed):
    rng = np.random.default_rng(seed)
    base = {0, n - 1, min(127, n - 1), min(128, n - 1), n // 2}
    extra = rng.choice(n, size=min(count, n), replace=False)
    return np.array(sorted(base | set(int(v) for v in extra)), dtype=np.int64)


def check_op(op, a, b, rot, nb, rnd=mx.ROUND_RNE, seed=0, sample=None):
    out = run_op(op, a, b, rot, nb, rnd, seed).cpu().numpy()
    (ca, na), (cb, nb_lines) = _operands(op, a, b)
    ia = None if sample is None else sample_lines(na, sample, 1)
    jb = None if sample is None else sample_lines(nb_lines, sample, 2)
    Aq, As = oracle.quantize(a, OC[ca], rot, nb, rnd, seed, 1, lines=ia)
    Bq, Bs = oracle.quantize(b, OC[cb], rot, nb, rnd, seed, 2, lines=jb)
    Cref, Cabs = oracle.gemm(Aq, As, Bq, Bs)
    got = out if sample is None else out[np.ix_(ia, jb)]
    return assert_gemm_close(got, Cref, Cabs, f"op {op} rot {rot}/{nb} rnd {rnd}")


def _par_gemm(Aq, As, Bq, Bs, split_b):
    """oracle.gemm partitioned over the host cores (the oracle's C code releases
    the GIL), by blocks of B's lines (output columns) or of A's lines (rows)."""
    from concurrent.futures import ThreadPoolExecutor
    n = (Bq if split_b else Aq).shape[0]
    parts = max(1, min(os.cpu_count() or 1, n // 8))
    edges = np.linspace(0, n, parts + 1).astype(int)
    def one(i):
        lo, hi = edges[i], edges[i + 1]
        if split_b:
            return oracle.gemm(Aq, As, Bq[lo:hi], Bs[lo:hi])
        return oracle.gemm(Aq[lo:hi], As[lo:hi], Bq, Bs)
    with ThreadPoolExecutor(parts) as ex:
        res = list(ex.map(one, range(parts)))
    axis = 1 if split_b else 0
    return np.concatenate([r[0] for r in res], axis), np.concatenate([r[1] for r in res], axis)


def check_op_rows_cols(op, a, b, rot, nb, rnd=mx.ROUND_RNE, seed=0, n_rows=64, n_cols=64,
                       n_rand=4096):
    """Full-size check: n_rows full output rows, n_cols full output columns and
    n_rand random entries, each computed by the oracle from every encoded line."""
    out = run_op(op, a, b, rot, nb, rnd, seed).cpu().numpy()
    (ca, na), (cb, nb_lines) = _operands(op, a, b)
    Aq, As = oracle.quantize(a, OC[ca], rot, nb, rnd, seed, 1)
    Bq, Bs = oracle.quantize(b, OC[cb], rot, nb, rnd, seed, 2)
    rows = sample_lines(na, n_rows, 11)
    cols = sample_lines(nb_lines, n_cols, 12)
    worst = 0.0
    Cr, Car = _par_gemm(Aq[rows], As[rows], Bq, Bs, split_b=True)
    worst = max(worst, assert_gemm_close(out[rows], Cr, Car, f"op {op}: {rows.size} full rows"))
    Cc, Cac = _par_gemm(Aq, As, Bq[cols], Bs[cols], split_b=False)
    worst = max(worst, assert_gemm_close(out[:, cols], Cc, Cac, f"op {op}: {cols.size} full cols"))
    rng = np.random.default_rng(13)
    ii, jj = rng.integers(0, na, n_rand), rng.integers(0, nb_lines, n_rand)
    Ce, Cae = oracle.gemm_entries(Aq, As, Bq, Bs, ii, jj)
    worst = max(worst, assert_gemm_close(out[ii, jj], Ce, Cae, f"op {op}: {n_rand} entries"))
    return worst


def _bits(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return bf16_bits(rng.standard_normal(shape).astype(np.float32) * np.float32(scale))


def test_tiny_wgrad_full():
    d = config_inputs("tiny", seed=0)
    worst = check_op(mx.OP_WGRAD, d["dY"], d["X"], mx.ROT_HADAMARD_DET, 32)
    assert worst < 1e-5


@pytest.mark.parametrize("rot,nb,rnd", [(mx.ROT_HADAMARD_DET, 32, mx.ROUND_RNE),
                                        (mx.ROT_NONE, 32, mx.ROUND_RNE),
                                        (mx.ROT_HADAMARD_RAND, 64, mx.ROUND_RNE),
                                        (mx.ROT_NONE, 32, mx.ROUND_SR),
                                        (mx.ROT_HADAMARD_DET, 256, mx.ROUND_SR)])
def test_small_ragged_all_ops(rot, nb, rnd):
    T, N, K = 1280, 200, 328
    dY, X = _bits((T, N), 1, 1e-3), _bits((T, K), 2)
    check_op(mx.OP_WGRAD, dY, X, rot, nb, rnd, seed=3)
    # Fprop: X [T', K'] W [N', K'] with contraction K' = 1280
    X2, W = _bits((200, 1280), 3), _bits((328, 1280), 4, 0.02)
    check_op(mx.OP_FPROP, X2, W, rot, nb, rnd, seed=3)
    # Dgrad: dY [T', N'] W [N', K'] with contraction N' = 1280
    dY2, W2 = _bits((200, 1280), 5, 1e-3), _bits((1280, 328), 6, 0.02)
    check_op(mx.OP_DGRAD, dY2, W2, rot, nb, rnd, seed=3)


def test_deterministic_bits():
    d = config_inputs("tiny", seed=0)
    a = run_op(mx.OP_WGRAD, d["dY"], d["X"], mx.ROT_HADAMARD_DET, 32, mx.ROUND_RNE, 0)
    b = run_op(mx.OP_WGRAD, d["dY"], d["X"], mx.ROT_HADAMARD_DET, 32, mx.ROUND_RNE, 0)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_timeout_path_reports_without_hanging():
    # the probe's barrier is never completed; its wait must give up and report
    assert mx.debug_timeout_probe(20000) == 6
    mx.check_status()                      # cleared: next status is OK
    d = config_inputs("tiny", seed=0)      # and the context is still usable
    check_op(mx.OP_WGRAD, d["dY"], d["X"], mx.ROT_HADAMARD_DET, 32)


# ---------------------------------------------------------------- full size
def _compare_codes(bits, contract, rot, nb, rnd, seed, lines=None):
    rows, cols = bits.shape
    L, n = (rows, cols) if contract == mx.CONTRACT_ROWS else (cols, rows)
    codes, scales = mx.quantize(_dev(bits), contract, rot, nb, rnd, seed)
    mx.check_status()
    codes, scales = codes.cpu().numpy(), untile_scales(scales.cpu().numpy(), n, L)
    oc, os_ = oracle.quantize(bits, OC[contract], rot, nb, rnd, seed, 1, lines=lines)
    if lines is not None:
        codes, scales = codes[lines], scales[lines]
    assert np.array_equal(codes, oc) and np.array_equal(scales, os_)


@pytest.mark.slow
def test_o_proj_full_size():
    d = config_inputs("o_proj", seed=0)
    for name in ("dY", "X"):
        _compare_codes(d[name], mx.CONTRACT_ROWS, mx.ROT_HADAMARD_DET, 32, mx.ROUND_RNE, 0)
    worst = check_op_rows_cols(mx.OP_WGRAD, d["dY"], d["X"], mx.ROT_HADAMARD_DET, 32)
    assert worst < 1e-5


def _par_oracle_quantize(bits, contract, rot, nb, rnd, seed, tag):
    """oracle.quantize of every line, partitioned by lines over the host cores
    (the oracle's C code releases the GIL); its arithmetic is unchanged."""
    from concurrent.futures import ThreadPoolExecutor
    n = bits.shape[1] if contract == mx.CONTRACT_ROWS else bits.shape[0]
    parts = max(1, min(os.cpu_count() or 1, n // 64))
    chunks = np.array_split(np.arange(n), parts)
    with ThreadPoolExecutor(parts) as ex:
        res = list(ex.map(lambda ln: oracle.quantize(bits, OC[contract], rot, nb, rnd, seed, tag,
                                                     lines=ln), chunks))
    return np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res])


def _compare_pair_all_lines(dY_bits, X_bits, rot, nb, rnd, seed):
    """Every code and scale byte of both Wgrad operands from the one-launch
    encode (mx_quantize_pair, SR tags 1 and 2) against the oracle."""
    (ca, sa), (cb, sb) = mx.quantize_pair(_dev(dY_bits), _dev(X_bits), rot, nb, rnd, seed)
    mx.check_status()
    T = dY_bits.shape[0]
    for bits, codes, scales, tag in ((dY_bits, ca, sa, 1), (X_bits, cb, sb, 2)):
        n = bits.shape[1]
        oc, os_ = _par_oracle_quantize(bits, mx.CONTRACT_ROWS, rot, nb, rnd, seed, tag)
        got_c = codes.cpu().numpy()
        got_s = untile_scales(scales.cpu().numpy(), n, T)
        bad = np.argwhere((got_c != oc).any(axis=1) | (got_s != os_).any(axis=1))
        assert bad.size == 0, f"rot {rot}/{nb} rnd {rnd}: {bad.size} of {n} lines differ, " \
                              f"first {bad[:5].ravel().tolist()}"


@pytest.mark.slow
def test_down_proj_rotation_sweep():
    # every line of both operands at every Hadamard size, plus sampled GEMM entries
    d = config_inputs("down_proj", seed=0)
    for nb in (16, 32, 64, 128, 256):
        _compare_pair_all_lines(d["dY"], d["X"], mx.ROT_HADAMARD_DET, nb, mx.ROUND_RNE, 0)
        check_op(mx.OP_WGRAD, d["dY"], d["X"], mx.ROT_HADAMARD_DET, nb, sample=24)


@pytest.mark.slow
def test_ablation_modes_full_size():
    d = config_inputs("ablation", seed=0)
    for rot, nb, rnd, seed in [(mx.ROT_NONE, 32, mx.ROUND_RNE, 0),
                               (mx.ROT_HADAMARD_RAND, 32, mx.ROUND_RNE, 1),
                               (mx.ROT_NONE, 32, mx.ROUND_SR, 1)]:
        _compare_pair_all_lines(d["dY"], d["X"], rot, nb, rnd, seed)
        check_op(mx.OP_WGRAD, d["dY"], d["X"], rot, nb, rnd, seed, sample=24)


@pytest.mark.slow
def test_qkv_gateup_all_three_gemms():
    d = config_inputs("qkv_gateup", seed=0)
    X = d["X"]
    for w, dy in (("W_qkv", "dY_qkv"), ("W_gu", "dY_gu")):
        W, dY = d[w], d[dy]
        # each GEMM: >= 64 full rows, >= 64 full columns and 4,096 random entries
        check_op_rows_cols(mx.OP_FPROP, X, W, mx.ROT_NONE, 32)
        check_op_rows_cols(mx.OP_DGRAD, dY, W, mx.ROT_NONE, 32)
        check_op_rows_cols(mx.OP_WGRAD, dY, X, mx.ROT_HADAMARD_DET, 32)


@pytest.mark.parametrize("T,N,K,rot,nb", [(1024, 512, 768, mx.ROT_HADAMARD_DET, 32),
                                          (2048, 256, 1280, mx.ROT_HADAMARD_DET, 16),
                                          (512, 768, 256, mx.ROT_NONE, 32),
                                          (4096, 2560, 2304, mx.ROT_HADAMARD_DET, 32)])
def test_wgrad_fused_launch_equals_separate_launches(T, N, K, rot, nb):
    """mx_linear_wgrad_fused runs these shapes as one launch whose encoder
    warps feed the GEMM; the result has the bits of mx_linear_wgrad's separate
    encode + GEMM launches (the same encode and the same accumulation order)
    and matches the oracle on sampled entries.  The last shape has more tiles
    than pairs."""
    assert mx.lib().mx_linear_wgrad_fused_supported(T, N, K, rot, nb, mx.ROUND_RNE) == 1
    dY_bits = _bits((T, N), 51, 1e-3)
    X_bits = _bits((T, K), 52)
    dY, X = _dev(dY_bits), _dev(X_bits)
    fused = mx.linear_wgrad_fused(dY, X, rot=rot, rot_block=nb, rnd=mx.ROUND_RNE, seed=0)
    mx.check_status()
    (aq, as_), (bq, bs) = mx.quantize_pair(dY, X, rot, nb, mx.ROUND_RNE, 0)
    sep = mx.gemm(aq, as_, bq, bs, N, K, T)
    mx.check_status()
    assert torch.equal(fused.view(torch.int32), sep.view(torch.int32))
    again = mx.linear_wgrad_fused(dY, X, rot=rot, rot_block=nb, rnd=mx.ROUND_RNE, seed=0)
    mx.check_status()
    assert torch.equal(fused.view(torch.int32), again.view(torch.int32))
    ref, ref_abs = _oracle_entries(dY_bits, X_bits, rot, nb)
    got = fused.cpu().numpy()
    ii, jj = ref[2], ref[3]
    assert np.all(np.abs(got[ii, jj].astype(np.float64) - ref[0]) <= 1e-5 * ref_abs)


def _oracle_entries(dY_bits, X_bits, rot, nb, n=2048):
    Aq, As = oracle.quantize(dY_bits, oracle.CONTRACT_ROWS, rot, nb, mx.ROUND_RNE, 0, 1)
    Bq, Bs = oracle.quantize(X_bits, oracle.CONTRACT_ROWS, rot, nb, mx.ROUND_RNE, 0, 2)
    rng = np.random.default_rng(9)
    ii, jj = rng.integers(0, Aq.shape[0], n), rng.integers(0, Bq.shape[0], n)
    C, Ca = oracle.gemm_entries(Aq, As, Bq, Bs, ii, jj)
    return (C, Ca, ii, jj), Ca


def test_wgrad_fused_rejects_modes_it_does_not_cover():
    dY = torch.zeros((1024, 256), dtype=torch.int16, device="cuda")
    X = torch.zeros((1024, 256), dtype=torch.int16, device="cuda")
    for rot, nb, rnd in [(mx.ROT_HADAMARD_RAND, 32, mx.ROUND_RNE), (mx.ROT_HADAMARD_DET, 64, mx.ROUND_RNE),
                         (mx.ROT_HADAMARD_DET, 32, mx.ROUND_SR)]:
        assert mx.lib().mx_linear_wgrad_fused_supported(1024, 256, 256, rot, nb, rnd) == 0
        with pytest.raises(mx.MXError):
            mx.linear_wgrad_fused(dY, X, rot=rot, rot_block=nb, rnd=rnd)
    assert mx.lib().mx_linear_wgrad_fused_supported(1000, 256, 256, 1, 32, 0) == 0   # T % 512
