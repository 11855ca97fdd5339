"""Host-only checks of the C-ABI library: it loads, exports every symbol that
include/mx.h declares, sizes buffers as documented, and rejects bad arguments
before launching anything (no GPU needed for any call here)."""
import ctypes
import os
import re

import numpy as np
import pytest

import mxfp4_precision_gb300 as mx
from mxfp4_precision_gb300 import build as mxbuild
from tests.mx_testutil import padded_dims, tile_scales, untile_scales

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    mxbuild.build()
    return mx.lib()


def _declared():
    with open(os.path.join(ROOT, "include", "mx.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mx_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert "mx_quantize" in names and "mx_gemm" in names and "mx_linear_wgrad" in names
    for n in names:
        assert hasattr(L, n), f"{n} declared in mx.h but not exported"
        ctypes.cast(getattr(L, n), ctypes.c_void_p)
    assert set(names) <= set(mx._binding.EXPORTED) | set(names)


def test_version_and_status_strings(L):
    assert mx.lib().mx_version() == 100
    for code, name in [(0, "MX_OK"), (1, "MX_ERR_INVALID_ARG"), (2, "MX_ERR_SHAPE"),
                       (3, "MX_ERR_ALIGN"), (4, "MX_ERR_WORKSPACE"), (5, "MX_ERR_CUDA"),
                       (6, "MX_ERR_TIMEOUT"), (7, "MX_ERR_UNSUPPORTED")]:
        assert mx.status_string(code) == name


def test_buffer_sizes(L):
    assert mx.codes_bytes(4096, 8192) == 4096 * 4096
    assert mx.scales_bytes(4096, 8192) == 4096 * 256
    assert mx.scales_bytes(200, 800) == 256 * 32     # lines -> 256, blocks -> 32
    assert mx.codes_bytes(0, 64) == 0 and mx.scales_bytes(5, 0) == 0
    T, N, K = 8192, 4096, 14336
    ws = mx.linear_workspace_bytes(mx.OP_WGRAD, T, N, K)
    # both encoded operands, plus one 4-byte counter per (256-line panel,
    # 512-token chunk) for the fused Wgrad launch
    counters = 4 * (N // 256 + K // 256) * (T // 512)
    assert ws == (N * T // 2 + N * T // 32) + (K * T // 2 + K * T // 32) + (counters + 255) // 256 * 256
    assert mx.linear_workspace_bytes(mx.OP_FPROP, T, N, K) == \
        (T * K // 2 + T * K // 32) + (N * K // 2 + N * K // 32)
    assert mx.linear_workspace_bytes(7, T, N, K) == 0


def test_scale_tiling_roundtrip_and_documented_offsets():
    rng = np.random.default_rng(0)
    for mn, k in [(128, 256), (200, 800), (4096, 8192 // 16)]:
        canon = rng.integers(0, 255, size=(mn, k // 32), dtype=np.uint8)
        flat = tile_scales(canon, mn, k)
        MP, KB = padded_dims(mn, k)
        assert flat.size == MP * KB
        assert np.array_equal(untile_scales(flat, mn, k), canon)
        for r, b in [(0, 0), (mn - 1, k // 32 - 1), (mn // 2, 1)]:
            off = ((r // 128) * (KB // 4) + b // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + b % 4
            assert flat[off] == canon[r, b]


V = ctypes.c_void_p


def _q(L, src=0x1000, rows=256, cols=64, contract=0, rot=1, nb=32, rnd=0, codes=0x2000,
       scales=0x3000):
    return L.mx_quantize(V(src), rows, cols, contract, rot, nb, rnd, 0, V(codes), V(scales), None)


def test_quantize_rejects_bad_arguments_before_launch(L):
    assert _q(L, contract=2) == 1
    assert _q(L, rot=3) == 1
    assert _q(L, nb=48) == 1
    assert _q(L, rnd=5) == 1
    assert _q(L, src=0) == 1
    assert _q(L, rows=-1) == 2
    assert _q(L, rows=100) == 2                   # contraction length not a multiple of 32
    assert _q(L, rows=96, nb=64) == 2              # rot_block must divide it
    assert _q(L, contract=1, cols=96, nb=64) == 2
    assert _q(L, src=0x1001) == 3
    assert _q(L, codes=0x2008) == 3
    assert _q(L, cols=60) == 3                     # rows not 16-byte aligned
    assert _q(L, rows=0) == 0 and _q(L, cols=0) == 0  # empty: nothing to do


def _qd(L, src=0x1000, T=256, N=128, rot=1, nb=32, rnd=0, ct=0x2000, st=0x3000, cn=0x4000,
        sn=0x5000):
    return L.mx_quantize_dual(src, T, N, rot, nb, rnd, 0, ct, st, cn, sn, None)


def test_quantize_dual_rejects_bad_arguments_before_launch(L):
    # the union of the column-direction and row-direction rules
    assert _qd(L, rot=3) == 1
    assert _qd(L, nb=48) == 1
    assert _qd(L, rnd=5) == 1
    assert _qd(L, src=0) == 1
    assert _qd(L, cn=0) == 1 and _qd(L, st=0) == 1
    assert _qd(L, T=-1) == 2
    assert _qd(L, T=100) == 2                      # contraction T not a multiple of 32
    assert _qd(L, T=96, nb=64) == 2                # rot_block must divide T
    assert _qd(L, N=72) == 2                       # contraction N not a multiple of 32
    assert _qd(L, src=0x1001) == 3 and _qd(L, sn=0x5008) == 3
    assert _qd(L, T=0) == 0 and _qd(L, N=0) == 0   # empty: nothing to do


def test_scales_to_canonical_rejects_bad_arguments_before_launch(L):
    f = lambda sc=0x1000, lines=128, k=256, out=0x2000: L.mx_scales_to_canonical(sc, lines, k, out,
                                                                               None)
    assert f(k=100) == 2 and f(lines=-1) == 2
    assert f(sc=0) == 1 and f(out=0) == 1
    assert f(lines=0) == 0 and f(k=0) == 0


def test_gemm_rejects_bad_arguments_before_launch(L):
    g = lambda **k: L.mx_gemm(V(k.get("a", 0x1000)), V(0x2000), V(0x3000), V(0x4000),
                              V(k.get("c", 0x5000)), k.get("M", 128), k.get("N", 256),
                              k.get("K", 256), None)
    assert g(M=-1) == 2
    assert g(K=48) == 2
    assert g(N=250) == 3
    assert g(c=0x5004) == 3
    assert g(a=0) == 1
    assert g(c=0) == 1
    assert g(M=0) == 0 and g(N=0) == 0


def test_linear_rejects_bad_arguments_before_launch(L):
    def w(ws=0x10000, ws_bytes=1 << 40, T=256, N=128, K=256, rot=1, nb=32, dW=0x5000):
        return L.mx_linear_wgrad(V(0x1000), V(0x2000), V(dW), T, N, K, rot, nb, 0, 0, V(ws),
                                 ws_bytes, None)
    assert w(ws_bytes=10) == 4
    assert w(ws=0) == 4
    assert w(ws=0x10010) == 3                      # workspace must be 256-byte aligned
    assert w(T=100) == 2
    assert w(nb=7) == 1
    assert w(dW=0) == 1
    assert w(K=250) == 3
    assert w(N=0) == 0


def test_noalloc_checks_arguments_before_the_scratch_limit(L):
    """The no-allocation Wgrad entry point reports the same status codes as
    mx_linear_wgrad for bad arguments, even when the request is also larger
    than its fixed scratch area; only otherwise-valid oversize requests get
    MX_ERR_WORKSPACE.  None of these calls reaches the GPU."""
    big = dict(T=16384, N=4096, K=4096)            # needs 71.3 MB > 64 MiB of scratch

    def na(T, N, K, rot=1, nb=32, rnd=0, dW=0x5000, dY=0x1000):
        return L.mx_linear_wgrad_noalloc(V(dY), V(0x2000), V(dW), T, N, K, rot, nb, rnd, 0, None)
    assert na(**big) == 4                          # valid, too large: MX_ERR_WORKSPACE
    assert na(**{**big, "T": 16384 - 16}) == 2     # T % 32 != 0: MX_ERR_SHAPE
    assert na(**{**big, "K": 4094}) == 3           # K % 8 != 0 (TMA rows): MX_ERR_ALIGN
    assert na(**big, rot=5) == 1                   # bad enum: MX_ERR_INVALID_ARG
    assert na(**big, nb=48) == 1
    assert na(**big, rnd=2) == 1
    assert na(**big, dW=0) == 1
    assert na(**big, dY=0x1008) == 3               # misaligned input
    assert na(T=256, N=0, K=256) == 0              # empty: nothing to do
    assert na(T=-1, N=128, K=256) == 2
