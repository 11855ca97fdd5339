"""Synthetic stand-ins for the Llama-3.1-8B / C4 tensors of the pages' study.

The study ("Neue Studie von AMD durchbricht die bestehende Erkenntnis",
section "Fehlerdiagnoseexperiment") pretrains Llama 3.1-8B on C4 with the
MLPerf setup; neither the dataset nor weights exist here, so every tensor is
drawn from a seeded distribution with the layer's shape:

* activations X: N(0, 1) with 1% of channels scaled x20 (outlier channels),
  or SiLU(g) * u with g, u ~ N(0, 1) for the FFN down-projection input;
* output gradients dY: Student-t with 3 degrees of freedom scaled to std 1e-3
  (heavy tails), drawn as z / sqrt(chi2_3 / 3) with chi2_3 = 2 * Gamma(1.5);
* weights W: N(0, 0.02^2).

All values are rounded to bf16 (round to nearest even) and returned as raw
uint16 bit patterns, so the oracle and the GPU path see identical inputs.
Draws are chunked by rows from one numpy PCG64 stream per tensor, keyed by
(seed, tensor id); the chunking is fixed, so outputs are reproducible.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

_CHUNK_ROWS = 512


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), int(tensor_id)]))


def _chunked(shape, draw) -> np.ndarray:
    rows, cols = shape
    out = np.empty((rows, cols), dtype=np.uint16)
    for r0 in range(0, rows, _CHUNK_ROWS):
        r1 = min(rows, r0 + _CHUNK_ROWS)
        out[r0:r1] = bf16_bits(draw((r1 - r0, cols)))
    return out


def normal_bf16(shape, std: float, seed: int, tensor_id: int) -> np.ndarray:
    g = _rng(seed, tensor_id)
    return _chunked(shape, lambda s: g.standard_normal(s, dtype=np.float32) * np.float32(std))


def student_t3_bf16(shape, std: float, seed: int, tensor_id: int) -> np.ndarray:
    """Student-t(nu=3) scaled so that its standard deviation is `std`."""
    g = _rng(seed, tensor_id)
    scale = np.float32(std / np.sqrt(3.0))

    def draw(s):
        z = g.standard_normal(s, dtype=np.float32)
        chi2 = np.float32(2.0) * g.standard_gamma(1.5, s, dtype=np.float32)
        return z / np.sqrt(chi2 / np.float32(3.0)) * scale
    return _chunked(shape, draw)


def outlier_channels_bf16(shape, seed: int, tensor_id: int, frac: float = 0.01,
                          factor: float = 20.0, n_outliers: int | None = None) -> np.ndarray:
    """N(0, 1) activations whose outlier channels (columns) are scaled by `factor`."""
    rows, cols = shape
    g = _rng(seed, tensor_id)
    k = n_outliers if n_outliers is not None else max(1, int(cols * frac))
    chosen = g.permutation(cols)[:k]
    mult = np.ones(cols, dtype=np.float32)
    mult[chosen] = np.float32(factor)
    return _chunked(shape, lambda s: g.standard_normal(s, dtype=np.float32) * mult)


def silu_gate_bf16(shape, seed: int, tensor_id: int) -> np.ndarray:
    """SiLU(g) * u with g, u ~ N(0, 1): the FFN down-projection input."""
    g = _rng(seed, tensor_id)

    def draw(s):
        a = g.standard_normal(s, dtype=np.float32)
        u = g.standard_normal(s, dtype=np.float32)
        return a / (np.float32(1.0) + np.exp(-a)) * u
    return _chunked(shape, draw)


@dataclass(frozen=True)
class WorkloadConfig:
    name: str
    description: str
    T: int
    tensors: dict = field(default_factory=dict)     # name -> (shape, kind, kwargs)
    rot_blocks: tuple = (32,)


# Tensor kinds: ("normal", std) | ("t3", std) | ("outlier", frac/n) | ("silu",)
CONFIGS = {
    "tiny": WorkloadConfig(
        "tiny", "Tiny Wgrad: dY [256,128] N(0,1e-3^2), X [256,256] N(0,1) with 2 of 256 "
        "channels x20; Hadamard 32 along T, RNE, seed 0", 256,
        {"dY": ((256, 128), "normal", 1e-3), "X": ((256, 256), "outlier", 2)}),
    "o_proj": WorkloadConfig(
        "o_proj", "Llama-3.1-8B attention o_proj Wgrad: T=8192, dY [8192,4096] Student-t(3) "
        "std 1e-3, X [8192,4096] N(0,1) with 1% outlier channels x20; Hadamard 32", 8192,
        {"dY": ((8192, 4096), "t3", 1e-3), "X": ((8192, 4096), "outlier", None)}),
    "down_proj": WorkloadConfig(
        "down_proj", "Llama-3.1-8B FFN down_proj Wgrad: T=8192, dY [8192,4096] Student-t(3) "
        "std 1e-3, X [8192,14336] SiLU(g)*u; Hadamard block swept 16/32/64/128/256", 8192,
        {"dY": ((8192, 4096), "t3", 1e-3), "X": ((8192, 14336), "silu", None)},
        rot_blocks=(16, 32, 64, 128, 256)),
    "qkv_gateup": WorkloadConfig(
        "qkv_gateup", "Llama-3.1-8B fused QKV + gate/up, Fprop/Dgrad/Wgrad: T=16384, "
        "X [16384,4096] N(0,1) 1% outliers x20, W [6144,4096] and [28672,4096] N(0,0.02^2), "
        "dY Student-t(3) std 1e-3", 16384,
        {"X": ((16384, 4096), "outlier", None),
         "W_qkv": ((6144, 4096), "normal", 0.02), "W_gu": ((28672, 4096), "normal", 0.02),
         "dY_qkv": ((16384, 6144), "t3", 1e-3), "dY_gu": ((16384, 28672), "t3", 1e-3)}),
    "ablation": WorkloadConfig(
        "ablation", "Rotation/rounding ablation at down_proj shape (T=8192, K=14336, N=4096)",
        8192,
        {"dY": ((8192, 4096), "t3", 1e-3), "X": ((8192, 14336), "silu", None)}),
}

_TENSOR_IDS = {"dY": 1, "X": 2, "W_qkv": 3, "W_gu": 4, "dY_qkv": 5, "dY_gu": 6}


def make_tensor(shape, kind, arg, seed: int, tensor_id: int) -> np.ndarray:
    if kind == "normal":
        return normal_bf16(shape, arg, seed, tensor_id)
    if kind == "t3":
        return student_t3_bf16(shape, arg, seed, tensor_id)
    if kind == "outlier":
        return outlier_channels_bf16(shape, seed, tensor_id, n_outliers=arg)
    if kind == "silu":
        return silu_gate_bf16(shape, seed, tensor_id)
    raise ValueError(kind)


def config_inputs(name: str, seed: int = 0, only=None, rows: int | None = None) -> dict:
    """bf16 bit patterns for a named workload; `rows` truncates T (for small cases)."""
    cfg = CONFIGS[name]
    out = {}
    for tname, (shape, kind, arg) in cfg.tensors.items():
        if only is not None and tname not in only:
            continue
        shp = shape
        if rows is not None and shape[0] == cfg.T:
            shp = (rows, shape[1])
        out[tname] = make_tensor(shp, kind, arg, seed, _TENSOR_IDS[tname])
    return out
