"""Seeded synthetic inputs shared by the tests, the oracle checks and the bench.

This module draws random numbers and shapes workloads; it holds none of the
quantization, dequantization or GEMV arithmetic.  Both the CPU oracle and the
CUDA path consume what it produces, so it is the only code they share.

Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) used counter-style: the i-th
64-bit draw of stream ``key`` is ``mix(key * 2**32 + i)`` through the
SplitMix64 output function, so any slice regenerates independently.  Normal
deviates come from the Box-Muller transform of two 53-bit uniforms in (0, 1].
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def draws(key: int, start: int, count: int) -> np.ndarray:
    """uint64 draws [start, start+count) of stream ``key`` (SplitMix64 sequence)."""
    base = np.uint64((key * (1 << 32)) & 0xFFFFFFFFFFFFFFFF)
    ctr = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(base + ctr * _GOLDEN)


def uniform(key: int, start: int, count: int) -> np.ndarray:
    """float64 uniforms in (0, 1] from the top 53 bits of each draw."""
    d = draws(key, start, count)
    return ((d >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def normal(key: int, n: int, std: float = 1.0, chunk: int = 1 << 24) -> np.ndarray:
    """float32 N(0, std^2): element 2p and 2p+1 from uniforms 2p, 2p+1 (Box-Muller)."""
    out = np.empty(n, np.float32)
    npairs = (n + 1) // 2
    for p0 in range(0, npairs, chunk):
        p1 = min(npairs, p0 + chunk)
        u = uniform(key, 2 * p0, 2 * (p1 - p0))
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log(u1)) * std
        t = 2.0 * np.pi * u2
        z = np.empty(2 * (p1 - p0), np.float64)
        z[0::2] = r * np.cos(t)
        z[1::2] = r * np.sin(t)
        e0, e1 = 2 * p0, min(n, 2 * p1)
        out[e0:e1] = z[: e1 - e0].astype(np.float32)
    return out


def distinct_indices(key: int, n: int, m: int) -> np.ndarray:
    """m distinct indices in [0, n): the m smallest draw values of stream ``key``."""
    if m <= 0:
        return np.zeros(0, np.int64)
    d = draws(key, 0, n)
    idx = np.argpartition(d, m - 1)[:m]
    return np.sort(idx.astype(np.int64))


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (finite inputs).

    Used only to shape the bf16 activation input x."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    return ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


# --------------------------------------------------------------------------
# workloads (shapes, sizes, distributions and seeds of the five configurations)

STD_W = 0.02


def weights(seed: int, n: int, outlier_frac: float = 0.0, outlier_seed: int | None = None,
            outlier_scale: float = 10.0) -> np.ndarray:
    """Weights ~ N(0, 0.02) as float32; optionally round(frac*n) distinct
    elements multiplied by ``outlier_scale`` (in float32)."""
    w = normal(seed, n, STD_W)
    if outlier_frac > 0.0:
        m = int(round(outlier_frac * n))
        idx = distinct_indices(outlier_seed if outlier_seed is not None else seed + 100, n, m)
        w[idx] = (w[idx] * np.float32(outlier_scale)).astype(np.float32)
    return w


def activations(seed: int, batch: int, K: int) -> np.ndarray:
    """x ~ N(0, 1), rounded to bf16, as uint16 bit patterns [batch, K]."""
    return to_bf16_bits(normal(seed, batch * K, 1.0)).reshape(batch, K)


@dataclass(frozen=True)
class Layer:
    name: str
    N: int
    K: int
    seed: int


QWEN_1P5B_LAYERS = (
    Layer("q_proj", 1536, 1536, 20), Layer("k_proj", 256, 1536, 21),
    Layer("v_proj", 256, 1536, 22), Layer("o_proj", 1536, 1536, 23),
    Layer("gate_proj", 8960, 1536, 24), Layer("up_proj", 8960, 1536, 25),
    Layer("down_proj", 1536, 8960, 26),
)
QWEN_X_SEED = 30

LLAMA_7B_LAYERS = (
    Layer("attn_proj", 4096, 4096, 40), Layer("gate_up_proj", 11008, 4096, 41),
    Layer("down_proj", 4096, 11008, 42),
)
LLAMA_BATCHES = (1, 4, 8)


def llama_x_seed(batch: int) -> int:
    return 50 + batch


@dataclass(frozen=True)
class DequantCase:
    name: str
    n: int
    seed: int
    outlier_frac: float = 0.0
    outlier_seed: int | None = None
    dtypes: tuple = ("bf16",)
    shape: tuple | None = None


CONFIG0 = DequantCase("1024x1024", 1024 * 1024, 0, shape=(1024, 1024))
CONFIG1 = DequantCase("4096x4096_outliers", 4096 * 4096, 1, 0.001, 101, ("bf16", "fp16"),
                      shape=(4096, 4096))
CONFIG4 = (
    (DequantCase("28672x8192", 28672 * 8192, 60, shape=(28672, 8192)),)
    + tuple(DequantCase(f"flat_2^{e}", 1 << e, 61 + i) for i, e in enumerate((20, 22, 24, 26, 28, 30)))
    + (DequantCase("ragged_64x256x1000+64x37", 64 * 256 * 1000 + 64 * 37, 67),)
)
