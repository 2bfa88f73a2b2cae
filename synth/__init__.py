"""Seeded synthetic inputs shared by the tests, the oracle checks and the bench.

This module draws random numbers and shapes workloads; it holds none of the
quantization, dequantization or GEMV arithmetic.  Both the CPU oracle and the
CUDA path consume what it produces, so it is the only code they share.

Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) used counter-style: draw i of
stream ``key`` is the SplitMix64 output mix of ``key * 2**32 + (i + 1) *
0x9E3779B97F4A7C15`` (mod 2**64), so any slice regenerates independently.
Normal deviates come from the Box-Muller transform of two 53-bit uniforms in
(0, 1].  The core is ``synth.c`` (threaded C, loaded with ctypes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "_synth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the generator core (C, pthreads)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                        "-shared", "-pthread", _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P, I64, U64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64
        lib.synth_normal_f32.argtypes = [U64, I64, I64, ctypes.c_double, P, ctypes.c_int]
        lib.synth_normal_bf16.argtypes = [U64, I64, I64, P, ctypes.c_int]
        lib.synth_draws.argtypes = [U64, I64, I64, P, ctypes.c_int]
        _lib = lib
    return _lib


def _threads() -> int:
    try:
        return max(1, min(32, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(32, os.cpu_count() or 1))


def draws(key: int, start: int, count: int) -> np.ndarray:
    """uint64 draws [start, start+count) of stream ``key`` (SplitMix64 sequence)."""
    out = np.empty(count, np.uint64)
    if count:
        _load().synth_draws(key, start, count, out.ctypes.data, _threads())
    return out


def normal(key: int, n: int, std: float = 1.0, start: int = 0) -> np.ndarray:
    """float32 N(0, std^2): element 2p and 2p+1 from uniforms 2p, 2p+1 (Box-Muller)."""
    out = np.empty(n, np.float32)
    if n:
        _load().synth_normal_f32(key, start, n, float(std), out.ctypes.data, _threads())
    return out


def normal_bf16(key: int, n: int) -> np.ndarray:
    """N(0, 1) rounded to bfloat16 (nearest even), as uint16 bit patterns."""
    out = np.empty(n, np.uint16)
    if n:
        _load().synth_normal_bf16(key, 0, n, out.ctypes.data, _threads())
    return out


def distinct_indices(key: int, n: int, m: int) -> np.ndarray:
    """m distinct indices in [0, n): the m smallest draw values of stream ``key``."""
    if m <= 0:
        return np.zeros(0, np.int64)
    d = draws(key, 0, n)
    idx = np.argpartition(d, m - 1)[:m]
    return np.sort(idx.astype(np.int64))


def code2_linear() -> np.ndarray:
    """The workloads' second-level table: binary16 of (i - 127.5) / 127.5, i < 256
    (binary64 value rounded once to binary16), as uint16 bit patterns."""
    return ((np.arange(256, dtype=np.float64) - 127.5) / 127.5).astype(np.float16).view(np.uint16)


def code2_dynamic() -> np.ndarray:
    """A non-linear second-level table for the table-generality cases:
    logarithmically spaced magnitudes, entry 128 + k = binary16(2^((k - 127) / 16))
    for k < 128 and entry 127 - k its negation, as uint16 bit patterns."""
    pos = np.exp2((np.arange(128, dtype=np.float64) - 127.0) / 16.0).astype(np.float16).view(np.uint16)
    out = np.zeros(256, np.uint16)
    out[128:] = pos
    out[:128] = (pos | 0x8000)[::-1]
    return out


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
    return normal_bf16(seed, batch * K).reshape(batch, K)


def bias(seed: int, N: int, dtype: str) -> np.ndarray:
    """Layer bias ~ N(0, 1) in the output type ("bf16", "fp16" or "f32") as bit
    patterns: uint16 for the 16-bit types (nearest even), uint32 for binary32."""
    if dtype == "bf16":
        return normal_bf16(seed, N)
    f = normal(seed, N)
    if dtype == "fp16":
        return f.astype(np.float16).view(np.uint16)
    if dtype == "f32":
        return f.view(np.uint32).copy()
    raise ValueError(dtype)


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
