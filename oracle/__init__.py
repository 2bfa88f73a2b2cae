"""CPU oracle for NF4 double-quantized dequantization and decode GEMV.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product path
(``w4a16_gemv_gb300`` and its CUDA library) never imports, links or runs it,
and this package imports nothing from the product path.

The arithmetic lives in ``nf4_oracle.c`` (plain single-threaded C, built with
floating-point contraction disabled); this module is argument marshalling with
ctypes and numpy.  Each function names the passage it follows:

* quantization: "NF4反量化算子优化", sections "双量化" (first and second level),
  and the report "NF4 双重量化反量化 CUDA Kernel 实现报告" section 1.2;
* dequantization: the report, section 1.3 (formula) and 2.2 (nibble order);
* GEMV: "RTX 4060 上的 LLM 量化实测", section "Fused kernel：把反量化搬到片上";
* the layer's output stage (bias added to the row sum, result stored in the
  layer's 16-bit type): the same section.

Every function here is pinned by tests under ``tests/`` (``-m "not gpu"``)
against values and properties the pages and the mathematics fix.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nf4_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_nf4_oracle.so")
_lib = None

BF16 = 0
FP16 = 1
F32 = 2


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (single translation unit, -ffp-contract=off)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.oracle_nf4_code.argtypes = [P]
    lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_f16.restype = ctypes.c_uint16
    lib.oracle_f64_to_f16.argtypes = [ctypes.c_double]
    lib.oracle_f64_to_f16.restype = ctypes.c_uint16
    lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_f32.restype = ctypes.c_float
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    lib.oracle_code2_linear.argtypes = [P]
    lib.oracle_code2_dynamic.argtypes = [P]
    lib.oracle_block_absmax.argtypes = [P, I64, I64, P]
    lib.oracle_nf4_nearest.argtypes = [ctypes.c_float]
    lib.oracle_nf4_nearest.restype = ctypes.c_int
    lib.oracle_nf4_encode.argtypes = [P, I64, I64, P, P]
    lib.oracle_code2_nearest.argtypes = [ctypes.c_float, P]
    lib.oracle_code2_nearest.restype = ctypes.c_int
    lib.oracle_double_quant.argtypes = [P, I64, I64, P, P, P, P]
    lib.oracle_block_scale.argtypes = [P, P, P, ctypes.c_float, I64, I64]
    lib.oracle_block_scale.restype = ctypes.c_float
    lib.oracle_dequant_f32.argtypes = [P, P, P, P, ctypes.c_float, I64, I64, I64, P]
    lib.oracle_dequant.argtypes = [P, P, P, P, ctypes.c_float, I64, I64, I64, ctypes.c_int, P]
    lib.oracle_dequant_at.argtypes = [P, P, P, P, ctypes.c_float, I64, I64, ctypes.c_int, P, I64, P]
    lib.oracle_gemv.argtypes = [P, P, P, P, ctypes.c_float, I64, I64, I64, I64, P, I64, P, I64, P, P]
    lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
    lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
    lib.oracle_f64_to_f32_bits.argtypes = [ctypes.c_double]
    lib.oracle_f64_to_f32_bits.restype = ctypes.c_uint32
    lib.oracle_round_f64.argtypes = [ctypes.c_double, ctypes.c_int]
    lib.oracle_round_f64.restype = ctypes.c_uint32
    lib.oracle_decode.argtypes = [ctypes.c_uint32, ctypes.c_int]
    lib.oracle_decode.restype = ctypes.c_double
    lib.oracle_gemv_output.argtypes = [P, I64, I64, P, P, ctypes.c_int, P, P]
    lib.oracle_gemv_abs.argtypes = [P, P, P, P, ctypes.c_float, I64, I64, I64, I64, P, I64, P]
    _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# --------------------------------------------------------------------------
# scalar conversions (IEEE-754 round to nearest even, written from the
# definition in C; pinned against numpy / torch CPU conversions in the tests)

def f32_to_bf16(v: float) -> int:
    return int(_load().oracle_f32_to_bf16(float(np.float32(v))))


def f32_to_f16(v: float) -> int:
    return int(_load().oracle_f32_to_f16(float(np.float32(v))))


def f64_to_f16(v: float) -> int:
    return int(_load().oracle_f64_to_f16(float(v)))


def f16_to_f32(h: int) -> float:
    return float(np.float32(_load().oracle_f16_to_f32(int(h))))


def bf16_to_f32(h: int) -> float:
    return float(np.float32(_load().oracle_bf16_to_f32(int(h))))


def nf4_code() -> np.ndarray:
    """The sixteen NF4 codes (binary32), "NF4反量化算子优化", section "NF4 table"."""
    out = np.zeros(16, np.float32)
    _load().oracle_nf4_code(_ptr(out))
    return out


def nf4_nearest(v: float) -> int:
    return int(_load().oracle_nf4_nearest(float(np.float32(v))))


def code2_linear() -> np.ndarray:
    """fp16[256] second-level table, entry i = (i - 127.5) / 127.5 (as uint16 bits)."""
    out = np.zeros(256, np.uint16)
    _load().oracle_code2_linear(_ptr(out))
    return out


def code2_dynamic() -> np.ndarray:
    """fp16[256] non-linear second-level table: entry 128 + k = 2^((k - 127) / 16),
    entry 127 - k its negation (as uint16 bits)."""
    out = np.zeros(256, np.uint16)
    _load().oracle_code2_dynamic(_ptr(out))
    return out


def code2_nearest(r: float, code2: np.ndarray) -> int:
    code2 = np.ascontiguousarray(code2, np.uint16)
    return int(_load().oracle_code2_nearest(float(np.float32(r)), _ptr(code2)))


# --------------------------------------------------------------------------
# quantization

@dataclass
class NF4Tensor:
    """Double-quantized NF4 tensor in the layout the CUDA library consumes."""
    packed: np.ndarray      # uint8 [ceil(n/2)], even element in the high nibble
    absmax_q: np.ndarray    # uint8 [ceil(n/bs)]
    absmax2: np.ndarray     # uint16 (fp16 bits) [ceil(nb/s2)]
    code2: np.ndarray       # uint16 (fp16 bits) [256]
    offset: float           # binary32 value
    n: int
    blocksize: int = 64
    s2_blocksize: int = 256


def block_absmax(w: np.ndarray, blocksize: int = 64) -> np.ndarray:
    w = np.ascontiguousarray(w, np.float32).reshape(-1)
    nb = (w.size + blocksize - 1) // blocksize
    out = np.zeros(nb, np.float32)
    _load().oracle_block_absmax(_ptr(w), w.size, blocksize, _ptr(out))
    return out


def nf4_encode(w: np.ndarray, absmax: np.ndarray, blocksize: int = 64) -> np.ndarray:
    w = np.ascontiguousarray(w, np.float32).reshape(-1)
    absmax = np.ascontiguousarray(absmax, np.float32)
    out = np.zeros((w.size + 1) // 2, np.uint8)
    _load().oracle_nf4_encode(_ptr(w), w.size, blocksize, _ptr(absmax), _ptr(out))
    return out


def double_quant(absmax: np.ndarray, s2_blocksize: int = 256, code2: np.ndarray | None = None):
    absmax = np.ascontiguousarray(absmax, np.float32)
    if code2 is None:
        code2 = code2_linear()
    code2 = np.ascontiguousarray(code2, np.uint16)
    nb = absmax.size
    ng = (nb + s2_blocksize - 1) // s2_blocksize
    absmax_q = np.zeros(nb, np.uint8)
    absmax2 = np.zeros(ng, np.uint16)
    off = np.zeros(1, np.float32)
    _load().oracle_double_quant(_ptr(absmax), nb, s2_blocksize, _ptr(code2), _ptr(absmax_q),
                                _ptr(absmax2), _ptr(off))
    return absmax_q, absmax2, float(off[0])


def quantize(w: np.ndarray, blocksize: int = 64, s2_blocksize: int = 256,
             code2: np.ndarray | None = None) -> NF4Tensor:
    """Full NF4 + double quantization of a binary32 tensor (flattened)."""
    w = np.ascontiguousarray(w, np.float32).reshape(-1)
    if code2 is None:
        code2 = code2_linear()
    absmax = block_absmax(w, blocksize)
    packed = nf4_encode(w, absmax, blocksize)
    absmax_q, absmax2, offset = double_quant(absmax, s2_blocksize, code2)
    return NF4Tensor(packed, absmax_q, absmax2, np.ascontiguousarray(code2, np.uint16), offset,
                     w.size, blocksize, s2_blocksize)


# --------------------------------------------------------------------------
# dequantization and GEMV

def block_scale(t: NF4Tensor, b: int) -> float:
    return float(np.float32(_load().oracle_block_scale(
        _ptr(t.absmax_q), _ptr(t.absmax2), _ptr(t.code2), ctypes.c_float(t.offset), b, t.s2_blocksize)))


def dequant_f32(t: NF4Tensor) -> np.ndarray:
    """binary32 dequantized values (before any 16-bit rounding)."""
    out = np.zeros(t.n, np.float32)
    _load().oracle_dequant_f32(_ptr(t.packed), _ptr(t.absmax_q), _ptr(t.absmax2), _ptr(t.code2),
                               ctypes.c_float(t.offset), t.n, t.blocksize, t.s2_blocksize, _ptr(out))
    return out


def dequant(t: NF4Tensor, dtype: int = BF16) -> np.ndarray:
    """16-bit dequantized output as uint16 bit patterns (dtype 0 bf16, 1 fp16)."""
    out = np.zeros(t.n, np.uint16)
    _load().oracle_dequant(_ptr(t.packed), _ptr(t.absmax_q), _ptr(t.absmax2), _ptr(t.code2),
                           ctypes.c_float(t.offset), t.n, t.blocksize, t.s2_blocksize, int(dtype),
                           _ptr(out))
    return out


def dequant_at(t: NF4Tensor, idx: np.ndarray, dtype: int = BF16) -> np.ndarray:
    idx = np.ascontiguousarray(idx, np.int64)
    out = np.zeros(idx.size, np.uint16)
    _load().oracle_dequant_at(_ptr(t.packed), _ptr(t.absmax_q), _ptr(t.absmax2), _ptr(t.code2),
                              ctypes.c_float(t.offset), t.blocksize, t.s2_blocksize, int(dtype),
                              _ptr(idx), idx.size, _ptr(out))
    return out


def gemv(t: NF4Tensor, N: int, K: int, x_bf16: np.ndarray, rows: np.ndarray | None = None):
    """fp64 reference y = W_hat x and S = sum |W_hat * x| for x bf16 bits [batch, K].

    Returns (y_ref, s_abs), each float64 [batch, nrows].
    """
    assert N * K <= t.n
    x = np.ascontiguousarray(x_bf16, np.uint16).reshape(-1, K)
    batch = x.shape[0]
    if rows is not None:
        rows = np.ascontiguousarray(rows, np.int64)
        count = rows.size
        rp = _ptr(rows)
    else:
        count = N
        rp = None
    y = np.zeros((batch, count), np.float64)
    s = np.zeros((batch, count), np.float64)
    _load().oracle_gemv(_ptr(t.packed), _ptr(t.absmax_q), _ptr(t.absmax2), _ptr(t.code2),
                        ctypes.c_float(t.offset), N, K, t.blocksize, t.s2_blocksize, _ptr(x), batch,
                        rp, count, _ptr(y), _ptr(s))
    return y, s


# --------------------------------------------------------------------------
# output stage of a layer: bias and the output type
# ("RTX 4060 上的 LLM 量化实测", section "Fused kernel：把反量化搬到片上")

def f64_to_bf16(v: float) -> int:
    return int(_load().oracle_f64_to_bf16(float(v)))


def f64_to_f32_bits(v: float) -> int:
    return int(_load().oracle_f64_to_f32_bits(float(v)))


def round_f64(v: float, dtype: int) -> int:
    """Pattern of dtype (BF16, FP16, F32) nearest the binary64 value v, ties to even."""
    return int(_load().oracle_round_f64(float(v), int(dtype)))


def decode(bits: int, dtype: int) -> float:
    """Exact value of a BF16 / FP16 / F32 pattern."""
    return float(_load().oracle_decode(int(bits), int(dtype)))


def gemv_output(y_ref: np.ndarray, dtype: int, bias_bits: np.ndarray | None = None,
                rows: np.ndarray | None = None):
    """v = y_ref + bias (binary64, bias widened exactly) and its nearest dtype pattern.

    y_ref is [batch, count] from ``gemv``; bias_bits is [N] (uint16 for BF16/FP16, uint32 for
    F32) or None. Returns (v float64 [batch, count], y_bits uint32 [batch, count]).
    """
    y_ref = np.ascontiguousarray(y_ref, np.float64)
    batch, count = y_ref.shape
    bp = None
    if bias_bits is not None:
        bias_bits = np.ascontiguousarray(bias_bits, np.uint32 if dtype == F32 else np.uint16)
        bp = _ptr(bias_bits)
    rp = None
    if rows is not None:
        rows = np.ascontiguousarray(rows, np.int64)
        rp = _ptr(rows)
    v = np.zeros((batch, count), np.float64)
    yb = np.zeros((batch, count), np.uint32)
    _load().oracle_gemv_output(_ptr(y_ref), batch, count, rp, bp, int(dtype), _ptr(v), _ptr(yb))
    return v, yb


def gemv_abs(t: NF4Tensor, N: int, K: int, e: np.ndarray) -> np.ndarray:
    """a[b, r] = sum_k |W_hat[r, k]| * e[b, k] (binary64) for e >= 0 [batch, K]: how far a
    perturbation of the input by at most e moves W_hat x."""
    assert N * K <= t.n
    e = np.ascontiguousarray(e, np.float64).reshape(-1, K)
    batch = e.shape[0]
    a = np.zeros((batch, N), np.float64)
    _load().oracle_gemv_abs(_ptr(t.packed), _ptr(t.absmax_q), _ptr(t.absmax2), _ptr(t.code2),
                            ctypes.c_float(t.offset), N, K, t.blocksize, t.s2_blocksize, _ptr(e),
                            batch, _ptr(a))
    return a
