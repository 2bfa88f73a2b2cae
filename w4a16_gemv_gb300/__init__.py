"""Python binding of libnf4 (NF4 double-quant dequant and fused decode GEMV on GB300).

Argument marshalling only: tensors are checked for device, dtype, size and
contiguity, then their device pointers and the current CUDA stream go to the C
ABI declared in ``include/nf4.h``. Every step of the computation runs in the
library's CUDA kernels; there is no fallback. Importing this package fails
loudly if ``libnf4.so`` has not been built (``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

__all__ = ["NF4Error", "NF4Weight", "nf4_dequant", "nf4_gemv", "nf4_gemv_ex", "DecodeStep", "nf4_quantize",
           "nf4_quantize_workspace_size", "nf4_quantize_noalloc", "nf4_version", "nf4_status_string",
           "nf4_device_error_flags", "LIB_PATH"]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libnf4.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built: run `python -c \"import __graft_entry__ as g; g.build()\"`")

_lib = ctypes.CDLL(LIB_PATH)
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_lib.nf4_version.restype = ctypes.c_int
_lib.nf4_status_string.argtypes = [ctypes.c_int]
_lib.nf4_status_string.restype = ctypes.c_char_p
_lib.nf4_last_cuda_error.restype = ctypes.c_int
_lib.nf4_dequant.argtypes = [_P, _P, _P, _P, ctypes.c_float, _I64, _I32, _I32, _P, ctypes.c_int, _P]
_lib.nf4_dequant.restype = ctypes.c_int
_lib.nf4_gemv.argtypes = [_P, _P, _P, _P, ctypes.c_float, _I64, _I64, _I32, _I32, _P, _I32, _P, _P]
_lib.nf4_gemv.restype = ctypes.c_int
_lib.nf4_gemv_ex.argtypes = [_P, _P, _P, _P, ctypes.c_float, _I64, _I64, _I32, _I32, _P, _I32, _P, _P,
                             ctypes.c_int, _P]
_lib.nf4_gemv_ex.restype = ctypes.c_int


class _GemvNode(ctypes.Structure):
    """nf4_gemv_node of include/nf4.h."""
    _fields_ = [("packed", _P), ("absmax_q", _P), ("absmax2", _P), ("code2", _P),
                ("offset", ctypes.c_float), ("N", _I64), ("K", _I64), ("blocksize", _I32),
                ("s2_blocksize", _I32), ("bias", _P), ("input", _I32), ("y", _P),
                ("y_dtype", ctypes.c_int)]


_lib.nf4_step_create.argtypes = [ctypes.POINTER(_GemvNode), _I32, _P, _I32, ctypes.POINTER(_P)]
_lib.nf4_step_create.restype = ctypes.c_int
_lib.nf4_step_launch.argtypes = [_P, _P]
_lib.nf4_step_launch.restype = ctypes.c_int
_lib.nf4_step_kernel_count.argtypes = [_P, ctypes.POINTER(_I32)]
_lib.nf4_step_kernel_count.restype = ctypes.c_int
_lib.nf4_step_destroy.argtypes = [_P]
_lib.nf4_step_destroy.restype = ctypes.c_int
_lib.nf4_quantize_workspace_size.argtypes = [_I64, _I32, _I32]
_lib.nf4_quantize_workspace_size.restype = ctypes.c_size_t
_lib.nf4_quantize.argtypes = [_P, _I64, _I32, _I32, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
_lib.nf4_quantize.restype = ctypes.c_int
_lib.nf4_quantize_noalloc.argtypes = [_P, _I64, _I32, _I32, _P, _P, _P, _P, _P, _P]
_lib.nf4_quantize_noalloc.restype = ctypes.c_int
_lib.nf4_device_error_flags.argtypes = [ctypes.POINTER(ctypes.c_uint)]
_lib.nf4_device_error_flags.restype = ctypes.c_int

NF4_BF16 = 0
NF4_FP16 = 1
NF4_F32 = 2
_DTYPES = {torch.bfloat16: NF4_BF16, torch.float16: NF4_FP16}
_Y_DTYPES = {torch.bfloat16: NF4_BF16, torch.float16: NF4_FP16, torch.float32: NF4_F32}


class NF4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        self.cuda_error = _lib.nf4_last_cuda_error() if status == 7 else 0
        msg = f"{where}: {nf4_status_string(status)}"
        if self.cuda_error:
            msg += f" (cudaError {self.cuda_error})"
        super().__init__(msg)


def nf4_version() -> int:
    return int(_lib.nf4_version())


def nf4_status_string(status: int) -> str:
    return _lib.nf4_status_string(int(status)).decode()


def nf4_device_error_flags() -> int:
    """Read and clear the device-side error flags (bit 0: a bounded wait ran out)."""
    f = ctypes.c_uint(0)
    _check(_lib.nf4_device_error_flags(ctypes.byref(f)), "nf4_device_error_flags")
    return int(f.value)


def _check(status: int, where: str) -> None:
    if status != 0:
        raise NF4Error(status, where)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: torch.Tensor | None, name: str, dtype, numel: int | None = None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} has {t.numel()} elements, needs {numel}")
    return t.data_ptr() if t.numel() > 0 else None


@dataclass
class NF4Weight:
    """A double-quantized NF4 tensor resident on the GPU (layout of include/nf4.h)."""
    packed: torch.Tensor      # uint8 [ceil(n/2)]
    absmax_q: torch.Tensor    # uint8 [nblocks]
    absmax2: torch.Tensor     # float16 [ngroups]
    code2: torch.Tensor       # float16 [256]
    offset: float             # binary32 value (host copy)
    n: int
    shape: tuple
    blocksize: int = 64
    s2_blocksize: int = 256

    def nblocks(self) -> int:
        return (self.n + self.blocksize - 1) // self.blocksize


def _sizes(n: int, blocksize: int, s2_blocksize: int):
    nb = (n + blocksize - 1) // blocksize
    return (n + 1) // 2, nb, (nb + s2_blocksize - 1) // s2_blocksize


def nf4_dequant(packed, absmax_q, absmax2, code2, offset: float, n: int, blocksize: int = 64,
                s2_blocksize: int = 256, out: torch.Tensor | None = None,
                out_dtype: torch.dtype = torch.bfloat16, stream=None) -> torch.Tensor:
    """Dequantize n NF4 elements to bf16/fp16 (bit-exact formula of include/nf4.h)."""
    if out_dtype not in _DTYPES:
        raise TypeError("out_dtype must be torch.bfloat16 or torch.float16")
    nbytes, nb, ng = _sizes(n, blocksize, s2_blocksize) if n > 0 else (0, 0, 0)
    if out is None:
        out = torch.empty(n, dtype=out_dtype, device=packed.device)
    st = _lib.nf4_dequant(_ptr(packed, "packed", torch.uint8, nbytes),
                          _ptr(absmax_q, "absmax_q", torch.uint8, nb),
                          _ptr(absmax2, "absmax2", torch.float16, ng),
                          _ptr(code2, "code2", torch.float16, 256), float(offset), int(n),
                          int(blocksize), int(s2_blocksize), _ptr(out, "out", out_dtype, n),
                          _DTYPES[out_dtype], _stream(stream))
    _check(st, "nf4_dequant")
    return out


def nf4_gemv(packed, absmax_q, absmax2, code2, offset: float, N: int, K: int, x: torch.Tensor,
             y: torch.Tensor | None = None, blocksize: int = 64, s2_blocksize: int = 256,
             stream=None) -> torch.Tensor:
    """y[b, r] = sum_k W_hat[r, k] x[b, k] for x bf16 [batch, K]; returns fp32 [batch, N]."""
    if x.dim() == 1:
        x = x.view(1, -1)
    batch = x.shape[0]
    if x.shape[1] != K:
        raise ValueError(f"x has {x.shape[1]} columns, expected K={K}")
    n = N * K
    nbytes, nb, ng = _sizes(n, blocksize, s2_blocksize) if n > 0 else (0, 0, 0)
    if y is None:
        y = torch.empty((batch, N), dtype=torch.float32, device=x.device)
    st = _lib.nf4_gemv(_ptr(packed, "packed", torch.uint8, nbytes),
                       _ptr(absmax_q, "absmax_q", torch.uint8, nb),
                       _ptr(absmax2, "absmax2", torch.float16, ng),
                       _ptr(code2, "code2", torch.float16, 256), float(offset), int(N), int(K),
                       int(blocksize), int(s2_blocksize), _ptr(x, "x", torch.bfloat16, batch * K),
                       int(batch), _ptr(y, "y", torch.float32, batch * N), _stream(stream))
    _check(st, "nf4_gemv")
    return y


def nf4_gemv_ex(packed, absmax_q, absmax2, code2, offset: float, N: int, K: int, x: torch.Tensor,
                bias: torch.Tensor | None = None, y: torch.Tensor | None = None,
                out_dtype: torch.dtype = torch.bfloat16, blocksize: int = 64,
                s2_blocksize: int = 256, stream=None) -> torch.Tensor:
    """y[b, r] = round(fp32(sum_k W_hat[r, k] x[b, k] + bias[r])) in out_dtype (bf16, fp16 or
    fp32); bias (optional) is [N] of out_dtype. Returns y [batch, N]."""
    if out_dtype not in _Y_DTYPES:
        raise TypeError("out_dtype must be torch.bfloat16, torch.float16 or torch.float32")
    if x.dim() == 1:
        x = x.view(1, -1)
    batch = x.shape[0]
    if x.shape[1] != K:
        raise ValueError(f"x has {x.shape[1]} columns, expected K={K}")
    n = N * K
    nbytes, nb, ng = _sizes(n, blocksize, s2_blocksize) if n > 0 else (0, 0, 0)
    if y is None:
        y = torch.empty((batch, N), dtype=out_dtype, device=x.device)
    st = _lib.nf4_gemv_ex(_ptr(packed, "packed", torch.uint8, nbytes),
                          _ptr(absmax_q, "absmax_q", torch.uint8, nb),
                          _ptr(absmax2, "absmax2", torch.float16, ng),
                          _ptr(code2, "code2", torch.float16, 256), float(offset), int(N), int(K),
                          int(blocksize), int(s2_blocksize), _ptr(x, "x", torch.bfloat16, batch * K),
                          int(batch), _ptr(bias, "bias", out_dtype, N),
                          _ptr(y, "y", out_dtype, batch * N), _Y_DTYPES[out_dtype], _stream(stream))
    _check(st, "nf4_gemv_ex")
    return y


class DecodeStep:
    """A fixed sequence of fused GEMV nodes recorded once into a CUDA graph
    (nf4_step_create) and replayed with ``launch()`` (nf4_step_launch).

    ``nodes`` is a list of dicts: ``weight`` (NF4Weight of shape (N, K)), ``y`` (CUDA tensor
    [batch, N] of bf16, fp16 or fp32), optional ``bias`` ([N], y's dtype) and ``input`` (-1 for
    the step input ``x``, else the index of an earlier node whose bf16 ``y`` is this node's x).
    The tensors are referenced, not copied: replays read their current contents.
    """

    def __init__(self, nodes: list, x: torch.Tensor):
        if x.dim() == 1:
            x = x.view(1, -1)
        batch = x.shape[0]
        arr = (_GemvNode * len(nodes))()
        self._keep = [x]
        for i, nd in enumerate(nodes):
            wt, y = nd["weight"], nd["y"]
            N, K = wt.shape
            inp = int(nd.get("input", -1))
            if y.dtype not in _Y_DTYPES:
                raise TypeError(f"node {i}: y must be bf16, fp16 or fp32")
            if inp == -1 and x.shape[1] != K:
                raise ValueError(f"node {i}: x has {x.shape[1]} columns, expected K={K}")
            n = N * K
            nbytes, nb, ng = _sizes(n, wt.blocksize, wt.s2_blocksize) if n > 0 else (0, 0, 0)
            bias = nd.get("bias")
            arr[i] = _GemvNode(_ptr(wt.packed, "packed", torch.uint8, nbytes),
                               _ptr(wt.absmax_q, "absmax_q", torch.uint8, nb),
                               _ptr(wt.absmax2, "absmax2", torch.float16, ng),
                               _ptr(wt.code2, "code2", torch.float16, 256), float(wt.offset), N, K,
                               wt.blocksize, wt.s2_blocksize, _ptr(bias, "bias", y.dtype, N), inp,
                               _ptr(y, "y", y.dtype, batch * N), _Y_DTYPES[y.dtype])
            self._keep += [wt, y, bias]
        h = _P()
        st = _lib.nf4_step_create(arr, len(nodes), _ptr(x, "x", torch.bfloat16, x.numel()),
                                  int(batch), ctypes.byref(h))
        _check(st, "nf4_step_create")
        self._h = h

    def launch(self, stream=None) -> None:
        _check(_lib.nf4_step_launch(self._h, _stream(stream)), "nf4_step_launch")

    def kernel_count(self) -> int:
        """Kernel launches per replay (grouped nodes share one)."""
        n = _I32(0)
        _check(_lib.nf4_step_kernel_count(self._h, ctypes.byref(n)), "nf4_step_kernel_count")
        return int(n.value)

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            _lib.nf4_step_destroy(self._h)
        self._h = None

    def __del__(self):
        self.close()


def nf4_quantize_workspace_size(n: int, blocksize: int = 64, s2_blocksize: int = 256) -> int:
    return int(_lib.nf4_quantize_workspace_size(int(n), int(blocksize), int(s2_blocksize)))


def nf4_quantize(w: torch.Tensor, code2: torch.Tensor, blocksize: int = 64, s2_blocksize: int = 256,
                 workspace: torch.Tensor | None = None, stream=None) -> NF4Weight:
    """NF4 + double quantization of a float32 CUDA tensor (flattened)."""
    n = w.numel()
    nbytes, nb, ng = _sizes(n, blocksize, s2_blocksize) if n > 0 else (0, 0, 0)
    dev = w.device
    packed = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    absmax_q = torch.empty(nb, dtype=torch.uint8, device=dev)
    absmax2 = torch.empty(ng, dtype=torch.float16, device=dev)
    offset = torch.zeros(1, dtype=torch.float32, device=dev)
    ws_bytes = nf4_quantize_workspace_size(n, blocksize, s2_blocksize)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 8), dtype=torch.uint8, device=dev)
    st = _lib.nf4_quantize(_ptr(w.reshape(-1), "w", torch.float32, n),
                           int(n), int(blocksize), int(s2_blocksize),
                           _ptr(code2, "code2", torch.float16, 256), _ptr(packed, "packed", torch.uint8),
                           _ptr(absmax_q, "absmax_q", torch.uint8), _ptr(absmax2, "absmax2", torch.float16),
                           offset.data_ptr(), _ptr(workspace, "workspace", torch.uint8),
                           workspace.numel(), _stream(stream))
    _check(st, "nf4_quantize")
    return NF4Weight(packed, absmax_q, absmax2, code2, float(offset.item()) if n > 0 else 0.0, n,
                     tuple(w.shape), blocksize, s2_blocksize)


def nf4_quantize_noalloc(w: torch.Tensor, code2: torch.Tensor, blocksize: int = 64,
                         s2_blocksize: int = 256, stream=None) -> NF4Weight:
    """nf4_quantize with the library's fixed device scratch (no workspace argument)."""
    n = w.numel()
    nbytes, nb, ng = _sizes(n, blocksize, s2_blocksize) if n > 0 else (0, 0, 0)
    dev = w.device
    packed = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    absmax_q = torch.empty(nb, dtype=torch.uint8, device=dev)
    absmax2 = torch.empty(ng, dtype=torch.float16, device=dev)
    offset = torch.zeros(1, dtype=torch.float32, device=dev)
    st = _lib.nf4_quantize_noalloc(_ptr(w.reshape(-1), "w", torch.float32, n),
                                   int(n), int(blocksize), int(s2_blocksize),
                                   _ptr(code2, "code2", torch.float16, 256),
                                   _ptr(packed, "packed", torch.uint8),
                                   _ptr(absmax_q, "absmax_q", torch.uint8),
                                   _ptr(absmax2, "absmax2", torch.float16),
                                   offset.data_ptr(), _stream(stream))
    _check(st, "nf4_quantize_noalloc")
    return NF4Weight(packed, absmax_q, absmax2, code2, float(offset.item()) if n > 0 else 0.0, n,
                     tuple(w.shape), blocksize, s2_blocksize)


def dequant(wt: NF4Weight, out_dtype: torch.dtype = torch.bfloat16, out=None, stream=None):
    return nf4_dequant(wt.packed, wt.absmax_q, wt.absmax2, wt.code2, wt.offset, wt.n, wt.blocksize,
                       wt.s2_blocksize, out=out, out_dtype=out_dtype, stream=stream)


def gemv(wt: NF4Weight, x: torch.Tensor, y=None, stream=None, bias=None, out_dtype=None):
    """Fused GEMV of an N x K weight: fp32 y by default; with a bias or an out_dtype, the fused
    output stage of nf4_gemv_ex."""
    N, K = wt.shape
    if bias is None and out_dtype in (None, torch.float32):
        return nf4_gemv(wt.packed, wt.absmax_q, wt.absmax2, wt.code2, wt.offset, N, K, x, y=y,
                        blocksize=wt.blocksize, s2_blocksize=wt.s2_blocksize, stream=stream)
    return nf4_gemv_ex(wt.packed, wt.absmax_q, wt.absmax2, wt.code2, wt.offset, N, K, x, bias=bias,
                       y=y, out_dtype=out_dtype or torch.float32, blocksize=wt.blocksize,
                       s2_blocksize=wt.s2_blocksize, stream=stream)
