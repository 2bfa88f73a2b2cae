"""nf4_quantize_noalloc (workspace in the library's fixed device array) against
nf4_quantize (caller workspace), both called through the C ABI: identical
outputs on consecutive calls with different inputs and block sizes, and at the
largest size the fixed array holds. Quantizer outputs are codes and bit
patterns, so the comparison is exact. This file is collected last so that it
also runs after every other GPU test in the same process."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIMIT = int(re.search(r"#define NF4_QUANTIZE_NOALLOC_SCRATCH_BYTES (\d+)",
                      open(os.path.join(ROOT, "include", "nf4.h")).read()).group(1))
P = ctypes.c_void_p


@pytest.fixture(scope="module")
def lib():
    import w4a16_gemv_gb300 as nf4
    lib = ctypes.CDLL(nf4.LIB_PATH)
    lib.nf4_quantize_noalloc.argtypes = [P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                         P, P, P, P, P, P]
    lib.nf4_quantize_noalloc.restype = ctypes.c_int
    lib.nf4_quantize.argtypes = [P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                 P, P, P, P, P, P, ctypes.c_size_t, P]
    lib.nf4_quantize.restype = ctypes.c_int
    lib.nf4_quantize_workspace_size.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]
    lib.nf4_quantize_workspace_size.restype = ctypes.c_size_t
    return lib


def _outputs(n, bs, s2):
    nb = (n + bs - 1) // bs
    ng = (nb + s2 - 1) // s2
    # filled with a pattern so that a missing write shows up
    return dict(packed=torch.full(((n + 1) // 2,), 0xA5, dtype=torch.uint8, device="cuda"),
                absmax_q=torch.full((nb,), 0x5A, dtype=torch.uint8, device="cuda"),
                absmax2=torch.full((ng,), -7.0, dtype=torch.float16, device="cuda"),
                offset=torch.full((1,), -3.0, dtype=torch.float32, device="cuda"))


def _noalloc(lib, w, code2, bs, s2):
    o = _outputs(w.numel(), bs, s2)
    st = lib.nf4_quantize_noalloc(P(w.data_ptr()), w.numel(), bs, s2, P(code2.data_ptr()),
                                  P(o["packed"].data_ptr()), P(o["absmax_q"].data_ptr()),
                                  P(o["absmax2"].data_ptr()), P(o["offset"].data_ptr()),
                                  P(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
    return o


def _with_workspace(lib, w, code2, bs, s2):
    o = _outputs(w.numel(), bs, s2)
    ws_bytes = lib.nf4_quantize_workspace_size(w.numel(), bs, s2)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    st = lib.nf4_quantize(P(w.data_ptr()), w.numel(), bs, s2, P(code2.data_ptr()),
                          P(o["packed"].data_ptr()), P(o["absmax_q"].data_ptr()),
                          P(o["absmax2"].data_ptr()), P(o["offset"].data_ptr()), P(ws.data_ptr()),
                          ws_bytes, P(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
    return o


def _same(a, b):
    for k in ("packed", "absmax_q"):
        assert torch.equal(a[k], b[k]), k
    assert torch.equal(a["absmax2"].view(torch.int16), b["absmax2"].view(torch.int16))
    assert torch.equal(a["offset"].view(torch.int32), b["offset"].view(torch.int32))


@pytest.fixture(scope="module")
def code2():
    return torch.from_numpy(synth.code2_linear().view(np.float16)).cuda()


def test_consecutive_calls_match_workspace_entry_point(lib, code2):
    c = synth.CONFIG1
    w1 = torch.from_numpy(synth.weights(c.seed, c.n, c.outlier_frac, c.outlier_seed)).cuda()
    w2 = torch.from_numpy(synth.weights(77, 64 * 256 * 37 + 65, 0.01, 78)).cuda()
    # two calls in a row on the same stream, different inputs and block sizes:
    # the second overwrites the scratch the first used
    a1 = _noalloc(lib, w1, code2, 64, 256)
    a2 = _noalloc(lib, w2, code2, 128, 4)
    b1 = _with_workspace(lib, w1, code2, 64, 256)
    b2 = _with_workspace(lib, w2, code2, 128, 4)
    torch.cuda.synchronize()
    _same(a1, b1)
    _same(a2, b2)
    # and the same input twice in a row gives the same result again
    a3 = _noalloc(lib, w1, code2, 64, 256)
    a4 = _noalloc(lib, w1, code2, 64, 256)
    torch.cuda.synchronize()
    _same(a3, b1)
    _same(a4, b1)


def test_largest_size_the_scratch_holds(lib, code2):
    n = 1 << 28
    assert lib.nf4_quantize_workspace_size(n, 64, 256) == LIMIT
    g = torch.Generator(device="cuda")
    g.manual_seed(91)
    w = torch.randn(n, generator=g, device="cuda", dtype=torch.float32) * 0.02
    a = _noalloc(lib, w, code2, 64, 256)
    b = _with_workspace(lib, w, code2, 64, 256)
    torch.cuda.synchronize()
    _same(a, b)
    del w, a, b
    torch.cuda.empty_cache()


def test_binding_name(code2):
    import w4a16_gemv_gb300 as nf4
    w = torch.from_numpy(synth.weights(5, 4096 + 3)).cuda()
    a = nf4.nf4_quantize_noalloc(w, code2)
    b = nf4.nf4_quantize(w, code2)
    torch.cuda.synchronize()
    assert torch.equal(a.packed, b.packed) and torch.equal(a.absmax_q, b.absmax_q)
    assert torch.equal(a.absmax2.view(torch.int16), b.absmax2.view(torch.int16))
    assert np.float32(a.offset).view(np.uint32) == np.float32(b.offset).view(np.uint32)
