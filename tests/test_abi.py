"""The C ABI without a GPU: the library loads, exports every symbol that
include/nf4.h declares, and rejects bad arguments on the host before any CUDA
call (so these calls are safe on a machine without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nf4.h")

OK, ERR_NULL, ERR_SIZE, ERR_BS, ERR_ALIGN, ERR_DTYPE, ERR_BATCH, ERR_CUDA, ERR_WS = range(9)


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__._build_module().build()
    import w4a16_gemv_gb300 as nf4
    return nf4._lib


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"NF4_API\s+[\w\s\*]+?\b(nf4_\w+)\s*\(", text)


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == {"nf4_version", "nf4_status_string", "nf4_last_cuda_error", "nf4_dequant",
                          "nf4_gemv", "nf4_gemv_ex", "nf4_quantize_workspace_size", "nf4_quantize",
                          "nf4_device_error_flags", "nf4_quantize_noalloc", "nf4_step_create",
                          "nf4_step_launch", "nf4_step_destroy", "nf4_step_kernel_count"}
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    text = open(HEADER).read()
    codes = dict((m.group(1), int(m.group(2))) for m in re.finditer(r"(NF4_(?:OK|ERR_\w+))\s*=\s*(\d+)", text))
    assert codes["NF4_OK"] == 0 and len(codes) == 9
    for name, v in codes.items():
        s = lib.nf4_status_string(v).decode()
        assert s.startswith(name), (name, s)
    assert lib.nf4_status_string(99).decode().startswith("NF4: unknown")
    assert lib.nf4_version() == 100
    assert lib.nf4_last_cuda_error() == 0
    assert lib.nf4_device_error_flags(None) == ERR_NULL


A = 0x100000  # a fake, well-aligned address: never dereferenced by these calls
P = ctypes.c_void_p


def dq(lib, n=128, packed=A, absmax_q=A, absmax2=A, code2=A, out=A, bs=64, s2=256, dtype=0):
    return lib.nf4_dequant(P(packed), P(absmax_q), P(absmax2), P(code2), 0.5, n, bs, s2, P(out),
                           dtype, None)


def gv(lib, N=16, K=64, x=A, y=A, batch=1, bs=64, s2=256, packed=A):
    return lib.nf4_gemv(P(packed), P(A), P(A), P(A), 0.0, N, K, bs, s2, P(x), batch, P(y), None)


def test_dequant_argument_errors(lib):
    assert dq(lib, n=-1) == ERR_SIZE
    assert dq(lib, n=(1 << 40) + 1) == ERR_SIZE
    for bs in (0, 1, 3, 48, 65, 1 << 21, -64):
        assert dq(lib, bs=bs) == ERR_BS, bs
    for s2 in (0, 3, 255, 1 << 21):
        assert dq(lib, s2=s2) == ERR_BS, s2
    assert dq(lib, dtype=2) == ERR_DTYPE
    assert dq(lib, dtype=-1) == ERR_DTYPE
    assert dq(lib, n=0, packed=0, absmax_q=0, absmax2=0, code2=0, out=0) == OK
    assert dq(lib, packed=0) == ERR_NULL
    assert dq(lib, absmax_q=0) == ERR_NULL
    assert dq(lib, absmax2=0) == ERR_NULL
    assert dq(lib, code2=0) == ERR_NULL
    assert dq(lib, out=0) == ERR_NULL
    assert dq(lib, out=A + 1) == ERR_ALIGN
    assert dq(lib, absmax2=A + 1) == ERR_ALIGN
    assert dq(lib, code2=A + 3) == ERR_ALIGN


def test_gemv_argument_errors(lib):
    assert gv(lib, N=-1) == ERR_SIZE
    assert gv(lib, K=-2) == ERR_SIZE
    assert gv(lib, K=63) == ERR_SIZE
    assert gv(lib, N=1 << 30, K=1 << 12) == ERR_SIZE
    assert gv(lib, bs=96) == ERR_BS
    for b in (0, 65, -1):
        assert gv(lib, batch=b) == ERR_BATCH, b
    assert gv(lib, N=0, y=0, x=0) == OK
    assert gv(lib, y=0) == ERR_NULL
    assert gv(lib, x=0) == ERR_NULL
    assert gv(lib, packed=0) == ERR_NULL
    assert gv(lib, y=A + 2) == ERR_ALIGN
    assert gv(lib, x=A + 1) == ERR_ALIGN


def test_gemv_ex_argument_errors(lib):
    def gx(N=16, K=64, x=A, y=A, bias=0, dtype=0, batch=1):
        return lib.nf4_gemv_ex(P(A), P(A), P(A), P(A), 0.0, N, K, 64, 256, P(x), batch, P(bias),
                               P(y), dtype, None)
    for d in (3, -1, 7):
        assert gx(dtype=d) == ERR_DTYPE, d
    assert gx(N=-1, dtype=3) == ERR_SIZE  # sizes are checked first
    assert gx(batch=65) == ERR_BATCH
    assert gx(N=0, y=0, x=0, dtype=2) == OK
    assert gx(y=0) == ERR_NULL
    assert gx(x=0, bias=A) == ERR_NULL
    # y and bias aligned to the output element size (2 bytes, or 4 for binary32)
    assert gx(y=A + 1, dtype=0) == ERR_ALIGN
    assert gx(y=A + 2, dtype=2) == ERR_ALIGN
    assert gx(bias=A + 1, dtype=1) == ERR_ALIGN
    assert gx(bias=A + 2, dtype=2) == ERR_ALIGN
    assert gx(x=A + 1, y=A + 2, bias=A + 6, dtype=0) == ERR_ALIGN  # x misaligned


def test_quantize_argument_errors_and_workspace_size(lib):
    lib.nf4_quantize_workspace_size.restype = ctypes.c_size_t
    ws = lib.nf4_quantize_workspace_size
    assert ws(0, 64, 256) == 0 and ws(-5, 64, 256) == 0 and ws(100, 63, 256) == 0
    # n = 64*256*3 + 1: 769 blocks (256-aligned float array) + 4 groups of binary64
    assert ws(64 * 256 * 3 + 1, 64, 256) == 3328 + 4 * 8
    assert ws(1 << 20, 64, 256) == 16384 * 4 + 64 * 8

    def q(n=1000, w=A, ws_ptr=A, ws_bytes=1 << 20, off=A, bs=64):
        return lib.nf4_quantize(P(w), n, bs, 256, P(A), P(A), P(A), P(A), P(off), P(ws_ptr),
                                ctypes.c_size_t(ws_bytes), None)
    assert q(n=-1) == ERR_SIZE
    assert q(bs=5) == ERR_BS
    assert q(n=0, w=0) == OK
    assert q(w=0) == ERR_NULL
    assert q(off=0) == ERR_NULL
    assert q(w=A + 2) == ERR_ALIGN
    assert q(ws_ptr=0) == ERR_WS
    assert q(ws_bytes=16) == ERR_WS
    assert q(ws_ptr=A + 4) == ERR_WS


def test_quantize_noalloc_argument_errors_and_limit(lib):
    text = open(HEADER).read()
    limit = int(re.search(r"#define NF4_QUANTIZE_NOALLOC_SCRATCH_BYTES (\d+)", text).group(1))
    lib.nf4_quantize_workspace_size.restype = ctypes.c_size_t
    # the stated limit is exactly the workspace of 2^28 elements at 64/256
    assert lib.nf4_quantize_workspace_size(1 << 28, 64, 256) == limit
    assert lib.nf4_quantize_workspace_size((1 << 28) + 1, 64, 256) > limit

    def q(n=1000, w=A, off=A, bs=64, s2=256):
        return lib.nf4_quantize_noalloc(P(w), n, bs, s2, P(A), P(A), P(A), P(A), P(off), None)
    assert q(n=-1) == ERR_SIZE
    assert q(bs=5) == ERR_BS
    assert q(n=0, w=0) == OK
    assert q(w=0) == ERR_NULL
    assert q(off=0) == ERR_NULL
    assert q(w=A + 2) == ERR_ALIGN
    # too large for the fixed scratch: rejected on the host before any CUDA call
    assert q(n=(1 << 28) + 1) == ERR_WS
    assert q(n=1 << 30, bs=2, s2=1) == ERR_WS


def test_gemv_node_layout_matches_the_header(tmp_path):
    """The binding's nf4_gemv_node mirrors the C struct (offsets from a C
    program compiled against include/nf4.h)."""
    import shutil
    import subprocess
    import w4a16_gemv_gb300 as nf4
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = [f[0] for f in nf4._GemvNode._fields_]
    src = tmp_path / "layout.c"
    body = " ".join(f'printf("%zu ", offsetof(nf4_gemv_node, {f}));' for f in fields)
    src.write_text("#include <stdio.h>\n#include <stddef.h>\n#include \"nf4.h\"\n"
                   f"int main(void) {{ {body} printf(\"%zu\\n\", sizeof(nf4_gemv_node)); return 0; }}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    want = [getattr(nf4._GemvNode, f).offset for f in fields] + [ctypes.sizeof(nf4._GemvNode)]
    assert got == want


def test_step_argument_errors(lib):
    """nf4_step_create validates every node on the host before any CUDA call."""
    import w4a16_gemv_gb300 as nf4
    Node = nf4._GemvNode

    def node(N=32, K=64, inp=-1, y=A, dtype=0, bias=0):
        return Node(A, A, A, A, 0.0, N, K, 64, 256, bias or None, inp, y or None, dtype)

    def create(nodes, x=A, batch=1, n=None):
        arr = (Node * max(len(nodes), 1))(*nodes)
        h = P()
        st = lib.nf4_step_create(arr if nodes else None, len(nodes) if n is None else n,
                                 P(x), batch, ctypes.byref(h))
        assert h.value is None
        return st
    assert lib.nf4_step_create(None, 1, P(A), 1, None) == ERR_NULL
    assert create([], n=0) == ERR_SIZE
    assert create([], n=2) == ERR_NULL
    assert create([node(inp=0)]) == ERR_SIZE              # its own output
    assert create([node(inp=-2)]) == ERR_SIZE
    assert create([node(), node(inp=2)]) == ERR_SIZE      # a later node
    assert create([node(dtype=1), node(K=32, inp=0)]) == ERR_DTYPE  # input must be bf16
    assert create([node(N=48), node(K=64, inp=0)]) == ERR_SIZE      # K != N of the input
    assert create([node(), node(K=32, inp=0, y=0)]) == ERR_NULL
    assert create([node(), node(K=32, inp=0, dtype=5)]) == ERR_DTYPE
    assert create([node()], batch=65) == ERR_BATCH
    assert create([node()], x=0) == ERR_NULL
    assert create([node(y=A + 1)]) == ERR_ALIGN
    assert create([node(K=63)]) == ERR_SIZE
    assert lib.nf4_step_launch(None, None) == ERR_NULL
    assert lib.nf4_step_destroy(None) == OK
    assert lib.nf4_step_kernel_count(None, None) == ERR_NULL



def test_cuda_failure_is_reported_as_a_status(lib):
    """Failure detection on the host: on a machine without a usable GPU every
    CUDA call fails, which stands in for a failing launch. Calls with valid
    arguments return NF4_ERR_CUDA, record the CUDA error code, and leave the
    library usable (argument checks still answer). Skipped where a GPU is
    present: the fake addresses would then reach a kernel."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert dq(lib) == ERR_CUDA
    assert lib.nf4_last_cuda_error() != 0
    assert gv(lib) == ERR_CUDA
    assert lib.nf4_last_cuda_error() != 0
    assert dq(lib, bs=48) == ERR_BS      # host checks are unaffected
    assert gv(lib, batch=0) == ERR_BATCH


def test_calls_from_many_host_threads(lib):
    """The host side keeps no unsynchronised state: argument checks (and, on
    a machine without a usable GPU, the CUDA-failure path with its per-thread
    error record and the per-device caches it passes through) answer the same
    from eight threads at once as from one."""
    import threading

    import torch
    no_gpu = not torch.cuda.is_available()
    cases = [lambda: gv(lib, batch=0), lambda: gv(lib, K=63), lambda: gv(lib, x=0),
             lambda: gv(lib, bs=48), lambda: dq(lib, dtype=2), lambda: dq(lib, out=A + 1),
             lambda: gv(lib, N=0, x=0, y=0)]
    if no_gpu:
        cases += [lambda: gv(lib), lambda: dq(lib), lambda: gv(lib, batch=4), lambda: gv(lib, batch=16)]
    expected = [c() for c in cases]
    errors = []

    def worker(seed):
        order = list(range(len(cases))) * 50
        for i in order[seed::3] + order:
            got = cases[i]()
            if got != expected[i]:
                errors.append((seed, i, got, expected[i]))
            if no_gpu and got == ERR_CUDA and lib.nf4_last_cuda_error() == 0:
                errors.append((seed, i, "no CUDA error recorded"))

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors[:5]
