"""Build libnf4.so in-tree with nvcc for sm_103a (one -gencode, sources in parallel)."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libnf4.so")
SOURCES = ("nf4_api.cu", "nf4_dequant.cu", "nf4_gemv.cu", "nf4_gemv_b1.cu", "nf4_gemv_stream.cu",
           "nf4_quantize.cu", "nf4_step.cu", "nf4_gemm_tc.cu")
GENCODE = "arch=compute_103a,code=sm_103a"


def nvcc_path() -> str:
    cand = shutil.which("nvcc")
    if cand:
        return cand
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    return os.path.join(home, "bin", "nvcc")


def nvcc_flags(extra: tuple[str, ...] = ()) -> list[str]:
    return ["-gencode", GENCODE, "-lineinfo", "-O3", "-std=c++17", "-ftz=false",
            "-prec-div=true", "-prec-sqrt=true", "-Xcompiler", "-fPIC,-O2,-fvisibility=hidden",
            "-I", INCLUDE, "-I", CSRC, *extra]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "nf4.h"),
                                                                  os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra: tuple[str, ...] = ()) -> str:
    """Compile every source to an object in parallel, then link libnf4.so."""
    if not force and not _stale():
        return LIB
    os.makedirs(OBJDIR, exist_ok=True)
    nvcc = nvcc_path()
    procs = []
    for src in SOURCES:
        obj = os.path.join(OBJDIR, src.replace(".cu", ".o"))
        cmd = [nvcc, *nvcc_flags(extra), "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, obj, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    objs = []
    failed = []
    for src, obj, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append((src, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"), file=sys.stderr)
        objs.append(obj)
    if failed:
        msg = "\n".join(f"--- {s}\n{o}" for s, o in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, "-gencode", GENCODE, "-shared", "-o", tmp, *objs]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
    print(LIB)
