"""Builds the CUDA library in-tree: invariant_rmsnorm_fwd_gb300/_lib/librmsnorm_bi.so.

sm_103a only (one -gencode), -fmad=false so no multiply-add is contracted
behind the explicit intrinsics, translation units compiled in parallel.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIBDIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIBDIR, "librmsnorm_bi.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-fmad=false", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fno-strict-aliasing", f"-I{INCLUDE}"]
SOURCES = ["rmsnorm_bi.cu", "rows_fwd.cu", "rows_dx.cu", "rows_dxdw.cu", "rows_adddxdw.cu", "gemm_dw.cu",
           "plan.cpp"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def _deps():
    out = [os.path.join(INCLUDE, "rmsnorm_bi.h"), __file__]
    out += [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    return out


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _build_into(out_lib: str, objdir: str, extra_flags=(), verbose: bool = False) -> str:
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(objdir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr, flush=True)
        return obj

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = out_lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out_lib)
    return out_lib


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and up_to_date():
        return LIB
    return _build_into(LIB, LIBDIR, extra_flags, verbose)


def build_test_variant(tag: str, defines: dict) -> str:
    """A separate copy of the library compiled with extra preprocessor defines,
    for tests only (e.g. a short wait limit); the product library is untouched.
    Written to _lib/variant_<tag>/librmsnorm_bi_<tag>.so."""
    d = os.path.join(LIBDIR, f"variant_{tag}")
    out = os.path.join(d, f"librmsnorm_bi_{tag}.so")
    if os.path.exists(out) and all(os.path.getmtime(p) <= os.path.getmtime(out) for p in _deps()):
        return out
    flags = [f"-D{k}={v}" if v is not None else f"-D{k}" for k, v in sorted(defines.items())]
    return _build_into(out, d, flags)


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "--ptxas" in sys.argv else []))
