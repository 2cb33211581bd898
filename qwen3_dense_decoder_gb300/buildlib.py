"""Build the sm_103a CUDA library (libq3.so) in-tree with nvcc.

Each translation unit under csrc/ compiles in parallel for
``-gencode arch=compute_103a,code=sm_103a``; the objects link into one shared
library with the CUDA runtime linked statically, so the library loads on a
host without a GPU (the CPU tests check its exported symbols).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libq3.so")

SOURCES = ["runtime.cu", "k_gemm.cu", "k_gemv.cu", "k_attn.cu", "k_attn_prefill.cu", "k_misc.cu",
           "noalloc.cu", "k_decode.cu", "k_attn_tc.cu", "k_gemv_a4.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", INCLUDE]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libq3.so")
    return path


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "q3.h"))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None) -> str:
    """Compile csrc/*.cu into libq3.so (skipped when up to date)."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    extra = list(extra or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


FAULT_LIB = os.path.join(BUILD, "faults", "libq3_faults.so")


def build_fault_variant(force: bool = False) -> str:
    """The test build of the mutation gate: runtime.cu compiled with
    -DQ3_TEST_FAULTS (the host then plants the addressing fault named by the
    Q3_FAULT environment variable in what it uploads) and linked with the
    product's kernel objects into a separate library.  Never the product."""
    build()
    out_dir = os.path.dirname(FAULT_LIB)
    obj = os.path.join(out_dir, "runtime.o")
    src = os.path.join(CSRC, "runtime.cu")
    if not force and os.path.exists(FAULT_LIB) and os.path.getmtime(FAULT_LIB) >= os.path.getmtime(LIB):
        return FAULT_LIB
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    r = subprocess.run([cc, *ARCH, *FLAGS, "-DQ3_TEST_FAULTS", "-c", src, "-o", obj], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on runtime.cu (fault build):\n{r.stdout}\n{r.stderr}")
    objs = [obj] + [os.path.join(BUILD, f.replace(".cu", ".o")) for f in SOURCES if f != "runtime.cu"]
    tmp = FAULT_LIB + f".tmp{os.getpid()}"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed (fault build):\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, FAULT_LIB)
    return FAULT_LIB


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas" in sys.argv else None
    print(build(force=True, verbose=v or bool(extra), extra=extra))
