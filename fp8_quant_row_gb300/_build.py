"""Ahead-of-time build of libfp8q.so for sm_103a (nvcc, in-tree; no JIT, no cmake)."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libfp8q.so")
SOURCES = [os.path.join(CSRC, "fp8q_capi.cu")]


def deps() -> list:
    """Every file the build reads: all of csrc/ (sources and the headers they include) and
    the public headers. Taken from the directories at call time, so a new or renamed kernel
    header can never be left out of the staleness check."""
    out = []
    for d in (CSRC, INCLUDE):
        for f in sorted(os.listdir(d)):
            if f.endswith((".cu", ".cuh", ".h", ".hpp")):
                out.append(os.path.join(d, f))
    return out


ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
# The CUDA runtime is linked shared (soname libcudart.so.13): inside a process that already
# loaded torch, the library binds to the same runtime instance torch uses.
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-Wall", "-cudart", "shared",
              "-Xlinker", f"-rpath,{os.path.join(CUDA_HOME, 'lib64')}", f"-I{INCLUDE}"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"),
                 os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc"),
                 shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set CUDA_HOME or NVCC)")


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in deps())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA sources into fp8_quant_row_gb300/libfp8q.so (sm_103a only)."""
    if not force and up_to_date():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc_path(), *ARCH, *NVCC_FLAGS, "-o", tmp, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB
