"""Builds ``libpagedkv.so`` (in-tree, next to this file) with nvcc for sm_103a.

The library links the CUDA runtime dynamically (``-cudart shared``), so a
process that also loads PyTorch shares one runtime instance with it; the
rpath points at the toolkit's ``lib64`` for processes that load the library
first.
"""

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libpagedkv.so")
SOURCES = [os.path.join(HERE, "csrc", "pagedkv.cu")]
DEPS = SOURCES + [os.path.join(HERE, "csrc", f) for f in ("kernels.cuh", "ptx.cuh")] + [
    os.path.join(ROOT, "include", "pagedkv.h")]


def nvcc_path():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def up_to_date():
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build_library(force=False, verbose=False, extra=()):
    if not force and up_to_date():
        return LIB
    nvcc = nvcc_path()
    cuda_home = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    tmp = LIB + ".tmp"
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo", "-O3", "-std=c++17",
           "-shared", "-Xcompiler", "-fPIC", "-cudart", "shared",
           "-Xlinker", f"-rpath,{os.path.join(cuda_home, 'lib64')}",
           "-I", os.path.join(ROOT, "include"), "-o", tmp, *SOURCES, *extra]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{res.stdout}\n{res.stderr}")
    if verbose and (res.stdout or res.stderr):
        print(res.stdout, res.stderr, file=sys.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    extra = [a for a in sys.argv[1:] if a.startswith("-D")]
    if "--ptxas-v" in sys.argv:
        extra += ["-Xptxas", "-v"]
    build_library(force="--force" in sys.argv, verbose=True, extra=extra)
    print(LIB)
