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
DEPS = SOURCES + [os.path.join(HERE, "csrc", f) for f in ("kernels.cuh", "ptx.cuh",
                                                              "varlen_tc.cuh", "prefill_tc.cuh")] + [
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


C_E2E_SRC = os.path.join(ROOT, "tests", "c_abi", "e2e_step.c")
C_E2E_EXE = os.path.join(HERE, "_build", "e2e_step")


def build_c_e2e(force=False):
    """Compiles the plain-C end-to-end driver (tests/c_abi/e2e_step.c)
    against libpagedkv.so and the CUDA runtime; returns the executable."""
    lib = build_library()
    if (not force and os.path.exists(C_E2E_EXE)
            and os.path.getmtime(C_E2E_EXE) >= max(os.path.getmtime(C_E2E_SRC),
                                                    os.path.getmtime(lib))):
        return C_E2E_EXE
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no C compiler")
    cuda_home = os.path.dirname(os.path.dirname(os.path.realpath(nvcc_path())))
    os.makedirs(os.path.dirname(C_E2E_EXE), exist_ok=True)
    cmd = [cc, "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", "-D_POSIX_C_SOURCE=199309L",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda_home, "include"),
           C_E2E_SRC, "-o", C_E2E_EXE, "-L", HERE, "-lpagedkv",
           "-L", os.path.join(cuda_home, "lib64"), "-lcudart",
           "-Wl,-rpath," + HERE, "-Wl,-rpath," + os.path.join(cuda_home, "lib64")]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"C driver build failed ({res.returncode}):\n{res.stderr}")
    return C_E2E_EXE


if __name__ == "__main__":
    extra = [a for a in sys.argv[1:] if a.startswith("-D")]
    if "--ptxas-v" in sys.argv:
        extra += ["-Xptxas", "-v"]
    build_library(force="--force" in sys.argv, verbose=True, extra=extra)
    print(LIB)
