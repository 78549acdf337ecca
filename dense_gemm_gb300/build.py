"""Build libgemm_f16.so in-tree with nvcc for sm_103a.

    python -m dense_gemm_gb300.build [--force] [--debug]

--debug builds libgemm_f16_debug.so instead: the same kernels with device-side
bounds and alignment checks (GEMM_DEBUG) that report GEMM_ERR_CHECK instead of
trapping. The binding loads it when GEMM_LIBRARY=debug.

One translation unit, one -gencode, static CUDA runtime; no cmake. The same
command works on x86-64 and aarch64 hosts.
"""
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libgemm_f16.so")
DEBUG_LIB = os.path.join(HERE, "libgemm_f16_debug.so")
SOURCES = [os.path.join(CSRC, "gemm_f16.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in ("gemm_kernel.cuh", "gemm_pair.cuh", "ptx.cuh")] + \
    [os.path.join(INCLUDE, "gemm_f16.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def command(out: str, verbose_ptxas: bool = False, debug: bool = False):
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-Wall", "-I", INCLUDE, "-I", CSRC, "-o", out, *SOURCES]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    if debug:
        cmd.insert(1, "-DGEMM_DEBUG")
    return cmd


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in DEPENDS)


def build(force: bool = False, verbose_ptxas: bool = False, debug: bool = False) -> str:
    lib = DEBUG_LIB if debug else LIB
    if not force and up_to_date(lib):
        return lib
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.run(command(tmp, verbose_ptxas, debug), check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, debug="--debug" in sys.argv))
