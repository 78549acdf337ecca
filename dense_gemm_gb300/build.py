"""Build libgemm_f16.so in-tree with nvcc for sm_103a.

    python -m dense_gemm_gb300.build [--force]

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
SOURCES = [os.path.join(CSRC, "gemm_f16.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in ("gemm_kernel.cuh", "gemm_pair.cuh", "ptx.cuh")] + \
    [os.path.join(INCLUDE, "gemm_f16.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def command(out: str, verbose_ptxas: bool = False):
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-Wall", "-I", INCLUDE, "-I", CSRC, "-o", out, *SOURCES]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in DEPENDS)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run(command(tmp, verbose_ptxas), check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
