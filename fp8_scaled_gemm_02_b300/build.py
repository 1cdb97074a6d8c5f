"""Build libfp8sgemm.so in-tree with nvcc for sm_103a (B300).

The library is a single translation unit (csrc/fp8sgemm.cu) exporting the C
ABI declared in include/fp8sgemm.h.  nvcc cross-compiles without a GPU.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
SRC = os.path.join(CSRC, "fp8sgemm.cu")
LIB = os.path.join(HERE, "libfp8sgemm.so")
HEADER = os.path.join(ROOT, "include", "fp8sgemm.h")

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-shared", "-Xcompiler", "-fPIC,-fvisibility=hidden",
         "-Xcompiler", "-Wall", "--expt-relaxed-constexpr"]


def sources():
    out = [HEADER]
    for f in sorted(os.listdir(CSRC)):
        if f.endswith((".cu", ".cuh", ".h")):
            out.append(os.path.join(CSRC, f))
    return out


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in sources())


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    if force or needs_build():
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [NVCC, *ARCH, *FLAGS, "-o", tmp, SRC]
        if verbose_ptxas:
            cmd.insert(1, "-Xptxas=-v")
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
