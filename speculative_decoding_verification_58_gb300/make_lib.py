"""Build ``libspecverify.so`` in-tree for GB300 (sm_103a) with nvcc.

One translation unit, one ``-gencode``; a cross-compile that needs no GPU.
"""

from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libspecverify.so")
SOURCES = [os.path.join(CSRC, "spec_verify.cu")]
GENCODE = "arch=compute_103a,code=sm_103a"


def _inputs() -> list[str]:
    files = list(SOURCES)
    for d in (CSRC, INCLUDE):
        for name in os.listdir(d):
            if name.endswith((".cuh", ".h", ".cu")):
                files.append(os.path.join(d, name))
    return files


def nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cuda, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile the library unless it is newer than every source; return its path."""
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(f) for f in _inputs())
        if os.path.getmtime(LIB) >= newest:
            return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), "-gencode", GENCODE, "-O3", "-lineinfo", "-std=c++17",
           "-Xcompiler", "-fPIC", "-shared", "-I", INCLUDE,
           *SOURCES, "-o", tmp, "-ldl"]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose_ptxas="-v" in sys.argv))
