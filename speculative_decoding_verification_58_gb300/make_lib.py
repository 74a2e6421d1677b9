"""Build ``libspecverify.so`` in-tree for GB300 (sm_103a) with nvcc.

One translation unit, one ``-gencode``; a cross-compile that needs no GPU.
The range-checking build (``-DSPEC_DEBUG``) compiles beside it.
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
# The same library with device-side range checks (-DSPEC_DEBUG).
LIB_DEBUG = os.path.join(HERE, "libspecverify_debug.so")
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


def _command(out: str, debug: bool, verbose_ptxas: bool) -> list[str]:
    cmd = [nvcc(), "-gencode", GENCODE, "-O3", "-lineinfo", "-std=c++17",
           "-Xcompiler", "-fPIC", "-shared", "-I", INCLUDE,
           *SOURCES, "-o", out, "-ldl"]
    if debug:
        cmd.insert(1, "-DSPEC_DEBUG")
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def _stale(path: str) -> bool:
    if not os.path.exists(path):
        return True
    newest = max(os.path.getmtime(f) for f in _inputs())
    return os.path.getmtime(path) < newest


def build(force: bool = False, verbose_ptxas: bool = False, debug: bool = False) -> str:
    """Compile one library (the range-checking one with debug) unless it is
    newer than every source; return its path."""
    lib = LIB_DEBUG if debug else LIB
    if not force and not _stale(lib):
        return lib
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.run(_command(tmp, debug, verbose_ptxas), check=True)
    os.replace(tmp, lib)
    return lib


def build_all(force: bool = False) -> list[str]:
    """Compile the release and the range-checking library side by side."""
    jobs = []
    for lib, debug in ((LIB, False), (LIB_DEBUG, True)):
        if force or _stale(lib):
            tmp = lib + f".tmp{os.getpid()}"
            jobs.append((subprocess.Popen(_command(tmp, debug, False)), tmp, lib))
    failed = []
    for proc, tmp, lib in jobs:
        if proc.wait() != 0:
            failed.append(lib)
        else:
            os.replace(tmp, lib)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    return [LIB, LIB_DEBUG]


if __name__ == "__main__":
    print(build(force=True, verbose_ptxas="-v" in sys.argv))
