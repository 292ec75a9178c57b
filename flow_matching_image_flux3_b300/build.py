"""Build libflux3.so in-tree with nvcc for sm_103a (B300)."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libflux3.so")
SRC = os.path.join(HERE, "csrc", "flux3.cu")
DEPS = [os.path.join(HERE, "csrc", f) for f in ("flux3.cu", "sm103.cuh", "gemm.cuh", "attention.cuh", "simt.cuh")] + \
    [os.path.join(ROOT, "include", "flux3.h")]


def nvcc_path() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found")
    return p


def command(out: str = LIB, extra=()) -> list:
    return [nvcc_path(), "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
            "-Xcompiler", "-fPIC", "-shared", "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"),
            *extra, "-o", out, SRC]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    if not force and up_to_date():
        return LIB
    cmd = command(extra=extra)
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + r.stdout + r.stderr)
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, file=sys.stderr)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, extra=tuple(a for a in sys.argv[1:] if a != "--force"))
