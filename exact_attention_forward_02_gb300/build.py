"""Build libfa.so (the CUDA library behind the C ABI in include/fa_fwd.h) in-tree.

One translation unit, one -gencode (sm_103a), linked against the static CUDA runtime;
the driver entry point for TMA tensor maps is fetched at run time, so no libcuda link.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "fa_fwd.cu")
DEPS = [SRC, os.path.join(PKG, "csrc", "sm103_ptx.cuh"), os.path.join(PKG, "csrc", "fa_bwd.cuh"),
        os.path.join(PKG, "csrc", "philox.cuh"), os.path.join(PKG, "csrc", "fa_fwd_kernel.cuh"),
        os.path.join(ROOT, "include", "fa_fwd.h")]
LIB = os.path.join(PKG, "libfa.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def compile_cmd(out: str, extra=()) -> list[str]:
    return [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
            "-I", os.path.join(ROOT, "include"), "-I", os.path.join(PKG, "csrc"),
            *extra, SRC, "-o", out]


def build(force: bool = False, verbose: bool = False, out: str = LIB, extra=()) -> str:
    stale = force or not os.path.exists(out) or any(
        os.path.getmtime(out) < os.path.getmtime(d) for d in DEPS)
    if stale:
        tmp = out + f".tmp{os.getpid()}"
        cmd = compile_cmd(tmp, (*extra, "-Xptxas", "-v") if verbose else extra)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("nvcc failed building libfa.so")
        if verbose:
            sys.stderr.write(r.stderr)
        os.replace(tmp, out)
    return out


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
