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


# The same library with device-side range checks of every stream-K workspace access
# (FA_DEBUG): an index outside the workspace's layout records FA_ERR_BOUNDS and the access
# is skipped. Used by the tests; the release library compiles the checks out.
DEBUG_LIB = os.path.join(PKG, "libfa_debug.so")
DEBUG_FLAGS = ("-DFA_DEBUG",)


def _stale(out: str) -> bool:
    return not os.path.exists(out) or any(os.path.getmtime(out) < os.path.getmtime(d) for d in DEPS)


def build(force: bool = False, verbose: bool = False, out: str = LIB, extra=()) -> str:
    return build_many([(out, extra)], force=force, verbose=verbose)[0]


def build_many(targets, force: bool = False, verbose: bool = False) -> list[str]:
    """Compile each (output, extra flags) target that is stale, all nvcc runs at once."""
    procs = []
    for out, extra in targets:
        if force or _stale(out):
            tmp = out + f".tmp{os.getpid()}"
            cmd = compile_cmd(tmp, (*extra, "-Xptxas", "-v") if verbose else extra)
            procs.append((out, tmp, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                                     text=True)))
    failed = []
    for out, tmp, pr in procs:
        so, se = pr.communicate()
        if pr.returncode != 0:
            sys.stderr.write(so + se)
            failed.append(os.path.basename(out))
            continue
        if verbose:
            sys.stderr.write(se)
        os.replace(tmp, out)
    if failed:
        raise RuntimeError(f"nvcc failed building {', '.join(failed)}")
    return [out for out, _ in targets]


def build_all(force: bool = False) -> list[str]:
    """The release library and its range-checked twin."""
    return build_many([(LIB, ()), (DEBUG_LIB, DEBUG_FLAGS)], force=force)


if __name__ == "__main__":
    if "--all" in sys.argv:
        build_all(force="--force" in sys.argv)
    else:
        build(force="--force" in sys.argv, verbose="-v" in sys.argv)
