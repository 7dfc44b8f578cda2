"""Build libspecverify.so in place with nvcc for sm_103a.

    python -m speculative_decoding_verification_31_gb300.build
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libspecverify.so")
CHECKED_LIB = os.path.join(PKG, "libspecverify_checked.so")  # SPECVERIFY_CHECKED: index checks
SOURCES = ["specverify.cu"]
DEPS = ["specverify.cu", "kernels.cuh", "vocab.cuh", "device_common.cuh", "philox.cuh", "lmhead.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home and os.path.exists(os.path.join(home, "bin", "nvcc")):
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def nvcc_command(out: str = LIB, extra=()) -> list:
    home = cuda_home()
    return [os.path.join(home, "bin", "nvcc"), *ARCH, "-O3", "-std=c++17", "-lineinfo",
            "--shared", "-Xcompiler", "-fPIC", "-cudart", "shared",
            f"-I{INCLUDE}", f"-I{CSRC}", "-Xlinker", f"-rpath={os.path.join(home, 'lib64')}",
            *extra, "-o", out, *[os.path.join(CSRC, s) for s in SOURCES]]


def up_to_date(out: str = LIB) -> bool:
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    deps = [os.path.join(CSRC, d) for d in DEPS] + [os.path.join(INCLUDE, "specverify.h")]
    return all(os.path.getmtime(d) <= t for d in deps)


def build(force: bool = False, verbose: bool = False, extra=(), checked: bool = True) -> str:
    """Compile libspecverify.so and (unless checked=False) its index-checked variant
    libspecverify_checked.so, the two nvcc runs side by side.  Returns the library's path."""
    jobs = []
    if force or not up_to_date(LIB):
        jobs.append(nvcc_command(out=LIB, extra=list(extra)))
    if checked and (force or not up_to_date(CHECKED_LIB)):
        jobs.append(nvcc_command(out=CHECKED_LIB, extra=["-DSPECVERIFY_CHECKED", *extra]))
    procs = []
    for cmd in jobs:
        if verbose:
            print(" ".join(cmd))
        procs.append((cmd, subprocess.Popen(cmd)))
    failed = [cmd for cmd, pr in procs if pr.wait() != 0]
    if failed:
        raise subprocess.CalledProcessError(1, failed[0])
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True,
          extra=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else [])
