"""Build libh3qk.so (the CUDA path, sm_103a only) in the package directory.

    python -m video_vae_decoder_qkv_gb300.build [--force] [-v]

nvcc flags: one -gencode for sm_103a; -fmad=false, IEEE division and square
root, no flush-to-zero (the kernels also use explicit _rn intrinsics at every
rounding point, so results do not depend on contraction); cudart linked
statically so the library needs nothing but the driver.
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
LIB = os.path.join(PKG, "libh3qk.so")
SOURCES = [os.path.join(CSRC, "h3qk_api.cu"), os.path.join(CSRC, "h3qk_vae_ops.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "h3qk_kernels.cuh"), os.path.join(CSRC, "h3qk_internal.h"),
                  os.path.join(INCLUDE, "h3qk.h")]

NVCC_FLAGS = [
    "-O3", "-std=c++17", "--threads", "0",
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo",
    "-fmad=false", "-prec-div=true", "-prec-sqrt=true", "-ftz=false",
    "-Xcompiler", "-fPIC", "-shared",
    "-cudart", "static",
]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None) -> str:
    if not force and up_to_date():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc_path(), *NVCC_FLAGS, *(extra or []), "-I", INCLUDE, "-I", CSRC, "-o", tmp, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
