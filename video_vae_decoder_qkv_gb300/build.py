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
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libh3qk.so")
# The same sources with the kernels' device-side bounds checks compiled in
# (H3QK_DEBUG_CHECKS=1; include/h3qk.h, "Debug builds").
LIB_DEBUG = os.path.join(PKG, "libh3qk_debug.so")
# The kernel instances of each input type sit in their own translation unit
# so that the sources compile in parallel.
SOURCES = [os.path.join(CSRC, f) for f in ("h3qk_api.cu", "h3qk_host.cu", "h3qk_launch_bf16.cu",
                                           "h3qk_launch_fp16.cu", "h3qk_vae_ops.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("h3qk_kernels.cuh", "h3qk_launch.cuh", "h3qk_internal.h")] + \
    [os.path.join(INCLUDE, "h3qk.h")]

COMPILE_FLAGS = [
    "-O3", "-std=c++17",
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo",
    "-fmad=false", "-prec-div=true", "-prec-sqrt=true", "-ftz=false",
    "-Xcompiler", "-fPIC",
]
LINK_FLAGS = ["-shared", "-cudart", "static", "-gencode", "arch=compute_103a,code=sm_103a"]
# One-shot form (all sources in one nvcc command), for tools that build variants.
NVCC_FLAGS = COMPILE_FLAGS + ["--threads", "0", "-shared", "-cudart", "static"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None, debug: bool = False) -> str:
    """Build libh3qk.so (or, with debug, libh3qk_debug.so with the device-side
    bounds checks) unless it is newer than every source."""
    out = LIB_DEBUG if debug else LIB
    if debug:
        extra = [*(extra or []), "-DH3QK_DEBUG_CHECKS=1"]
    if not force and up_to_date(out):
        return out
    tag = f".tmp{os.getpid()}{'d' if debug else ''}"
    objs = [os.path.join(PKG, os.path.basename(src) + tag + ".o") for src in SOURCES]

    def compile_one(src_obj):
        src, obj = src_obj
        cmd = [nvcc_path(), *COMPILE_FLAGS, *(extra or []), "-I", INCLUDE, "-I", CSRC, "-c", "-o", obj, src]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode:
            sys.stdout.write(r.stdout)
            sys.stderr.write(r.stderr)
        r.check_returncode()

    try:
        with ThreadPoolExecutor(len(SOURCES)) as ex:
            list(ex.map(compile_one, zip(SOURCES, objs)))
        tmp = out + tag
        subprocess.run([nvcc_path(), *LINK_FLAGS, "-o", tmp, *objs], check=True)
        os.replace(tmp, out)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
