"""Build the CUDA library libbil.so in-tree, for sm_103a (GB300).

    python -m invariant_token_log_gb300.build        # build if out of date
    python -m invariant_token_log_gb300.build --force

The library is built per machine architecture under ``_build/<machine>/`` so
that an x86_64 build and an aarch64 build of the same tree never mix.
Contraction of floating-point multiply-adds is off (``--fmad=false``): every
operation whose rounding matters is written out explicitly in the source.
"""
from __future__ import annotations

import os
import platform
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SOURCES = [os.path.join(HERE, "csrc", f) for f in ("bil.cu", "linear.cu")]
HEADERS = [os.path.join(ROOT, "include", "bil.h")] + [
    os.path.join(HERE, "csrc", f) for f in ("device_common.cuh", "logp_device.cuh", "internal.h")]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "--fmad=false", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-Wall"]


def library_path() -> str:
    return os.path.join(HERE, "_build", platform.machine(), "libbil.so")


def nvcc() -> str:
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def up_to_date(out: str) -> bool:
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(f) <= t for f in SOURCES + HEADERS + [__file__])


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile each source to an object file (in parallel), then link libbil.so."""
    out = library_path()
    if not force and up_to_date(out):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tag = f"tmp{os.getpid()}"
    objs = [os.path.join(os.path.dirname(out), os.path.basename(src) + f".{tag}.o") for src in SOURCES]
    procs = [subprocess.Popen([nvcc(), *ARCH_FLAGS, *NVCC_FLAGS, *(["-Xptxas", "-v"] if verbose else []),
                               "-c", src, "-o", obj]) for src, obj in zip(SOURCES, objs)]
    codes = [p.wait() for p in procs]
    try:
        if any(codes):
            raise subprocess.CalledProcessError(max(codes), "nvcc")
        tmp = f"{out}.{tag}"
        subprocess.run([nvcc(), *ARCH_FLAGS, "-shared", *objs, "-ldl", "-o", tmp], check=True)
        os.replace(tmp, out)
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
