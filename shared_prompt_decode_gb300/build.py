"""Build librelay.so (the CUDA library behind include/relay.h) for sm_103a."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "librelay.so")
SOURCES = [os.path.join(CSRC, "relay.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "relay_kernels.cuh"), os.path.join(CSRC, "sys_tc.cuh"),
                  os.path.join(INCLUDE, "relay.h")]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librelay")


def build(force: bool = False, verbose: bool = False, variant: str = "", defines=()) -> str:
    """Build librelay.so.  A named variant (tests only) is the same sources
    with extra -D definitions, built to librelay_<variant>.so."""
    os.makedirs(OUT_DIR, exist_ok=True)
    lib = LIB if not variant else os.path.join(OUT_DIR, f"librelay_{variant}.so")
    if not force and os.path.exists(lib):
        t = os.path.getmtime(lib)
        if all(os.path.getmtime(f) <= t for f in DEPS):
            return lib
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "-o", tmp] + [f"-D{d}" for d in defines] + SOURCES
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + r.stdout + r.stderr)
    if verbose:
        print(r.stdout + r.stderr)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
