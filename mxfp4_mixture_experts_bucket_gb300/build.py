"""Builds the in-tree shared library libmoe_mxfp4.so for sm_103a with nvcc.

Each translation unit compiles in parallel into _build/, then one link step
produces the library next to this file. Rebuilds only when a source or header
is newer than the library. No GPU is needed to build.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmoe_mxfp4.so")
# the checked build: the same sources with -DMOE_CHECKED (device-side bounds checks)
BUILD_CHECKED = os.path.join(HERE, "_build_checked")
LIB_CHECKED = os.path.join(HERE, "libmoe_mxfp4_checked.so")

SOURCES = ["abi.cu", "route_bucket.cu", "gemv.cu", "decode.cu", "decode_mx.cu", "prepack.cu", "grouped_mm.cu",
           "grouped_mx.cu", "noalloc.cu", "selftest.cu", "q8.cu", "grouped_mx4.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "-I" + INCLUDE, "-I" + CSRC] + ARCH


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe_mxfp4.so")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return files


def needs_build(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Builds libmoe_mxfp4.so, or with checked=True libmoe_mxfp4_checked.so (-DMOE_CHECKED)."""
    lib = LIB_CHECKED if checked else LIB
    out_dir = BUILD_CHECKED if checked else BUILD
    if not force and not needs_build(lib):
        return lib
    nvcc = _nvcc()
    os.makedirs(out_dir, exist_ok=True)
    flags = NVCC_FLAGS + (["-DMOE_CHECKED"] if checked else [])

    def compile_one(src: str) -> str:
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = [nvcc] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as pool:
        objs = list(pool.map(compile_one, SOURCES))
    tmp = lib + ".tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked="--checked" in sys.argv))
