"""Builds libmamba3.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

    python -m selective_state_space_134_b300.build [--force]

Every translation unit is compiled to an object in parallel, then linked into
one shared library with the CUDA runtime linked statically, so the library
loads on a machine without a GPU driver (its calls then report M3_ERR_CUDA).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libmamba3.so")
OBJDIR = os.path.join(ROOT, "_build", "mamba3")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmamba3.so")
    return exe


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(ROOT, "include", "mamba3.h"),
                                                                   os.path.abspath(__file__)]


# the sources each kernel family is built from (its kernels, launch code and shared headers)
KERNEL_SOURCES = {
    "prefill_output": ("m3_scan_tc*.cu", "m3_scan_tc.cuh", "m3_tc.cuh", "m3_internal.cuh"),
    "decode": ("m3_decode.cu", "m3_tc.cuh", "m3_internal.cuh"),
}


def source_digest(kernel: str = "") -> str:
    """Short hash of the library sources (kernels, host code, public header), or of the sources one
    kernel family is built from (a KERNEL_SOURCES key)."""
    import hashlib
    h = hashlib.sha256()
    if kernel:
        files = [p for pat in KERNEL_SOURCES[kernel] for p in glob.glob(os.path.join(CSRC, pat))]
    else:
        files = sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
    for p in sorted(set(files) | {os.path.join(ROOT, "include", "mamba3.h")}):
        h.update(os.path.basename(p).encode())
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(OBJDIR, os.path.basename(src) + ".o")
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + (["-Xptxas", "-v"] if verbose else []) + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(OBJDIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), sources()))
    tmp = LIB + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
