"""Builds the CUDA library libswa_sdpa_bwd.so in-tree with nvcc (sm_103a only).

Each translation unit is compiled in parallel, then linked into one shared
library that exports the C ABI of include/sdpa_bwd.h. build(debug_bounds=True)
builds the range-checked variant libswa_sdpa_bwd_dbg.so (-DSDPA_DEBUG_BOUNDS:
every raw global index is checked against its buffer and an out-of-range one
is reported as SDPA_ERR_BOUNDS instead of being accessed).
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libswa_sdpa_bwd.so")
LIB_DBG = os.path.join(BUILD, "libswa_sdpa_bwd_dbg.so")
DEBUG_BOUNDS = ("-DSDPA_DEBUG_BOUNDS",)
SOURCES = ["api.cu", "aux_kernels.cu", "main_kernel.cu", "fwd_kernel.cu"]
HEADERS = ["ptx.cuh", "seq.cuh", "sdpa_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _flags(extra=()):
    return [*ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
            "-I", os.path.join(ROOT, "include"), *extra]


def _digest(extra) -> str:
    h = hashlib.sha256()
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    for name in sorted(os.listdir(os.path.join(ROOT, "include"))):
        with open(os.path.join(ROOT, "include", name), "rb") as f:
            h.update(f.read())
    h.update(" ".join(_flags(extra)).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, extra=(), debug_bounds: bool = False) -> str:
    """Compile and link the library if any source changed; returns its path."""
    if debug_bounds:
        extra = tuple(extra) + DEBUG_BOUNDS
    lib_path = LIB_DBG if debug_bounds else LIB
    objdir = os.path.join(BUILD, "dbg") if debug_bounds else BUILD
    os.makedirs(objdir, exist_ok=True)
    stamp = os.path.join(objdir, "stamp")
    digest = _digest(extra)
    if not force and os.path.exists(lib_path) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return lib_path
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [nvcc, *_flags(extra), "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            print(log)
    tmp = lib_path + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-lcudart"],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    with open(stamp, "w") as f:
        f.write(digest)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug_bounds="--debug-bounds" in sys.argv))
