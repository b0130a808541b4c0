"""In-tree build of libgqa_attn.so for sm_103a with nvcc (no cmake, no torch extension).

Each translation unit is compiled in parallel with `-gencode arch=compute_103a,
code=sm_103a -lineinfo -O3`, then linked with `nvcc -shared` (static CUDA runtime, so
the library loads on a machine without a GPU and needs no libcuda at link time).
Extra nvcc flags may be given in the GQA_NVCC_FLAGS environment variable.

`build(debug=True)` makes a second library, libgqa_attn_debug.so (objects in _build_debug),
compiled with -DGQA_DEBUG_BOUNDS: every global access whose index comes from device-side
data is checked first, and a failed check records GQA_ERR_DEVICE_BOUNDS instead of
accessing memory.  It is slower and meant for testing; the normal library has no checks.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgqa_attn.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libgqa_attn_debug.so")
SOURCES = ["api.cu", "rope.cu", "kv.cu", "decode.cu", "prefill.cu", "prefill_stream.cu",
           "prefill_wide.cu", "prefill_pair.cu", "qknorm.cu", "chunk.cu", "watchdog.cu"]
HEADERS = ["ptx.cuh", "internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
         "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgqa_attn.so")


def _newest_input() -> float:
    paths = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    paths.append(os.path.join(INCLUDE, "gqa_attn.h"))
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def up_to_date(lib: str = LIB) -> bool:
    return os.path.exists(lib) and os.path.getmtime(lib) >= _newest_input()


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    lib, bdir = (LIB_DEBUG, BUILD_DEBUG) if debug else (LIB, BUILD)
    if debug:
        extra_flags = (*extra_flags, "-DGQA_DEBUG_BOUNDS")
    if not force and up_to_date(lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(bdir, os.path.splitext(src)[0] + ".o")
        env_flags = os.environ.get("GQA_NVCC_FLAGS", "").split()
        cmd = [cc, *ARCH, *FLAGS, *extra_flags, *env_flags, "-c", os.path.join(CSRC, src),
               "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    verbose = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas" in sys.argv else []
    print(build(force=True, verbose=verbose or bool(extra), extra_flags=extra))
