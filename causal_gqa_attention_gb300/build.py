"""Build the CUDA library ``_build/libgqa_attn.so`` from ``csrc/`` with nvcc for sm_103a.

Each translation unit compiles in its own nvcc process (in parallel), then one link step makes
the shared library. The CUDA runtime is linked statically and the driver is reached through the
runtime's entry-point query, so the library loads on machines without a GPU driver too.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libgqa_attn.so")
# the same sources with device-side index checks compiled in (GQA_ATTN_DEBUG); built on demand
DEBUG_LIB = os.path.join(BUILD, "libgqa_attn_debug.so")
SOURCES = ["api.cu", "prefill_tc.cu", "prefill_f32.cu", "decode.cu", "decode_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps_mtime() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    paths.append(os.path.join(ROOT, "include", "gqa_attn.h"))
    return max(os.path.getmtime(p) for p in paths)


def _compile(src: str, verbose: bool, debug: bool = False) -> str:
    obj = os.path.join(BUILD, src.replace(".cu", "_debug.o" if debug else ".o"))
    cmd = [nvcc(), *ARCH, *FLAGS, *(["-DGQA_ATTN_DEBUG"] if debug else []), "-c",
           os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile and link the library (or with debug=True its debug build) if any source is
    newer than it. Returns its path."""
    lib = DEBUG_LIB if debug else LIB
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime():
        return lib
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, debug), SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
