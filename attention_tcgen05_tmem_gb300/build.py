"""Build the CUDA library ``libattn_train.so`` in-tree for sm_103a.

Each ``csrc/*.cu`` translation unit is compiled by nvcc in parallel, then
linked into one shared library next to this file.  No CMake, no torch
extension machinery: the library exposes a plain C ABI
(``include/attn_train.h``) that ``binding.py`` loads with ctypes.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libattn_train.so")
BUILD_DIR = os.path.join(ROOT, "_build")
SOURCES = ["api.cu", "fwd.cu", "fwd_split.cu", "bwd.cu", "aux.cu", "loss.cu", "host_step.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "attn_train.h"))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


TRACE_LIB = os.path.join(HERE, "libattn_train_trace.so")
DEBUG_LIB = os.path.join(HERE, "libattn_train_debug.so")


def build_trace(force: bool = False) -> str:
    """Same library built with -DATTN_TRACE (pipeline timeline probes on), as
    libattn_train_trace.so; used by pipeline_trace.py, never by the product."""
    return build(force=force, trace=True)


def build_debug(force: bool = False) -> str:
    """Same library built with -DATTN_DEBUG (device-side checks of tile
    coordinates, work items and workspace slots), as libattn_train_debug.so:
    a bring-up aid, loaded explicitly (binding.load(DEBUG_LIB))."""
    return build(force=force, debug=True)


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False,
          trace: bool = False, debug: bool = False) -> str:
    lib = TRACE_LIB if trace else DEBUG_LIB if debug else LIB
    if not force and os.path.exists(lib) and all(
            os.path.getmtime(f) <= os.path.getmtime(lib) for f in _deps()):
        return lib
    bdir = BUILD_DIR + ("_trace" if trace else "_debug" if debug else "")
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_v else []
    if trace:
        extra.append("-DATTN_TRACE")
    if debug:
        extra.append("-DATTN_DEBUG")

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_v:
        for _, log in results:
            if log:
                sys.stderr.write(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_v="--ptxas-v" in sys.argv)
    print(LIB)
