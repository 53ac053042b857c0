"""Build libdflash.so in-tree: every csrc/*.cu compiled for sm_103a in parallel, then linked.

Run as `python -m speculative_decoding_drafter_dflash_gb300.build` or through
`__graft_entry__.build()`. nvcc cross-compiles without a GPU.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libdflash.so")
# The debug build: device-side index checks that write DF_EINVAL to the status word (DF_DEBUG).
DEBUG_LIB = os.path.join(PKG, "libdflash_debug.so")
# The trace build: per-CTA kernel spans in one device buffer (DF_TRACE; relocatable device code).
TRACE_LIB = os.path.join(PKG, "libdflash_trace.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _cuda_home(nvcc: str) -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def build(verbose: bool = False, force: bool = False, debug: bool = False,
          trace: bool = False) -> str:
    nvcc = _nvcc()
    lib = DEBUG_LIB if debug else (TRACE_LIB if trace else LIB)
    objdir = os.path.join(BUILD, "debug" if debug else "trace") if (debug or trace) else BUILD
    os.makedirs(objdir, exist_ok=True)
    srcs = sources()
    deps = srcs + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    deps.append(os.path.join(INCLUDE, "dflash.h"))
    if not force and os.path.exists(lib):
        t_lib = os.path.getmtime(lib)
        if all(os.path.getmtime(d) <= t_lib for d in deps):
            return lib
    flags = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
             "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC] + ARCH
    if debug:
        flags.append("-DDF_DEBUG=1")
    if trace:
        flags += ["-DDF_TRACE=1", "-rdc=true"]

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [nvcc] + flags + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    cuda_lib = os.path.join(_cuda_home(nvcc), "lib64")
    tmp = lib + ".tmp"
    cmd = [nvcc, "-shared", "-cudart", "shared", "-o", tmp] + (["-rdc=true"] if trace else []) + \
        objs + ARCH + [
        "-Xlinker", f"-rpath={cuda_lib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose=True, force="--force" in sys.argv, debug="--debug" in sys.argv,
                trace="--trace" in sys.argv))
