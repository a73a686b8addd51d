"""Builds libvarlen_attn.so in-tree for sm_103a with nvcc.

``--bounds`` (``build(bounds=True)``) builds the bounds-checking variant into
``_build/bounds/libvarlen_attn.so``: the same sources compiled with
-DVARLEN_DEBUG_BOUNDS, whose kernels check every plain global access against
its operand's extent (load it by setting VARLEN_ATTN_LIB to that path).

Each .cu translation unit compiles in parallel to an object file, then nvcc
links them into one shared library with the CUDA runtime linked statically
(the library depends on no CUDA shared object at load time; the driver API
entry points it needs are fetched at run time).

    python -m packed_variable_length_varlen_gb300.build
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libvarlen_attn.so")
BOUNDS_LIB = os.path.join(BUILD, "bounds", "libvarlen_attn.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libvarlen_attn")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))] + [
        os.path.join(INCLUDE, "varlen_attn.h"), os.path.abspath(__file__)]


def up_to_date(lib: str | None = None) -> bool:
    lib = lib or LIB
    stamp = lib + ".arch"
    if not (os.path.exists(lib) and os.path.exists(stamp)):
        return False
    with open(stamp) as f:
        if f.read().strip() != platform.machine():
            return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(src: str, verbose: bool, out_dir: str, defines=()) -> str:
    obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *defines, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
    log = os.path.join(out_dir, os.path.basename(src)[:-3] + ".ptxas.txt")
    with open(log, "w") as f:
        f.write(r.stdout + r.stderr)
    if verbose:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, bounds: bool = False) -> str:
    """Compile and link; returns the library path.  Skips work when the
    library is newer than every source and was built on this machine type.
    ``bounds`` builds the bounds-checking variant (BOUNDS_LIB) instead."""
    lib = BOUNDS_LIB if bounds else LIB
    if not force and up_to_date(lib):
        return lib
    out_dir = os.path.dirname(lib)
    os.makedirs(out_dir, exist_ok=True)
    defines = ["-DVARLEN_DEBUG_BOUNDS"] if bounds else []
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, out_dir, defines), sources()))
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)
    with open(lib + ".arch", "w") as f:
        f.write(platform.machine())
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, bounds="--bounds" in sys.argv))
