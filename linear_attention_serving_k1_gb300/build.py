"""Builds the in-tree CUDA library ``_build/libkda.so`` for sm_103a with nvcc,
and its bounds-checking debug build ``_build/debug/libkda_debug.so`` (the
same sources with ``-DKDA_DEBUG``: every data-dependent global index checked
before the access, failures reported by the C ABI as KDA_ERR_BOUNDS).

Each translation unit under ``csrc/`` compiles, for both builds at once, in
parallel to an object file; each build's objects link into one shared library
with the CUDA runtime linked statically, so the library exports only the C
ABI of ``include/kda.h``.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libkda.so")
DEBUG_BUILD = os.path.join(BUILD, "debug")
DEBUG_LIB = os.path.join(DEBUG_BUILD, "libkda_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-v"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found (CUDA toolkit required to build libkda.so)")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(ROOT, "include", "kda.h"),
                                                                 os.path.abspath(__file__)]


def library_path() -> str:
    return LIB


def debug_library_path() -> str:
    return DEBUG_LIB


# (library, object directory, extra nvcc flags) of the two builds
VARIANTS = ((LIB, BUILD, []), (DEBUG_LIB, DEBUG_BUILD, ["-DKDA_DEBUG"]))


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _deps())


def is_stale() -> bool:
    return any(_stale(lib) for lib, _, _ in VARIANTS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every .cu under csrc/ for both builds and link libkda.so and
    libkda_debug.so (each skipped when up to date); returns libkda.so's path."""
    todo = [v for v in VARIANTS if force or _stale(v[0])]
    if not todo:
        return LIB
    nv = nvcc()
    procs = []
    links = []
    for lib, objdir, extra in todo:
        os.makedirs(objdir, exist_ok=True)
        objs = []
        for src in sources():
            obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
            log = obj + ".log"
            cmd = [nv, *ARCH, *NVCC_FLAGS, *extra, "-I", os.path.join(ROOT, "include"), "-c", src, "-o", obj]
            procs.append((src, log, subprocess.Popen(cmd, stdout=open(log, "w"), stderr=subprocess.STDOUT)))
            objs.append(obj)
        links.append((lib, objs))
    failed = []
    for src, log, p in procs:
        if p.wait() != 0:
            failed.append((src, open(log).read()))
        elif verbose:
            sys.stdout.write(open(log).read())
    if failed:
        msg = "\n".join(f"--- {s}\n{l}" for s, l in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    for lib, objs in links:
        tmp = lib + f".tmp{os.getpid()}"
        subprocess.run([nv, *ARCH, "-shared", "--cudart", "static", *objs, "-o", tmp], check=True)
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
