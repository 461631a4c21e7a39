"""In-tree build of libhalo.so for sm_103a with nvcc (no cmake, no torch build
machinery).  Translation units compile in parallel, then link into one shared
library next to this file."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIBRARY = os.path.join(PKG, "libhalo.so")
# debug variant: every kernel checks its slot indices (-DHALO_DEBUG, HALO_EBOUNDS)
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIBRARY_DEBUG = os.path.join(PKG, "libhalo_debug.so")
SOURCES = ["halo_api.cu", "halo_build.cu", "halo_exchange.cu", "halo_modes.cu", "halo_noalloc.cu",
           "stencil.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, extra_flags=(), force: bool = False, debug: bool = False) -> str:
    """Compile every source (in parallel) and link the library; debug=True
    builds the bounds-checking variant libhalo_debug.so instead."""
    build_dir = BUILD_DEBUG if debug else BUILD
    library = LIBRARY_DEBUG if debug else LIBRARY
    if debug:
        extra_flags = (*extra_flags, "-DHALO_DEBUG")
    os.makedirs(build_dir, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    objs, procs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s, *headers, __file__]):
            cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra_flags, "-c", s, "-o", o]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose and out:
            print(out, file=sys.stderr)
        if p.returncode != 0:
            failed.append((src, out))
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join("%s:\n%s" % f for f in failed))
    if force or _stale(library, objs):
        tmp = library + ".tmp%d" % os.getpid()
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout)
        os.replace(tmp, library)
    return library


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
