"""Build libmala.so in-tree with nvcc for sm_103a.

Each .cu file under csrc/ compiles to its own object in parallel, then nvcc
links the shared library next to this file.  Objects are rebuilt only when a
source or header is newer.  Run as ``python -m mass_adaptive_sparse_gb300.build``
(``--debug`` for the bounds-checked variant only).

The bounds-checked variant, libmala_debug.so, is the same source compiled with
-DMALA_DEBUG: every TMA box origin and global index of the tensor-core and
decode kernels is checked against the extents the host validated, and a
violation sets bit 8 of the device status word and skips the access.  The
binding loads it instead of libmala.so when MALA_LIBRARY=debug.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmala.so")
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libmala_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmala.so")


def _newest(paths) -> float:
    return max((os.path.getmtime(p) for p in paths), default=0.0)


def build(verbose: bool = False, force: bool = False, variants=("release", "debug")) -> str:
    """Compile the listed variants (objects of all of them in one parallel
    pool), link each library, and return the release library's path."""
    nvcc = _nvcc()
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    hdr_time = _newest(headers)
    layout = {"release": (BUILD, LIB, []), "debug": (BUILD_DEBUG, LIB_DEBUG, ["-DMALA_DEBUG"])}
    jobs = []
    for v in variants:
        bdir, _, extra = layout[v]
        os.makedirs(bdir, exist_ok=True)
        jobs += [(src, bdir, extra) for src in sources]

    def compile_one(job):
        src, bdir, extra = job
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        if not force and os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), hdr_time):
            return obj
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{res.stdout}\n{res.stderr}")
        return obj

    with ThreadPoolExecutor(max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, jobs))
    for v in variants:
        bdir, lib, _ = layout[v]
        vobjs = [o for o in objs if os.path.dirname(o) == bdir]
        if force or not os.path.exists(lib) or os.path.getmtime(lib) < _newest(vobjs):
            tmp = lib + ".tmp"
            cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *vobjs]
            res = subprocess.run(cmd, capture_output=True, text=True)
            if res.returncode != 0:
                raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
            os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    only_debug = "--debug" in sys.argv
    print(build(verbose="-v" in sys.argv, force="--force" in sys.argv,
                variants=("debug",) if only_debug else ("release", "debug")))
