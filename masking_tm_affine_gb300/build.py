"""Build ``libtm.so`` in-tree with nvcc for sm_103a (GB300).

Each ``csrc/*.cu`` translation unit compiles in parallel into ``_build/``;
they link into ``masking_tm_affine_gb300/lib/libtm.so`` against the shared CUDA
runtime (``libcudart.so.13``).  A process that already loaded the runtime --
torch does at import -- shares that one instance with libtm, so the current
device, streams and contexts are the caller's; otherwise the RUNPATH to the
toolkit's lib64 finds it.  No fast-math and no flush-to-zero: the maps must match the
oracle bit for bit.  ``ptxas -v`` reports (registers, spills, shared memory)
land in ``_build/*.ptxas.txt``.

Usage: ``python -m masking_tm_affine_gb300.build [--force]``.
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
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libtm.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "--ftz=false",
              "--prec-div=true", "--prec-sqrt=true", "--fmad=true", "-Xptxas", "-v",
              "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtm")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))) + \
        [os.path.join(INCLUDE, "tm.h"), os.path.abspath(__file__)]


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str) -> str:
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
    log = os.path.join(BUILD, os.path.basename(src)[:-3] + ".ptxas.txt")
    hdrs = [d for d in _deps() if not d.endswith(".cu")]
    if _stale(obj, [src] + hdrs):
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        with open(log, "w") as f:
            f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s" % (os.path.basename(src), r.stderr[-6000:]))
    return obj


def build(force: bool = False) -> str:
    """Compile and link libtm.so if any source changed; return its path."""
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    if force:
        for o in glob.glob(os.path.join(BUILD, "*.o")):
            os.remove(o)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(_compile, srcs))
    if force or _stale(LIB, objs):
        tmp = LIB + ".tmp%d" % os.getpid()
        libdir = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc()))), "lib64")
        # --no-undefined: a symbol some unit uses but none defines fails the build, not the first load
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-Xlinker", "-rpath," + libdir, "-Xlinker", "--no-undefined",
               "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link of libtm.so failed:\n%s" % r.stderr[-6000:])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
