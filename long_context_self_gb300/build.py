"""Build libmagicdec.so in-tree for sm_103a with nvcc (no cmake, no torch extension machinery).

Each .cu under csrc/ compiles to an object in parallel; the objects link into
``long_context_self_gb300/libmagicdec.so`` with the CUDA runtime linked
statically.  ``python -m long_context_self_gb300.build`` rebuilds when a source
or header is newer than the library.

``build(debug=True)`` (``--debug``) builds ``libmagicdec_debug.so`` from the
same sources with ``-DMAGICDEC_DEBUG_CHECKS``: the kernels also record a
length or index outside its range in the device error word (code 4) before
clamping or skipping it as the release build does.  The binding loads it when
``MAGICDEC_LIBRARY=debug``.
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
OUT = os.path.join(PKG, "libmagicdec.so")
OUT_DEBUG = os.path.join(PKG, "libmagicdec_debug.so")
BUILD_DIR = os.path.join(PKG, "_build")
BUILD_DIR_DEBUG = os.path.join(PKG, "_build_debug")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmagicdec")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(ROOT, "include", "magicdec.h"),
                                                                   os.path.abspath(__file__)]


def up_to_date(out: str = OUT) -> bool:
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False, debug: bool = False) -> str:
    out = OUT_DEBUG if debug else OUT
    if not force and up_to_date(out):
        return out
    bdir = BUILD_DIR_DEBUG if debug else BUILD_DIR
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    extra = (["-Xptxas", "-v"] if ptxas_v else []) + (["-DMAGICDEC_DEBUG_CHECKS"] if debug else [])

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        results = list(ex.map(compile_one, _sources()))
    if verbose or ptxas_v:
        for obj, log in results:
            if log.strip():
                print(f"--- {os.path.basename(obj)}\n{log}", file=sys.stderr)
    tmp = out + f".{os.getpid()}.tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_v="--ptxas-v" in sys.argv,
                debug="--debug" in sys.argv))
