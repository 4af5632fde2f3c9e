"""Build libkvdecode.so (all CUDA sources, sm_103a) in-tree.

Each translation unit is compiled in parallel with nvcc, then linked into one shared
library next to this file. Intermediate objects go to ``_build/`` at the repo root.
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libkvdecode.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvdecode.so")


def flags(ptxas_verbose: bool = False):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC, "-Xptxas",
                   "-v" if ptxas_verbose else "-O3"]


def _compile(src: str, obj: str, verbose: bool) -> tuple[str, str]:
    cmd = [nvcc(), "-c", src, "-o", obj] + flags(verbose)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    return src, r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every CUDA source and link libkvdecode.so (skipped when it is up to date);
    `verbose` prints ptxas register / shared-memory / spill figures per kernel."""
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    deps = srcs + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    if not force and os.path.exists(LIB):
        lib_t = os.path.getmtime(LIB)
        if all(os.path.getmtime(d) <= lib_t for d in deps):
            return LIB
    os.makedirs(BUILD, exist_ok=True)
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in srcs]
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        for src, log in ex.map(lambda so: _compile(so[0], so[1], verbose), zip(srcs, objs)):
            if verbose and log:
                print(f"== {os.path.basename(src)}\n{log}", file=sys.stderr)
    tmp = LIB + f".tmp{os.getpid()}"
    # -z defs: an unresolved symbol fails the build here, not the first import on the GPU machine
    cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-Xlinker", "-z", "-Xlinker", "defs"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
