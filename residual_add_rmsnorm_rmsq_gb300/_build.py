"""Build librmsq.so in-tree: nvcc for sm_103a only, one object per translation
unit compiled in parallel, linked with the static CUDA runtime.

Floating-point flags: no --use_fast_math; IEEE division and square root and no
flush-to-zero are nvcc's defaults and are stated explicitly below.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "librmsq.so")

UNITS = ["rmsq_api.cu", "rmsq_rows_bf16.cu", "rmsq_rows_fp16.cu", "rmsq_noalloc.cu", "rmsq_act.cu", "rmsq_qk.cu",
         "rmsq_allreduce.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-ftz=false", "-prec-div=true",
                     "-prec-sqrt=true", "-fmad=true", "-Xcompiler", "-fPIC,-O2",
                     "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librmsq")


def source_digest() -> str:
    """sha256 over every source that goes into the library (for staleness checks)."""
    h = hashlib.sha256()
    files = sorted(os.listdir(CSRC)) + ["../../include/rmsq.h"]
    for f in files:
        p = os.path.normpath(os.path.join(CSRC, f))
        if os.path.isfile(p) and p.endswith((".cu", ".cuh", ".h")):
            h.update(os.path.basename(p).encode())
            with open(p, "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()


def _compile(unit: str, verbose: bool, build_dir: str = BUILD, extra: list | None = None) -> str:
    obj = os.path.join(build_dir, unit.replace(".cu", ".o"))
    cmd = [nvcc()] + NVCC_FLAGS + (extra or []) + (["-Xptxas", "-v"] if verbose else []) + \
        ["-c", os.path.join(CSRC, unit), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {unit}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    digest = source_digest()
    stamp = os.path.join(LIBDIR, "librmsq.sha256")
    if not force and os.path.exists(LIB) and os.path.exists(stamp):
        with open(stamp) as fh:
            if fh.read().strip() == digest:
                return LIB
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        objs = list(ex.map(lambda u: _compile(u, verbose), UNITS))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as fh:
        fh.write(digest + "\n")
    return LIB


def build_variant(name: str, defines: dict) -> str:
    """Build a separately named copy of the library with compile-time tuning
    macros set (e.g. {"RMSQ_PIPE_MIN_BLOCKS": 2}), for launch-shape
    experiments; returns its path.  Results do not depend on these macros."""
    bdir = os.path.join(BUILD, name)
    os.makedirs(bdir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    extra = [f"-D{k}={v}" for k, v in sorted(defines.items())]
    with cf.ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        objs = list(ex.map(lambda u: _compile(u, False, bdir, extra), UNITS))
    out = os.path.join(LIBDIR, f"librmsq_{name}.so")
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", out] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
