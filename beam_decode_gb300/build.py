"""Build libgrbeam.so (sm_103a) in-tree with nvcc.

The three translation units compile in parallel; the shared library links the
CUDA runtime statically, so it needs no torch headers and no -lcuda (the
tensor-map encoder is fetched through the runtime's driver entry point).
"""
from __future__ import annotations

import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libgrbeam.so")
UNITS = ["api.cu", "k_topk.cu", "k_attn.cu", "k_attn_pair.cu", "k_noalloc.cu"]
HEADERS = [os.path.join(SRC, "grbeam_internal.h"), os.path.join(SRC, "topk_dev.cuh"), os.path.join(SRC, "attn_dev.cuh"),
           os.path.join(os.path.dirname(HERE), "include", "grbeam.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgrbeam")


def _stamp() -> str:
    return f"{platform.machine()}|{' '.join(ARCH + FLAGS)}"


def _up_to_date() -> bool:
    stamp = os.path.join(BUILD, "stamp.txt")
    if not (os.path.exists(LIB) and os.path.exists(stamp)):
        return False
    if open(stamp).read() != _stamp():
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in [os.path.join(SRC, u) for u in UNITS] + HEADERS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link; returns the library path."""
    if not force and _up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(unit: str) -> str:
        obj = os.path.join(BUILD, unit.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, "-c", os.path.join(SRC, unit), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {unit}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        objs = list(ex.map(compile_one, UNITS))
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(os.path.join(BUILD, "stamp.txt"), "w") as f:
        f.write(_stamp())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
