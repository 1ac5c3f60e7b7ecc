"""Build libattn.so (the CUDA kernels and the C ABI) in-tree with nvcc for sm_103a.

    python -m causal_scaled_dot_gb300.build        # build (or rebuild if stale)
    python -m causal_scaled_dot_gb300.build --force --verbose

The library lands in ``causal_scaled_dot_gb300/_build/libattn.so``.  It links
the CUDA runtime dynamically (the same libcudart that PyTorch loads) and
reaches the driver's tensor-map encoder through the runtime's entry-point
query, so it needs no ``-lcuda`` at link time.
"""
from __future__ import annotations

import argparse
import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIBRARY = os.path.join(BUILD_DIR, "libattn.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    cand = [os.environ.get("NVCC", ""), shutil.which("nvcc") or "", "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libattn")


def _cuda_home(nvcc: str) -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + sorted(glob.glob(os.path.join(CSRC, "*.h"))) + [
        os.path.join(INCLUDE, "attn.h"), os.path.abspath(__file__)]


def is_stale() -> bool:
    if not os.path.exists(LIBRARY):
        return True
    t = os.path.getmtime(LIBRARY)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _run(cmd: list[str], verbose: bool) -> subprocess.CompletedProcess:
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{res.stdout}\n{res.stderr}")
    return res


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile every .cu under csrc/ into one shared library; returns its path.

    Each source is its own translation unit (no device code is shared across
    them), so they compile in parallel to objects and are linked once."""
    if not force and not is_stale():
        return LIBRARY
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()
    cuda_lib = os.path.join(_cuda_home(nvcc), "lib64")
    tmp_dir = os.path.join(BUILD_DIR, f"obj.tmp{os.getpid()}")
    os.makedirs(tmp_dir, exist_ok=True)
    tmp = LIBRARY + f".tmp{os.getpid()}"
    flags = [ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", f"-I{INCLUDE}"]
    if ptxas_verbose:
        flags.insert(0, "-Xptxas=-v")
    try:
        srcs = sources()
        objs = [os.path.join(tmp_dir, os.path.basename(f)[:-3] + ".o") for f in srcs]
        with concurrent.futures.ThreadPoolExecutor(max_workers=len(srcs)) as pool:
            outs = list(pool.map(lambda so: _run([nvcc, *flags, "-c", so[0], "-o", so[1]], verbose),
                                 zip(srcs, objs)))
        _run([nvcc, ARCH, "-shared", "-cudart", "shared", "-Xlinker", f"-rpath,{cuda_lib}", "-o", tmp, *objs],
             verbose)
        if verbose or ptxas_verbose:
            for res in outs:
                sys.stdout.write(res.stdout + res.stderr)
        os.replace(tmp, LIBRARY)
    finally:
        shutil.rmtree(tmp_dir, ignore_errors=True)
        if os.path.exists(tmp):
            os.remove(tmp)
    return LIBRARY


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true", help="print registers/spills per kernel")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, ptxas_verbose=a.ptxas_verbose))


if __name__ == "__main__":
    main()
