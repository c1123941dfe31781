"""Builds libpgqa.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each ``csrc/*.cu`` compiles to an object in parallel, then nvcc links the
shared library next to this file.  The CUDA runtime is linked statically; the
driver is reached only through ``cudaGetDriverEntryPointByVersion``.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpgqa.so")
VARIANTS = {"": [], "trace": ["-DPGQA_TRACE"]}


def lib_path(variant: str = "") -> str:
    """The shared library of a build variant ("" = normal, "trace" = with phase timestamps)."""
    return LIB if not variant else os.path.join(HERE, f"libpgqa_{variant}.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))
            + [os.path.abspath(__file__)])


def stale(variant: str = "") -> bool:
    lib = lib_path(variant)
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(d) > t for d in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False, variant: str = "") -> str:
    """Compile every CUDA source for sm_103a and link ``libpgqa.so`` (or a variant); returns its path."""
    lib = lib_path(variant)
    if not force and not stale(variant):
        return lib
    bdir = os.path.join(BUILD, variant or "default")
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()
    extra = (["-Xptxas", "-v"] if ptxas_v else []) + VARIANTS[variant]
    procs = []
    objs = []
    for src in _sources():
        obj = os.path.join(bdir, os.path.splitext(os.path.basename(src))[0] + ".o")
        objs.append(obj)
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if out and (verbose or ptxas_v or p.returncode != 0):
            print(out, file=sys.stderr)
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    variant = "trace" if "--trace" in sys.argv else ""
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, ptxas_v="--ptxas-v" in sys.argv,
                variant=variant))
