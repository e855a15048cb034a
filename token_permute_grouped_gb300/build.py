"""Builds the CUDA library liba2av_gmm.so in-tree with nvcc (sm_103a only)."""

from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "liba2av_gmm.so")
# Debug variant: device-side bounds checks that record a status bit instead
# of trapping (-DA2AV_CHECKS).  Only the sources the checks touch are built
# again; the others are linked from the ordinary build.
CHECKS_LIB = os.path.join(PKG, "liba2av_gmm_checks.so")
CHECKS_SOURCES = ["api.cu", "permute.cu", "grouped_gemm.cu"]
SOURCES = ["api.cu", "permute.cu", "grouped_gemm.cu", "grouped_gemm_mx.cu", "amp.cu", "quant_reduce.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        path = os.path.join(cand, "bin", "nvcc") if cand else ""
        if path and os.path.exists(path):
            return path
    return "nvcc"


def _inputs_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return max(os.path.getmtime(f) for f in files)


def up_to_date(lib: str = LIB) -> bool:
    return os.path.exists(lib) and os.path.getmtime(lib) >= _inputs_mtime()


def build(verbose: bool = False, ptxas_info: bool = False, force: bool = False, checks: bool = False) -> str:
    """Compile every translation unit in parallel, then link the shared library.

    checks=True builds the debug variant CHECKS_LIB (after the ordinary one)."""
    if checks:
        build(verbose, ptxas_info, force)
        if not force and up_to_date(CHECKS_LIB):
            return CHECKS_LIB
    elif not force and up_to_date():
        return LIB
    out_dir = os.path.join(BUILD, "checks") if checks else BUILD
    os.makedirs(out_dir, exist_ok=True)
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    if checks:
        flags += ["-DA2AV_CHECKS"]
    if ptxas_info:
        flags += ["-Xptxas", "-v"]

    def compile_one(src: str) -> str:
        if checks and src not in CHECKS_SOURCES:
            return os.path.join(BUILD, src.replace(".cu", ".o"))
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = [nvcc(), *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or ptxas_info or r.returncode:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError(f"nvcc failed on {src}")
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    lib = CHECKS_LIB if checks else LIB
    tmp = lib + ".tmp"
    subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    build(verbose=True, ptxas_info="-v" in sys.argv, force=True)
    print(LIB)
