"""Builds libvsf.so in-tree with nvcc for sm_103a (no torch extension machinery).

build(variant="bounds") builds libvsf_bounds.so instead: the same library
with -DVSF_DEBUG_BOUNDS, whose kernels check every range they index against
the packed buffers' extent and record a failed check in the device error
word (bit 4) instead of accessing; load it with VSF_LIBRARY=<path>."""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libvsf.so")
BUILD = os.path.join(PKG, "_build")
VARIANTS = {None: ("libvsf.so", []), "bounds": ("libvsf_bounds.so", ["-DVSF_DEBUG_BOUNDS"])}

SOURCES = ["plan.cpp", "vsf_kernels.cu", "muon.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _inputs():
    files = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))
             if f.endswith((".cu", ".cuh", ".cpp", ".h"))]
    return files + [os.path.join(INCLUDE, "vsf.h")]


def lib_path(variant: str | None = None) -> str:
    return os.path.join(PKG, VARIANTS[variant][0])


def up_to_date(variant: str | None = None) -> bool:
    out = lib_path(variant)
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          variant: str | None = None) -> str:
    out = lib_path(variant)
    if not force and up_to_date(variant):
        return out
    objdir = os.path.join(BUILD, variant or "release")
    os.makedirs(objdir, exist_ok=True)
    # -fmad=false: no floating-point multiply-add contraction anywhere in
    # device code, so every fp32 operation of the update rounds once, in the
    # order written (explicit __fmaf_rn calls stay fused).
    common = ["-O3", "-std=c++17", "-lineinfo", "-fmad=false", "-Xcompiler",
              "-fPIC,-O2,-ffp-contract=off", "-I", INCLUDE, "-I", CSRC] + ARCH + VARIANTS[variant][1]
    if ptxas_info:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [nvcc(), "-c", os.path.join(CSRC, src), "-o", obj] + common
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for _, err in results:
            sys.stderr.write(err)
    tmp = out + ".tmp"
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(nvcc())), "lib64")
    cmd = [nvcc(), "-shared", "-o", tmp] + [o for o, _ in results] + ARCH + [
        "-lcudart_static", "-L" + cuda_lib, "-Xlinker", "-rpath=" + cuda_lib]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="-v" in sys.argv))
