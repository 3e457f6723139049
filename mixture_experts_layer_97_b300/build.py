"""Build libmoe_b300.so in-tree with nvcc for sm_103a (B300).

    python -m mixture_experts_layer_97_b300.build [--force] [--ptxas-info]

The library is a single translation unit (csrc/moe_b300.cu includes the
kernel headers) so that the device error word is one symbol per device.
cudart is linked statically; the driver's tensor-map encoder is reached
through cudaGetDriverEntryPointByVersion, so there is no -lcuda.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libmoe_b300.so")
# the benchmark's fp32 FMA microbenchmark (the route kernel's roofline denominator)
PEAK_LIB = os.path.join(PKG, "libmoe_fma_peak.so")
PEAK_SRC = os.path.join(CSRC, "fma_peak.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the CUDA library cannot be built")
    return p


def _sources():
    return ([os.path.join(CSRC, "moe_b300.cu")] + sorted(glob.glob(os.path.join(CSRC, "*.cuh")))
            + [os.path.join(ROOT, "include", "moe.h")])


def build_fma_peak(force: bool = False) -> str:
    """The fp32 FMA microbenchmark library (separate from the MoE library)."""
    if not force and os.path.exists(PEAK_LIB) and os.path.getmtime(PEAK_LIB) >= os.path.getmtime(PEAK_SRC):
        return PEAK_LIB
    tmp = PEAK_LIB + f".tmp{os.getpid()}"
    cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-shared", "-o", tmp,
           PEAK_SRC]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed ({r.returncode}):\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, PEAK_LIB)
    return PEAK_LIB


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(s) <= t for s in _sources())


def build(force: bool = False, ptxas_info: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-shared",
           "-I", os.path.join(ROOT, "include"), "-o", tmp, os.path.join(CSRC, "moe_b300.cu")]
    if ptxas_info:
        cmd += ["-Xptxas", "-v"]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed ({r.returncode}):\n{r.stdout}\n{r.stderr}")
    if ptxas_info or verbose:
        sys.stderr.write(r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, ptxas_info="--ptxas-info" in sys.argv, verbose=True)
    build_fma_peak(force="--force" in sys.argv)
    print(LIB)
