"""Builds libbsa_fp8.so in-tree with nvcc for sm_103a (GB300)."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libbsa_fp8.so")
SOURCES = [os.path.join(CSRC, "bsa_fp8.cu")]
HEADERS = [os.path.join(CSRC, f) for f in ("ptx_sm103.cuh", "bsa_common.cuh", "bsa_attention.cuh",
                                           "bsa_attention_wide.cuh", "bsa_quant.cuh")] + [
    os.path.join(INCLUDE, "bsa_fp8.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in SOURCES + HEADERS)


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "-I", CSRC, "-o", LIB, *SOURCES]
    if ptxas_info:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or r.returncode != 0:
        print(" ".join(cmd))
        print(r.stdout)
        print(r.stderr)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed building libbsa_fp8.so")
    return LIB


if __name__ == "__main__":
    build(verbose=True, ptxas_info=True)
