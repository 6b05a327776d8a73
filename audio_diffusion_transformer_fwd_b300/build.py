"""Build libh3dit.so in-tree with nvcc for sm_103a.

    python -m audio_diffusion_transformer_fwd_b300.build [--verbose-ptxas]

The library is a single translation unit (csrc/h3dit_api.cu includes every
kernel file) linked against the static CUDA runtime, so the .so carries no
dependency beyond the driver.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libh3dit.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh")))


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = sources() + [os.path.join(ROOT, "include", "h3dit.h")]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, ptxas_verbose: bool = False) -> str:
    if not force and not needs_build():
        return LIB
    cmd = [
        NVCC, "-O3", "-std=c++17", "-lineinfo",
        "-gencode", "arch=compute_103a,code=sm_103a",
        "-Xcompiler", "-fPIC", "-shared", "-cudart", "static",
        "-I", os.path.join(ROOT, "include"),
        os.path.join(CSRC, "h3dit_api.cu"),
        "-o", LIB + ".tmp",
    ]
    if ptxas_verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    build(force=True, ptxas_verbose="--verbose-ptxas" in sys.argv)
    print(LIB)
