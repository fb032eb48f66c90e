"""Build the CUDA library libvssm.so in-tree (sm_103a).

    python bidirectional_selective_scan_vssm_b300/build.py [--force] [-v]

This file is standalone (it does not import the package, whose import needs
the library).

nvcc cross-compiles without a GPU. The library has a plain C ABI
(include/vssm.h); the Python binding in this package loads it with ctypes.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libvssm.so")
SOURCES = [os.path.join(CSRC, "vssm_api.cu")]
HEADERS = [os.path.join(CSRC, f) for f in ("scan_kernel.cuh", "scan_warp.cuh", "scan_grad.cuh", "ncssd.cuh", "ptx.cuh")] + [
    os.path.join(ROOT, "include", "vssm.h")]
NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-shared",
         "--expt-relaxed-constexpr"]


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in SOURCES + HEADERS)


def build(force: bool = False, verbose: bool = False, out: str = LIB, defines=()) -> str:
    if not force and not needs_build() and out == LIB:
        return LIB
    cmd = [NVCC, *ARCH, *FLAGS, "-I", os.path.join(ROOT, "include"), "-o", out + ".tmp",
           *[f"-D{d}" for d in defines], *SOURCES, "-lcudart"]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    if verbose:
        sys.stderr.write(r.stdout + r.stderr)
    os.replace(out + ".tmp", out)
    return out


PROBE_SRC = os.path.join(CSRC, "ceiling_probe.cu")
PROBE = os.path.join(PKG, "ceiling_probe")


def build_probe() -> str:
    """The MUFU / FMA-pipe ceiling probe (a standalone program)."""
    cmd = [NVCC, *ARCH, "-O3", "-std=c++17", "-o", PROBE, PROBE_SRC]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return PROBE


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
    if "--probe" in sys.argv:
        print(build_probe())
