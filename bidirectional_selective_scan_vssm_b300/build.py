"""Build the CUDA library libvssm.so in-tree (sm_103a).

    python bidirectional_selective_scan_vssm_b300/build.py [--force] [-v]

This file is standalone (it does not import the package, whose import needs
the library).

nvcc cross-compiles without a GPU. Each kernel family is its own translation
unit; the units compile in parallel into _build/ and link into one shared
library with a plain C ABI (include/vssm.h), which the Python binding in this
package loads with ctypes.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libvssm.so")
UNITS = ["vssm_api.cu", "k_warp.cu", "k_warp_plain.cu", "k_warp_sp.cu", "k_warp_conv.cu",
         "k_warp_spconv.cu", "k_general.cu", "k_grad.cu", "k_ncssd.cu"]
SOURCES = [os.path.join(CSRC, f) for f in UNITS]
HEADERS = [os.path.join(CSRC, f) for f in ("common.cuh", "scan_kernel.cuh", "scan_warp.cuh", "scan_grad.cuh",
                                            "ncssd.cuh", "ptx.cuh", "launch.h", "k_warp_opts.cuh", "grad_ext.cuh")] + [
    os.path.join(ROOT, "include", "vssm.h")]
NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr"]


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in SOURCES + HEADERS)


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False, out: str = LIB, defines=()) -> str:
    if not force and not needs_build() and out == LIB:
        return LIB
    bdir = os.path.join(ROOT, "_build", os.path.basename(out).replace(".so", ""))
    os.makedirs(bdir, exist_ok=True)
    common = [NVCC, *ARCH, *FLAGS, "-I", os.path.join(ROOT, "include"), *[f"-D{d}" for d in defines]]
    if verbose:
        common.insert(1, "-Xptxas=-v")
    objs = [os.path.join(bdir, os.path.basename(s).replace(".cu", ".o")) for s in SOURCES]
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        logs = list(ex.map(lambda so: _run([*common, "-c", so[0], "-o", so[1]]), zip(SOURCES, objs)))
    if verbose:
        sys.stderr.write("".join(logs))
    _run([NVCC, *ARCH, "-shared", "-o", out + ".tmp", *objs, "-lcudart"])
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
