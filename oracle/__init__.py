"""fp64 CPU oracle for the bidirectional selective scan -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (the CUDA library and
its binding) never imports, links or runs anything here, and this package
shares no code with it: the only module both sides use is ``workloads`` (seeded
input generation, no scan arithmetic).

Contents:
  * ``vssm_oracle.c`` -- the recurrence written out in plain C, fp64, OpenMP
    over (batch, channel) rows. See its header for the equations and the pages
    they follow.
  * ``quadform.py`` -- the SSD page's quadratic (matrix) form, NumPy, used only
    to pin the recurrence on tiny inputs.
  * ``scan()``, ``scan_grad()``, ``conv_silu()`` and ``ncssd()`` below --
    ctypes bindings of the C oracle.

Pins (in ``tests/test_oracle_pins.py``): the quadratic form, a hand-worked
two-step example from the SSD page's linear-form section, closed forms for
A = 0 (prefix sum), vanishing decay, Δ = 0 and C = 0, L = 1, the
backward-equals-flipped-forward invariant, folded-equals-per-segment, the
silu gate against scipy's logistic function, linearity in x, the fused step
map against the closed-form inverse of softplus (and softplus(0) = ln 2), the
per-direction step as a sum of single-direction scans, the directional
convolution's taps against shifted inputs (forward, backward, across folded
segment edges) and its feed into each direction, the adjoint gradients
against central finite differences of the forward oracle, NC-SSD against the
VSSD page's matrix form and its token-order independence, and a mutation test
that plants mistakes in a copy of the C source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vssm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

DIR_FWD, DIR_BWD, DIR_BOTH = 1, 2, 3


def compile_c(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the C oracle (or a copy of it) into a shared library."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True)
    return out


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        compile_c()
    return _LIB_PATH


def load_library(path: str):
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.oracle_scan.restype = ctypes.c_int
    lib.oracle_scan.argtypes = [dp] * 12 + [ctypes.c_long] * 4 + [
        ctypes.c_int, ctypes.c_long, ctypes.c_int]
    lib.oracle_scan_ex.restype = ctypes.c_int
    lib.oracle_scan_ex.argtypes = [dp] * 14 + [ctypes.c_int, dp, dp] + [ctypes.c_long] * 4 + [
        ctypes.c_int, ctypes.c_long, ctypes.c_int]
    lib.oracle_scan_grad.restype = ctypes.c_int
    lib.oracle_scan_grad.argtypes = [dp] * 23 + [ctypes.c_long] * 4 + [ctypes.c_int, ctypes.c_long]
    lib.oracle_scan_grad_ex.restype = ctypes.c_int
    lib.oracle_scan_grad_ex.argtypes = ([dp] * 14 + [ctypes.c_int] + [dp] * 4 + [ctypes.c_long] +
                                        [dp] * 19 + [ctypes.c_long] * 4 + [ctypes.c_int, ctypes.c_long])
    lib.oracle_ncssd.restype = ctypes.c_int
    lib.oracle_ncssd.argtypes = [dp] * 7 + [ctypes.c_long] * 4
    lib.oracle_conv_silu.restype = ctypes.c_int
    lib.oracle_conv_silu.argtypes = [dp] * 4 + [ctypes.c_long] * 4 + [ctypes.c_int, ctypes.c_long]
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def _get_lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def max_threads() -> int:
    return int(_get_lib().oracle_max_threads())


def _as_f64(a):
    if a is None:
        return None, None
    arr = np.ascontiguousarray(a, dtype=np.float64)
    return arr, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def scan(x, delta, A_fwd, A_bwd, B, C, D_fwd=None, D_bwd=None, z=None,
         B_bwd=None, C_bwd=None, dirs: int = DIR_BOTH, seg_len: int = 0,
         nthreads: int = 0, lib=None, delta_bwd=None, delta_bias=None,
         delta_bias_bwd=None, delta_softplus: bool = False, conv_w=None, conv_b=None,
         conv_w_bwd=None, conv_b_bwd=None) -> np.ndarray:
    """Run the fp64 oracle. Arrays may be any float dtype; they are widened to
    float64 exactly. Shapes: x, delta, z (batch, dim, L); B, C (batch, L, N);
    A (dim, N); D (dim,). Returns out (batch, dim, L) float64.

    delta_bwd: the backward direction's step (None = delta). With
    delta_softplus each direction's step is softplus(its delta + its bias[d])
    (delta_bias, delta_bias_bwd: (dim,); None = 0 / = delta_bias).

    conv_w (dim, K) and conv_b (dim,): the directional depthwise convolution +
    SiLU in front of the scan (``conv_silu``); each direction reads its own
    convolution of x (conv_w_bwd, conv_b_bwd: None = the forward one)."""
    lib = lib or _get_lib()
    x_bwd = None
    if conv_w is not None:
        cw_b = conv_w if conv_w_bwd is None else conv_w_bwd
        cb_b = conv_b if conv_b_bwd is None else conv_b_bwd
        x_in = x
        x = conv_silu(x_in, conv_w, conv_b, reverse=False, seg_len=seg_len, lib=lib)
        x_bwd = conv_silu(x_in, cw_b, cb_b, reverse=True, seg_len=seg_len, lib=lib)
    if delta_bwd is not None or delta_bias is not None or delta_bias_bwd is not None \
            or delta_softplus or x_bwd is not None:
        return _scan_ex(lib, x, delta, A_fwd, A_bwd, B, C, D_fwd, D_bwd, z, B_bwd, C_bwd,
                        dirs, seg_len, nthreads, delta_bwd, delta_bias, delta_bias_bwd,
                        delta_softplus, x_bwd)
    x = np.asarray(x)
    batch, dim, L = x.shape
    N = np.asarray(B).shape[-1]
    if A_fwd is None and A_bwd is None:
        raise ValueError("need A for the selected direction(s)")
    keep = []
    ptrs = []
    for a in (x, delta, z, B, C, B_bwd, C_bwd, A_fwd, A_bwd, D_fwd, D_bwd):
        arr, p = _as_f64(a)
        keep.append(arr)
        ptrs.append(p)
    out = np.empty((batch, dim, L), dtype=np.float64)
    pout = out.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    rc = lib.oracle_scan(*ptrs, pout, batch, dim, L, N, int(dirs), int(seg_len),
                         int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_scan rejected its arguments (status {rc})")
    return out


def ncssd(x, B, C, m, D=None, z=None, lib=None) -> np.ndarray:
    """NC-SSD (C oracle ``oracle_ncssd``): x, z (batch, dim, L); B, C
    (batch, L, N); m (batch, L) token weights; D (dim,) or None. float64."""
    lib = lib or _get_lib()
    x = np.asarray(x)
    batch, dim, L = x.shape
    N = np.asarray(B).shape[-1]
    keep, ptrs = [], []
    for a in (x, z, B, C, m, D):
        arr, p = _as_f64(a)
        keep.append(arr)
        ptrs.append(p)
    out = np.empty((batch, dim, L), dtype=np.float64)
    rc = lib.oracle_ncssd(*ptrs, out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                          batch, dim, L, N)
    if rc != 0:
        raise ValueError(f"oracle_ncssd rejected its arguments (status {rc})")
    return out


def conv_silu(x, w, b=None, reverse: bool = False, seg_len: int = 0, lib=None) -> np.ndarray:
    """Directional depthwise convolution + SiLU (C oracle ``oracle_conv_silu``):
    x (batch, dim, L), w (dim, K), b (dim,) or None. reverse=False is the
    causal (forward) convolution, True the backward one."""
    lib = lib or _get_lib()
    x = np.asarray(x)
    batch, dim, L = x.shape
    w = np.asarray(w)
    K = w.shape[-1]
    xa, px = _as_f64(x)
    wa, pw = _as_f64(w)
    ba, pb = _as_f64(b)
    out = np.empty((batch, dim, L), dtype=np.float64)
    rc = lib.oracle_conv_silu(px, pw, pb, out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                              batch, dim, L, K, int(bool(reverse)), int(seg_len))
    if rc != 0:
        raise ValueError(f"oracle_conv_silu rejected its arguments (status {rc})")
    return out


def _scan_ex(lib, x, delta, A_fwd, A_bwd, B, C, D_fwd, D_bwd, z, B_bwd, C_bwd, dirs, seg_len,
             nthreads, delta_bwd, delta_bias, delta_bias_bwd, delta_softplus, x_bwd=None):
    x = np.asarray(x)
    batch, dim, L = x.shape
    N = np.asarray(B).shape[-1]
    keep, ptrs = [], []
    for a in (x, delta, z, B, C, B_bwd, C_bwd, A_fwd, A_bwd, D_fwd, D_bwd,
              delta_bwd, delta_bias, delta_bias_bwd):
        arr, p = _as_f64(a)
        keep.append(arr)
        ptrs.append(p)
    xb, pxb = _as_f64(x_bwd)
    out = np.empty((batch, dim, L), dtype=np.float64)
    pout = out.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    rc = lib.oracle_scan_ex(*ptrs, int(bool(delta_softplus)), pxb, pout, batch, dim, L, N,
                            int(dirs), int(seg_len), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_scan_ex rejected its arguments (status {rc})")
    return out


def scan_grad(x, delta, A_fwd, A_bwd, B, C, D_fwd=None, D_bwd=None, z=None, dout=None,
              B_bwd=None, C_bwd=None, dirs: int = DIR_BOTH, seg_len: int = 0, lib=None,
              delta_bwd=None, delta_bias=None, delta_bias_bwd=None, delta_softplus: bool = False,
              conv_w=None, conv_b=None, conv_w_bwd=None, conv_b_bwd=None) -> dict:
    """Gradients of L = sum(dout * scan(...)) (C oracle ``oracle_scan_grad_ex``),
    for the plain scan or with the step options and the convolution of
    ``scan``: dict with dx, ddelta, dz (None without z), dB, dC, dB_bwd / dC_bwd
    (None when the backward direction shares B / C), dA_fwd, dA_bwd, dD_fwd,
    dD_bwd (None for a direction that is not run), ddelta_bwd (with
    delta_bwd), ddelta_bias / ddelta_bias_bwd (with softplus; the backward
    one only with its own bias), dconv_w, dconv_b, dconv_w_bwd, dconv_b_bwd
    (with the convolution; each only for a given parameter). float64. A
    backward parameter that is not given is the forward one, and its
    gradient is included in the forward one's."""
    lib = lib or _get_lib()
    x = np.asarray(x)
    batch, dim, L = x.shape
    N = np.asarray(B).shape[-1]
    K = 0 if conv_w is None else np.asarray(conv_w).shape[-1]
    keep, ptrs = [], []
    for a in (x, delta, z, B, C, B_bwd, C_bwd, A_fwd, A_bwd, D_fwd, D_bwd, delta_bwd,
              delta_bias, delta_bias_bwd):
        arr, p = _as_f64(a)
        keep.append(arr)
        ptrs.append(p)
    cptrs = []
    for a in (conv_w, conv_b, conv_w_bwd, conv_b_bwd):
        arr, p = _as_f64(a)
        keep.append(arr)
        cptrs.append(p)
    dout_arr, dout_p = _as_f64(dout)
    act = lambda: np.zeros((batch, dim, L))
    bc = lambda: np.zeros((batch, L, N))
    sp = bool(delta_softplus)
    g = dict(dx=act(), ddelta=act(), dz=act() if z is not None else None, dB=bc(), dC=bc(),
             dB_bwd=bc() if B_bwd is not None else None, dC_bwd=bc() if C_bwd is not None else None,
             dA_fwd=np.zeros((dim, N)) if dirs & DIR_FWD else None,
             dA_bwd=np.zeros((dim, N)) if dirs & DIR_BWD else None,
             dD_fwd=np.zeros(dim) if dirs & DIR_FWD else None,
             dD_bwd=np.zeros(dim) if dirs & DIR_BWD else None,
             ddelta_bwd=act() if delta_bwd is not None else None,
             ddelta_bias=np.zeros(dim) if sp else None,
             ddelta_bias_bwd=np.zeros(dim) if sp and delta_bias_bwd is not None else None,
             dconv_w=np.zeros((dim, K)) if K else None,
             dconv_b=np.zeros(dim) if K and conv_b is not None else None,
             dconv_w_bwd=np.zeros((dim, K)) if K and conv_w_bwd is not None else None,
             dconv_b_bwd=np.zeros(dim) if K and conv_b_bwd is not None else None)
    outp = [_as_f64(g[k])[1] if g[k] is not None else None
            for k in ("dx", "ddelta", "dz", "dB", "dC", "dB_bwd", "dC_bwd", "dA_fwd", "dA_bwd",
                      "dD_fwd", "dD_bwd", "ddelta_bwd", "ddelta_bias", "ddelta_bias_bwd",
                      "dconv_w", "dconv_b", "dconv_w_bwd", "dconv_b_bwd")]
    # _as_f64 returns the same array for float64 C-contiguous input, so the
    # pointers above write into g's arrays
    rc = lib.oracle_scan_grad_ex(*ptrs, int(sp), *cptrs, K, dout_p, *outp, batch, dim, L, N,
                                 int(dirs), int(seg_len))
    if rc != 0:
        raise ValueError(f"oracle_scan_grad_ex rejected its arguments (status {rc})")
    return g


def scan_inputs(inp, dirs: Optional[int] = None, seg_len: Optional[int] = None,
                nthreads: int = 0) -> np.ndarray:
    """Oracle on a ``workloads.Inputs`` set (its exact, possibly bf16-rounded
    values)."""
    wl = inp.wl
    return scan(inp.x, inp.delta, inp.A_fwd, inp.A_bwd, inp.B, inp.C,
                inp.D_fwd, inp.D_bwd, inp.z,
                dirs=wl.dirs if dirs is None else dirs,
                seg_len=wl.seg_len if seg_len is None else seg_len,
                nthreads=nthreads)


def scan_rows(inp, rows, nthreads: int = 0) -> np.ndarray:
    """Oracle outputs of selected (b, d) rows only: returns (len(rows), L)."""
    wl = inp.wl
    out = np.empty((len(rows), wl.seqlen), dtype=np.float64)
    for i, (b, d) in enumerate(rows):
        sl = (slice(b, b + 1), slice(d, d + 1))
        out[i] = scan(inp.x[sl], inp.delta[sl], inp.A_fwd[d:d + 1], inp.A_bwd[d:d + 1],
                      inp.B[b:b + 1], inp.C[b:b + 1], inp.D_fwd[d:d + 1],
                      inp.D_bwd[d:d + 1], inp.z[sl], dirs=wl.dirs,
                      seg_len=wl.seg_len, nthreads=nthreads)[0, 0]
    return out
