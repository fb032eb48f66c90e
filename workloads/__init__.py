"""Seeded synthetic inputs for the bidirectional selective scan.

This module is shared by the fp64 oracle's tests and by the CUDA path's tests
and benchmark. It holds no arithmetic of the scan itself: it only draws random
tensors with the shapes and value distributions of the vision-Mamba workloads
and rounds them to the storage dtype.

Workloads (shapes from the Vim page "Vision Mamba (Vim) 双向SSM设计详解", §2.1
token construction, and the SF-Mamba page "SF-Mamba：高效视觉Mamba与辅助Patch交换",
section "批量折叠与周期性状态重置"):

==========  =====  =====  ====  ==  ======  ====  ===========  =========
name        batch  L      dim   N   dtype   dirs  seg_len      Δ mean
==========  =====  =====  ====  ==  ======  ====  ===========  =========
vim_ti_224  1      197    384   16  f32     both  -            -2
vim_s_224   128    197    768   16  bf16    both  -            -2
vim_s_512   32     1025   768   16  bf16    both  -            -2
sf_folded   1      52224  1024  16  bf16    fwd   51           -2
vim_s_1024  8      4097   768   16  bf16    both  -            -3
==========  =====  =====  ====  ==  ======  ====  ===========  =========

Value distributions (all workloads): x, z ~ N(0, 1); Δ = softplus(N(μ, 0.5));
A = -exp(U[ln 0.5, ln 16]) per (channel, state); B_t, C_t ~ N(0, 1)/sqrt(N);
D ~ N(0, 1). Forward and backward A and D are drawn independently. Draw order:
x, Δ, z, B, C, A_fwd, A_bwd, D_fwd, D_bwd from numpy's PCG64 ``default_rng``.

Layouts: x, delta, z, out are (batch, dim, L) with L fastest; B, C are
(batch, L, N) with N fastest; A is (dim, N); D is (dim,).

Fused-step variant (``fused_step=True``, any workload): the step is passed
before its positivity map, per direction. The draw at Δ's position is kept as
the pre-activation v ~ N(μ, 0.5); after D_bwd come bias_fwd, bias_bwd ~
U[-0.5, 0.5] per channel and the backward pre-activation v_b ~ N(μ, 0.5).
The stored steps are delta = v - bias_fwd and delta_bwd = v_b - bias_bwd, so
softplus(delta + bias) has the plain workloads' distribution in each direction.

Convolution variant (``conv=K``, any workload): after everything above come
the forward taps and bias, then the backward taps and bias, each ~
U[-1/sqrt(K), 1/sqrt(K)] (the usual fan-in initialisation of a depthwise
convolution with K taps); shapes (dim, K) and (dim,).

NC-SSD variant (``ncssd=True``): after everything above come the per-token
weights m ~ U[0.5, 1.5], shape (batch, L) (the VSSD page's m_j = 1/A_j, here
drawn directly).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np

DIR_FWD = 1
DIR_BWD = 2
DIR_BOTH = 3


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seqlen: int
    dim: int
    dstate: int
    dtype: str          # "f32" or "bf16": storage type of x, delta, z, B, C, out
    dirs: int           # DIR_FWD, DIR_BWD or DIR_BOTH
    seg_len: int = 0    # > 0: batch-folded sequence, state reset every seg_len tokens
    delta_mu: float = -2.0
    delta_sigma: float = 0.5
    description: str = ""
    fused_step: bool = False   # per-direction pre-activation steps + biases (softplus inside)
    conv: int = 0              # taps of the directional convolution + SiLU in front (0: none)
    ncssd: bool = False        # also draw the NC-SSD per-token weights m

    @property
    def tokch(self) -> int:
        """Token-channel count (the work unit): batch * seqlen * dim."""
        return self.batch * self.seqlen * self.dim

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("vim_ti_224", 1, 197, 384, 16, "f32", DIR_BOTH,
                 description="Vim-Ti 224^2: 14x14 patches + mid CLS, fp32 I/O"),
        Workload("vim_s_224", 128, 197, 768, 16, "bf16", DIR_BOTH,
                 description="Vim-S 224^2: batch 128, bf16 I/O, fp32 state"),
        Workload("vim_s_512", 32, 1025, 768, 16, "bf16", DIR_BOTH,
                 description="Vim-S 512^2: 32x32 patches + CLS, bf16 I/O"),
        Workload("sf_folded", 1, 52224, 1024, 16, "bf16", DIR_FWD, seg_len=51,
                 description="SF-Mamba batch-folded: 1024 sequences of 51 tokens "
                             "(7x7 patches + 2 aux) folded into one, reset every 51"),
        Workload("vim_s_1024", 8, 4097, 768, 16, "bf16", DIR_BOTH, delta_mu=-3.0,
                 description="high-res 1024^2: 64x64 patches + CLS, long-range decay"),
    ]
}
ORDER = ["vim_ti_224", "vim_s_224", "vim_s_512", "sf_folded", "vim_s_1024"]


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even).

    Returns the uint16 bit patterns. Inputs here are finite.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact float32 values of bfloat16 bit patterns."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class Inputs:
    """One seeded input set. ``*_f32`` arrays hold the exact values the scan
    consumes (bf16-rounded where the workload stores bf16); ``*_bits`` hold the
    bf16 bit patterns (None for f32 workloads)."""
    wl: Workload
    x: np.ndarray
    delta: np.ndarray
    z: np.ndarray
    B: np.ndarray
    C: np.ndarray
    A_fwd: np.ndarray
    A_bwd: np.ndarray
    D_fwd: np.ndarray
    D_bwd: np.ndarray
    bits: Optional[Dict[str, np.ndarray]] = None
    delta_bwd: Optional[np.ndarray] = None        # fused-step workloads only
    delta_bias: Optional[np.ndarray] = None
    delta_bias_bwd: Optional[np.ndarray] = None
    conv_w: Optional[np.ndarray] = None           # convolution workloads only
    conv_b: Optional[np.ndarray] = None
    conv_w_bwd: Optional[np.ndarray] = None
    conv_b_bwd: Optional[np.ndarray] = None
    m: Optional[np.ndarray] = None                # NC-SSD workloads only

    def storage(self, name: str) -> np.ndarray:
        """The array as stored for the device: uint16 bits (bf16) or float32."""
        if self.bits is not None and name in self.bits:
            return self.bits[name]
        return getattr(self, name)


def _softplus(v: np.ndarray) -> np.ndarray:
    v64 = v.astype(np.float64)
    return (np.maximum(v64, 0.0) + np.log1p(np.exp(-np.abs(v64)))).astype(np.float32)


def make_inputs(wl: Workload, seed: int = 0) -> Inputs:
    """Draw the inputs of workload ``wl`` with ``seed`` (order fixed above)."""
    rng = np.random.default_rng(seed)
    b, L, D, N = wl.batch, wl.seqlen, wl.dim, wl.dstate
    x = rng.standard_normal((b, D, L), dtype=np.float32)
    v = (rng.standard_normal((b, D, L), dtype=np.float32) * np.float32(wl.delta_sigma)
         + np.float32(wl.delta_mu))
    delta = v if wl.fused_step else _softplus(v)
    z = rng.standard_normal((b, D, L), dtype=np.float32)
    scale = np.float32(1.0 / np.sqrt(N))
    B = rng.standard_normal((b, L, N), dtype=np.float32) * scale
    C = rng.standard_normal((b, L, N), dtype=np.float32) * scale
    lo, hi = np.log(0.5), np.log(16.0)
    A_fwd = (-np.exp(rng.uniform(lo, hi, size=(D, N)))).astype(np.float32)
    A_bwd = (-np.exp(rng.uniform(lo, hi, size=(D, N)))).astype(np.float32)
    D_fwd = rng.standard_normal(D, dtype=np.float32)
    D_bwd = rng.standard_normal(D, dtype=np.float32)
    extra = {}
    if wl.fused_step:
        bias_f = rng.uniform(-0.5, 0.5, size=D).astype(np.float32)
        bias_b = rng.uniform(-0.5, 0.5, size=D).astype(np.float32)
        v_b = (rng.standard_normal((b, D, L), dtype=np.float32) * np.float32(wl.delta_sigma)
               + np.float32(wl.delta_mu))
        delta = (v - bias_f[None, :, None]).astype(np.float32)
        extra = dict(delta_bwd=(v_b - bias_b[None, :, None]).astype(np.float32),
                     delta_bias=bias_f, delta_bias_bwd=bias_b)
    if wl.conv:
        lim = 1.0 / np.sqrt(wl.conv)
        for sfx in ("", "_bwd"):
            extra["conv_w" + sfx] = rng.uniform(-lim, lim, size=(D, wl.conv)).astype(np.float32)
            extra["conv_b" + sfx] = rng.uniform(-lim, lim, size=D).astype(np.float32)
    if wl.ncssd:
        extra["m"] = rng.uniform(0.5, 1.5, size=(b, L)).astype(np.float32)
    bits = None
    if wl.dtype == "bf16":
        bits = {}
        for name, arr in (("x", x), ("delta", delta), ("z", z), ("B", B), ("C", C)):
            bits[name] = bf16_round(arr)
        x, delta, z, B, C = (bf16_to_f32(bits[k]) for k in ("x", "delta", "z", "B", "C"))
        if "delta_bwd" in extra:
            bits["delta_bwd"] = bf16_round(extra["delta_bwd"])
            extra["delta_bwd"] = bf16_to_f32(bits["delta_bwd"])
    elif wl.dtype != "f32":
        raise ValueError(f"unknown dtype {wl.dtype}")
    return Inputs(wl, x, delta, z, B, C, A_fwd, A_bwd, D_fwd, D_bwd, bits, **extra)


def algorithmic_bytes(wl: Workload) -> int:
    """Bytes a scan must move at least once: x, delta, z read and out written
    (4 * tokch elements), B and C read once per token, A and D per direction."""
    e = 4 if wl.dtype == "f32" else 2
    ndir = (1 if wl.dirs & DIR_FWD else 0) + (1 if wl.dirs & DIR_BWD else 0)
    n = (4 * wl.tokch * e + 2 * wl.batch * wl.seqlen * wl.dstate * e
         + ndir * (wl.dim * wl.dstate + wl.dim) * 4)
    if wl.fused_step:   # the backward step tensor and the per-direction biases
        n += (wl.tokch * e if wl.dirs & DIR_BWD else 0) + ndir * wl.dim * 4
    if wl.conv:         # taps and bias per direction
        n += ndir * wl.dim * (wl.conv + 1) * 4
    return n


def exp_count(wl: Workload) -> int:
    """Decay exponentials the recurrence evaluates: one per (token, channel,
    state, direction)."""
    ndir = (1 if wl.dirs & DIR_FWD else 0) + (1 if wl.dirs & DIR_BWD else 0)
    return wl.tokch * wl.dstate * ndir
