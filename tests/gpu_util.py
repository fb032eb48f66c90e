"""Helpers shared by the GPU tests: upload seeded inputs, compare with the
oracle. Holds no scan arithmetic."""
from __future__ import annotations

import numpy as np
import torch


def to_device(inp, device="cuda"):
    """Device tensors of a workloads.Inputs set in its storage dtype."""
    def act(name):
        a = inp.storage(name)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    t = {k: act(k) for k in ("x", "delta", "z", "B", "C")}
    for k in ("A_fwd", "A_bwd", "D_fwd", "D_bwd"):
        t[k] = torch.from_numpy(getattr(inp, k)).to(device)
    if inp.delta_bwd is not None:          # fused-step inputs
        t["delta_bwd"] = act("delta_bwd")
        t["delta_bias"] = torch.from_numpy(inp.delta_bias).to(device)
        t["delta_bias_bwd"] = torch.from_numpy(inp.delta_bias_bwd).to(device)
    if inp.conv_w is not None:             # convolution inputs
        for k in ("conv_w", "conv_b", "conv_w_bwd", "conv_b_bwd"):
            t[k] = torch.from_numpy(getattr(inp, k)).to(device)
    return t


def normwise_rel(got, ref):
    """max_i |g_i - r_i| / max_i |r_i| (the gated parity metric)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    den = float(np.max(np.abs(ref)))
    num = float(np.max(np.abs(got - ref)))
    if not np.all(np.isfinite(got)):
        return float("inf")
    return num / den if den > 0 else num


def elementwise_rel(got, ref):
    """max_i |g_i - r_i| / max(|r_i|, 1e-3 * rms(r)) (reported, not gated)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    floor = 1e-3 * float(np.sqrt(np.mean(ref ** 2))) + 1e-300
    return float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), floor)))


TOL = {"f32": 1e-4, "bf16": 2e-2}
