"""SSD quadratic form of the selective scan -- TEST INFRASTRUCTURE (pin only).

The VSSD page ("VSSD: Vision Mamba with Non-Causal State Space Duality",
§4.2.1.1 "SSD的矩阵变换形式" and §4.2.1.2 "标量化后的SSD二次形式") writes the
scan as one matrix acting on the whole input sequence: y = F x with F lower
triangular, F[t, s] = C_t · (product of the decays strictly after s up to t) ·
B_s. The page states it for a scalar A; with A per (channel, state) the same
form holds separately for every state index n, and the per-state results add:

    y_t = sum_n sum_{s <= t} C_t[n] * M_n[t, s] * B_s[n] * delta_s * x_s + D * x_t
    M_n[t, s] = prod_{k = s+1 .. t} Abar_k[n]   (1 when s = t, 0 when s > t)
    Abar_k[n] = exp(delta_k * A[n])             (0 at a folded segment start)

The page's own index bounds on the product are garbled (one version starts the
product at i+2, the other writes an empty range for i > j); the reading above
is the one under which this form equals the recurrence. This materialises an
L x L matrix per (row, n), so it is for tiny inputs only.
"""
from __future__ import annotations

import numpy as np
from scipy.special import expit


def decay_matrix(abar: np.ndarray) -> np.ndarray:
    """M[t, s] = prod_{k=s+1}^{t} abar[k] for s <= t, else 0 (explicit products)."""
    L = abar.shape[0]
    M = np.zeros((L, L), dtype=np.float64)
    for t in range(L):
        for s in range(t + 1):
            M[t, s] = np.prod(abar[s + 1:t + 1])
    return M


def scan_direction(x, delta, A, B, C, D, seg_len: int = 0, reverse: bool = False):
    """One direction for one (batch, channel) row via the quadratic form.

    x, delta: (L,); A: (N,); B, C: (L, N); D: scalar. reverse=True evaluates the
    backward direction as the forward form on the reversed sequence.
    """
    x = np.asarray(x, np.float64)
    delta = np.asarray(delta, np.float64)
    B = np.asarray(B, np.float64)
    C = np.asarray(C, np.float64)
    A = np.asarray(A, np.float64)
    L, N = B.shape
    idx = np.arange(L)
    if reverse:
        x, delta, B, C = x[::-1], delta[::-1], B[::-1], C[::-1]
        pos = idx[::-1]
    else:
        pos = idx
    y = np.zeros(L, dtype=np.float64)
    for n in range(N):
        abar = np.exp(delta * A[n])
        if seg_len > 0:
            start = (pos % seg_len == seg_len - 1) if reverse else (pos % seg_len == 0)
            abar = np.where(start, 0.0, abar)
        M = decay_matrix(abar)
        F = C[:, n][:, None] * M * B[:, n][None, :]
        y += F @ (delta * x)
    y += float(D) * x
    return y[::-1] if reverse else y


def scan(x, delta, A_fwd, A_bwd, B, C, D_fwd, D_bwd, z=None, dirs: int = 3,
         seg_len: int = 0):
    """Full bidirectional scan via the quadratic form; shapes as in the oracle."""
    x = np.asarray(x, np.float64)
    batch, dim, L = x.shape
    out = np.zeros((batch, dim, L), dtype=np.float64)
    for b in range(batch):
        for d in range(dim):
            y = np.zeros(L)
            if dirs & 1:
                y += scan_direction(x[b, d], delta[b, d], A_fwd[d], B[b], C[b],
                                    0.0 if D_fwd is None else D_fwd[d], seg_len, False)
            if dirs & 2:
                y += scan_direction(x[b, d], delta[b, d], A_bwd[d], B[b], C[b],
                                    0.0 if D_bwd is None else D_bwd[d], seg_len, True)
            if z is not None:
                zz = np.asarray(z[b, d], np.float64)
                y = y * zz * expit(zz)
            out[b, d] = y
    return out
