"""Pins for the fp64 oracle, written as functions of a loaded oracle library so
that the same checks can run against deliberately broken copies of the C
source (see test_oracle_pins.test_planted_mistakes_are_caught).

Every check compares the oracle with something other than itself: a value
worked by hand from the pages, a closed form, a second formulation (the SSD
quadratic form), or an invariant the pages state.
"""
from __future__ import annotations

import os

import numpy as np
from scipy.special import expit

import oracle
from oracle import quadform

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rand_problem(rng, batch, dim, L, N, gate=True, A_scale=1.0):
    x = rng.standard_normal((batch, dim, L))
    delta = np.log1p(np.exp(rng.normal(-1.0, 0.5, size=(batch, dim, L))))
    z = rng.standard_normal((batch, dim, L)) if gate else None
    B = rng.standard_normal((batch, L, N)) / np.sqrt(N)
    C = rng.standard_normal((batch, L, N)) / np.sqrt(N)
    A_f = -np.exp(rng.uniform(np.log(0.5), np.log(16), size=(dim, N))) * A_scale
    A_b = -np.exp(rng.uniform(np.log(0.5), np.log(16), size=(dim, N))) * A_scale
    D_f = rng.standard_normal(dim)
    D_b = rng.standard_normal(dim)
    return dict(x=x, delta=delta, z=z, B=B, C=C, A_fwd=A_f, A_bwd=A_b,
                D_fwd=D_f, D_bwd=D_b)


def _run(lib, p, **kw):
    return oracle.scan(p["x"], p["delta"], p["A_fwd"], p["A_bwd"], p["B"], p["C"],
                       p["D_fwd"], p["D_bwd"], p["z"], lib=lib, **kw)


def _close(a, b, tol):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    return bool(np.all(np.isfinite(a))) and float(np.max(np.abs(a - b), initial=0.0)) <= tol * scale


def read_golden(name="ssd_linear_form_worked_example.txt"):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            vals[k.strip()] = np.array([float(t) for t in v.split()])
    return vals


# ---------------------------------------------------------------- the pins

def pin_worked_example(lib):
    g = read_golden()
    x = g["x"].reshape(1, 1, -1)
    L = x.shape[-1]
    delta = np.ones_like(x)
    A = np.array([[np.log(g["abar"][0])]])
    B = np.full((1, L, 1), g["dbx_scale"][0])
    C = np.ones((1, L, 1))
    ok = True
    for key, dirs, seg in (("fwd", 1, 0), ("bwd", 2, 0), ("fwd_fold2", 1, 2), ("bwd_fold2", 2, 2)):
        out = oracle.scan(x, delta, A, A, B, C, None, None, None, dirs=dirs,
                          seg_len=seg, lib=lib)
        ok &= _close(out[0, 0], g[key], 1e-12)
    return ok


def pin_quadratic_form(lib):
    rng = np.random.default_rng(11)
    ok = True
    for L, N, dirs, seg in ((1, 1, 3, 0), (5, 4, 1, 0), (7, 3, 2, 0), (17, 4, 3, 0),
                            (12, 2, 3, 4), (13, 3, 1, 5), (40, 4, 3, 8)):
        p = _rand_problem(rng, 2, 3, L, N)
        got = _run(lib, p, dirs=dirs, seg_len=seg)
        ref = quadform.scan(p["x"], p["delta"], p["A_fwd"], p["A_bwd"], p["B"], p["C"],
                            p["D_fwd"], p["D_bwd"], p["z"], dirs=dirs, seg_len=seg)
        ok &= _close(got, ref, 1e-12)
    return ok


def pin_A_zero_prefix_sum(lib):
    """A = 0: every decay is exactly 1, so h_t is the running sum of
    delta_s B_s x_s (a textbook prefix sum)."""
    rng = np.random.default_rng(12)
    p = _rand_problem(rng, 2, 3, 33, 4, gate=False)
    p["A_fwd"] = np.zeros_like(p["A_fwd"])
    p["A_bwd"] = np.zeros_like(p["A_bwd"])
    got = _run(lib, p, dirs=3)
    ref = np.empty_like(got)
    for b in range(2):
        for d in range(3):
            u = (p["delta"][b, d] * p["x"][b, d])[:, None] * p["B"][b]     # (L, N)
            hf = np.cumsum(u, axis=0)
            hb = np.cumsum(u[::-1], axis=0)[::-1]
            ref[b, d] = (np.sum(p["C"][b] * hf, axis=1) + np.sum(p["C"][b] * hb, axis=1)
                         + (p["D_fwd"][d] + p["D_bwd"][d]) * p["x"][b, d])
    return _close(got, ref, 1e-12)


def pin_vanishing_decay(lib):
    """Decay exactly 0 (exp underflows): h_t = delta_t B_t x_t, so
    y_t = (C_t . B_t) delta_t x_t + D x_t in each direction."""
    rng = np.random.default_rng(13)
    p = _rand_problem(rng, 1, 4, 9, 4, gate=False)
    p["A_fwd"] = np.full_like(p["A_fwd"], -1e308)
    p["A_bwd"] = np.full_like(p["A_bwd"], -1e308)
    got = _run(lib, p, dirs=3)
    cb = np.sum(p["C"][0] * p["B"][0], axis=1)
    ref = (2 * cb[None, :] * p["delta"][0] * p["x"][0]
           + (p["D_fwd"] + p["D_bwd"])[:, None] * p["x"][0])
    return _close(got[0], ref, 1e-12)


def pin_zero_input_paths(lib):
    """delta = 0 or C = 0 leaves only the skip: out = (D_f + D_b) x silu(z)."""
    rng = np.random.default_rng(14)
    ok = True
    for which in ("delta", "C"):
        p = _rand_problem(rng, 2, 3, 10, 4)
        p[which] = np.zeros_like(p[which])
        got = _run(lib, p, dirs=3)
        ref = ((p["D_fwd"] + p["D_bwd"])[None, :, None] * p["x"]
               * p["z"] * expit(p["z"]))
        ok &= _close(got, ref, 1e-12)
    return ok


def pin_single_token(lib):
    """L = 1: y = (C . B) delta x + D x per direction (no history)."""
    rng = np.random.default_rng(15)
    p = _rand_problem(rng, 3, 5, 1, 4, gate=False)
    got = _run(lib, p, dirs=3)
    cb = np.sum(p["C"][:, 0, :] * p["B"][:, 0, :], axis=1)          # (batch,)
    ref = (2 * cb[:, None, None] * p["delta"] * p["x"]
           + (p["D_fwd"] + p["D_bwd"])[None, :, None] * p["x"])
    return _close(got, ref, 1e-12)


def pin_backward_is_flipped_forward(lib):
    """Vim page §2.2: the backward path is the forward scan of the reversed
    sequence (with the backward A, D)."""
    rng = np.random.default_rng(16)
    p = _rand_problem(rng, 2, 3, 23, 4)
    bwd = _run(lib, p, dirs=2)
    q = dict(p)
    for k in ("x", "delta", "z"):
        q[k] = p[k][:, :, ::-1]
    for k in ("B", "C"):
        q[k] = p[k][:, ::-1, :]
    q["A_fwd"], q["D_fwd"] = p["A_bwd"], p["D_bwd"]
    fwd_of_flip = _run(lib, q, dirs=1)
    return _close(bwd, fwd_of_flip[:, :, ::-1], 1e-13)


def pin_folded_equals_segments(lib):
    """SF-Mamba page: the folded output equals the unfolded output. Fold B2
    sequences of T tokens into one row with a reset every T tokens."""
    rng = np.random.default_rng(17)
    ok = True
    T, B2, dim, N = 6, 5, 3, 4
    p = _rand_problem(rng, B2, dim, T, N)           # B2 independent sequences
    for dirs in (1, 2, 3):
        ref = _run(lib, p, dirs=dirs)                # (B2, dim, T)
        f = {}
        for k in ("x", "delta", "z"):                # (1, dim, B2*T)
            f[k] = p[k].transpose(1, 0, 2).reshape(1, dim, B2 * T)
        for k in ("B", "C"):                         # (1, B2*T, N)
            f[k] = p[k].reshape(1, B2 * T, N)
        for k in ("A_fwd", "A_bwd", "D_fwd", "D_bwd"):
            f[k] = p[k]
        got = _run(lib, f, dirs=dirs, seg_len=T)
        ok &= _close(got.reshape(dim, B2, T).transpose(1, 0, 2), ref, 1e-13)
    return ok


def pin_reset_first_token(lib):
    """A reset at t = 0 of every segment gives h_t = delta_t B_t x_t there."""
    rng = np.random.default_rng(18)
    p = _rand_problem(rng, 1, 2, 12, 4, gate=False)
    p["D_fwd"] = np.zeros_like(p["D_fwd"])
    got = _run(lib, p, dirs=1, seg_len=4)
    ok = True
    for t in (0, 4, 8):
        cb = np.sum(p["C"][0, t] * p["B"][0, t])
        ok &= _close(got[0, :, t], cb * p["delta"][0, :, t] * p["x"][0, :, t], 1e-13)
    return ok


def pin_gate(lib):
    """out = y * z * sigmoid(z): compare to the ungated run times scipy's
    logistic function; z = 0 gives exactly 0."""
    rng = np.random.default_rng(19)
    p = _rand_problem(rng, 2, 3, 8, 4)
    gated = _run(lib, p, dirs=3)
    q = dict(p)
    q["z"] = None
    plain = _run(lib, q, dirs=3)
    ok = _close(gated, plain * p["z"] * expit(p["z"]), 1e-13)
    q["z"] = np.zeros_like(p["z"])
    ok &= bool(np.all(_run(lib, q, dirs=3) == 0.0))
    return ok


def pin_linearity(lib):
    """For fixed delta, B, C, z the scan is linear in x."""
    rng = np.random.default_rng(20)
    p = _rand_problem(rng, 2, 3, 15, 4)
    x1, x2 = p["x"], rng.standard_normal(p["x"].shape)
    a, b = 0.7, -1.3
    q = dict(p)
    y1 = _run(lib, p, dirs=3)
    q["x"] = x2
    y2 = _run(lib, q, dirs=3)
    q["x"] = a * x1 + b * x2
    y3 = _run(lib, q, dirs=3)
    return _close(y3, a * y1 + b * y2, 1e-12)


def _softplus_inverse(step):
    """The pre-activation whose softplus is `step` (> 0): log(exp(step) - 1),
    from the closed form of the inverse."""
    return np.log(np.expm1(step))


def pin_softplus_step(lib):
    """Fused step map: softplus(delta + bias) per direction, checked against
    targets built with the closed-form inverse of softplus. A direction fed
    raw = log(expm1(s)) - bias must scan exactly like the plain oracle fed the
    step s; both directions together (no gate) are the sum of the two
    single-direction scans, each with its own step and bias."""
    rng = np.random.default_rng(31)
    p = _rand_problem(rng, 2, 5, 23, 6, gate=False)
    s_f = np.exp(rng.normal(-1.5, 0.6, size=p["x"].shape))      # target steps, > 0
    s_b = np.exp(rng.normal(-1.0, 0.6, size=p["x"].shape))
    bias_f = rng.normal(0.0, 1.0, size=5)
    bias_b = rng.normal(0.0, 1.0, size=5)
    raw_f = _softplus_inverse(s_f) - bias_f[None, :, None]
    raw_b = _softplus_inverse(s_b) - bias_b[None, :, None]
    ok = True
    for dirs in (1, 2, 3):
        got = oracle.scan(p["x"], raw_f, p["A_fwd"], p["A_bwd"], p["B"], p["C"], p["D_fwd"],
                          p["D_bwd"], None, dirs=dirs, lib=lib, delta_bwd=raw_b,
                          delta_bias=bias_f, delta_bias_bwd=bias_b, delta_softplus=True)
        want = 0.0
        if dirs & 1:
            want = want + oracle.scan(p["x"], s_f, p["A_fwd"], p["A_bwd"], p["B"], p["C"],
                                      p["D_fwd"], p["D_bwd"], None, dirs=1, lib=lib)
        if dirs & 2:
            want = want + oracle.scan(p["x"], s_b, p["A_fwd"], p["A_bwd"], p["B"], p["C"],
                                      p["D_fwd"], p["D_bwd"], None, dirs=2, lib=lib)
        ok = ok and _close(got, want, 1e-10)
    # softplus(0) = ln 2: raw = -bias gives the constant step ln 2
    zero = -np.broadcast_to(bias_f[None, :, None], p["x"].shape)
    got = oracle.scan(p["x"], zero, p["A_fwd"], p["A_bwd"], p["B"], p["C"], p["D_fwd"],
                      p["D_bwd"], None, dirs=1, lib=lib, delta_bias=bias_f, delta_softplus=True)
    want = oracle.scan(p["x"], np.full(p["x"].shape, np.log(2.0)), p["A_fwd"], p["A_bwd"],
                       p["B"], p["C"], p["D_fwd"], p["D_bwd"], None, dirs=1, lib=lib)
    ok = ok and _close(got, want, 1e-12)
    # large pre-activations: softplus(v) = v to within exp(-v); no overflow at 800
    for v in (40.0, 800.0):
        big = np.full(p["x"].shape, v)
        got = oracle.scan(p["x"], big, p["A_fwd"], p["A_bwd"], p["B"], p["C"], p["D_fwd"],
                          p["D_bwd"], None, dirs=1, lib=lib, delta_softplus=True)
        want = oracle.scan(p["x"], big, p["A_fwd"], p["A_bwd"], p["B"], p["C"], p["D_fwd"],
                           p["D_bwd"], None, dirs=1, lib=lib)
        ok = ok and _close(got, want, 1e-12)
    return ok


def pin_per_direction_step(lib):
    """The backward direction with its own step: both directions (no gate) are
    the forward scan with delta plus the backward scan with delta_bwd, and the
    backward scan with delta_bwd is the forward scan of the flipped sequence
    (A_bwd, D_bwd, flipped delta_bwd, x, B, C)."""
    rng = np.random.default_rng(37)
    p = _rand_problem(rng, 2, 4, 19, 5, gate=False)
    d_b = np.log1p(np.exp(rng.normal(-0.5, 0.5, size=p["x"].shape)))
    both = oracle.scan(p["x"], p["delta"], p["A_fwd"], p["A_bwd"], p["B"], p["C"], p["D_fwd"],
                       p["D_bwd"], None, dirs=3, lib=lib, delta_bwd=d_b)
    fwd = oracle.scan(p["x"], p["delta"], p["A_fwd"], p["A_bwd"], p["B"], p["C"], p["D_fwd"],
                      p["D_bwd"], None, dirs=1, lib=lib)
    bwd = oracle.scan(p["x"], p["delta"], p["A_fwd"], p["A_bwd"], p["B"], p["C"], p["D_fwd"],
                      p["D_bwd"], None, dirs=2, lib=lib, delta_bwd=d_b)
    fl = lambda a: np.ascontiguousarray(a[..., ::-1])
    fB = np.ascontiguousarray(p["B"][:, ::-1, :])
    fC = np.ascontiguousarray(p["C"][:, ::-1, :])
    flipped = fl(oracle.scan(fl(p["x"]), fl(d_b), p["A_bwd"], p["A_bwd"], fB, fC, p["D_bwd"],
                             p["D_bwd"], None, dirs=1, lib=lib))
    return _close(both, fwd + bwd, 1e-12) and _close(bwd, flipped, 1e-12)


def _shift(a, s):
    """a[..., t - s] along the last axis, zero where t - s falls outside."""
    out = np.zeros_like(a)
    L = a.shape[-1]
    if s >= 0:
        out[..., s:] = a[..., :L - s] if s < L else 0.0
    else:
        out[..., :L + s] = a[..., -s:] if -s < L else 0.0
    return out


def _silu(v):
    return v * expit(v)


def pin_conv_taps(lib):
    """Directional convolution + SiLU against shifted inputs: a one-hot tap k
    of K = 4 reads x[t - 3 + k] going forward and x[t + 3 - k] going
    backward (zero outside the row, and outside the segment on a folded
    row); two taps add; a bias alone gives silu(bias)."""
    rng = np.random.default_rng(41)
    x = rng.standard_normal((2, 3, 17))
    ok = True
    for k in range(4):
        w = np.zeros((3, 4))
        w[:, k] = 1.0
        ok = ok and _close(oracle.conv_silu(x, w, lib=lib), _silu(_shift(x, 3 - k)), 1e-14)
        ok = ok and _close(oracle.conv_silu(x, w, reverse=True, lib=lib),
                           _silu(_shift(x, k - 3)), 1e-14)
    w = np.zeros((3, 4))
    w[:, 0], w[:, 3] = 0.5, -2.0
    ok = ok and _close(oracle.conv_silu(x, w, lib=lib),
                       _silu(0.5 * _shift(x, 3) - 2.0 * x), 1e-14)
    bias = rng.standard_normal(3)
    ok = ok and _close(oracle.conv_silu(x, np.zeros((3, 4)), bias, lib=lib),
                       np.broadcast_to(_silu(bias)[None, :, None], x.shape), 1e-14)
    # folded rows: segments of 5, the taps stop at segment edges
    w = np.zeros((3, 4))
    w[:, 1] = 1.0                     # x[t - 2] forward, x[t + 2] backward
    seg = 5
    t = np.arange(17)
    keep_f = (t % seg) >= 2
    keep_b = (t % seg) <= seg - 3
    keep_b &= t + 2 < 17
    ok = ok and _close(oracle.conv_silu(x, w, seg_len=seg, lib=lib),
                       _silu(_shift(x, 2) * keep_f), 1e-14)
    ok = ok and _close(oracle.conv_silu(x, w, reverse=True, seg_len=seg, lib=lib),
                       _silu(_shift(x, -2) * keep_b), 1e-14)
    return ok


def pin_conv_feeds_each_direction(lib):
    """With the convolution on, both directions (no gate) are the forward
    scan of the forward convolution plus the backward scan of the backward
    convolution, each with its own weights."""
    rng = np.random.default_rng(43)
    p = _rand_problem(rng, 2, 4, 21, 5, gate=False)
    w_f, w_b = rng.standard_normal((4, 4)) * 0.5, rng.standard_normal((4, 4)) * 0.5
    b_f, b_b = rng.standard_normal(4) * 0.3, rng.standard_normal(4) * 0.3
    both = oracle.scan(p["x"], p["delta"], p["A_fwd"], p["A_bwd"], p["B"], p["C"], p["D_fwd"],
                       p["D_bwd"], None, dirs=3, lib=lib, conv_w=w_f, conv_b=b_f,
                       conv_w_bwd=w_b, conv_b_bwd=b_b)
    u_f = oracle.conv_silu(p["x"], w_f, b_f, lib=lib)
    u_b = oracle.conv_silu(p["x"], w_b, b_b, reverse=True, lib=lib)
    fwd = oracle.scan(u_f, p["delta"], p["A_fwd"], p["A_bwd"], p["B"], p["C"], p["D_fwd"],
                      p["D_bwd"], None, dirs=1, lib=lib)
    bwd = oracle.scan(u_b, p["delta"], p["A_fwd"], p["A_bwd"], p["B"], p["C"], p["D_fwd"],
                      p["D_bwd"], None, dirs=2, lib=lib)
    return _close(both, fwd + bwd, 1e-12)


def _grad_fd_ok(lib, rng, dirs, gate, seg_len, own_bc, L=6):
    """Every entry of every gradient of L = sum(dout * out) against a central
    finite difference of the (pinned) forward oracle."""
    b, d, N = 1, 2, 3
    p = _rand_problem(rng, b, d, L, N, gate=gate)
    if own_bc:
        p["B_bwd"] = rng.standard_normal((b, L, N)) / np.sqrt(N)
        p["C_bwd"] = rng.standard_normal((b, L, N)) / np.sqrt(N)
    dout = rng.standard_normal((b, d, L))
    keys = ("x", "delta", "A_fwd", "A_bwd", "B", "C", "D_fwd", "D_bwd", "z", "B_bwd", "C_bwd")

    def loss(q):
        out = oracle.scan(q["x"], q["delta"], q["A_fwd"], q["A_bwd"], q["B"], q["C"], q["D_fwd"],
                          q["D_bwd"], q.get("z"), B_bwd=q.get("B_bwd"), C_bwd=q.get("C_bwd"),
                          dirs=dirs, seg_len=seg_len, lib=lib)
        return float(np.sum(dout * out))

    g = oracle.scan_grad(p["x"], p["delta"], p["A_fwd"], p["A_bwd"], p["B"], p["C"], p["D_fwd"],
                         p["D_bwd"], p.get("z"), dout, B_bwd=p.get("B_bwd"),
                         C_bwd=p.get("C_bwd"), dirs=dirs, seg_len=seg_len, lib=lib)
    names = {"x": "dx", "delta": "ddelta", "z": "dz", "B": "dB", "C": "dC", "B_bwd": "dB_bwd",
             "C_bwd": "dC_bwd", "A_fwd": "dA_fwd", "A_bwd": "dA_bwd", "D_fwd": "dD_fwd",
             "D_bwd": "dD_bwd"}
    eps = 1e-6
    for k in keys:
        if p.get(k) is None:
            continue
        if k.endswith("_fwd") and not dirs & 1 or k.endswith("_bwd") and not dirs & 2:
            continue
        fd = np.zeros_like(p[k])
        for idx in np.ndindex(p[k].shape):
            q = {kk: (vv.copy() if isinstance(vv, np.ndarray) else vv) for kk, vv in p.items()}
            q[k][idx] += eps
            lp = loss(q)
            q[k][idx] -= 2 * eps
            fd[idx] = (lp - loss(q)) / (2 * eps)
        if not _close(g[names[k]], fd, 1e-6):
            return False
    return True


def _grad_opts_fd_ok(lib, rng, dirs, seg_len, sp, own_step, own_bias, K, own_conv, L=7):
    """As _grad_fd_ok, with the fused step (softplus(delta + bias), the
    backward direction's own delta and bias) and the directional convolution
    (own backward taps and bias or shared): every entry of every gradient,
    the raw steps, biases and taps included, against a central finite
    difference of the forward oracle with the same options."""
    b, d, N = 1, 2, 3
    p = _rand_problem(rng, b, d, L, N, gate=True)
    p["delta"] = rng.normal(-1.0, 0.6, (b, d, L))            # raw step (pre-softplus when sp)
    if not sp:
        p["delta"] = np.abs(p["delta"]) * 0.5 + 0.05
    if own_step:
        p["delta_bwd"] = (rng.normal(-1.0, 0.6, (b, d, L)) if sp
                          else rng.uniform(0.05, 0.6, (b, d, L)))
    if sp:
        p["delta_bias"] = rng.uniform(-0.5, 0.5, d)
        if own_bias:
            p["delta_bias_bwd"] = rng.uniform(-0.5, 0.5, d)
    if K:
        p["conv_w"] = rng.uniform(-0.8, 0.8, (d, K))
        p["conv_b"] = rng.uniform(-0.3, 0.3, d)
        if own_conv:
            p["conv_w_bwd"] = rng.uniform(-0.8, 0.8, (d, K))
            p["conv_b_bwd"] = rng.uniform(-0.3, 0.3, d)
    dout = rng.standard_normal((b, d, L))
    opt_keys = ("delta_bwd", "delta_bias", "delta_bias_bwd", "conv_w", "conv_b", "conv_w_bwd",
                "conv_b_bwd")

    def opts(q):
        o = {k: q.get(k) for k in opt_keys}
        o["delta_softplus"] = sp
        return o

    def loss(q):
        out = oracle.scan(q["x"], q["delta"], q["A_fwd"], q["A_bwd"], q["B"], q["C"], q["D_fwd"],
                          q["D_bwd"], q["z"], dirs=dirs, seg_len=seg_len, lib=lib, **opts(q))
        return float(np.sum(dout * out))

    g = oracle.scan_grad(p["x"], p["delta"], p["A_fwd"], p["A_bwd"], p["B"], p["C"], p["D_fwd"],
                         p["D_bwd"], p["z"], dout, dirs=dirs, seg_len=seg_len, lib=lib, **opts(p))
    names = {"x": "dx", "delta": "ddelta", "z": "dz", "B": "dB", "C": "dC", "A_fwd": "dA_fwd",
             "A_bwd": "dA_bwd", "D_fwd": "dD_fwd", "D_bwd": "dD_bwd", "delta_bwd": "ddelta_bwd",
             "delta_bias": "ddelta_bias", "delta_bias_bwd": "ddelta_bias_bwd", "conv_w": "dconv_w",
             "conv_b": "dconv_b", "conv_w_bwd": "dconv_w_bwd", "conv_b_bwd": "dconv_b_bwd"}
    eps = 1e-6
    for k, name in names.items():
        if p.get(k) is None:
            continue
        if k in ("A_fwd", "D_fwd") and not dirs & 1 or k in ("A_bwd", "D_bwd") and not dirs & 2:
            continue
        if g.get(name) is None:
            return False
        fd = np.zeros_like(p[k])
        for idx in np.ndindex(p[k].shape):
            q = {kk: (vv.copy() if isinstance(vv, np.ndarray) else vv) for kk, vv in p.items()}
            q[k][idx] += eps
            lp = loss(q)
            q[k][idx] -= 2 * eps
            fd[idx] = (lp - loss(q)) / (2 * eps)
        if not _close(g[name], fd, 1e-6):
            return False
    return True


def pin_gradient_step_options_fd(lib):
    """The gradient through the fused step map softplus(delta + bias) (the
    raw step and the bias), with a shared step, the backward direction's own
    step, and its own bias, on plain and folded rows, against central finite
    differences of the forward oracle."""
    rng = np.random.default_rng(61)
    ok = True
    for dirs, seg, sp, own_step, own_bias in ((3, 0, True, False, False), (3, 0, True, True, True),
                                              (3, 0, False, True, False), (2, 0, True, True, False),
                                              (3, 4, True, True, True)):
        ok = ok and _grad_opts_fd_ok(lib, rng, dirs, seg, sp, own_step, own_bias, 0, False,
                                     L=2 * seg if seg else 7)
    return ok


def pin_gradient_conv_fd(lib):
    """The gradient through the directional convolution + SiLU (x through
    the taps of both directions, the taps and the biases, shared or per
    direction), alone and with the fused step, on plain rows and on folded
    rows whose taps stop at segment edges, against central finite
    differences of the forward oracle."""
    rng = np.random.default_rng(67)
    ok = True
    for dirs, seg, sp, own_step, K, own_conv in ((3, 0, False, False, 4, False),
                                                 (3, 0, False, False, 3, True),
                                                 (1, 0, False, False, 2, False),
                                                 (3, 0, True, True, 4, True),
                                                 (3, 4, False, False, 3, True)):
        ok = ok and _grad_opts_fd_ok(lib, rng, dirs, seg, sp, own_step, False, K, own_conv,
                                     L=2 * seg if seg else 7)
    return ok


def pin_gradient_finite_differences(lib):
    """The adjoint gradients (dx, ddelta, dz, dB, dC, per-direction dB/dC,
    dA, dD) equal central finite differences of the forward oracle, for each
    direction alone and both, with and without the gate, on folded rows, and
    with the backward direction's own B and C."""
    rng = np.random.default_rng(47)
    ok = True
    for dirs, gate, seg, own in ((1, True, 0, False), (2, True, 0, False), (3, True, 0, False),
                                 (3, False, 0, False), (3, True, 3, False), (3, True, 0, True),
                                 (1, True, 2, False)):
        ok = ok and _grad_fd_ok(lib, rng, dirs, gate, seg, own)
    return ok


def _ncssd_problem(rng, b=2, d=5, L=9, N=4):
    return dict(x=rng.standard_normal((b, d, L)), B=rng.standard_normal((b, L, N)),
                C=rng.standard_normal((b, L, N)), m=rng.uniform(0.2, 3.0, (b, L)),
                D=rng.standard_normal(d), z=rng.standard_normal((b, d, L)))


def pin_ncssd_matrix_form(lib):
    """NC-SSD against the VSSD page's simplified form Y = C (B^T (X m))
    (§4.2.5.2), evaluated with numpy matrix products, plus the skip and the
    gate: out = (Y + D x) silu(z). With C = 0 only the gated skip remains."""
    rng = np.random.default_rng(53)
    p = _ncssd_problem(rng)
    got = oracle.ncssd(p["x"], p["B"], p["C"], p["m"], p["D"], p["z"], lib=lib)
    ok = True
    for bb in range(p["x"].shape[0]):
        X = p["x"][bb].T                               # (L, dim)
        H = p["B"][bb].T @ (X * p["m"][bb][:, None])   # (N, dim)
        Y = p["C"][bb] @ H                             # (L, dim)
        want = (Y + X * p["D"][None, :]) * (p["z"][bb].T * expit(p["z"][bb].T))
        ok = ok and _close(got[bb], want.T, 1e-12)
    zero = oracle.ncssd(p["x"], p["B"], np.zeros_like(p["C"]), p["m"], p["D"], p["z"], lib=lib)
    ok = ok and _close(zero, p["D"][None, :, None] * p["x"] * p["z"] * expit(p["z"]), 1e-13)
    return ok


def pin_ncssd_token_order(lib):
    """The global state does not depend on where the tokens sit (VSSD page
    §4.2.4): permuting the tokens (x, B, C, m, z together) permutes the
    output's token axis the same way; the output is linear in m."""
    rng = np.random.default_rng(59)
    p = _ncssd_problem(rng, L=11)
    perm = rng.permutation(11)
    base = oracle.ncssd(p["x"], p["B"], p["C"], p["m"], p["D"], p["z"], lib=lib)
    q = dict(x=p["x"][..., perm], B=p["B"][:, perm], C=p["C"][:, perm], m=p["m"][:, perm],
             z=p["z"][..., perm])
    moved = oracle.ncssd(np.ascontiguousarray(q["x"]), np.ascontiguousarray(q["B"]),
                         np.ascontiguousarray(q["C"]), np.ascontiguousarray(q["m"]), p["D"],
                         np.ascontiguousarray(q["z"]), lib=lib)
    ok = _close(moved, base[..., perm], 1e-12)
    m2 = rng.uniform(0.2, 3.0, p["m"].shape)
    f = lambda m: oracle.ncssd(p["x"], p["B"], p["C"], m, None, None, lib=lib)
    ok = ok and _close(f(p["m"] + 2.0 * m2), f(p["m"]) + 2.0 * f(m2), 1e-12)
    return ok


PINS = [pin_worked_example, pin_quadratic_form, pin_A_zero_prefix_sum,
        pin_vanishing_decay, pin_zero_input_paths, pin_single_token,
        pin_backward_is_flipped_forward, pin_folded_equals_segments,
        pin_reset_first_token, pin_gate, pin_linearity, pin_softplus_step,
        pin_per_direction_step, pin_conv_taps, pin_conv_feeds_each_direction,
        pin_gradient_finite_differences, pin_gradient_step_options_fd, pin_gradient_conv_fd,
        pin_ncssd_matrix_form, pin_ncssd_token_order]


def failing_pins(lib):
    failed = []
    for pin in PINS:
        try:
            ok = pin(lib)
        except Exception:  # a crash or a rejected call counts as a failure
            ok = False
        if not ok:
            failed.append(pin.__name__)
    return failed
