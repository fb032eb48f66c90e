"""Gradient of the scan (vssm_scan_grad) vs the fp64 oracle's adjoint, which
is itself pinned against finite differences of the forward oracle.

Tolerances (normwise, max|g - r| / max|r|): the per-token gradients dx,
ddelta, dz are rounded to the I/O dtype, so they take the forward's bars
(1e-4 for float32, 2e-2 for bfloat16); the float32 sums dB, dC, dA, dD take
1e-4 with float32 inputs and 1e-3 with bfloat16 inputs (their inputs are the
same exact values, the sums run over up to batch x tokens terms in fp32).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL, normwise_rel, to_device
from workloads import DIR_BOTH, DIR_BWD, DIR_FWD, WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import bidirectional_selective_scan_vssm_b300 as vssm  # noqa: E402  (fails loudly if unbuilt)

SUM_TOL = {"f32": 1e-4, "bf16": 1e-3}


def _dout(inp, seed):
    """An upstream gradient in the I/O dtype: device tensor and its exact values."""
    rng = np.random.default_rng(seed)
    g = rng.standard_normal(inp.x.shape).astype(np.float32)
    dt = torch.float32 if inp.wl.dtype == "f32" else torch.bfloat16
    t = torch.from_numpy(g).to("cuda").to(dt)
    return t, t.float().cpu().numpy().astype(np.float64)


def _run(inp, dirs, seg_len=0, gate=True, skip=True, own_bc=None, seed=0):
    t = to_device(inp)
    dout_t, dout = _dout(inp, seed)
    kw = {}
    okw = {}
    if own_bc is not None:
        kw = dict(B_bwd=torch.from_numpy(own_bc[0]).to("cuda").to(t["B"].dtype),
                  C_bwd=torch.from_numpy(own_bc[1]).to("cuda").to(t["C"].dtype))
        okw = dict(B_bwd=kw["B_bwd"].float().cpu().numpy(), C_bwd=kw["C_bwd"].float().cpu().numpy())
    got = vssm.scan_grad(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"],
                         t["D_fwd"] if skip else None, t["D_bwd"] if skip else None,
                         t["z"] if gate else None, dout=dout_t, dirs=dirs, seg_len=seg_len, **kw)
    ref = oracle.scan_grad(inp.x, inp.delta, inp.A_fwd, inp.A_bwd, inp.B, inp.C,
                           inp.D_fwd if skip else None, inp.D_bwd if skip else None,
                           inp.z if gate else None, dout, dirs=dirs, seg_len=seg_len, **okw)
    return got, ref


def _compare(got, ref, dtype, what):
    for k, r in ref.items():
        if r is None:
            assert got[k] is None, f"{what}: {k} should be absent"
            continue
        g = got[k].float().cpu().numpy()
        tol = TOL[dtype] if k in ("dx", "ddelta", "dz") else SUM_TOL[dtype]
        err = normwise_rel(g, r)
        assert err <= tol, f"{what}: {k} normwise rel err {err:.3e} > {tol}"


SHAPES = [(1, 40, 1), (2, 40, 5), (1, 33, 8), (2, 40, 9), (1, 64, 17), (2, 33, 64),
          (1, 40, 197)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_grad(dtype, dirs, shape):
    b, d, L = shape
    wl = WORKLOADS["vim_ti_224"].scaled(batch=b, dim=d, seqlen=L, dtype=dtype)
    inp = make_inputs(wl, seed=800 + L)
    got, ref = _run(inp, dirs, seed=L)
    _compare(got, ref, dtype, f"{shape} dirs={dirs}")


@pytest.mark.parametrize("gate,skip", [(False, True), (True, False), (False, False)])
def test_grad_without_gate_or_skip(gate, skip):
    wl = WORKLOADS["vim_ti_224"].scaled(batch=2, dim=40, seqlen=45)
    inp = make_inputs(wl, seed=810)
    got, ref = _run(inp, DIR_BOTH, gate=gate, skip=skip)
    _compare(got, ref, "f32", f"gate={gate} skip={skip}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
@pytest.mark.parametrize("seg,nseg", [(1, 12), (5, 9), (51, 4), (16, 3)])
def test_grad_folded(dtype, dirs, seg, nseg):
    wl = WORKLOADS["sf_folded"].scaled(batch=2, dim=40, seqlen=seg * nseg, seg_len=seg,
                                       dtype=dtype, dirs=dirs)
    inp = make_inputs(wl, seed=820 + seg)
    got, ref = _run(inp, dirs, seg_len=seg)
    _compare(got, ref, dtype, f"seg={seg}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
def test_grad_long_rows_cut_into_ranges(dtype, dirs):
    """Two 32-channel groups of 1001-token rows: too few groups to fill the
    GPU, so the adjoint runs each row as 15 ranges of 17 chunks (the last one
    ragged), joined by the adjoint summaries."""
    wl = WORKLOADS["vim_ti_224"].scaled(batch=1, dim=40, seqlen=1001, dtype=dtype, dirs=dirs)
    inp = make_inputs(wl, seed=840)
    got, ref = _run(inp, dirs)
    _compare(got, ref, dtype, "ranges")


@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
@pytest.mark.parametrize("seg,nseg", [(51, 20), (5, 200), (1, 700)])
def test_grad_long_folded_rows_cut_into_ranges(dirs, seg, nseg):
    """Folded rows with few channel groups: the adjoint (and the checkpoint
    pass) cut each row into independent ranges at segment starts, where the
    reset stops the adjoint in both directions. Ranges are multiples of
    lcm(seg, 4) tokens: 204 for 51-token segments, 20 for 5, 4 for 1."""
    wl = WORKLOADS["sf_folded"].scaled(batch=1, dim=40, seqlen=seg * nseg, seg_len=seg, dtype="f32",
                                       dirs=dirs)
    inp = make_inputs(wl, seed=850 + seg)
    got, ref = _run(inp, dirs, seg_len=seg)
    _compare(got, ref, "f32", f"folded ranges seg={seg}")


def test_grad_folded_row_shorter_than_a_segment_uses_summaries():
    """A forward-only folded call whose one (partial) segment is longer than
    the row: no segment start to cut at, so the ranges are joined by the
    adjoint summaries, with the reset only at token 0."""
    wl = WORKLOADS["sf_folded"].scaled(batch=1, dim=40, seqlen=1001, seg_len=4096, dtype="f32",
                                       dirs=DIR_FWD)
    inp = make_inputs(wl, seed=855)
    got, ref = _run(inp, DIR_FWD, seg_len=4096)
    _compare(got, ref, "f32", "folded, summaries")


def test_grad_long_workload_sampled():
    """The 1024² workload (8 x 4097 tokens x 768 channels, 192 groups, rows run as
    ranges): dB, dC of one batch entry and dx of sampled rows against the oracle."""
    wl = WORKLOADS["vim_s_1024"]
    inp = make_inputs(wl, seed=0)
    t = to_device(inp)
    dout_t, dout = _dout(inp, 3)
    got = vssm.scan_grad(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"], t["D_fwd"],
                         t["D_bwd"], t["z"], dout=dout_t)
    b = 5
    sl = slice(b, b + 1)
    ref = oracle.scan_grad(inp.x[sl], inp.delta[sl], inp.A_fwd, inp.A_bwd, inp.B[sl], inp.C[sl],
                           inp.D_fwd, inp.D_bwd, inp.z[sl], dout[sl])
    for k in ("dB", "dC"):
        err = normwise_rel(got[k][b].cpu().numpy(), ref[k][0])
        assert err <= SUM_TOL["bf16"], f"{k}: {err:.3e}"
    for d in (0, 31, 32, 400, 767):
        for k in ("dx", "ddelta", "dz"):
            err = normwise_rel(got[k][b, d].float().cpu().numpy(), ref[k][0, d])
            assert err <= TOL["bf16"], f"{k} row ({b}, {d}): {err:.3e}"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_grad_backward_own_B_C(dtype):
    wl = WORKLOADS["vim_ti_224"].scaled(batch=2, dim=48, seqlen=70, dtype=dtype)
    inp = make_inputs(wl, seed=830)
    other = make_inputs(wl, seed=831)
    got, ref = _run(inp, DIR_BOTH, own_bc=(other.B, other.C))
    _compare(got, ref, dtype, "own B/C")


def test_grad_workload_size_sampled():
    """Vim-S 224² at full size: dA, dD against the oracle on sampled
    channels, dx on sampled rows, dB / dC on one batch entry."""
    wl = WORKLOADS["vim_s_224"]
    inp = make_inputs(wl, seed=0)
    t = to_device(inp)
    dout_t, dout = _dout(inp, 1)
    got = vssm.scan_grad(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"], t["D_fwd"],
                         t["D_bwd"], t["z"], dout=dout_t)
    rng = np.random.default_rng(2)
    b = int(rng.integers(0, wl.batch))
    chans = rng.integers(0, wl.dim, 6)
    # one batch entry, all channels: dB, dC of that entry; dx of sampled rows
    sl = slice(b, b + 1)
    ref = oracle.scan_grad(inp.x[sl], inp.delta[sl], inp.A_fwd, inp.A_bwd, inp.B[sl], inp.C[sl],
                           inp.D_fwd, inp.D_bwd, inp.z[sl], dout[sl])
    for k in ("dB", "dC"):
        err = normwise_rel(got[k][b].cpu().numpy(), ref[k][0])
        assert err <= SUM_TOL["bf16"], f"{k}: {err:.3e}"
    for d in chans:
        err = normwise_rel(got["dx"][b, d].float().cpu().numpy(), ref["dx"][0, d])
        assert err <= TOL["bf16"], f"dx row ({b}, {d}): {err:.3e}"
    # dA, dD sum over every batch entry: compare on a channel slice
    dsl = slice(int(chans[0]), int(chans[0]) + 1)
    refA = oracle.scan_grad(inp.x[:, dsl], inp.delta[:, dsl], inp.A_fwd[dsl], inp.A_bwd[dsl],
                            inp.B, inp.C, inp.D_fwd[dsl], inp.D_bwd[dsl], inp.z[:, dsl],
                            dout[:, dsl])
    for k in ("dA_fwd", "dA_bwd", "dD_fwd", "dD_bwd"):
        err = normwise_rel(got[k][dsl].cpu().numpy(), refA[k])
        assert err <= SUM_TOL["bf16"], f"{k}: {err:.3e}"
