"""Token ranges joined by the carry (vssm_scan_chunked) vs the fp64 oracle.

Each row is cut into ranges; every range but the last in a direction is
summarised from a zero state as (decay, end state), the summaries are composed
associatively into each range's incoming state, and every range is scanned
from that state (Vim page §3.1, parallel scan). In exact arithmetic this is
the unsplit scan, so the oracle's plain recurrence is the reference. The
cases span one-token rows, ranges shorter than, equal to and one past the
16-token copy chunk, one-token ranges, the 4097-token rows of the 1024²
workload, folded rows cut off segment boundaries, and the library's own
choice of cut for few rows.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL, elementwise_rel, normwise_rel, to_device
from workloads import DIR_BOTH, DIR_BWD, DIR_FWD, WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import bidirectional_selective_scan_vssm_b300 as vssm  # noqa: E402  (fails loudly if unbuilt)


def _chunked(t, dirs, pieces, seg_len=0):
    return vssm.scan_chunked(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"],
                             t["D_fwd"], t["D_bwd"], t["z"], pieces=pieces, seg_len=seg_len,
                             dirs=dirs)


def _oracle(inp, dirs, seg_len=0):
    return oracle.scan(inp.x, inp.delta, inp.A_fwd, inp.A_bwd, inp.B, inp.C, inp.D_fwd,
                       inp.D_bwd, inp.z, dirs=dirs, seg_len=seg_len)


def _check(got, ref, dtype, what=""):
    g = got.float().cpu().numpy()
    err = normwise_rel(g, ref)
    assert err <= TOL[dtype], f"{what}: normwise rel err {err:.3e} > {TOL[dtype]} " \
                              f"(elementwise {elementwise_rel(g, ref):.3e})"


ROWS = [(1, 40, 1), (1, 40, 5), (1, 40, 16), (1, 40, 17), (2, 40, 33), (1, 33, 197),
        (1, 40, 1025), (2, 33, 4097)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
@pytest.mark.parametrize("pieces", [2, 3, 8, 64])
@pytest.mark.parametrize("shape", ROWS, ids=lambda s: "x".join(map(str, s)))
def test_chunked_matches_oracle(dtype, dirs, pieces, shape):
    b, d, L = shape
    wl = WORKLOADS["vim_ti_224"].scaled(batch=b, dim=d, seqlen=L, dtype=dtype)
    inp = make_inputs(wl, seed=300 + L + pieces)
    got = _chunked(to_device(inp), dirs, pieces)
    _check(got, _oracle(inp, dirs), dtype, f"{shape} pieces={pieces} dirs={dirs}")


@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
@pytest.mark.parametrize("L", [2, 17, 40])
def test_one_token_ranges(dirs, L):
    """pieces = L: every range is one token, so every state is carried."""
    wl = WORKLOADS["vim_ti_224"].scaled(batch=1, dim=35, seqlen=L)
    inp = make_inputs(wl, seed=400 + L)
    got = _chunked(to_device(inp), dirs, L)
    _check(got, _oracle(inp, dirs), "f32", f"L={L} dirs={dirs}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
@pytest.mark.parametrize("seg,nseg,pieces", [(5, 9, 4), (51, 20, 7), (16, 8, 3), (1, 30, 4)])
def test_chunked_folded(dtype, dirs, seg, nseg, pieces):
    """Folded rows cut off segment boundaries: a range holding a reset carries
    nothing past it (its decay is 0)."""
    wl = WORKLOADS["sf_folded"].scaled(batch=2, dim=40, seqlen=seg * nseg, seg_len=seg,
                                       dtype=dtype, dirs=dirs)
    inp = make_inputs(wl, seed=500 + seg + nseg)
    got = _chunked(to_device(inp), dirs, pieces, seg_len=seg)
    _check(got, _oracle(inp, dirs, seg_len=seg), dtype, f"seg={seg} nseg={nseg} P={pieces}")


def test_chunked_folded_forward_partial_last_segment():
    wl = WORKLOADS["sf_folded"].scaled(batch=1, dim=33, seqlen=51 * 7 + 20, dtype="f32")
    inp = make_inputs(wl, seed=23)
    got = _chunked(to_device(inp), DIR_FWD, 5, seg_len=51)
    _check(got, _oracle(inp, DIR_FWD, seg_len=51), "f32")


def test_one_piece_equals_unsplit_bitwise():
    """pieces = 1 runs the unsplit scan: bit-identical to a call whose plan
    does not cut (rows enough to fill the GPU)."""
    wl = WORKLOADS["vim_s_224"].scaled(batch=32, dim=768, seqlen=197)
    t = to_device(make_inputs(wl, seed=24))
    ref = vssm.scan_bidir(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"],
                          t["D_fwd"], t["D_bwd"], t["z"])
    got = _chunked(t, DIR_BOTH, 1)
    assert torch.equal(got, ref)


def _step_opts(src, sp, conv):
    get = (lambda k: src[k]) if isinstance(src, dict) else (lambda k: getattr(src, k))
    kw = {}
    if sp:
        kw.update(delta_bwd=get("delta_bwd"), delta_bias=get("delta_bias"),
                  delta_bias_bwd=get("delta_bias_bwd"), delta_softplus=True)
    if conv:
        kw.update(conv_w=get("conv_w"), conv_b=get("conv_b"), conv_w_bwd=get("conv_w_bwd"),
                  conv_b_bwd=get("conv_b_bwd"))
    return kw


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
@pytest.mark.parametrize("L,sp,conv,seg", [(257, False, False, 0), (1001, False, False, 0),
                                           (1030, True, False, 0), (1001, False, True, 0),
                                           (1001, True, True, 0), (1020, False, False, 51)],
                         ids=str)
def test_uncut_long_rows(dtype, dirs, L, sp, conv, seg):
    """Rows longer than 256 tokens forced uncut (pieces = 1): the forward
    kernel's wider-unroll variant, element by element, with ragged tails
    (L mod 4 = 1, 2), the fused step, the convolution (single directions
    take the wider unroll with it; both directions keep the narrow one), and
    folded rows."""
    name = "sf_folded" if seg else "vim_ti_224"
    wl = WORKLOADS[name].scaled(batch=2, dim=40, seqlen=L, dtype=dtype, dirs=dirs,
                                fused_step=sp, conv=4 if conv else 0)
    inp = make_inputs(wl, seed=310 + L + 2 * sp + conv)
    t = to_device(inp)
    got = vssm.scan_chunked(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"],
                            t["D_fwd"], t["D_bwd"], t["z"], pieces=1, seg_len=seg, dirs=dirs,
                            **_step_opts(t, sp, conv))
    ref = oracle.scan(inp.x, inp.delta, inp.A_fwd, inp.A_bwd, inp.B, inp.C, inp.D_fwd,
                      inp.D_bwd, inp.z, dirs=dirs, seg_len=seg, **_step_opts(inp, sp, conv))
    _check(got, ref, dtype, f"L={L} sp={sp} conv={conv} seg={seg} dirs={dirs}")


@pytest.mark.parametrize("workload", ["vim_ti_224", "vim_s_1024"])
def test_library_choice_for_few_rows(workload):
    """The default entry point cuts few long rows by itself; its result
    matches the oracle. vim_s_1024 at batch 1 has 24 channel groups."""
    wl = WORKLOADS[workload].scaled(batch=1)
    inp = make_inputs(wl, seed=25)
    t = to_device(inp)
    a = vssm.make_args(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"],
                       t["D_fwd"], t["D_bwd"], t["z"], torch.empty_like(t["x"]))
    assert vssm.workspace_size(a) > vssm.workspace_size(a, pieces=1), "expected a carry plan"
    got = vssm.scan_bidir(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"],
                          t["D_fwd"], t["D_bwd"], t["z"])
    _check(got, _oracle(inp, DIR_BOTH), wl.dtype, workload)


def test_chunked_close_to_unsplit():
    """Same inputs, split and unsplit: equal up to fp32 rounding order."""
    wl = WORKLOADS["vim_ti_224"].scaled(batch=2, dim=64, seqlen=999)
    t = to_device(make_inputs(wl, seed=26))
    one = _chunked(t, DIR_BOTH, 1).double()
    for P in (2, 5, 31):
        got = _chunked(t, DIR_BOTH, P).double()
        err = float((got - one).abs().max() / one.abs().max())
        assert err < 2e-6, f"pieces={P}: {err:.3e}"
