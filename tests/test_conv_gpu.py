"""Directional depthwise convolution + SiLU in front of the scan vs the fp64
oracle (Vim page §2.3: forward and backward paths use 1D convolutions of
opposite directions; SF-Mamba page: SiLU of a depthwise convolution feeds the
SSM, and on folded rows the convolution never crosses a segment boundary).

Cases: both kernels (N = 16 and N < 16), 1 to 4 taps, single directions,
rows with partial chunks and odd halves (the history crosses the
meet-in-the-middle point), folded rows with segments shorter than the taps,
ranges joined by the carry (the history reaches back into the previous
range), and the convolution together with the fused step.
"""
import pytest
import torch

import oracle
from gpu_util import TOL, elementwise_rel, normwise_rel, to_device
from workloads import DIR_BOTH, DIR_BWD, DIR_FWD, WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import bidirectional_selective_scan_vssm_b300 as vssm  # noqa: E402  (fails loudly if unbuilt)


def _args(t):
    return (t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"], t["D_fwd"], t["D_bwd"],
            t["z"])


def _conv_kw(t, own_bwd=True):
    kw = dict(conv_w=t["conv_w"], conv_b=t["conv_b"])
    if own_bwd:
        kw.update(conv_w_bwd=t["conv_w_bwd"], conv_b_bwd=t["conv_b_bwd"])
    return kw


def _step_kw(t):
    if "delta_bwd" not in t:
        return {}
    return dict(delta_bwd=t["delta_bwd"], delta_bias=t["delta_bias"],
                delta_bias_bwd=t["delta_bias_bwd"], delta_softplus=True)


def _oracle(inp, dirs, seg_len=0, own_bwd=True):
    kw = dict(conv_w=inp.conv_w, conv_b=inp.conv_b)
    if own_bwd:
        kw.update(conv_w_bwd=inp.conv_w_bwd, conv_b_bwd=inp.conv_b_bwd)
    if inp.delta_bwd is not None:
        kw.update(delta_bwd=inp.delta_bwd, delta_bias=inp.delta_bias,
                  delta_bias_bwd=inp.delta_bias_bwd, delta_softplus=True)
    return oracle.scan(inp.x, inp.delta, inp.A_fwd, inp.A_bwd, inp.B, inp.C, inp.D_fwd,
                       inp.D_bwd, inp.z, dirs=dirs, seg_len=seg_len, **kw)


def _check(got, ref, dtype, what=""):
    g = got.float().cpu().numpy()
    err = normwise_rel(g, ref)
    assert err <= TOL[dtype], f"{what}: normwise rel err {err:.3e} > {TOL[dtype]} " \
                              f"(elementwise {elementwise_rel(g, ref):.3e})"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
@pytest.mark.parametrize("K", [1, 2, 4])
@pytest.mark.parametrize("shape", [(2, 40, 3, 16), (1, 64, 33, 16), (3, 33, 197, 16),
                                   (2, 24, 61, 8)], ids=lambda s: "x".join(map(str, s)))
def test_conv(dtype, dirs, K, shape):
    b, d, L, N = shape
    wl = WORKLOADS["vim_ti_224"].scaled(batch=b, dim=d, seqlen=L, dstate=N, dtype=dtype, conv=K)
    inp = make_inputs(wl, seed=700 + L + K)
    t = to_device(inp)
    got = vssm.scan_bidir(*_args(t), dirs=dirs, **_conv_kw(t))
    _check(got, _oracle(inp, dirs), dtype, f"{shape} K={K} dirs={dirs}")


def test_conv_shared_backward_weights():
    """conv_w_bwd / conv_b_bwd NULL: the backward direction uses the forward
    taps, applied in its own (reversed) direction."""
    wl = WORKLOADS["vim_ti_224"].scaled(batch=2, dim=40, seqlen=90, conv=4)
    inp = make_inputs(wl, seed=710)
    t = to_device(inp)
    got = vssm.scan_bidir(*_args(t), **_conv_kw(t, own_bwd=False))
    _check(got, _oracle(inp, DIR_BOTH, own_bwd=False), "f32")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
@pytest.mark.parametrize("seg,nseg", [(1, 20), (2, 15), (3, 11), (51, 9), (16, 7)])
def test_conv_folded(dtype, dirs, seg, nseg):
    """The taps stop at segment edges, also for segments shorter than the taps."""
    wl = WORKLOADS["sf_folded"].scaled(batch=2, dim=40, seqlen=seg * nseg, seg_len=seg,
                                       dtype=dtype, dirs=dirs, conv=4)
    inp = make_inputs(wl, seed=720 + seg)
    t = to_device(inp)
    got = vssm.scan_folded(*_args(t), seg_len=seg, dirs=dirs, **_conv_kw(t))
    _check(got, _oracle(inp, dirs, seg_len=seg), dtype, f"seg={seg}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
@pytest.mark.parametrize("pieces", [2, 7, 40])
def test_conv_with_carry(dtype, dirs, pieces):
    """Ranges joined by the carry: each range's first tokens take their
    convolution history from the range before (after, going backward)."""
    wl = WORKLOADS["vim_ti_224"].scaled(batch=1, dim=40, seqlen=203, dtype=dtype, conv=4)
    inp = make_inputs(wl, seed=730 + pieces)
    t = to_device(inp)
    got = vssm.scan_chunked(*_args(t), pieces=pieces, dirs=dirs, **_conv_kw(t))
    _check(got, _oracle(inp, dirs), dtype, f"pieces={pieces}")


def test_conv_folded_with_carry():
    """Folded rows cut off segment boundaries, with the convolution."""
    wl = WORKLOADS["sf_folded"].scaled(batch=1, dim=40, seqlen=51 * 8, seg_len=51,
                                       dirs=DIR_BOTH, dtype="f32", conv=4)
    inp = make_inputs(wl, seed=740)
    t = to_device(inp)
    got = vssm.scan_chunked(*_args(t), pieces=5, seg_len=51, dirs=DIR_BOTH, **_conv_kw(t))
    _check(got, _oracle(inp, DIR_BOTH, seg_len=51), "f32")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_conv_with_fused_step(dtype):
    wl = WORKLOADS["vim_ti_224"].scaled(batch=2, dim=48, seqlen=150, dtype=dtype, conv=4,
                                        fused_step=True)
    inp = make_inputs(wl, seed=750)
    t = to_device(inp)
    got = vssm.scan_bidir(*_args(t), **_conv_kw(t), **_step_kw(t))
    _check(got, _oracle(inp, DIR_BOTH), dtype)
