"""Gradient of the scan with the fused step and the directional convolution
(vssm_scan_grad with delta_softplus, delta_bwd, conv_k > 0) vs the fp64
oracle's chain rule, which is itself pinned against finite differences of the
forward oracle.

The step of direction k is softplus(v_k + bias_k) (Vim page §2.2, one SSM
module per direction; Mamba2D page, dt_proj with bias) and its input is
silu of a causal (forward) or reversed (backward) depthwise convolution of x
(Vim page §2.3), segment bounded on folded rows (SF-Mamba page). Cases: each
option alone and together, shared and own steps, biases and taps, defaulted
biases, 1 to 4 taps, single directions, both I/O dtypes, folded rows with
segments shorter than the taps, rows cut into adjoint ranges, and the 224²
workload at full size on sampled outputs.

Tolerances as the plain gradient's: per-token gradients (dx, ddelta,
ddelta_bwd, dz) are rounded to the I/O dtype and take the forward's bars;
the float32 sums (dB, dC, dA, dD, the step biases', the taps' and the
convolution biases' gradients) take 1e-4 with float32 inputs and 1e-3 with
bfloat16 inputs.
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
TOKEN_KEYS = ("dx", "ddelta", "ddelta_bwd", "dz")


def _dout(inp, seed):
    rng = np.random.default_rng(seed)
    g = rng.standard_normal(inp.x.shape).astype(np.float32)
    dt = torch.float32 if inp.wl.dtype == "f32" else torch.bfloat16
    t = torch.from_numpy(g).to("cuda").to(dt)
    return t, t.float().cpu().numpy().astype(np.float64)


def _options(src, softplus=True, own_step=True, bias=True, bias_bwd=True, conv=True,
             own_taps=True, conv_bias=True):
    """The option keyword arguments, taken from ``src`` (device tensors or
    the inputs' arrays)."""
    get = (lambda k: src[k]) if isinstance(src, dict) else (lambda k: getattr(src, k))
    kw = {}
    if own_step:
        kw["delta_bwd"] = get("delta_bwd")
    if softplus:
        kw["delta_softplus"] = True
        if bias:
            kw["delta_bias"] = get("delta_bias")
        if bias_bwd:
            kw["delta_bias_bwd"] = get("delta_bias_bwd")
    if conv:
        kw["conv_w"] = get("conv_w")
        if conv_bias:
            kw["conv_b"] = get("conv_b")
        if own_taps:
            kw["conv_w_bwd"] = get("conv_w_bwd")
            if conv_bias:
                kw["conv_b_bwd"] = get("conv_b_bwd")
    return kw


def _run(inp, dirs, seg_len=0, seed=0, **opts):
    t = to_device(inp)
    dout_t, dout = _dout(inp, seed)
    got = vssm.scan_grad(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"], t["D_fwd"],
                         t["D_bwd"], t["z"], dout=dout_t, dirs=dirs, seg_len=seg_len,
                         **_options(t, **opts))
    ref = oracle.scan_grad(inp.x, inp.delta, inp.A_fwd, inp.A_bwd, inp.B, inp.C, inp.D_fwd,
                           inp.D_bwd, inp.z, dout, dirs=dirs, seg_len=seg_len,
                           **_options(inp, **opts))
    return got, ref


def _compare(got, ref, dtype, what):
    for k, g in got.items():
        if g is None:
            continue
        assert ref.get(k) is not None, f"{what}: {k} returned without a reference"
        tol = TOL[dtype] if k in TOKEN_KEYS else SUM_TOL[dtype]
        err = normwise_rel(g.float().cpu().numpy(), ref[k])
        assert err <= tol, f"{what}: {k} normwise rel err {err:.3e} > {tol}"


def _workload(dtype, shape, conv=4, seg_len=0, dirs=DIR_BOTH, name="vim_ti_224", fused=True):
    """A small workload; ``fused``: the steps are pre-activations (softplus
    inside), else positive steps used as given."""
    b, d, L = shape
    kw = dict(batch=b, dim=d, seqlen=L, dtype=dtype, fused_step=fused, conv=conv, dirs=dirs)
    if seg_len:
        kw["seg_len"] = seg_len
    return WORKLOADS[name].scaled(**kw)


SHAPES = [(1, 40, 1), (2, 40, 9), (1, 33, 64), (2, 40, 197)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_grad_step_and_conv(dtype, dirs, shape):
    """Every option at once: own steps and biases, own taps and biases, K = 4."""
    inp = make_inputs(_workload(dtype, shape, dirs=dirs), seed=900 + shape[2])
    got, ref = _run(inp, dirs, seed=shape[2])
    _compare(got, ref, dtype, f"{shape} dirs={dirs}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
def test_grad_fused_step_only(dtype, dirs):
    inp = make_inputs(_workload(dtype, (2, 40, 70), conv=0, dirs=dirs), seed=910)
    got, ref = _run(inp, dirs, conv=False)
    _compare(got, ref, dtype, "step")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("own_step,bias,bias_bwd", [
    (False, True, False),     # one step, one bias: ddelta and ddelta_bias hold both directions'
    (False, True, True),      # one step, own biases
    (True, False, False),     # no bias (0)
    (True, False, True),      # forward bias 0, backward its own
    (False, False, False)])   # one step, no bias
def test_grad_step_sharing_and_default_biases(dtype, own_step, bias, bias_bwd):
    inp = make_inputs(_workload(dtype, (2, 40, 45), conv=0), seed=920)
    got, ref = _run(inp, DIR_BOTH, conv=False, own_step=own_step, bias=bias, bias_bwd=bias_bwd)
    _compare(got, ref, dtype, f"own_step={own_step} bias={bias} bias_bwd={bias_bwd}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_grad_backward_step_without_softplus(dtype):
    """A backward step of its own, both steps used as given (made positive by
    taking the absolute value of the pre-activations)."""
    inp = make_inputs(_workload(dtype, (2, 40, 45), conv=0), seed=925)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    t = to_device(inp)
    for k in ("delta", "delta_bwd"):
        t[k] = torch.from_numpy(np.abs(getattr(inp, k)) * np.float32(0.2)).to("cuda").to(dt)
        setattr(inp, k, t[k].float().cpu().numpy())     # the values the device holds
    dout_t, dout = _dout(inp, 1)
    got = vssm.scan_grad(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"], t["D_fwd"],
                         t["D_bwd"], t["z"], dout=dout_t, delta_bwd=t["delta_bwd"])
    ref = oracle.scan_grad(inp.x, inp.delta, inp.A_fwd, inp.A_bwd, inp.B, inp.C, inp.D_fwd,
                           inp.D_bwd, inp.z, dout, delta_bwd=inp.delta_bwd)
    _compare(got, ref, dtype, "raw backward step")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_grad_conv_only(dtype, dirs, K):
    inp = make_inputs(_workload(dtype, (2, 40, 33), conv=K, dirs=dirs, fused=False), seed=930 + K)
    got, ref = _run(inp, dirs, softplus=False, own_step=False)
    _compare(got, ref, dtype, f"K={K}")


@pytest.mark.parametrize("own_taps,conv_bias", [(False, True), (True, False), (False, False)])
def test_grad_conv_shared_taps_and_no_bias(own_taps, conv_bias):
    inp = make_inputs(_workload("f32", (2, 40, 50), conv=3), seed=940)
    got, ref = _run(inp, DIR_BOTH, own_taps=own_taps, conv_bias=conv_bias)
    _compare(got, ref, "f32", f"own_taps={own_taps} conv_bias={conv_bias}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
@pytest.mark.parametrize("seg,nseg", [(1, 12), (3, 11), (5, 9), (51, 4)])
def test_grad_options_folded(dtype, dirs, seg, nseg):
    """Folded rows: the resets and the segment-bounded taps (segments of 1 and
    3 tokens are shorter than the 4 taps)."""
    wl = _workload(dtype, (2, 40, seg * nseg), seg_len=seg, dirs=dirs, name="sf_folded")
    inp = make_inputs(wl, seed=950 + seg)
    got, ref = _run(inp, dirs, seg_len=seg)
    _compare(got, ref, dtype, f"seg={seg}")


@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
def test_grad_options_long_rows_cut_into_ranges(dirs):
    """1001-token rows of two channel groups: each direction's adjoint runs as
    token ranges joined by the adjoint summaries."""
    inp = make_inputs(_workload("bf16", (1, 40, 1001), dirs=dirs), seed=960)
    got, ref = _run(inp, dirs)
    _compare(got, ref, "bf16", "ranges")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
@pytest.mark.parametrize("b,L,seg,K", [(1, 2100, 0, 4), (1, 1024, 0, 2), (1, 2100, 7, 4),
                                       (1, 2100, 300, 4), (1, 1024, 1, 4), (1, 1530, 51, 1),
                                       (2, 1100, 0, 0), (2, 1100, 50, 2)], ids=str)
def test_grad_options_long_tiles(dtype, dirs, b, L, seg, K):
    """Rows of 1024 tokens or more, where the preparation and chain-rule
    kernels take four tokens per thread in 1024-token tiles: halos across
    tile edges, a ragged last tile, segments that do not divide the
    256-token thread stride (7, 51), segments longer than it (300),
    one-token segments, the fused step alone (K = 0) and two batch
    entries."""
    wl = _workload(dtype, (b, 40, L), conv=K, seg_len=seg, dirs=dirs,
                   name="sf_folded" if seg else "vim_ti_224")
    inp = make_inputs(wl, seed=970 + b + L + seg + K)
    got, ref = _run(inp, dirs, seg_len=seg, conv=K > 0)
    _compare(got, ref, dtype, f"b={b} L={L} seg={seg} K={K}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_grad_options_long_tiles_partial_segment(dtype):
    """Forward only (a backward reset needs whole segments): a 2101-token
    folded row of 300 segments of 7 tokens and one of 1, in 1024-token tiles."""
    wl = _workload(dtype, (1, 40, 2101), conv=3, seg_len=7, dirs=DIR_FWD, name="sf_folded")
    inp = make_inputs(wl, seed=990)
    got, ref = _run(inp, DIR_FWD, seg_len=7)
    _compare(got, ref, dtype, "partial segment")


def test_grad_options_workload_size_sampled():
    """Vim-S 224² (128 x 197 tokens x 768 channels, bfloat16) with own steps,
    biases and 4 taps per direction: the token gradients of one batch entry,
    and the per-channel sums on a channel slice, against the oracle."""
    wl = WORKLOADS["vim_s_224"].scaled(fused_step=True, conv=4)
    inp = make_inputs(wl, seed=0)
    t = to_device(inp)
    dout_t, dout = _dout(inp, 5)
    got = vssm.scan_grad(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"], t["D_fwd"],
                         t["D_bwd"], t["z"], dout=dout_t, **_options(t))
    b = 77
    sl = slice(b, b + 1)
    opts = _options(inp)
    ref = oracle.scan_grad(inp.x[sl], inp.delta[sl], inp.A_fwd, inp.A_bwd, inp.B[sl], inp.C[sl],
                           inp.D_fwd, inp.D_bwd, inp.z[sl], dout[sl],
                           **{k: (v[sl] if k == "delta_bwd" else v) for k, v in opts.items()})
    for k in ("dB", "dC"):
        err = normwise_rel(got[k][b].cpu().numpy(), ref[k][0])
        assert err <= SUM_TOL["bf16"], f"{k}: {err:.3e}"
    for k in TOKEN_KEYS:
        err = normwise_rel(got[k][b].float().cpu().numpy(), ref[k][0])
        assert err <= TOL["bf16"], f"{k} of batch entry {b}: {err:.3e}"
    d0 = 500
    dsl = slice(d0, d0 + 2)
    chan = {k: (v[:, dsl] if k == "delta_bwd" else v[dsl]) for k, v in opts.items()
            if k != "delta_softplus"}
    refc = oracle.scan_grad(inp.x[:, dsl], inp.delta[:, dsl], inp.A_fwd[dsl], inp.A_bwd[dsl],
                            inp.B, inp.C, inp.D_fwd[dsl], inp.D_bwd[dsl], inp.z[:, dsl],
                            dout[:, dsl], delta_softplus=True, **chan)
    for k in ("dA_fwd", "dA_bwd", "dD_fwd", "dD_bwd", "ddelta_bias", "ddelta_bias_bwd",
              "dconv_w", "dconv_b", "dconv_w_bwd", "dconv_b_bwd"):
        err = normwise_rel(got[k][dsl].cpu().numpy(), refc[k])
        assert err <= SUM_TOL["bf16"], f"{k}: {err:.3e}"


def test_grad_options_folded_workload_sampled():
    """The SF-Mamba batch-folded shape (1024 segments of 51 tokens in one
    52 224-token row, 1024 channels, bfloat16, forward only) with its own
    step, bias and 4 taps, in the launch configuration of the training
    step: a channel's token gradients and per-channel sums depend only on its
    own parameters and the shared B and C, so a two-channel slice of the
    oracle checks them exactly."""
    wl = WORKLOADS["sf_folded"].scaled(fused_step=True, conv=4)
    inp = make_inputs(wl, seed=0)
    t = to_device(inp)
    dout_t, dout = _dout(inp, 6)
    got = vssm.scan_grad(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"], t["D_fwd"],
                         t["D_bwd"], t["z"], dout=dout_t, dirs=wl.dirs, seg_len=wl.seg_len,
                         **_options(t))
    opts = _options(inp)
    dsl = slice(700, 702)
    chan = {k: (v[:, dsl] if k == "delta_bwd" else v[dsl]) for k, v in opts.items()
            if k != "delta_softplus"}
    refc = oracle.scan_grad(inp.x[:, dsl], inp.delta[:, dsl], inp.A_fwd[dsl], inp.A_bwd[dsl],
                            inp.B, inp.C, inp.D_fwd[dsl], inp.D_bwd[dsl], inp.z[:, dsl],
                            dout[:, dsl], dirs=wl.dirs, seg_len=wl.seg_len, delta_softplus=True,
                            **chan)
    for k in ("dx", "ddelta", "dz"):
        err = normwise_rel(got[k][:, dsl].float().cpu().numpy(), refc[k])
        assert err <= TOL["bf16"], f"{k} of channels 700-701: {err:.3e}"
    for k in ("dA_fwd", "dD_fwd", "ddelta_bias", "dconv_w", "dconv_b"):
        err = normwise_rel(got[k][dsl].cpu().numpy(), refc[k])
        assert err <= SUM_TOL["bf16"], f"{k}: {err:.3e}"


def test_grad_options_rejects_missing_and_extra_outputs():
    """The option gradients go exactly with their inputs: the binding fills
    them, so call the ABI through the binding's own argument structs."""
    import ctypes
    inp = make_inputs(_workload("f32", (1, 32, 16), conv=2), seed=970)
    t = to_device(inp)
    dout_t, _ = _dout(inp, 0)
    a = vssm.make_args(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"], t["D_fwd"],
                       t["D_bwd"], t["z"], **_options(t))
    need = vssm.grad_workspace_size(a)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    a.workspace, a.workspace_bytes = ws.data_ptr(), need
    keep = []

    def buf(*shape):
        x = torch.zeros(*shape, dtype=torch.float32, device="cuda")
        keep.append(x)
        return x.data_ptr()

    full = dict(dout=dout_t.data_ptr(), dx=buf(1, 32, 16), ddelta=buf(1, 32, 16),
                dz=buf(1, 32, 16), dB=buf(1, 16, 16), dC=buf(1, 16, 16), dA_fwd=buf(32, 16),
                dA_bwd=buf(32, 16), dD_fwd=buf(32), dD_bwd=buf(32), ddelta_bwd=buf(1, 32, 16),
                ddelta_bias=buf(32), ddelta_bias_bwd=buf(32), dconv_w=buf(32, 2), dconv_b=buf(32),
                dconv_w_bwd=buf(32, 2), dconv_b_bwd=buf(32))
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call(**drop):
        g = vssm.GradArgs()
        for k, v in full.items():
            setattr(g, k, None if k in drop else v)
        return vssm.lib.vssm_scan_grad(ctypes.byref(a), ctypes.byref(g), 0, s)

    code = {name: c for c, name in vssm.STATUS.items()}
    assert call() == code["VSSM_OK"]
    for k in ("ddelta_bwd", "ddelta_bias", "ddelta_bias_bwd", "dconv_w", "dconv_b",
              "dconv_w_bwd", "dconv_b_bwd"):
        assert call(**{k: True}) == code["VSSM_ERR_INVALID_ARG"], k
    torch.cuda.synchronize()
