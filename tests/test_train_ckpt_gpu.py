"""Training forward (vssm_scan_train): its output is the plain scan's, its
checkpoints are the recurrence's states, and the gradient computed from them
matches the fp64 oracle.

The checkpoint of 4-token chunk j is the state entering the chunk in the
direction's scan order (VSSD page §4.2.1.3): h after token 4j - 1 going
forward, h after token min(L, 4j + 4) going backward (Vim page §2.2), zero
where no token precedes and, on folded rows, where the chunk's first token
in scan order starts a segment (the recurrence restarts there; SF-Mamba
page, periodic state reset). The oracle states come from the oracle scan itself:
with C_t = e_n for every token, no skip and no gate, a single direction's
output y_t is its state h_t[n].
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


def _args(t, skip=True, gate=True):
    return (t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"],
            t["D_fwd"] if skip else None, t["D_bwd"] if skip else None, t["z"] if gate else None)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
@pytest.mark.parametrize("shape,seg", [((2, 40, 9), 0), ((1, 33, 197), 0), ((2, 64, 50), 5),
                                       ((1, 40, 4097), 0)], ids=str)
def test_train_output_is_the_scan(dtype, dirs, shape, seg):
    """Same output as vssm_scan_bidir / vssm_scan_folded, bit for bit (the
    1 x 40 x 4097 rows are cut into ranges joined by the carry)."""
    b, d, L = shape
    wl = WORKLOADS["vim_ti_224"].scaled(batch=b, dim=d, seqlen=L, dtype=dtype, dirs=dirs)
    t = to_device(make_inputs(wl, seed=1000 + L))
    out, ckpt = vssm.scan_train(*_args(t), seg_len=seg, dirs=dirs)
    if seg:
        ref = vssm.scan_folded(*_args(t), seg_len=seg, dirs=dirs)
    else:
        ref = vssm.scan_bidir(*_args(t), dirs=dirs)
    assert torch.equal(out.view(torch.int16 if dtype == "bf16" else torch.int32),
                       ref.view(torch.int16 if dtype == "bf16" else torch.int32))
    assert ckpt.numel() * 4 >= vssm.ckpt_size(vssm.make_args(*_args(t), dirs=dirs))


def _oracle_states(inp, dirs, seg):
    """h[direction][b][d][t][n] of each direction run, from the oracle scan
    with one-hot C (no skip, no gate)."""
    b, d, L = inp.x.shape
    out = {}
    for k, dflag in ((0, DIR_FWD), (1, DIR_BWD)):
        if not dirs & dflag:
            continue
        h = np.zeros((b, d, L, 16))
        for n in range(16):
            C = np.zeros_like(inp.C)
            C[:, :, n] = 1.0
            h[..., n] = oracle.scan(inp.x, inp.delta, inp.A_fwd, inp.A_bwd, inp.B, C, None, None,
                                    None, dirs=dflag, seg_len=seg)
        out[k] = h
    return out


@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
@pytest.mark.parametrize("shape,seg", [((2, 40, 23), 0), ((1, 33, 16), 0), ((1, 40, 30), 5),
                                       ((1, 40, 24), 3)], ids=str)
def test_checkpoints_are_the_states(dirs, shape, seg):
    b, d, L = shape
    wl = WORKLOADS["vim_ti_224"].scaled(batch=b, dim=d, seqlen=L, dtype="f32", dirs=dirs)
    inp = make_inputs(wl, seed=1100 + L)
    t = to_device(inp)
    _, ckpt = vssm.scan_train(*_args(t), seg_len=seg, dirs=dirs)
    ck = ckpt.cpu().numpy()
    rg, nch = (d + 31) // 32, (L + 3) // 4
    ndir = 2 if dirs == DIR_BOTH else 1
    ck = ck[:ndir * b * rg * nch * 512].reshape(ndir, b, rg, nch, 16, 32)
    states = _oracle_states(inp, dirs, seg)
    for k, h in states.items():
        slot = k if dirs == DIR_BOTH else 0
        got = np.zeros((b, d, nch, 16))
        ref = np.zeros((b, d, nch, 16))
        for j in range(nch):
            # the token whose state enters chunk j in this direction's order
            src = 4 * j - 1 if k == 0 else min(L, 4 * j + 4)
            # (on a folded row the recurrence restarts at a segment start: a
            # chunk whose first token in scan order starts a segment enters
            # with zero)
            first = 4 * j if k == 0 else min(L, 4 * j + 4) - 1
            restart = seg > 0 and first % seg == (0 if k == 0 else seg - 1)
            if 0 <= src < L and not restart:
                ref[:, :, j, :] = h[:, :, src, :]
            for g in range(rg):
                lanes = min(32, d - 32 * g)
                got[:, 32 * g:32 * g + lanes, j, :] = ck[slot, :, g, j, :, :lanes].transpose(0, 2, 1)
        err = normwise_rel(got, ref)
        assert err <= TOL["f32"], f"direction {k}: normwise rel err {err:.3e}"


def _dout(inp, seed):
    rng = np.random.default_rng(seed)
    g = rng.standard_normal(inp.x.shape).astype(np.float32)
    dt = torch.float32 if inp.wl.dtype == "f32" else torch.bfloat16
    tt = torch.from_numpy(g).to("cuda").to(dt)
    return tt, tt.float().cpu().numpy().astype(np.float64)


def _compare(got, ref, dtype, what):
    for k, g in got.items():
        if g is None:
            continue
        tol = TOL[dtype] if k in TOKEN_KEYS else SUM_TOL[dtype]
        err = normwise_rel(g.float().cpu().numpy(), ref[k])
        assert err <= tol, f"{what}: {k} normwise rel err {err:.3e} > {tol}"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
@pytest.mark.parametrize("shape,seg", [((2, 40, 9), 0), ((1, 33, 197), 0), ((2, 40, 60), 5),
                                       ((1, 40, 1001), 0)], ids=str)
def test_grad_from_train_checkpoints(dtype, dirs, shape, seg):
    b, d, L = shape
    wl = WORKLOADS["vim_ti_224"].scaled(batch=b, dim=d, seqlen=L, dtype=dtype, dirs=dirs)
    inp = make_inputs(wl, seed=1200 + L)
    t = to_device(inp)
    dout_t, dout = _dout(inp, L)
    _, ckpt = vssm.scan_train(*_args(t), seg_len=seg, dirs=dirs)
    got = vssm.scan_grad(*_args(t), dout=dout_t, dirs=dirs, seg_len=seg, ckpt=ckpt)
    ref = oracle.scan_grad(inp.x, inp.delta, inp.A_fwd, inp.A_bwd, inp.B, inp.C, inp.D_fwd,
                           inp.D_bwd, inp.z, dout, dirs=dirs, seg_len=seg)
    _compare(got, ref, dtype, f"{shape} seg={seg} dirs={dirs}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape,seg,dirs", [((2, 40, 70), 0, DIR_BOTH), ((1, 40, 2100), 0, DIR_BOTH),
                                            ((1, 40, 2100), 7, DIR_BOTH), ((1, 40, 2101), 7, DIR_FWD)],
                         ids=str)
def test_grad_from_train_checkpoints_with_options(dtype, shape, seg, dirs):
    """The composed gradient (own steps with softplus and biases, 4 taps per
    direction) reads each direction's checkpoints from the training forward:
    short rows; 2100-token rows of two channel groups, which the forward
    cuts into carry-joined ranges (the convolution's history and the
    checkpoints continue across them); folded rows of 7-token segments,
    whole (both directions) and with a partial last one (forward only)."""
    b, d, L = shape
    wl = WORKLOADS["vim_ti_224"].scaled(batch=b, dim=d, seqlen=L, dtype=dtype, fused_step=True,
                                        conv=4, dirs=dirs)
    inp = make_inputs(wl, seed=1300 + L + seg)
    t = to_device(inp)
    opts = dict(delta_bwd=t["delta_bwd"], delta_bias=t["delta_bias"],
                delta_bias_bwd=t["delta_bias_bwd"], delta_softplus=True, conv_w=t["conv_w"],
                conv_b=t["conv_b"], conv_w_bwd=t["conv_w_bwd"], conv_b_bwd=t["conv_b_bwd"])
    dout_t, dout = _dout(inp, 7)
    _, ckpt = vssm.scan_train(*_args(t), seg_len=seg, dirs=dirs, **opts)
    got = vssm.scan_grad(*_args(t), dout=dout_t, seg_len=seg, dirs=dirs, ckpt=ckpt, **opts)
    ref = oracle.scan_grad(inp.x, inp.delta, inp.A_fwd, inp.A_bwd, inp.B, inp.C, inp.D_fwd,
                           inp.D_bwd, inp.z, dout, dirs=dirs, seg_len=seg, delta_bwd=inp.delta_bwd,
                           delta_bias=inp.delta_bias, delta_bias_bwd=inp.delta_bias_bwd,
                           delta_softplus=True, conv_w=inp.conv_w, conv_b=inp.conv_b,
                           conv_w_bwd=inp.conv_w_bwd, conv_b_bwd=inp.conv_b_bwd)
    _compare(got, ref, dtype, f"options {shape} seg={seg} dirs={dirs}")


def test_train_rejects_short_or_missing_checkpoints():
    wl = WORKLOADS["vim_ti_224"].scaled(batch=1, dim=32, seqlen=16)
    t = to_device(make_inputs(wl, seed=1400))
    a = vssm.make_args(*_args(t), out=torch.empty_like(t["x"]))
    n = vssm.ckpt_size(a)
    assert n == 2 * 1 * 1 * 4 * 512 * 4
    ck = torch.empty(n // 4, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    import ctypes
    code = {name: c for c, name in vssm.STATUS.items()}
    assert vssm.lib.vssm_scan_train(ctypes.byref(a), 0, None, 0, ctypes.c_void_p(s)) == \
        code["VSSM_ERR_INVALID_ARG"]
    assert vssm.lib.vssm_scan_train(ctypes.byref(a), 0, ctypes.c_void_p(ck.data_ptr()), n - 4,
                                    ctypes.c_void_p(s)) == code["VSSM_ERR_INVALID_ARG"]
    assert vssm.lib.vssm_scan_train(ctypes.byref(a), 0, ctypes.c_void_p(ck.data_ptr() + 8), n,
                                    ctypes.c_void_p(s)) == code["VSSM_ERR_MISALIGNED"]
    torch.cuda.synchronize()
