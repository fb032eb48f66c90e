"""Step options vs the fp64 oracle: a backward step of its own and the fused
step map softplus(delta + bias) per direction (Vim page §2.2, one SSM module
per direction; Mamba2D page, dt_proj with bias). Covers both kernels (N = 16
and N < 16), single directions, partial chunks, ranges joined by the carry,
folded rows and defaulted biases.
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


def _step_kw(t, softplus=True, bias=True, bias_bwd=True):
    kw = dict(delta_bwd=t["delta_bwd"], delta_softplus=softplus)
    if softplus and bias:
        kw["delta_bias"] = t["delta_bias"]
        if bias_bwd:
            kw["delta_bias_bwd"] = t["delta_bias_bwd"]
    return kw


def _oracle(inp, dirs, seg_len=0, softplus=True, bias=True, bias_bwd=True):
    kw = dict(delta_bwd=inp.delta_bwd, delta_softplus=softplus)
    if softplus and bias:
        kw["delta_bias"] = inp.delta_bias
        if bias_bwd:
            kw["delta_bias_bwd"] = inp.delta_bias_bwd
    return oracle.scan(inp.x, inp.delta, inp.A_fwd, inp.A_bwd, inp.B, inp.C, inp.D_fwd,
                       inp.D_bwd, inp.z, dirs=dirs, seg_len=seg_len, **kw)


def _args(t):
    return (t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"], t["D_fwd"], t["D_bwd"],
            t["z"])


def _check(got, ref, dtype, what=""):
    g = got.float().cpu().numpy()
    err = normwise_rel(g, ref)
    assert err <= TOL[dtype], f"{what}: normwise rel err {err:.3e} > {TOL[dtype]} " \
                              f"(elementwise {elementwise_rel(g, ref):.3e})"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
@pytest.mark.parametrize("shape", [(2, 40, 17, 16), (1, 64, 33, 16), (3, 33, 197, 16),
                                   (2, 24, 100, 8), (1, 16, 45, 1)],
                         ids=lambda s: "x".join(map(str, s)))
def test_fused_step(dtype, dirs, shape):
    b, d, L, N = shape
    wl = WORKLOADS["vim_ti_224"].scaled(batch=b, dim=d, seqlen=L, dstate=N, dtype=dtype,
                                        fused_step=True)
    inp = make_inputs(wl, seed=600 + L + N)
    t = to_device(inp)
    got = vssm.scan_bidir(*_args(t), dirs=dirs, **_step_kw(t))
    _check(got, _oracle(inp, dirs), dtype, f"{shape} dirs={dirs}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_step_without_softplus(dtype):
    """A backward step of its own, both steps used as given (made positive
    here by taking the absolute value of the pre-activations)."""
    wl = WORKLOADS["vim_ti_224"].scaled(batch=2, dim=48, seqlen=150, dtype=dtype,
                                        fused_step=True)
    inp = make_inputs(wl, seed=610)
    inp.delta = np.abs(inp.delta) * 0.2
    inp.delta_bwd = np.abs(inp.delta_bwd) * 0.2
    t = to_device(inp)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    t["delta"] = torch.from_numpy(inp.delta).to("cuda").to(dt)
    t["delta_bwd"] = torch.from_numpy(inp.delta_bwd).to("cuda").to(dt)
    # the device tensors round to bf16 again; feed the oracle the same values
    inp.delta = t["delta"].float().cpu().numpy()
    inp.delta_bwd = t["delta_bwd"].float().cpu().numpy()
    got = vssm.scan_bidir(*_args(t), **_step_kw(t, softplus=False))
    _check(got, _oracle(inp, DIR_BOTH, softplus=False), dtype)


@pytest.mark.parametrize("bias,bias_bwd", [(False, False), (True, False)])
def test_default_biases(bias, bias_bwd):
    """delta_bias NULL means 0; delta_bias_bwd NULL means delta_bias."""
    wl = WORKLOADS["vim_ti_224"].scaled(batch=1, dim=40, seqlen=77, fused_step=True)
    inp = make_inputs(wl, seed=620)
    t = to_device(inp)
    got = vssm.scan_bidir(*_args(t), **_step_kw(t, bias=bias, bias_bwd=bias_bwd))
    _check(got, _oracle(inp, DIR_BOTH, bias=bias, bias_bwd=bias_bwd), "f32")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("pieces", [3, 16])
def test_fused_step_with_carry(dtype, pieces):
    wl = WORKLOADS["vim_ti_224"].scaled(batch=1, dim=40, seqlen=301, dtype=dtype,
                                        fused_step=True)
    inp = make_inputs(wl, seed=630 + pieces)
    t = to_device(inp)
    got = vssm.scan_chunked(*_args(t), pieces=pieces, **_step_kw(t))
    _check(got, _oracle(inp, DIR_BOTH), dtype, f"pieces={pieces}")


@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BOTH])
def test_fused_step_folded(dirs):
    wl = WORKLOADS["sf_folded"].scaled(batch=2, dim=40, seqlen=51 * 9, seg_len=51, dirs=dirs,
                                       fused_step=True)
    inp = make_inputs(wl, seed=640)
    t = to_device(inp)
    got = vssm.scan_folded(*_args(t), seg_len=51, dirs=dirs, **_step_kw(t))
    _check(got, _oracle(inp, dirs, seg_len=51), "bf16")


def test_fused_step_at_workload_size_sampled_rows():
    """The Vim-S 224² shape with the fused step, checked on sampled rows."""
    wl = WORKLOADS["vim_s_224"].scaled(fused_step=True)
    inp = make_inputs(wl, seed=0)
    t = to_device(inp)
    got = vssm.scan_bidir(*_args(t), **_step_kw(t)).float().cpu().numpy()
    rng = np.random.default_rng(1)
    for b, d in zip(rng.integers(0, wl.batch, 12), rng.integers(0, wl.dim, 12)):
        sl = (slice(b, b + 1), slice(d, d + 1))
        ref = oracle.scan(inp.x[sl], inp.delta[sl], inp.A_fwd[d:d + 1], inp.A_bwd[d:d + 1],
                          inp.B[b:b + 1], inp.C[b:b + 1], inp.D_fwd[d:d + 1], inp.D_bwd[d:d + 1],
                          inp.z[sl], dirs=DIR_BOTH, delta_bwd=inp.delta_bwd[sl],
                          delta_bias=inp.delta_bias[d:d + 1],
                          delta_bias_bwd=inp.delta_bias_bwd[d:d + 1], delta_softplus=True)
        err = normwise_rel(got[b, d], ref[0, 0])
        assert err <= TOL["bf16"], f"row ({b}, {d}): {err:.3e}"
