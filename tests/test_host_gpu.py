"""vssm_scan_host: the scan with inputs and output in host memory, sliced
over batch entries or channel ranges and pipelined over three streams. The
result must match the fp64 oracle like the device entry points do."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL, normwise_rel
from workloads import DIR_BOTH, DIR_FWD, WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import bidirectional_selective_scan_vssm_b300 as vssm  # noqa: E402  (fails loudly if unbuilt)


def _host(inp, pinned=True):
    def act(name):
        a = inp.storage(name)
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 \
            else torch.from_numpy(np.ascontiguousarray(a))
        t = t.contiguous()
        return t.pin_memory() if pinned else t
    t = {k: act(k) for k in ("x", "delta", "z", "B", "C")}
    for k in ("A_fwd", "A_bwd", "D_fwd", "D_bwd"):
        t[k] = torch.from_numpy(getattr(inp, k)).contiguous()
    return t


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape,slices", [((3, 40, 77), 0), ((16, 64, 50), 4), ((1, 384, 197), 0),
                                          ((5, 33, 20), 2), ((2, 100, 33), 7)],
                         ids=lambda v: str(v))
def test_host_pipeline(dtype, shape, slices):
    b, d, L = shape
    wl = WORKLOADS["vim_ti_224"].scaled(batch=b, dim=d, seqlen=L, dtype=dtype)
    inp = make_inputs(wl, seed=950 + L)
    t = _host(inp)
    got = vssm.scan_host(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"], t["D_fwd"],
                         t["D_bwd"], t["z"], slices=slices)
    err = normwise_rel(got.float().numpy(), oracle.scan_inputs(inp))
    assert err <= TOL[dtype], f"{shape} slices={slices}: {err:.3e}"


@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BOTH])
def test_host_pipeline_folded_pageable(dirs):
    wl = WORKLOADS["sf_folded"].scaled(batch=2, dim=40, seqlen=51 * 6, seg_len=51, dirs=dirs)
    inp = make_inputs(wl, seed=960)
    t = _host(inp, pinned=False)
    got = vssm.scan_host(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"], t["D_fwd"],
                         t["D_bwd"], t["z"], dirs=dirs, seg_len=51, slices=3)
    err = normwise_rel(got.float().numpy(), oracle.scan_inputs(inp))
    assert err <= TOL["bf16"], f"{err:.3e}"


def test_host_pipeline_matches_device_call():
    """Same inputs through the device entry point: equal up to fp32 rounding
    order (the slices may be planned differently from the whole call)."""
    wl = WORKLOADS["vim_s_224"].scaled(batch=24)
    inp = make_inputs(wl, seed=970)
    t = _host(inp)
    got = vssm.scan_host(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"], t["D_fwd"],
                         t["D_bwd"], t["z"]).float()
    dev = {k: v.cuda() for k, v in t.items()}
    ref = vssm.scan_bidir(dev["x"], dev["delta"], dev["A_fwd"], dev["A_bwd"], dev["B"], dev["C"],
                          dev["D_fwd"], dev["D_bwd"], dev["z"]).float().cpu()
    assert float((got - ref).abs().max()) <= 2e-2 * float(ref.abs().max())


def test_host_pipeline_rejects_device_tensors():
    wl = WORKLOADS["vim_ti_224"].scaled(batch=1, dim=8, seqlen=5)
    t = _host(make_inputs(wl, seed=1))
    with pytest.raises(TypeError):
        vssm.scan_host(t["x"].cuda(), t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"])
