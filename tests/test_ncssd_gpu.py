"""NC-SSD (vssm_ncssd), the VSSD page's non-causal global-state form, vs the
fp64 oracle (itself pinned against the page's matrix form and its
token-order independence). Covers ragged channel tiles, one-token rows, rows
split over clusters of 2, 4 and 8 CTAs (joined through distributed shared
memory), optional skip and gate, run-to-run determinism, and the Vim-S 224²
size on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL, normwise_rel, to_device
from workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import bidirectional_selective_scan_vssm_b300 as vssm  # noqa: E402  (fails loudly if unbuilt)


def _run(inp, skip=True, gate=True):
    t = to_device(inp)
    m = torch.from_numpy(inp.m).cuda()
    got = vssm.ncssd(t["x"], t["B"], t["C"], m, t["D_fwd"] if skip else None,
                     t["z"] if gate else None)
    ref = oracle.ncssd(inp.x, inp.B, inp.C, inp.m, inp.D_fwd if skip else None,
                       inp.z if gate else None)
    return got.float().cpu().numpy(), ref


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
# bf16 kernels: rows resident in shared memory for (2, 40, 9), (3, 64, 1),
# (8, 48, 100), (44, 768, 197) and (44, 768, 256) (one CTA per 32 rows, dim a
# multiple of 8, L <= 256); otherwise tiles, with 1 CTA per cluster for
# (44, 768, 257), (1, 130, 1), (1, 130, 33) and 2, 4, 8, 8 for the rest.
# fp32: the FMA-pipe kernel.
@pytest.mark.parametrize("shape", [(2, 40, 9), (3, 64, 1), (8, 48, 100), (44, 768, 197),
                                   (44, 768, 256), (44, 768, 257), (1, 130, 1), (1, 130, 33),
                                   (3, 64, 197), (2, 200, 300), (1, 64, 5000), (1, 33, 1100)],
                         ids=lambda s: "x".join(map(str, s)))
def test_ncssd(dtype, shape):
    b, d, L = shape
    wl = WORKLOADS["vim_ti_224"].scaled(batch=b, dim=d, seqlen=L, dtype=dtype, ncssd=True)
    got, ref = _run(make_inputs(wl, seed=1000 + L))
    err = normwise_rel(got, ref)
    assert err <= TOL[dtype], f"{shape}: {err:.3e}"


@pytest.mark.parametrize("skip,gate", [(False, False), (True, False), (False, True)])
@pytest.mark.parametrize("dtype,dim", [("f32", 70), ("bf16", 70), ("bf16", 64)])
def test_ncssd_optional_skip_gate(skip, gate, dtype, dim):
    wl = WORKLOADS["vim_ti_224"].scaled(batch=2, dim=dim, seqlen=50, dtype=dtype, ncssd=True)
    got, ref = _run(make_inputs(wl, seed=1100), skip=skip, gate=gate)
    assert normwise_rel(got, ref) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ncssd_deterministic(dtype):
    wl = WORKLOADS["vim_ti_224"].scaled(batch=1, dim=96, seqlen=3000, dtype=dtype, ncssd=True)
    inp = make_inputs(wl, seed=1200)
    t = to_device(inp)
    m = torch.from_numpy(inp.m).cuda()
    a = vssm.ncssd(t["x"], t["B"], t["C"], m, t["D_fwd"], t["z"])
    b = vssm.ncssd(t["x"], t["B"], t["C"], m, t["D_fwd"], t["z"])
    assert torch.equal(a, b)


def test_ncssd_vim_s_224_sampled():
    wl = WORKLOADS["vim_s_224"].scaled(ncssd=True)
    inp = make_inputs(wl, seed=0)
    t = to_device(inp)
    got = vssm.ncssd(t["x"], t["B"], t["C"], torch.from_numpy(inp.m).cuda(), t["D_fwd"], t["z"])
    bs = [0, 77, 127]
    ref = oracle.ncssd(inp.x[bs], inp.B[bs], inp.C[bs], inp.m[bs], inp.D_fwd, inp.z[bs])
    err = normwise_rel(got[bs].float().cpu().numpy(), ref)
    assert err <= TOL["bf16"], f"{err:.3e}"
