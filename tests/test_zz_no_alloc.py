"""vssm_scan_bidir_noalloc, the entry point for callers that cannot allocate
device memory, against vssm_scan_bidir and the fp64 oracle (needs a B300).

Some callers have no device allocator to hand this library a workspace (a
plain C host program, a serving loop that must not call cudaMalloc once it
runs). For them the library takes the scratch of bidirectional calls from a
fixed array of VSSM_NOALLOC_SCRATCH_BYTES in device memory. These tests call
it through the C ABI, twice in a row on the same scratch, and compare each
result with vssm_scan_bidir given its own workspace and with the oracle. A
call whose default plan (rows cut into ranges) needs more than the built-in
scratch runs with uncut rows when those fit; a call that fits neither is
refused. The file sorts last so that a run stopping at its first failure has
run every other test first.
"""
import ctypes

import pytest
import torch

import oracle
from gpu_util import TOL, normwise_rel, to_device
from workloads import DIR_BOTH, WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import bidirectional_selective_scan_vssm_b300 as vssm  # noqa: E402  (fails loudly if unbuilt)


def _noalloc(t, out):
    a = vssm.make_args(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"],
                       t["D_fwd"], t["D_bwd"], t["z"], out, dirs=DIR_BOTH)
    stream = torch.cuda.current_stream()
    return vssm.lib.vssm_scan_bidir_noalloc(ctypes.byref(a), ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_matches_scan_bidir_on_two_calls(dtype):
    wl = WORKLOADS["vim_s_224"].scaled(batch=4, dim=96, seqlen=197, dtype=dtype)
    inp = make_inputs(wl, seed=41)
    _check_two_calls(inp, dtype)


def _check_two_calls(inp, dtype):
    t = to_device(inp)
    ref = vssm.scan_bidir(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"],
                          t["D_fwd"], t["D_bwd"], t["z"], dirs=DIR_BOTH)
    torch.cuda.synchronize()
    r = ref.float().cpu().numpy()
    o = oracle.scan_inputs(inp, dirs=DIR_BOTH)
    for call in range(2):
        out = torch.full_like(t["x"], float("nan"))
        status = _noalloc(t, out)
        assert status == 0, vssm.lib.vssm_last_error().decode()
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        err = normwise_rel(got, r)
        assert err <= TOL[dtype], f"call {call}: normwise rel err {err:.3e} vs vssm_scan_bidir"
        err = normwise_rel(got, o)
        assert err <= TOL[dtype], f"call {call}: normwise rel err {err:.3e} vs the oracle"


def test_noalloc_falls_back_to_uncut_rows():
    """Few long rows: the default plan cuts them into ranges and needs more
    than the built-in scratch (stored y plus range summaries); uncut rows need
    only the stored y, which fits, so the call runs uncut."""
    wl = WORKLOADS["vim_s_1024"].scaled(batch=1, dim=992, seqlen=4097, dtype="bf16")
    inp = make_inputs(wl, seed=43)
    t = to_device(inp)
    a = vssm.make_args(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"],
                       t["D_fwd"], t["D_bwd"], t["z"], torch.empty_like(t["x"]), dirs=DIR_BOTH)
    # checked on the host first: the sizes exercise the fallback
    assert vssm.workspace_size(a, 0) > vssm.NOALLOC_SCRATCH_BYTES
    assert vssm.workspace_size(a, 0, pieces=1) <= vssm.NOALLOC_SCRATCH_BYTES
    _check_two_calls(inp, "bf16")


def test_noalloc_rejects_calls_beyond_the_scratch():
    # 4 bytes of scratch per token-channel: 64 x 768 x 1025 needs about 201 MB.
    wl = WORKLOADS["vim_s_512"].scaled(batch=64, dim=768, seqlen=1025, dtype="bf16")
    small = WORKLOADS["vim_s_224"].scaled(batch=1, dim=32, seqlen=8, dtype="bf16")
    t = to_device(make_inputs(small, seed=42))
    a = vssm.make_args(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"],
                       t["D_fwd"], t["D_bwd"], t["z"], torch.empty_like(t["x"]), dirs=DIR_BOTH)
    a.batch, a.dim, a.seqlen = wl.batch, wl.dim, wl.seqlen     # sizes only; nothing is launched
    # The sizes no longer match the buffers, so make sure on the host first
    # that this call is one the entry point must refuse.
    assert vssm.workspace_size(a, 0) > vssm.NOALLOC_SCRATCH_BYTES
    status = vssm.lib.vssm_scan_bidir_noalloc(ctypes.byref(a), None)
    assert status == -2
    assert "built-in scratch" in vssm.lib.vssm_last_error().decode()
