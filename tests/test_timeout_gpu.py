"""The bounded-wait path on the GPU: a wait that runs out records a timeout
that the host reads as VSSM_ERR_TIMEOUT, the word is cleared by the read, and
the device stays usable (a scan right after matches the oracle). The wait
runs out because its second arrival never comes; nothing faults or hangs."""
import ctypes

import pytest
import torch

import oracle
from gpu_util import TOL, normwise_rel, to_device
from workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import bidirectional_selective_scan_vssm_b300 as vssm  # noqa: E402  (fails loudly if unbuilt)


def test_expired_wait_is_reported_and_device_stays_usable():
    s = torch.cuda.current_stream()
    vssm.device_error(s)                                   # start from a clear word
    assert vssm.lib.vssm_selftest_wait_timeout(20000, ctypes.c_void_p(s.cuda_stream)) == 0
    with pytest.raises(vssm.VssmError) as e:
        vssm.device_error(s)
    assert e.value.status == -5                            # VSSM_ERR_TIMEOUT
    vssm.device_error(s)                                   # cleared by the read
    wl = WORKLOADS["vim_ti_224"].scaled(batch=1, dim=40, seqlen=50)
    inp = make_inputs(wl, seed=900)
    t = to_device(inp)
    got = vssm.scan_bidir(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"],
                          t["D_fwd"], t["D_bwd"], t["z"]).float().cpu().numpy()
    ref = oracle.scan_inputs(inp)
    assert normwise_rel(got, ref) <= TOL["f32"]
    vssm.device_error(s)


def test_selftest_rejects_bad_limits():
    assert vssm.lib.vssm_selftest_wait_timeout(0, None) == -1
    assert vssm.lib.vssm_selftest_wait_timeout(2000000, None) == -1
