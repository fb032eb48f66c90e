"""The C-ABI library on the host: it loads, exports every symbol the header
declares, and rejects invalid calls before launching anything. No call here
reaches the GPU (validation fails first, or the problem is empty)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vssm.h")


@pytest.fixture(scope="module")
def v():
    import __graft_entry__
    __graft_entry__.build()
    import bidirectional_selective_scan_vssm_b300 as v
    return v


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(vssm_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("vssm_scan_bidir", "vssm_scan_folded", "vssm_scan_workspace_size",
              "vssm_status_string", "vssm_last_error", "vssm_version"):
        assert n in names


def test_library_exports_every_declared_symbol(v):
    lib = ctypes.CDLL(v.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in vssm.h but not exported"
    assert set(v.EXPORTS) <= set(declared_functions())
    assert v.version() == 100


def test_args_struct_layout_matches_header(v):
    # 13 pointers + size_t, then 5 ints and an unsigned -> 8*14 + 4*6 = 136 bytes
    assert ctypes.sizeof(v.ScanArgs) == 136


def _args(v, **kw):
    a = v.ScanArgs()
    base = 1 << 20                       # fake, 16-byte aligned addresses; never dereferenced
    a.x, a.delta, a.z, a.B, a.C = base, base * 2, base * 3, base * 4, base * 5
    a.A_fwd, a.A_bwd, a.D_fwd, a.D_bwd = base * 6, base * 7, base * 8, base * 9
    a.out = base * 10
    a.batch, a.dim, a.seqlen, a.dstate, a.dtype, a.dir_flags = 1, 4, 8, 16, 1, 3
    for k, val in kw.items():
        setattr(a, k, val)
    return a


def _call(v, a, seg=None):
    if seg is None:
        return v.lib.vssm_scan_bidir(ctypes.byref(a), None)
    return v.lib.vssm_scan_folded(ctypes.byref(a), seg, None)


@pytest.mark.parametrize("kw,status", [
    (dict(x=None), -1), (dict(out=None), -1), (dict(A_fwd=None), -1),
    (dict(batch=-1), -1), (dict(dstate=0), -2), (dict(dstate=17), -2), (dict(dtype=7), -2),
    (dict(dir_flags=0), -1), (dict(dir_flags=4), -1), (dict(x=(1 << 20) + 2), -3),
    (dict(out=(1 << 20) * 2), -1),                    # out aliases delta
])
def test_invalid_calls_are_rejected(v, kw, status):
    assert _call(v, _args(v, **kw)) == status
    assert v.lib.vssm_last_error().decode() != ""


def test_folded_validation(v):
    assert _call(v, _args(v, seqlen=10), seg=0) == -1
    assert _call(v, _args(v, seqlen=10), seg=4) == -1          # backward needs L % seg == 0
    assert v.lib.vssm_status_string(-1).decode() == "invalid argument"


def test_workspace_required_for_long_rows(v):
    a = _args(v, seqlen=4097, dim=64)
    n = ctypes.c_size_t()
    assert v.lib.vssm_scan_workspace_size(ctypes.byref(a), 0, ctypes.byref(n)) == 0
    assert n.value == 64 * 4097 * 4
    assert _call(v, a) == -6                                     # no workspace given
    a.workspace, a.workspace_bytes = (1 << 20) * 11, n.value - 16
    assert _call(v, a) == -6                                     # too small


def test_workspace_sizes(v):
    n = ctypes.c_size_t(123)
    # general kernel (dstate != 16): short rows keep the y-buffer in shared memory
    a = _args(v, seqlen=197, dim=768, batch=128, dstate=8)
    assert v.lib.vssm_scan_workspace_size(ctypes.byref(a), 0, ctypes.byref(n)) == 0
    assert n.value == 0
    # warp kernel (dstate == 16): one fp32 partial output per token and channel
    a = _args(v, seqlen=197, dim=768, batch=128)
    assert v.lib.vssm_scan_workspace_size(ctypes.byref(a), 0, ctypes.byref(n)) == 0
    assert n.value == 128 * 768 * 197 * 4
    # a single direction needs none
    a = _args(v, seqlen=197, dim=768, batch=128, dir_flags=1)
    assert v.lib.vssm_scan_workspace_size(ctypes.byref(a), 0, ctypes.byref(n)) == 0
    assert n.value == 0


def test_empty_problem_launches_nothing(v):
    assert _call(v, _args(v, batch=0)) == 0
    assert _call(v, _args(v, seqlen=0, x=None, out=None)) == 0
