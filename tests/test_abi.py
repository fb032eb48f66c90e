"""The C-ABI library on the host: it loads, exports every symbol the header
declares, and rejects invalid calls before launching anything. No call here
reaches the GPU (validation fails first, or the problem is empty)."""
import ctypes
import subprocess
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
    for n in ("vssm_scan_bidir", "vssm_scan_folded", "vssm_scan_chunked",
              "vssm_scan_workspace_size", "vssm_scan_chunked_workspace_size",
              "vssm_status_string", "vssm_last_error", "vssm_version"):
        assert n in names


def test_library_exports_every_declared_symbol(v):
    lib = ctypes.CDLL(v.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in vssm.h but not exported"
    assert set(v.EXPORTS) <= set(declared_functions())
    declared = re.search(r"#define\s+VSSM_VERSION\s+(\d+)", open(HEADER).read())
    assert declared and v.version() == int(declared.group(1))


def test_args_struct_layout_matches_header(v):
    # 13 pointers + size_t, 5 ints and an unsigned (136 bytes); 3 pointers and
    # an int padded to 8 (32); 4 pointers and an int padded to 8 (40) -> 208
    assert ctypes.sizeof(v.ScanArgs) == 208


@pytest.mark.parametrize("struct,cname", [("ScanArgs", "vssm_scan_args"),
                                          ("GradArgs", "vssm_grad_args"),
                                          ("NcssdArgs", "vssm_ncssd_args")])
def test_args_struct_matches_c_header(v, tmp_path, struct, cname):
    """Compile a C program against include/vssm.h and compare the struct's
    size and field offsets with the ctypes mirror."""
    mirror = getattr(v, struct)
    src = tmp_path / "layout.c"
    fields = [f[0] for f in mirror._fields_]
    src.write_text("#include <stdio.h>\n#include <stddef.h>\n#include \"vssm.h\"\n"
                   f"int main(void) {{\n  printf(\"%zu\\n\", sizeof({cname}));\n" +
                   "".join(f"  printf(\"%zu\\n\", offsetof({cname}, {f}));\n"
                           for f in fields) + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), "-o", str(exe), str(src)],
                   check=True, capture_output=True)
    got = [int(t) for t in subprocess.run([str(exe)], check=True, capture_output=True,
                                          text=True).stdout.split()]
    assert got[0] == ctypes.sizeof(mirror)
    assert got[1:] == [getattr(mirror, f).offset for f in fields]


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
    (dict(delta_softplus=2), -1), (dict(delta_bwd=(1 << 20) * 12 + 4), -3),
    (dict(delta_bwd=(1 << 20) * 10), -1),             # out aliases delta_bwd
    (dict(delta_bias=(1 << 20) * 12 + 8), -3),
    (dict(conv_k=5, conv_w=(1 << 20) * 13), -2), (dict(conv_k=-1), -2),
    (dict(conv_k=4), -1),                             # conv_w missing
    (dict(conv_k=4, conv_w=(1 << 20) * 13 + 4), -3),
])
def test_invalid_calls_are_rejected(v, kw, status):
    assert _call(v, _args(v, **kw)) == status
    assert v.lib.vssm_last_error().decode() != ""


def test_folded_validation(v):
    assert _call(v, _args(v, seqlen=10), seg=0) == -1
    assert _call(v, _args(v, seqlen=10), seg=4) == -1          # backward needs L % seg == 0
    assert v.lib.vssm_status_string(-1).decode() == "invalid argument"


def test_workspace_required_for_long_rows(v):
    far = 1 << 32                                                # fake tensors may not overlap
    a = _args(v, batch=32, seqlen=1025, dim=768, **{k: far * (i + 1) for i, k in enumerate(
        ("x", "delta", "z", "B", "C", "A_fwd", "A_bwd", "D_fwd", "D_bwd", "out"))})  # no cuts
    n = ctypes.c_size_t()
    assert v.lib.vssm_scan_workspace_size(ctypes.byref(a), 0, ctypes.byref(n)) == 0
    assert n.value == 32 * 768 * 1025 * 4
    assert _call(v, a) == -6                                     # no workspace given
    a.workspace, a.workspace_bytes = far * 11, n.value - 16
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


def _chunked_ws(v, a, seg, pieces):
    n = ctypes.c_size_t(7)
    st = v.lib.vssm_scan_chunked_workspace_size(ctypes.byref(a), seg, pieces, ctypes.byref(n))
    return st, n.value


def test_chunked_workspace_sizes(v):
    a = _args(v, batch=1, dim=384, seqlen=197, dtype=0)        # 12 channel groups
    # one piece: one fp32 partial output per token and channel
    assert _chunked_ws(v, a, 0, 1) == (0, 384 * 197 * 4)
    # 4 pieces of 50 tokens: partial outputs per range (rounded to 32-channel
    # groups), then 2 directions x 12 groups x 4 summaries of 17 x 32 floats
    assert _chunked_ws(v, a, 0, 4) == (0, 12 * 4 * 50 * 32 * 4 + 2 * 12 * 4 * 17 * 32 * 4)
    # 5 requested pieces of 6 tokens on 26 tokens leave 5 pieces; 3 on 5 leave 3
    a1 = _args(v, batch=1, dim=32, seqlen=26, dir_flags=1)
    assert _chunked_ws(v, a1, 0, 5) == (0, 1 * 5 * 17 * 32 * 4)
    a2 = _args(v, batch=1, dim=32, seqlen=5, dir_flags=2)
    assert _chunked_ws(v, a2, 0, 4) == (0, 1 * 3 * 17 * 32 * 4)  # ceil(5/ceil(5/4)) = 3
    # more pieces than tokens: one token each
    a3 = _args(v, batch=1, dim=32, seqlen=3, dir_flags=1)
    assert _chunked_ws(v, a3, 0, 64) == (0, 3 * 17 * 32 * 4)
    # the library's choice for few rows includes summaries; for many rows it does not
    n = ctypes.c_size_t()
    assert v.lib.vssm_scan_workspace_size(ctypes.byref(a), 0, ctypes.byref(n)) == 0
    assert n.value > 384 * 197 * 4
    big = _args(v, batch=128, dim=768, seqlen=197)
    assert v.lib.vssm_scan_workspace_size(ctypes.byref(big), 0, ctypes.byref(n)) == 0
    assert n.value == 128 * 768 * 197 * 4


def test_chunked_validation(v):
    a = _args(v)
    assert v.lib.vssm_scan_chunked(ctypes.byref(a), 0, -1, None) == -1
    assert _chunked_ws(v, a, 0, -1)[0] == -1
    assert _chunked_ws(v, a, -2, 2)[0] == -1
    a8 = _args(v, dstate=8)
    assert v.lib.vssm_scan_chunked(ctypes.byref(a8), 0, 2, None) == -2   # carry needs dstate 16
    assert "dstate" in v.lib.vssm_last_error().decode()
    assert v.lib.vssm_scan_chunked(ctypes.byref(_args(v, seqlen=10)), 4, 2, None) == -1  # L % seg


def _plan(v, a, seg=0, pieces=0):
    r, n = ctypes.c_int(-1), ctypes.c_int(-1)
    st = v.lib.vssm_scan_plan_query(ctypes.byref(a), seg, pieces, ctypes.byref(r), ctypes.byref(n))
    return st, r.value, n.value


def test_plan_query(v):
    # rows enough to fill the GPU: one range, one launch
    assert _plan(v, _args(v, batch=128, dim=768, seqlen=197)) == (0, 1, 1)
    # the 1024^2 workload (8 x 24 channel groups per direction, one warp per
    # scheduler at most) is cut into ranges joined by the carry: summary
    # pass + scan
    st, r, n = _plan(v, _args(v, batch=8, dim=768, seqlen=4097))
    assert st == 0 and 2 <= r <= 16 and n == 2
    # so is a single 197-token row of 384 channels (the 224^2 Vim-Ti case)
    st, r, n = _plan(v, _args(v, batch=1, dim=384, seqlen=197))
    assert st == 0 and r > 1 and n == 2
    # explicit pieces
    assert _plan(v, _args(v, seqlen=26), 0, 5) == (0, 5, 2)
    assert _plan(v, _args(v, seqlen=26), 0, 1) == (0, 1, 1)
    # folded rows with many segments: independent ranges at segment starts, as
    # many as fill two waves of the warps resident at once (the SF-Mamba shape
    # in bf16 on 148 SMs: 128 ranges of 8 segments, one launch)
    st, r, n = _plan(v, _args(v, batch=1, dim=1024, seqlen=52224, dir_flags=1, dtype=1), 51)
    assert (st, r, n) == (0, 128, 1)
    # empty problem, bad arguments
    assert _plan(v, _args(v, batch=0)) == (0, 0, 0)
    assert _plan(v, _args(v), 0, -1)[0] == -1
    assert _plan(v, _args(v, dstate=8), 0, 2)[0] == -2


@pytest.mark.parametrize("b,d,nseg,seg,dirs,dt", [(1, 1024, 1024, 51, 1, 1), (2, 40, 20, 51, 3, 1),
                                                  (8, 768, 64, 51, 3, 0), (1, 64, 300, 7, 1, 0),
                                                  (4, 256, 1, 197, 3, 1), (1, 32, 4096, 1, 2, 1)])
def test_folded_plan_whole_segments(v, b, d, nseg, seg, dirs, dt):
    """The default folded plan cuts each row into independent ranges of whole
    segments (the last one possibly shorter), one launch, at least one range
    and at most one per segment."""
    st, r, n = _plan(v, _args(v, batch=b, dim=d, seqlen=nseg * seg, dir_flags=dirs, dtype=dt), seg)
    assert st == 0 and n == 1 and 1 <= r <= nseg
    per = -(-nseg // r)                                  # segments per range
    assert -(-nseg // per) == r


def _grad_args(v, **kw):
    g = v.GradArgs()
    base = 1 << 30                      # fake, aligned, far from the inputs of _args
    for i, name in enumerate(("dout", "dx", "ddelta", "dz", "dB", "dC", "dA_fwd", "dA_bwd",
                              "dD_fwd", "dD_bwd")):
        setattr(g, name, base * (i + 1))
    for k, val in kw.items():
        setattr(g, k, val)
    return g


def test_grad_workspace_size(v):
    a = _args(v, batch=1, dim=384, seqlen=197, dtype=0)
    n = ctypes.c_size_t()
    assert v.lib.vssm_scan_grad_workspace_size(ctypes.byref(a), 0, ctypes.byref(n)) == 0
    # checkpoints: 2 directions x 12 groups x 50 chunks of 4 tokens x 16 x 32 floats,
    # then partial dx, ddelta, dz: 12 groups x 197 tokens x 3 x 32 floats; 12 groups
    # are too few to fill the GPU, so each row is cut into 3 ranges of 17 chunks for the
    # adjoint, with a (P, q) summary of 2 x 16 x 32 floats per direction, group and range
    assert n.value == 2 * 12 * 50 * 512 * 4 + 12 * 197 * 96 * 4 + 2 * 12 * 3 * 1024 * 4
    a1 = _args(v, batch=1, dim=384, seqlen=197, dtype=0, dir_flags=1)
    assert v.lib.vssm_scan_grad_workspace_size(ctypes.byref(a1), 0, ctypes.byref(n)) == 0
    assert n.value == 12 * 50 * 512 * 4 + 12 * 3 * 1024 * 4
    # enough groups (128 x 24 = 3072): whole rows, no summaries
    a2 = _args(v, batch=128, dim=768, seqlen=197)
    assert v.lib.vssm_scan_grad_workspace_size(ctypes.byref(a2), 0, ctypes.byref(n)) == 0
    assert n.value == 2 * 3072 * 50 * 512 * 4 + 3072 * 197 * 96 * 4
    # short rows (fewer than 32 chunks) are never cut
    a3 = _args(v, batch=1, dim=384, seqlen=100)
    assert v.lib.vssm_scan_grad_workspace_size(ctypes.byref(a3), 0, ctypes.byref(n)) == 0
    assert n.value == 2 * 12 * 25 * 512 * 4 + 12 * 100 * 96 * 4


def test_grad_validation(v):
    def call(a, g, seg=0):
        return v.lib.vssm_scan_grad(ctypes.byref(a), ctypes.byref(g), seg, None)
    assert call(_args(v, dstate=8), _grad_args(v)) == -2
    # the option gradients go exactly with their inputs
    assert call(_args(v, delta_softplus=1), _grad_args(v)) == -6          # valid; no workspace
    assert call(_args(v, delta_softplus=1), _grad_args(v, ddelta_bias=(1 << 20) * 20)) == -1
    assert call(_args(v, delta_bwd=(1 << 20) * 12), _grad_args(v)) == -1  # ddelta_bwd missing
    assert call(_args(v, conv_k=4, conv_w=(1 << 20) * 13), _grad_args(v)) == -1  # dconv_w missing
    assert call(_args(v, conv_k=4, conv_w=(1 << 20) * 13),
                _grad_args(v, dconv_w=(1 << 20) * 20, dconv_b=(1 << 20) * 21)) == -1  # no conv_b
    assert call(_args(v, conv_k=4, conv_w=(1 << 20) * 13),
                _grad_args(v, dconv_w=(1 << 20) * 20 + 4)) == -3
    assert call(_args(v), _grad_args(v, dout=None)) == -1
    assert call(_args(v), _grad_args(v, dz=None)) == -1          # the call has z
    assert call(_args(v, B_bwd=(1 << 20) * 14), _grad_args(v)) == -1  # dB_bwd missing
    assert call(_args(v), _grad_args(v, dA_bwd=None)) == -1
    assert call(_args(v), _grad_args(v, dx=(1 << 30) + 4)) == -3
    ws = dict(workspace=(1 << 20) * 15, workspace_bytes=1 << 20)
    assert call(_args(v, **ws), _grad_args(v, dx=(1 << 20) * 2)) == -1  # dx overlaps delta
    assert call(_args(v, **ws), _grad_args(v, dB=(1 << 20) * 15)) == -1  # dB overlaps workspace
    assert call(_args(v), _grad_args(v), seg=-1) == -1
    assert call(_args(v), _grad_args(v)) == -6                    # no workspace
    assert call(_args(v, batch=0), _grad_args(v)) == 0            # empty: nothing to do


def _nc_args(v, **kw):
    a = v.NcssdArgs()
    base = dict(x=(1 << 20) * 1, z=(1 << 20) * 2, B=(1 << 20) * 3, C=(1 << 20) * 4,
                m=(1 << 20) * 5, D=(1 << 20) * 6, out=(1 << 20) * 7,
                batch=2, dim=64, seqlen=50, dstate=16, dtype=1)
    base.update(kw)
    for k, val in base.items():
        setattr(a, k, val)
    return a


def test_ncssd_needs_no_workspace(v):
    n = ctypes.c_size_t(123)
    assert v.lib.vssm_ncssd_workspace_size(ctypes.byref(_nc_args(v)), ctypes.byref(n)) == 0
    assert n.value == 0
    assert v.lib.vssm_ncssd_workspace_size(ctypes.byref(_nc_args(v, batch=-1)), ctypes.byref(n)) == -1


def test_ncssd_validation(v):
    def call(**kw):
        return v.lib.vssm_ncssd(ctypes.byref(_nc_args(v, **kw)), None)
    assert v.lib.vssm_ncssd(None, None) == -1
    assert call(batch=-1) == -1
    assert call(dstate=8) == -2
    assert call(dtype=7) == -2
    assert call(batch=70000) == -2
    far = {k: (1 << 36) * (i + 1) for i, k in enumerate(("x", "z", "B", "C", "m", "D", "out"))}
    assert call(dim=65536 * 32, **far) == -2             # more channel blocks than a grid row
    for k in ("x", "B", "C", "m", "out"):
        assert call(**{k: None}) == -1, k
    assert call(z=(1 << 20) * 2 + 4) == -3               # misaligned
    assert call(out=(1 << 20) * 2) == -1                 # out overlaps z
    assert call(batch=0) == 0                            # empty: nothing to do
    assert call(seqlen=0) == 0


def _al256(n):
    return (n + 255) // 256 * 256


def _host_ws(v, a, slices=0, seg=0):
    n = ctypes.c_size_t(0)
    st = v.lib.vssm_scan_host_workspace_size(ctypes.byref(a), seg, slices, ctypes.byref(n))
    return st, n.value


def _scan_ws(v, a, seg=0):
    n = ctypes.c_size_t(0)
    assert v.lib.vssm_scan_workspace_size(ctypes.byref(a), seg, ctypes.byref(n)) == 0
    return n.value


@pytest.mark.parametrize("batch,dim,slices", [(128, 768, 0), (128, 768, 16), (3, 768, 0), (1, 100, 4)])
def test_host_pipeline_workspace(v, batch, dim, slices):
    """vssm_scan_host's device workspace: the up-front parameters, then three
    ring slots, each holding one slice's five activation arrays and that
    slice's own scan workspace. Slices are whole batch entries when there are
    at least as many entries as slices, else 32-channel-aligned ranges."""
    L, es = 197, 2
    a = _args(v, batch=batch, dim=dim, seqlen=L)
    st, total = _host_ws(v, a, slices)
    assert st == 0
    S = slices or 8
    if batch >= S:
        per_b = -(-batch // S)
        rows_b, rows_d = per_b, dim
        nsl = -(-batch // per_b)
        last = (batch - (nsl - 1) * per_b, dim)
    else:
        per_entry = max(1, -(-S // batch))
        per_d = max(32, (-(-dim // per_entry) + 31) // 32 * 32)
        rows_b, rows_d = 1, per_d
        last = (1, dim % per_d or per_d)
    ws = max(_scan_ws(v, _args(v, batch=rows_b, dim=min(rows_d, dim), seqlen=L)),
             _scan_ws(v, _args(v, batch=last[0], dim=last[1], seqlen=L)))
    slot = _al256(5 * _al256(rows_b * rows_d * L * es) + ws)
    up = 4 * _al256(batch * L * 16 * es) + 2 * _al256(dim * 16 * 4) + 6 * _al256(dim * 4) + 2 * _al256(dim * 4)
    assert total == up + 3 * slot


def test_host_pipeline_validation(v):
    assert _host_ws(v, _args(v), slices=-1)[0] == -1
    assert _host_ws(v, _args(v, batch=0))[1] == 0
    assert v.lib.vssm_scan_host(ctypes.byref(_args(v)), 0, 0, None) == -6      # no workspace


def test_grad_workspace_sizes_with_options(v):
    """The plain gradient: 16 x 32 fp32 checkpoints per 4-token chunk, channel
    group of 32 and direction, plus 96 fp32 per token and channel group
    exchanged between the directions. With the step options or the
    convolution: float32 intermediates per direction (input, step, the two
    token gradients, the gate's share), float32
    copies of z, dout, B and C for bfloat16 I/O, then one direction's plain
    workspace."""
    n = ctypes.c_size_t(0)
    a = _args(v, batch=2, dim=64, seqlen=40, dtype=0)            # float32, both directions
    assert v.lib.vssm_scan_grad_workspace_size(ctypes.byref(a), 0, ctypes.byref(n)) == 0
    ck = 2 * 2 * 2 * 10 * 512 * 4                       # dirs x batch x groups x 4-token chunks
    part = 2 * 2 * 40 * 96 * 4
    assert n.value == ck + part
    one = ck // 2                                                 # one direction's checkpoints
    tok = 2 * 64 * 40 * 4
    r = lambda b: (b + 255) // 256 * 256
    # float32, convolution: per direction u, du, dst, dz (the raw step is read as given)
    a = _args(v, batch=2, dim=64, seqlen=40, dtype=0, conv_k=2, conv_w=(1 << 20) * 13)
    assert v.lib.vssm_scan_grad_workspace_size(ctypes.byref(a), 0, ctypes.byref(n)) == 0
    assert n.value == 2 * 4 * r(tok) + r(one)
    # bfloat16, softplus with one shared step: one u and one st for both directions, then
    # du, dst, dz per direction, B and C copies (shared), z and dout copies
    bc = 2 * 40 * 16 * 4
    a = _args(v, batch=2, dim=64, seqlen=40, dtype=1, delta_softplus=1)
    assert v.lib.vssm_scan_grad_workspace_size(ctypes.byref(a), 0, ctypes.byref(n)) == 0
    assert n.value == (2 + 2 * 3 + 2) * r(tok) + 2 * r(bc) + r(one)


def test_checkpoint_size(v):
    """vssm_scan_ckpt_size: 16 fp32 per 4-token chunk, 32-channel group lane
    and direction: 64 * directions * batch * ceil(dim / 32) * 32 * ceil(L / 4)."""
    n = ctypes.c_size_t(0)
    a = _args(v, batch=3, dim=40, seqlen=9)                      # both directions
    assert v.lib.vssm_scan_ckpt_size(ctypes.byref(a), ctypes.byref(n)) == 0
    assert n.value == 64 * 2 * 3 * 2 * 32 * 3
    a = _args(v, batch=3, dim=40, seqlen=9, dir_flags=2)
    assert v.lib.vssm_scan_ckpt_size(ctypes.byref(a), ctypes.byref(n)) == 0
    assert n.value == 64 * 1 * 3 * 2 * 32 * 3
    assert v.lib.vssm_scan_ckpt_size(ctypes.byref(_args(v, dir_flags=0)), ctypes.byref(n)) == -1


def test_train_validation(v):
    """The training forward validates its checkpoint buffer before launching
    (fake device addresses: nothing is launched)."""
    a = _args(v)                                                  # 1 x 4 x 8, both directions
    n = ctypes.c_size_t(0)
    assert v.lib.vssm_scan_ckpt_size(ctypes.byref(a), ctypes.byref(n)) == 0
    ck = (1 << 20) * 30
    assert v.lib.vssm_scan_train(ctypes.byref(a), 0, None, n.value, None) == -1        # NULL
    assert v.lib.vssm_scan_train(ctypes.byref(a), 0, ck, n.value - 4, None) == -1     # short
    assert v.lib.vssm_scan_train(ctypes.byref(a), 0, ck + 8, n.value, None) == -3     # misaligned
    assert v.lib.vssm_scan_train(ctypes.byref(a), 0, (1 << 20) * 10, n.value, None) == -1  # on out
    assert v.lib.vssm_scan_train(ctypes.byref(_args(v, dstate=8)), 0, ck, n.value, None) == -2
    assert v.lib.vssm_scan_train(ctypes.byref(a), -1, ck, n.value, None) == -1


def test_grad_plan_query(v):
    """Launch counts of the gradient for given arguments (no device touched):
    the zero-fills of the accumulated outputs, the checkpoint pass unless
    checkpoints are given, the summaries when rows are cut and joined, the
    adjoint; with the step options also the preparation, the bf16 widening
    of B and C and the chain rule, and the passes once per direction."""
    r, n = ctypes.c_int(0), ctypes.c_int(0)

    def query(a, g, seg=0):
        assert v.lib.vssm_scan_grad_plan_query(ctypes.byref(a), ctypes.byref(g), seg, ctypes.byref(r),
                                               ctypes.byref(n)) == 0
        return r.value, n.value

    # 128 x 768 x 197 both directions: enough groups, whole rows. Zero-fills of
    # dB, dC, dA_fwd, dA_bwd, dD_fwd, dD_bwd (6), checkpoints, adjoint
    a = _args(v, batch=128, dim=768, seqlen=197)
    g = _grad_args(v)
    assert query(a, g) == (1, 8)
    g.ckpt = (1 << 20) * 30
    assert query(a, g) == (1, 7)
    # few groups, long rows: ranges joined by the summaries (one more launch)
    a = _args(v, batch=1, dim=384, seqlen=197)
    g = _grad_args(v)
    assert query(a, g) == (3, 9)
    # folded rows with few groups: independent ranges at segment starts, no summaries
    a = _args(v, batch=1, dim=40, seqlen=51 * 20)
    ranges, launches = query(a, g, seg=51)
    assert ranges > 1 and launches == 8
    # bf16 with softplus, shared step and B/C: 6 zero-fills + ddelta_bias, prep,
    # widen B and C once, per direction checkpoints + adjoint, post
    a = _args(v, batch=128, dim=768, seqlen=197, dtype=1, delta_softplus=1, delta_bias=(1 << 20) * 11)
    g = _grad_args(v, ddelta_bias=(1 << 20) * 20)
    assert query(a, g) == (1, 7 + 1 + 2 + 2 * 2 + 1)
    # empty problem
    assert query(_args(v, batch=0), _grad_args(v)) == (0, 0)


def test_train_and_grad_empty_problems(v):
    """An empty problem is a no-op: the training forward needs no checkpoint
    buffer, the sizes are 0, and nothing is launched."""
    a = _args(v, batch=0)
    n = ctypes.c_size_t(123)
    assert v.lib.vssm_scan_ckpt_size(ctypes.byref(a), ctypes.byref(n)) == 0 and n.value == 0
    assert v.lib.vssm_scan_train(ctypes.byref(a), 0, None, 0, None) == 0
    assert v.lib.vssm_scan_grad_workspace_size(ctypes.byref(a), 0, ctypes.byref(n)) == 0 and n.value == 0


def test_grad_workspace_folded_rows_need_no_summaries(v):
    """Folded rows with few channel groups are cut at segment starts into
    independent ranges: the workspace is the checkpoints and the partial
    gradients only (no range summaries), whatever the number of ranges."""
    n = ctypes.c_size_t(0)
    L = 51 * 20
    a = _args(v, batch=1, dim=40, seqlen=L, dtype=0)            # both directions, 2 groups
    assert v.lib.vssm_scan_grad_workspace_size(ctypes.byref(a), 51, ctypes.byref(n)) == 0
    nch = (L + 3) // 4
    ck = 2 * 2 * nch * 512 * 4
    part = 2 * L * 96 * 4
    r = lambda b: (b + 255) // 256 * 256
    assert n.value == r(ck) + part
    # the same rows unfolded are cut and joined by summaries: more workspace
    m = ctypes.c_size_t(0)
    assert v.lib.vssm_scan_grad_workspace_size(ctypes.byref(a), 0, ctypes.byref(m)) == 0
    assert m.value > n.value
