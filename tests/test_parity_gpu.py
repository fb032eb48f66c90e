"""CUDA path vs the fp64 oracle, element by element (needs a B300).

Tolerance (normwise max relative error, max|g-r| / max|r|): 1e-4 for float32
I/O and 2e-2 for bfloat16 I/O with fp32 state. The oracle reads the same
(bf16-rounded) input values, so only arithmetic and the final rounding count.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL, elementwise_rel, normwise_rel, to_device
from workloads import DIR_BOTH, DIR_BWD, DIR_FWD, ORDER, WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import bidirectional_selective_scan_vssm_b300 as vssm  # noqa: E402  (fails loudly if unbuilt)


def _run(t, dirs, seg_len=0, gate=True, skip=True, bc_bwd=None):
    kw = dict(D_fwd=t["D_fwd"] if skip else None, D_bwd=t["D_bwd"] if skip else None,
              z=t["z"] if gate else None, dirs=dirs)
    if bc_bwd is not None:
        kw["B_bwd"], kw["C_bwd"] = bc_bwd
    if seg_len:
        return vssm.scan_folded(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"],
                                seg_len=seg_len, **kw)
    return vssm.scan_bidir(t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"], **kw)


def _oracle(inp, dirs, seg_len=0, gate=True, skip=True, bc_bwd=None):
    return oracle.scan(inp.x, inp.delta, inp.A_fwd, inp.A_bwd, inp.B, inp.C,
                       inp.D_fwd if skip else None, inp.D_bwd if skip else None,
                       inp.z if gate else None,
                       B_bwd=None if bc_bwd is None else bc_bwd[0],
                       C_bwd=None if bc_bwd is None else bc_bwd[1],
                       dirs=dirs, seg_len=seg_len)


def _check(got, ref, dtype, what=""):
    g = got.float().cpu().numpy()
    err = normwise_rel(g, ref)
    assert err <= TOL[dtype], f"{what}: normwise rel err {err:.3e} > {TOL[dtype]} " \
                              f"(elementwise {elementwise_rel(g, ref):.3e})"
    return err


SHAPES = [  # (batch, dim, L, N): ragged channel blocks, chunk edges, both y-buffer paths
    (1, 1, 1, 16), (2, 40, 31, 16), (2, 40, 33, 16), (1, 64, 64, 16), (3, 33, 197, 16),
    (1, 32, 385, 16), (1, 32, 513, 16), (1, 8, 1025, 16), (2, 16, 100, 4), (1, 24, 7, 1),
    (1, 96, 2, 16), (1, 70, 4097, 16),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes(dtype, dirs, shape):
    b, d, L, N = shape
    wl = WORKLOADS["vim_ti_224"].scaled(batch=b, dim=d, seqlen=L, dstate=N, dtype=dtype)
    inp = make_inputs(wl, seed=100 + L)
    got = _run(to_device(inp), dirs)
    _check(got, _oracle(inp, dirs), dtype, f"{shape} dirs={dirs}")


@pytest.mark.parametrize("gate,skip", [(False, True), (True, False), (False, False)])
def test_gate_and_skip_optional(gate, skip):
    wl = WORKLOADS["vim_ti_224"].scaled(batch=2, dim=40, seqlen=77)
    inp = make_inputs(wl, seed=7)
    got = _run(to_device(inp), DIR_BOTH, gate=gate, skip=skip)
    _check(got, _oracle(inp, DIR_BOTH, gate=gate, skip=skip), "f32")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_separate_backward_B_C(dtype):
    wl = WORKLOADS["vim_ti_224"].scaled(batch=2, dim=48, seqlen=150, dtype=dtype)
    inp = make_inputs(wl, seed=8)
    other = make_inputs(wl, seed=9)
    t = to_device(inp)
    t2 = to_device(other)
    got = _run(t, DIR_BOTH, bc_bwd=(t2["B"], t2["C"]))
    _check(got, _oracle(inp, DIR_BOTH, bc_bwd=(other.B, other.C)), dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BWD, DIR_BOTH])
@pytest.mark.parametrize("seg,nseg", [(1, 40), (5, 9), (51, 64), (51, 1), (64, 33)])
def test_folded(dtype, dirs, seg, nseg):
    wl = WORKLOADS["sf_folded"].scaled(batch=2, dim=40, seqlen=seg * nseg, seg_len=seg,
                                       dtype=dtype, dirs=dirs)
    inp = make_inputs(wl, seed=seg + nseg)
    got = _run(to_device(inp), dirs, seg_len=seg)
    _check(got, _oracle(inp, dirs, seg_len=seg), dtype, f"seg={seg} nseg={nseg}")


def test_folded_forward_partial_last_segment():
    wl = WORKLOADS["sf_folded"].scaled(batch=1, dim=33, seqlen=51 * 7 + 20, dtype="f32")
    inp = make_inputs(wl, seed=21)
    got = _run(to_device(inp), DIR_FWD, seg_len=51)
    _check(got, _oracle(inp, DIR_FWD, seg_len=51), "f32")


@pytest.mark.parametrize("dirs", [DIR_FWD, DIR_BOTH])
def test_folded_equals_unfolded_on_gpu(dirs):
    """SF-Mamba page: the folded output equals the unfolded output. B2
    sequences of T tokens scanned as a batch vs folded into one row."""
    T, B2, dim = 51, 24, 64
    wl = WORKLOADS["vim_s_224"].scaled(batch=B2, dim=dim, seqlen=T)
    t = to_device(make_inputs(wl, seed=22))
    ref = _run(t, dirs)                                          # (B2, dim, T)
    f = dict(t)
    for k in ("x", "delta", "z"):
        f[k] = t[k].permute(1, 0, 2).reshape(1, dim, B2 * T).contiguous()
    for k in ("B", "C"):
        f[k] = t[k].reshape(1, B2 * T, -1).contiguous()
    got = _run(f, dirs, seg_len=T).reshape(dim, B2, T).permute(1, 0, 2)
    assert torch.equal(got, ref)


def test_deterministic_and_stream():
    wl = WORKLOADS["vim_s_224"].scaled(batch=4, dim=96)
    t = to_device(make_inputs(wl, seed=30))
    a = _run(t, DIR_BOTH)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = _run(t, DIR_BOTH)
    s.synchronize()
    assert torch.equal(a, b)


def test_empty_problem_is_noop():
    wl = WORKLOADS["vim_s_224"].scaled(batch=2, dim=8)
    t = to_device(make_inputs(wl, seed=31))
    for k in ("x", "delta", "z"):
        t[k] = t[k][:0]
    t["B"], t["C"] = t["B"][:0], t["C"][:0]
    out = _run(t, DIR_BOTH)
    assert out.shape[0] == 0


def test_misaligned_pointer_is_rejected():
    wl = WORKLOADS["vim_ti_224"].scaled(batch=1, dim=4, seqlen=10)
    t = to_device(make_inputs(wl, seed=32))
    big = torch.zeros(4 * 10 + 1, device="cuda")
    x = big[1:].view(1, 4, 10)                     # 4-byte offset from an aligned base
    with pytest.raises(vssm.VssmError) as e:
        vssm.scan_bidir(x, t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"])
    assert e.value.status == -3


# ---------------------------------------------------------------- full-size workloads

def _sample_rows(wl, k, seed):
    rng = np.random.default_rng(seed)
    rows = {(0, 0), (wl.batch - 1, wl.dim - 1), (0, wl.dim - 1), (wl.batch - 1, 0)}
    while len(rows) < k:
        rows.add((int(rng.integers(wl.batch)), int(rng.integers(wl.dim))))
    return sorted(rows)


@pytest.mark.parametrize("name", ORDER)
def test_full_workload(name):
    """Each workload at full size in the benchmark's launch configuration;
    the small one compared in full, the others on sampled rows."""
    wl = WORKLOADS[name]
    inp = make_inputs(wl, seed=0)
    t = to_device(inp)
    got = _run(t, wl.dirs, seg_len=wl.seg_len)
    torch.cuda.synchronize()
    if wl.tokch <= 1_000_000:
        _check(got, oracle.scan_inputs(inp), wl.dtype, name)
        return
    rows = _sample_rows(wl, 48, seed=1)
    ref = oracle.scan_rows(inp, rows)
    g = torch.stack([got[b, d] for b, d in rows]).float().cpu().numpy()
    err = normwise_rel(g, ref)
    assert err <= TOL[wl.dtype], f"{name}: sampled rows normwise rel err {err:.3e}"
    assert torch.isfinite(got.float()).all()
