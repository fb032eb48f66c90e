"""Bidirectional selective scan (S6) on NVIDIA B300 -- Python binding.

A thin ctypes layer over the C ABI in ``include/vssm.h`` (library
``libvssm.so`` built in-tree by ``build.py``). It only marshals arguments:
every step of the scan runs in the CUDA kernels. PyTorch supplies device
memory and streams. There is no CPU fallback: importing this package fails
if the library is missing, and the scan functions refuse CPU tensors.

    out = scan_bidir(x, delta, A_fwd, A_bwd, B, C, D_fwd, D_bwd, z)
    out = scan_folded(x, delta, A_fwd, None, B, C, D_fwd, None, z, seg_len=51,
                      dirs=DIR_FWD)

Shapes: x, delta, z, out (batch, dim, L); B, C (batch, L, N); A (dim, N)
float32; D (dim,) float32. x, delta, z, B, C share one dtype (float32 or
bfloat16), which is also the output dtype.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch


DIR_FWD, DIR_BWD, DIR_BOTH = 1, 2, 3
VSSM_F32, VSSM_BF16 = 0, 1
STATUS = {0: "VSSM_OK", -1: "VSSM_ERR_INVALID_ARG", -2: "VSSM_ERR_UNSUPPORTED",
          -3: "VSSM_ERR_MISALIGNED", -4: "VSSM_ERR_CUDA", -5: "VSSM_ERR_TIMEOUT",
          -6: "VSSM_ERR_WORKSPACE"}

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libvssm.so")
EXPORTS = ["vssm_scan_bidir", "vssm_scan_bidir_noalloc", "vssm_scan_folded",
           "vssm_scan_chunked", "vssm_scan_workspace_size", "vssm_scan_chunked_workspace_size",
           "vssm_scan_plan_query", "vssm_scan_grad", "vssm_scan_grad_workspace_size",
           "vssm_selftest_wait_timeout", "vssm_scan_host", "vssm_scan_host_workspace_size",
           "vssm_ncssd", "vssm_ncssd_workspace_size", "vssm_scan_train", "vssm_scan_ckpt_size",
           "vssm_scan_grad_plan_query",
           "vssm_device_error", "vssm_status_string", "vssm_last_error", "vssm_version"]
NOALLOC_SCRATCH_BYTES = 16 << 20


class ScanArgs(ctypes.Structure):
    """Mirror of ``vssm_scan_args`` (include/vssm.h)."""
    _fields_ = [
        ("x", ctypes.c_void_p), ("delta", ctypes.c_void_p), ("z", ctypes.c_void_p),
        ("B", ctypes.c_void_p), ("C", ctypes.c_void_p),
        ("B_bwd", ctypes.c_void_p), ("C_bwd", ctypes.c_void_p),
        ("A_fwd", ctypes.c_void_p), ("A_bwd", ctypes.c_void_p),
        ("D_fwd", ctypes.c_void_p), ("D_bwd", ctypes.c_void_p),
        ("out", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("batch", ctypes.c_int), ("dim", ctypes.c_int), ("seqlen", ctypes.c_int),
        ("dstate", ctypes.c_int), ("dtype", ctypes.c_int), ("dir_flags", ctypes.c_uint),
        ("delta_bwd", ctypes.c_void_p), ("delta_bias", ctypes.c_void_p),
        ("delta_bias_bwd", ctypes.c_void_p), ("delta_softplus", ctypes.c_int),
        ("conv_w", ctypes.c_void_p), ("conv_b", ctypes.c_void_p),
        ("conv_w_bwd", ctypes.c_void_p), ("conv_b_bwd", ctypes.c_void_p), ("conv_k", ctypes.c_int),
    ]


class GradArgs(ctypes.Structure):
    """Mirror of ``vssm_grad_args`` (include/vssm.h)."""
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "dout", "dx", "ddelta", "dz", "dB", "dC", "dB_bwd", "dC_bwd", "dA_fwd", "dA_bwd",
        "dD_fwd", "dD_bwd", "ddelta_bwd", "ddelta_bias", "ddelta_bias_bwd", "dconv_w", "dconv_b",
        "dconv_w_bwd", "dconv_b_bwd", "ckpt")] + [("ckpt_bytes", ctypes.c_size_t)]


class NcssdArgs(ctypes.Structure):
    """Mirror of ``vssm_ncssd_args`` (include/vssm.h)."""
    _fields_ = [
        ("x", ctypes.c_void_p), ("z", ctypes.c_void_p), ("B", ctypes.c_void_p),
        ("C", ctypes.c_void_p), ("m", ctypes.c_void_p), ("D", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("batch", ctypes.c_int), ("dim", ctypes.c_int), ("seqlen", ctypes.c_int),
        ("dstate", ctypes.c_int), ("dtype", ctypes.c_int),
    ]


class VssmError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with "
            "`python bidirectional_selective_scan_vssm_b300/build.py` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(ScanArgs)
    lib.vssm_scan_bidir.argtypes = [P, ctypes.c_void_p]
    lib.vssm_scan_bidir.restype = ctypes.c_int
    lib.vssm_scan_bidir_noalloc.argtypes = [P, ctypes.c_void_p]
    lib.vssm_scan_bidir_noalloc.restype = ctypes.c_int
    lib.vssm_scan_folded.argtypes = [P, ctypes.c_int, ctypes.c_void_p]
    lib.vssm_scan_folded.restype = ctypes.c_int
    lib.vssm_scan_chunked.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    lib.vssm_scan_chunked.restype = ctypes.c_int
    lib.vssm_scan_workspace_size.argtypes = [P, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]
    lib.vssm_scan_workspace_size.restype = ctypes.c_int
    lib.vssm_scan_chunked_workspace_size.argtypes = [P, ctypes.c_int, ctypes.c_int,
                                                     ctypes.POINTER(ctypes.c_size_t)]
    lib.vssm_scan_chunked_workspace_size.restype = ctypes.c_int
    lib.vssm_scan_plan_query.argtypes = [P, ctypes.c_int, ctypes.c_int,
                                         ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
    lib.vssm_scan_plan_query.restype = ctypes.c_int
    lib.vssm_scan_grad.argtypes = [P, ctypes.POINTER(GradArgs), ctypes.c_int, ctypes.c_void_p]
    lib.vssm_scan_grad.restype = ctypes.c_int
    lib.vssm_scan_train.argtypes = [P, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.vssm_scan_train.restype = ctypes.c_int
    lib.vssm_scan_ckpt_size.argtypes = [P, ctypes.POINTER(ctypes.c_size_t)]
    lib.vssm_scan_ckpt_size.restype = ctypes.c_int
    lib.vssm_scan_grad_plan_query.argtypes = [P, ctypes.POINTER(GradArgs), ctypes.c_int,
                                              ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
    lib.vssm_scan_grad_plan_query.restype = ctypes.c_int
    lib.vssm_scan_host.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    lib.vssm_scan_host.restype = ctypes.c_int
    lib.vssm_scan_host_workspace_size.argtypes = [P, ctypes.c_int, ctypes.c_int,
                                                  ctypes.POINTER(ctypes.c_size_t)]
    lib.vssm_scan_host_workspace_size.restype = ctypes.c_int
    NP = ctypes.POINTER(NcssdArgs)
    lib.vssm_ncssd.argtypes = [NP, ctypes.c_void_p]
    lib.vssm_ncssd.restype = ctypes.c_int
    lib.vssm_ncssd_workspace_size.argtypes = [NP, ctypes.POINTER(ctypes.c_size_t)]
    lib.vssm_ncssd_workspace_size.restype = ctypes.c_int
    lib.vssm_selftest_wait_timeout.argtypes = [ctypes.c_uint, ctypes.c_void_p]
    lib.vssm_selftest_wait_timeout.restype = ctypes.c_int
    lib.vssm_scan_grad_workspace_size.argtypes = [P, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]
    lib.vssm_scan_grad_workspace_size.restype = ctypes.c_int
    lib.vssm_status_string.argtypes = [ctypes.c_int]
    lib.vssm_status_string.restype = ctypes.c_char_p
    lib.vssm_last_error.argtypes = []
    lib.vssm_last_error.restype = ctypes.c_char_p
    lib.vssm_device_error.argtypes = [ctypes.c_void_p]
    lib.vssm_device_error.restype = ctypes.c_int
    lib.vssm_version.argtypes = []
    lib.vssm_version.restype = ctypes.c_int
    return lib


lib = _load()


def _check(status: int):
    if status != 0:
        raise VssmError(status, lib.vssm_last_error().decode())


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dev_tensor(name, t, dtype=None, shape=None, device=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def make_args(x, delta, A_fwd, A_bwd, B, C, D_fwd=None, D_bwd=None, z=None, out=None,
              B_bwd=None, C_bwd=None, dirs: int = DIR_BOTH, delta_bwd=None, delta_bias=None,
              delta_bias_bwd=None, delta_softplus: bool = False, conv_w=None, conv_b=None,
              conv_w_bwd=None, conv_b_bwd=None) -> ScanArgs:
    """Validate tensors and fill a ``vssm_scan_args`` (no workspace yet).

    delta_bwd: the backward direction's step (None = delta). delta_softplus:
    each direction's step is softplus(its delta + its bias[d]) (delta_bias,
    delta_bias_bwd: (dim,) float32; None = 0 / = delta_bias).

    conv_w (dim, K) float32, K <= 4, conv_b (dim,): the directional depthwise
    convolution + SiLU in front of the scan (causal forward, reversed
    backward); conv_w_bwd, conv_b_bwd: the backward direction's (None = the
    forward ones)."""
    x = _dev_tensor("x", x)
    if x.dtype not in (torch.float32, torch.bfloat16) or x.dim() != 3:
        raise TypeError("x must be a 3-D float32 or bfloat16 tensor (batch, dim, L)")
    batch, dim, L = x.shape
    N = B.shape[-1]
    dev, dt = x.device, x.dtype
    _dev_tensor("delta", delta, dt, x.shape, dev)
    _dev_tensor("delta_bwd", delta_bwd, dt, x.shape, dev)
    _dev_tensor("z", z, dt, x.shape, dev)
    _dev_tensor("out", out, dt, x.shape, dev)
    for n, t in (("B", B), ("C", C), ("B_bwd", B_bwd), ("C_bwd", C_bwd)):
        _dev_tensor(n, t, dt, (batch, L, N), dev)
    for n, t in (("A_fwd", A_fwd), ("A_bwd", A_bwd)):
        _dev_tensor(n, t, torch.float32, (dim, N), dev)
    for n, t in (("D_fwd", D_fwd), ("D_bwd", D_bwd), ("delta_bias", delta_bias),
                 ("delta_bias_bwd", delta_bias_bwd), ("conv_b", conv_b),
                 ("conv_b_bwd", conv_b_bwd)):
        _dev_tensor(n, t, torch.float32, (dim,), dev)
    K = 0
    if conv_w is not None:
        if conv_w.dim() != 2 or conv_w.shape[0] != dim:
            raise ValueError(f"conv_w must be (dim, K), got {tuple(conv_w.shape)}")
        K = int(conv_w.shape[1])
        _dev_tensor("conv_w", conv_w, torch.float32, (dim, K), dev)
        _dev_tensor("conv_w_bwd", conv_w_bwd, torch.float32, (dim, K), dev)
    elif conv_w_bwd is not None or conv_b is not None or conv_b_bwd is not None:
        raise ValueError("conv_w is required with the other convolution arguments")
    a = ScanArgs()
    a.x, a.delta, a.z = _ptr(x), _ptr(delta), _ptr(z)
    a.B, a.C, a.B_bwd, a.C_bwd = _ptr(B), _ptr(C), _ptr(B_bwd), _ptr(C_bwd)
    a.A_fwd, a.A_bwd, a.D_fwd, a.D_bwd = _ptr(A_fwd), _ptr(A_bwd), _ptr(D_fwd), _ptr(D_bwd)
    a.out = _ptr(out)
    a.batch, a.dim, a.seqlen, a.dstate = batch, dim, L, N
    a.dtype = VSSM_F32 if dt == torch.float32 else VSSM_BF16
    a.dir_flags = dirs
    a.delta_bwd, a.delta_bias, a.delta_bias_bwd = _ptr(delta_bwd), _ptr(delta_bias), _ptr(delta_bias_bwd)
    a.delta_softplus = 1 if delta_softplus else 0
    a.conv_w, a.conv_b, a.conv_w_bwd, a.conv_b_bwd = (_ptr(conv_w), _ptr(conv_b), _ptr(conv_w_bwd),
                                                      _ptr(conv_b_bwd))
    a.conv_k = K
    return a


def workspace_size(a: ScanArgs, seg_len: int = 0, pieces: Optional[int] = None) -> int:
    """Workspace bytes for the call (``pieces`` given: for ``vssm_scan_chunked``)."""
    n = ctypes.c_size_t(0)
    if pieces is None:
        _check(lib.vssm_scan_workspace_size(ctypes.byref(a), seg_len, ctypes.byref(n)))
    else:
        _check(lib.vssm_scan_chunked_workspace_size(ctypes.byref(a), seg_len, pieces,
                                                    ctypes.byref(n)))
    return int(n.value)


def plan(a: ScanArgs, seg_len: int = 0, pieces: int = 0):
    """(token ranges per row, kernel launches) of the call (``vssm_scan_plan_query``)."""
    r, n = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib.vssm_scan_plan_query(ctypes.byref(a), seg_len, pieces, ctypes.byref(r),
                                    ctypes.byref(n)))
    return int(r.value), int(n.value)


def grad_plan(a: ScanArgs, g: GradArgs, seg_len: int = 0):
    """(adjoint token ranges per row, kernel launches) of the gradient call
    (``vssm_scan_grad_plan_query``)."""
    r, n = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib.vssm_scan_grad_plan_query(ctypes.byref(a), ctypes.byref(g), seg_len, ctypes.byref(r),
                                         ctypes.byref(n)))
    return int(r.value), int(n.value)


_ws_cache = {}


def _workspace(device: torch.device, stream, nbytes: int) -> Optional[torch.Tensor]:
    """A scratch buffer per (device, stream), grown on demand (device memory
    via torch). Calls on one stream run in order, so they can share it."""
    if nbytes == 0:
        return None
    key = (device, stream.cuda_stream)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def _launch(fn, a: ScanArgs, seg_len: Optional[int], device, workspace, stream,
            pieces: Optional[int] = None):
    need = workspace_size(a, seg_len or 0, pieces)
    stream = stream if stream is not None else torch.cuda.current_stream(device)
    if workspace is None:
        workspace = _workspace(device, stream, need)
    if workspace is not None:
        a.workspace = workspace.data_ptr()
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    s = stream.cuda_stream
    if pieces is not None:
        _check(fn(ctypes.byref(a), int(seg_len or 0), int(pieces), ctypes.c_void_p(s)))
    elif seg_len is None:
        _check(fn(ctypes.byref(a), ctypes.c_void_p(s)))
    else:
        _check(fn(ctypes.byref(a), int(seg_len), ctypes.c_void_p(s)))


def scan_bidir(x, delta, A_fwd, A_bwd, B, C, D_fwd=None, D_bwd=None, z=None,
               dirs: int = DIR_BOTH, out=None, B_bwd=None, C_bwd=None,
               stream: Optional[torch.cuda.Stream] = None, workspace=None,
               **step) -> torch.Tensor:
    """Selective scan over independent sequences (``vssm_scan_bidir``).
    ``step``: delta_bwd, delta_bias, delta_bias_bwd, delta_softplus (see
    :func:`make_args`)."""
    if out is None:
        out = torch.empty_like(x)
    a = make_args(x, delta, A_fwd, A_bwd, B, C, D_fwd, D_bwd, z, out, B_bwd, C_bwd, dirs, **step)
    _launch(lib.vssm_scan_bidir, a, None, x.device, workspace, stream)
    return out


def scan_bidir_noalloc(x, delta, A_fwd, A_bwd, B, C, D_fwd=None, D_bwd=None, z=None,
                       dirs: int = DIR_BOTH, out=None, B_bwd=None, C_bwd=None,
                       stream: Optional[torch.cuda.Stream] = None, **step) -> torch.Tensor:
    """``vssm_scan_bidir_noalloc``: the same scan as :func:`scan_bidir` with the
    library's built-in scratch instead of a workspace (for callers that cannot
    allocate device memory; calls share the scratch, so keep them on one
    stream). ``out`` is allocated here only when not given."""
    if out is None:
        out = torch.empty_like(x)
    a = make_args(x, delta, A_fwd, A_bwd, B, C, D_fwd, D_bwd, z, out, B_bwd, C_bwd, dirs, **step)
    stream = stream if stream is not None else torch.cuda.current_stream(x.device)
    _check(lib.vssm_scan_bidir_noalloc(ctypes.byref(a), ctypes.c_void_p(stream.cuda_stream)))
    return out


def scan_folded(x, delta, A_fwd, A_bwd, B, C, D_fwd=None, D_bwd=None, z=None, *,
                seg_len: int, dirs: int = DIR_FWD, out=None, B_bwd=None, C_bwd=None,
                stream: Optional[torch.cuda.Stream] = None, workspace=None,
                **step) -> torch.Tensor:
    """Batch-folded scan with a state reset every ``seg_len`` tokens
    (``vssm_scan_folded``)."""
    if out is None:
        out = torch.empty_like(x)
    a = make_args(x, delta, A_fwd, A_bwd, B, C, D_fwd, D_bwd, z, out, B_bwd, C_bwd, dirs, **step)
    _launch(lib.vssm_scan_folded, a, seg_len, x.device, workspace, stream)
    return out


def ckpt_size(a: ScanArgs) -> int:
    """Bytes of the checkpoints ``vssm_scan_train`` stores for this call."""
    n = ctypes.c_size_t(0)
    _check(lib.vssm_scan_ckpt_size(ctypes.byref(a), ctypes.byref(n)))
    return int(n.value)


def scan_train(x, delta, A_fwd, A_bwd, B, C, D_fwd=None, D_bwd=None, z=None, *,
               seg_len: int = 0, dirs: int = DIR_BOTH, out=None, ckpt=None, B_bwd=None, C_bwd=None,
               stream: Optional[torch.cuda.Stream] = None, workspace=None, **step):
    """``vssm_scan_train``: the forward scan (folded with ``seg_len`` > 0)
    that also stores the gradient's state checkpoints. Returns (out, ckpt);
    pass ckpt to :func:`scan_grad` for the same arguments. ``ckpt`` (float32,
    at least ``ckpt_size`` bytes) is allocated here when not given."""
    if out is None:
        out = torch.empty_like(x)
    a = make_args(x, delta, A_fwd, A_bwd, B, C, D_fwd, D_bwd, z, out, B_bwd, C_bwd, dirs, **step)
    n = ckpt_size(a)
    if ckpt is None:
        ckpt = torch.empty(max(1, n // 4), dtype=torch.float32, device=x.device)
    _dev_tensor("ckpt", ckpt, torch.float32, None, x.device)
    stream = stream if stream is not None else torch.cuda.current_stream(x.device)
    need = workspace_size(a, seg_len)
    if workspace is None:
        workspace = _workspace(x.device, stream, need)
    if workspace is not None:
        a.workspace = workspace.data_ptr()
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib.vssm_scan_train(ctypes.byref(a), int(seg_len), ctypes.c_void_p(ckpt.data_ptr()),
                               ckpt.numel() * 4, ctypes.c_void_p(stream.cuda_stream)))
    return out, ckpt


def scan_chunked(x, delta, A_fwd, A_bwd, B, C, D_fwd=None, D_bwd=None, z=None, *,
                 pieces: int, seg_len: int = 0, dirs: int = DIR_BOTH, out=None, B_bwd=None,
                 C_bwd=None, stream: Optional[torch.cuda.Stream] = None,
                 workspace=None, **step) -> torch.Tensor:
    """``vssm_scan_chunked``: the scan with each row cut into ``pieces`` token
    ranges joined by the exact carry (0 = the library's choice). ``seg_len``
    > 0 makes it the folded scan."""
    if out is None:
        out = torch.empty_like(x)
    a = make_args(x, delta, A_fwd, A_bwd, B, C, D_fwd, D_bwd, z, out, B_bwd, C_bwd, dirs, **step)
    _launch(lib.vssm_scan_chunked, a, seg_len, x.device, workspace, stream, pieces)
    return out


def grad_workspace_size(a: ScanArgs, seg_len: int = 0) -> int:
    n = ctypes.c_size_t(0)
    _check(lib.vssm_scan_grad_workspace_size(ctypes.byref(a), seg_len, ctypes.byref(n)))
    return int(n.value)


def scan_grad(x, delta, A_fwd, A_bwd, B, C, D_fwd=None, D_bwd=None, z=None, *, dout,
              dirs: int = DIR_BOTH, seg_len: int = 0, B_bwd=None, C_bwd=None,
              stream: Optional[torch.cuda.Stream] = None, workspace=None, ckpt=None, **step) -> dict:
    """``vssm_scan_grad``: gradients of sum(dout * out) for the forward call
    with these arguments (``seg_len`` > 0: the folded scan; ``step``: the step
    options and the convolution of :func:`make_args`). Returns a dict with dx,
    ddelta, dz (None without z) in x's dtype and float32 dB, dC, dB_bwd, dC_bwd
    (None when shared), dA_fwd, dA_bwd, dD_fwd, dD_bwd (None for a direction
    that is not run); with the options also ddelta_bwd (x's dtype),
    ddelta_bias, ddelta_bias_bwd, dconv_w, dconv_b, dconv_w_bwd, dconv_b_bwd
    (float32), each None unless the matching input is given. ``ckpt``: the
    checkpoints :func:`scan_train` stored for the same arguments (None: the
    gradient recomputes them). Output tensors are allocated here."""
    a = make_args(x, delta, A_fwd, A_bwd, B, C, D_fwd, D_bwd, z, None, B_bwd, C_bwd, dirs, **step)
    _dev_tensor("dout", dout, x.dtype, x.shape, x.device)
    batch, dim, L = x.shape
    N = B.shape[-1]
    f32 = dict(dtype=torch.float32, device=x.device)
    sp = bool(step.get("delta_softplus"))
    cw = step.get("conv_w")
    K = int(cw.shape[1]) if cw is not None else 0

    def given(name):
        return step.get(name) is not None

    out = dict(dx=torch.empty_like(x), ddelta=torch.empty_like(x),
               dz=torch.empty_like(x) if z is not None else None,
               dB=torch.empty(batch, L, N, **f32), dC=torch.empty(batch, L, N, **f32),
               dB_bwd=torch.empty(batch, L, N, **f32) if B_bwd is not None else None,
               dC_bwd=torch.empty(batch, L, N, **f32) if C_bwd is not None else None,
               dA_fwd=torch.empty(dim, N, **f32) if dirs & DIR_FWD else None,
               dA_bwd=torch.empty(dim, N, **f32) if dirs & DIR_BWD else None,
               dD_fwd=torch.empty(dim, **f32) if dirs & DIR_FWD else None,
               dD_bwd=torch.empty(dim, **f32) if dirs & DIR_BWD else None,
               ddelta_bwd=torch.empty_like(x) if given("delta_bwd") else None,
               ddelta_bias=torch.empty(dim, **f32) if sp and given("delta_bias") else None,
               ddelta_bias_bwd=torch.empty(dim, **f32) if sp and given("delta_bias_bwd") else None,
               dconv_w=torch.empty(dim, K, **f32) if K else None,
               dconv_b=torch.empty(dim, **f32) if K and given("conv_b") else None,
               dconv_w_bwd=torch.empty(dim, K, **f32) if K and given("conv_w_bwd") else None,
               dconv_b_bwd=torch.empty(dim, **f32) if K and given("conv_b_bwd") else None)
    g = GradArgs()
    g.dout = dout.data_ptr()
    for k, v in out.items():
        setattr(g, k, _ptr(v))
    if ckpt is not None:
        _dev_tensor("ckpt", ckpt, torch.float32, None, x.device)
        g.ckpt, g.ckpt_bytes = ckpt.data_ptr(), ckpt.numel() * 4
    stream = stream if stream is not None else torch.cuda.current_stream(x.device)
    need = grad_workspace_size(a, seg_len)
    if workspace is None:
        workspace = _workspace(x.device, stream, need)
    if workspace is not None:
        a.workspace = workspace.data_ptr()
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib.vssm_scan_grad(ctypes.byref(a), ctypes.byref(g), int(seg_len),
                              ctypes.c_void_p(stream.cuda_stream)))
    return out


def ncssd(x, B, C, m, D=None, z=None, *, out=None, stream: Optional[torch.cuda.Stream] = None,
          workspace=None) -> torch.Tensor:
    """``vssm_ncssd``: the VSSD page's non-causal global-state form,
    out = (C (B^T (x m)) + D x) silu(z); m is (batch, L) float32."""
    x = _dev_tensor("x", x)
    if x.dtype not in (torch.float32, torch.bfloat16) or x.dim() != 3:
        raise TypeError("x must be a 3-D float32 or bfloat16 tensor (batch, dim, L)")
    batch, dim, L = x.shape
    N = B.shape[-1]
    dev, dt = x.device, x.dtype
    _dev_tensor("z", z, dt, x.shape, dev)
    _dev_tensor("B", B, dt, (batch, L, N), dev)
    _dev_tensor("C", C, dt, (batch, L, N), dev)
    _dev_tensor("m", m, torch.float32, (batch, L), dev)
    _dev_tensor("D", D, torch.float32, (dim,), dev)
    if out is None:
        out = torch.empty_like(x)
    _dev_tensor("out", out, dt, x.shape, dev)
    a = NcssdArgs()
    a.x, a.z, a.B, a.C, a.m, a.D, a.out = (_ptr(x), _ptr(z), _ptr(B), _ptr(C), _ptr(m), _ptr(D),
                                           _ptr(out))
    a.batch, a.dim, a.seqlen, a.dstate = batch, dim, L, N
    a.dtype = VSSM_F32 if dt == torch.float32 else VSSM_BF16
    stream = stream if stream is not None else torch.cuda.current_stream(dev)
    n = ctypes.c_size_t(0)
    _check(lib.vssm_ncssd_workspace_size(ctypes.byref(a), ctypes.byref(n)))
    if workspace is None:
        workspace = _workspace(dev, stream, int(n.value))
    if workspace is not None:
        a.workspace = workspace.data_ptr()
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib.vssm_ncssd(ctypes.byref(a), ctypes.c_void_p(stream.cuda_stream)))
    return out


def _host_tensor(name, t, dtype=None, shape=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError(f"{name} must be a host (CPU) tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def scan_host(x, delta, A_fwd, A_bwd, B, C, D_fwd=None, D_bwd=None, z=None, *, out=None,
              dirs: int = DIR_BOTH, seg_len: int = 0, slices: int = 0, B_bwd=None, C_bwd=None,
              device=None, stream: Optional[torch.cuda.Stream] = None, workspace=None,
              sync: bool = True) -> torch.Tensor:
    """``vssm_scan_host``: the scan with every tensor in host memory (use
    page-locked tensors, ``pin_memory()``, for overlapped copies); the output
    is written to the host tensor ``out`` (allocated here, pinned, when not
    given). The device workspace comes from ``workspace`` or the per-stream
    cache. With ``sync`` the call waits for the stream before returning."""
    batch, dim, L = x.shape
    N = B.shape[-1]
    dt = x.dtype
    if dt not in (torch.float32, torch.bfloat16):
        raise TypeError("x must be float32 or bfloat16")
    for n, t in (("x", x), ("delta", delta), ("z", z)):
        _host_tensor(n, t, dt, (batch, dim, L))
    for n, t in (("B", B), ("C", C), ("B_bwd", B_bwd), ("C_bwd", C_bwd)):
        _host_tensor(n, t, dt, (batch, L, N))
    for n, t in (("A_fwd", A_fwd), ("A_bwd", A_bwd)):
        _host_tensor(n, t, torch.float32, (dim, N))
    for n, t in (("D_fwd", D_fwd), ("D_bwd", D_bwd)):
        _host_tensor(n, t, torch.float32, (dim,))
    if out is None:
        out = torch.empty_like(x).pin_memory()
    _host_tensor("out", out, dt, (batch, dim, L))
    a = ScanArgs()
    a.x, a.delta, a.z = _ptr(x), _ptr(delta), _ptr(z)
    a.B, a.C, a.B_bwd, a.C_bwd = _ptr(B), _ptr(C), _ptr(B_bwd), _ptr(C_bwd)
    a.A_fwd, a.A_bwd, a.D_fwd, a.D_bwd = _ptr(A_fwd), _ptr(A_bwd), _ptr(D_fwd), _ptr(D_bwd)
    a.out = _ptr(out)
    a.batch, a.dim, a.seqlen, a.dstate = batch, dim, L, N
    a.dtype = VSSM_F32 if dt == torch.float32 else VSSM_BF16
    a.dir_flags = dirs
    device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    stream = stream if stream is not None else torch.cuda.current_stream(device)
    n = ctypes.c_size_t(0)
    _check(lib.vssm_scan_host_workspace_size(ctypes.byref(a), int(seg_len), int(slices), ctypes.byref(n)))
    if workspace is None:
        workspace = _workspace(device, stream, int(n.value))
    if workspace is not None:
        a.workspace = workspace.data_ptr()
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(device):
        _check(lib.vssm_scan_host(ctypes.byref(a), int(seg_len), int(slices),
                                  ctypes.c_void_p(stream.cuda_stream)))
    if sync:
        stream.synchronize()
    return out


def device_error(stream: Optional[torch.cuda.Stream] = None) -> None:
    """Synchronise ``stream`` and raise VssmError(VSSM_ERR_TIMEOUT) if a scan
    kernel stopped on an expired device-side wait since the last check."""
    stream = stream if stream is not None else torch.cuda.current_stream()
    _check(lib.vssm_device_error(ctypes.c_void_p(stream.cuda_stream)))


def version() -> int:
    return int(lib.vssm_version())
