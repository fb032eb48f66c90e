#!/usr/bin/env python
"""Benchmark: bidirectional selective scan on one B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one scan of the whole workload (default vim_s_224: Vim-S at 224^2,
batch 128, 197 tokens, 768 channels, 16 states, bf16 I/O, both directions,
silu gate). Prints ONE JSON line (rank 0). ``value`` is algorithmic GB/s of
the whole job (inputs resident in HBM); ``e2e`` is the same metric with the
host<->device copies of every step's inputs and output inside the timed
region; ``roofline`` relates the scan kernel to the bound that limits it.

Under torchrun (N > 1) every rank scans its own full workload (weak scaling,
no collective on the data path: rows are independent); the timed region is
bracketed by barriers and the slowest rank's time is used.

``--impl reference`` times the fp64 CPU oracle on the host cores instead
(a bounded sample of the same workload per step).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import (DIR_BOTH, DIR_BWD, DIR_FWD, ORDER, WORKLOADS,  # noqa: E402
                       algorithmic_bytes, exp_count, make_inputs)

METRIC = "bidir selective-scan GB/s and Gtoken·ch/s, % of HBM roofline, 1×B300"
L2_BYTES = 126 * 1024 * 1024
FALLBACK_MAX_SM_MHZ = 2032.0   # B300 maximum SM clock, used only when the driver reports none
EX2_PER_CLK_SM = 32        # MUFU ex2.approx.f32 per clock per SM, measured on B300
FMA_PER_CLK_SM = 128       # fp32 FMA-pipe lane operations per clock per SM
FALLBACK_HBM_GBS = 6400.0
SPEC_HBM_GBS = 8000.0
PROFILES = os.path.join(ROOT, "profiles")


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--workload", default="vim_s_224", choices=ORDER)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target CPU time of the oracle sample (the reference arm: at most this "
                        "per step)")
    p.add_argument("--fused-step", action="store_true",
                   help="pass per-direction steps before softplus, with biases (the kernel "
                        "applies softplus(delta + bias))")
    p.add_argument("--grad", action="store_true",
                   help="time a training step: the training forward (vssm_scan_train, "
                        "which also stores the state checkpoints) plus the gradient "
                        "(vssm_scan_grad) from them, for a seeded upstream gradient")
    p.add_argument("--ncssd", action="store_true",
                   help="time the NC-SSD global-state variant (vssm_ncssd) on the workload's "
                        "shapes instead of the scan")
    p.add_argument("--conv", type=int, default=0, choices=[0, 1, 2, 3, 4],
                   help="taps of the directional depthwise convolution + SiLU in front of "
                        "the scan (0: none)")
    return p.parse_args(argv)


def selected_workload(args):
    wl = WORKLOADS[args.workload]
    if args.fused_step:
        wl = wl.scaled(fused_step=True)
    if args.conv:
        wl = wl.scaled(conv=args.conv)
    return wl


def variant_key(wl):
    """Workload name plus its options, the key of the committed traffic record."""
    return wl.name + ("+fused_step" if wl.fused_step else "") + (f"+conv{wl.conv}" if wl.conv else "")


STEP_KEYS = ("delta_bwd", "delta_bias", "delta_bias_bwd")


def step_kwargs(t, wl):
    """Options of the call: per-direction steps and biases with softplus
    inside, and the directional convolution."""
    kw = {}
    if wl.fused_step:
        kw.update(delta_bwd=t["delta_bwd"], delta_bias=t["delta_bias"],
                  delta_bias_bwd=t["delta_bias_bwd"], delta_softplus=True)
    if wl.conv:
        kw.update(conv_w=t["conv_w"], conv_b=t["conv_b"], conv_w_bwd=t["conv_w_bwd"],
                  conv_b_bwd=t["conv_b_bwd"])
    return kw


# ------------------------------------------------------------------ distributed

def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def dist_init(backend):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, world


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_max(value: float) -> float:
    """Max of a float over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput under weak scaling: all ranks' units / slowest time."""
    return units_per_rank * world / max_seconds


# ------------------------------------------------------------------ clocks

class _Nvml:
    """Read-only NVML through ctypes (clock and clock-event-reason queries
    only; nothing is ever set). Looks for the driver's libnvidia-ml in the
    loader path and in the usual driver directories."""
    SM = 1   # NVML_CLOCK_SM

    def __init__(self, uuid: str):
        import glob
        names = ["libnvidia-ml.so.1", "libnvidia-ml.so"]
        for d in ("/usr/lib/x86_64-linux-gnu", "/usr/lib64", "/usr/lib", "/usr/local/nvidia/lib64",
                  "/usr/local/nvidia/lib", "/usr/lib/x86_64-linux-gnu/nvidia/current"):
            names += sorted(glob.glob(os.path.join(d, "libnvidia-ml.so*")))
        self.lib, err = None, None
        for n in names:
            try:
                self.lib = ctypes.CDLL(n)
                break
            except OSError as e:
                err = e
        if self.lib is None:
            raise OSError(f"libnvidia-ml not found ({err})")
        init = getattr(self.lib, "nvmlInit_v2", None) or self.lib.nvmlInit
        if init() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        get = getattr(self.lib, "nvmlDeviceGetHandleByUUID")
        if get(uuid.encode(), ctypes.byref(self.h)) != 0:
            raise OSError(f"no NVML device with uuid {uuid}")
        self._reasons = (getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
                         or self.lib.nvmlDeviceGetCurrentClocksThrottleReasons)

    def sm_mhz(self):
        v = ctypes.c_uint()
        return v.value if self.lib.nvmlDeviceGetClockInfo(self.h, self.SM, ctypes.byref(v)) == 0 else None

    def max_sm_mhz(self):
        v = ctypes.c_uint()
        return v.value if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.SM, ctypes.byref(v)) == 0 else None

    def reasons(self):
        v = ctypes.c_ulonglong()
        return int(v.value) if self._reasons(self.h, ctypes.byref(v)) == 0 else 0


class ClockSampler:
    """Samples the SM clock and the clock-event reasons of one GPU during the
    timed region: NVML (read-only, through ctypes) every half millisecond when
    the library can be loaded, else a streaming nvidia-smi at its shortest
    period. It only reads clocks; it never sets them."""
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, uuid: str, period_ms: float = 0.5):
        self.uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        self.period_ms = period_ms
        self.samples = []
        self.max_mhz = None
        self.err = None
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        try:
            self.nv = _Nvml(self.uuid)
            self.max_mhz = self.nv.max_sm_mhz()
            self.source = "nvml"
        except Exception as e:
            self.nv = None
            self.err = f"nvml: {e!r}"

    @property
    def ok(self):
        return True

    def _nvml_sample(self):
        self.samples.append((self.nv.sm_mhz(), self.nv.reasons()))

    def _nvml_loop(self):
        while not self._stop.is_set():
            self._nvml_sample()
            time.sleep(self.period_ms / 1000)

    def _smi_loop(self):
        for line in self._proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 3:
                continue
            try:
                mhz, mx = float(parts[0]), float(parts[1])
                reasons = int(parts[2], 16)
            except ValueError:
                continue
            self.max_mhz = mx
            self.samples.append((mhz, reasons))
            if self._stop.is_set():
                break

    def start(self):
        """Begin sampling; returns once the first sample has arrived (or failed)."""
        if self.nv is not None:
            self._nvml_sample()
            # the launching thread holds the interpreter most of the time: a
            # short switch interval lets the sampler run every period
            self._switch = sys.getswitchinterval()
            sys.setswitchinterval(self.period_ms / 2000)
            self._thread = threading.Thread(target=self._nvml_loop, daemon=True)
            self._thread.start()
            return
        import subprocess
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.uuid,
                 "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", f"-lms={max(10, int(self.period_ms))}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError as e:
            self.err = (self.err or "") + f"; nvidia-smi: {e!r}"
            return
        self.source = "nvidia-smi"
        self._thread = threading.Thread(target=self._smi_loop, daemon=True)
        self._thread.start()
        t0 = time.time()
        while not self.samples and time.time() - t0 < 10:
            time.sleep(0.01)

    def stop(self):
        self._stop.set()
        if getattr(self, "_switch", None):
            sys.setswitchinterval(self._switch)
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def summary(self, first_in_region: int = 0):
        """Median SM clock and the union of the reasons over the samples taken
        from index first_in_region on (the timed region)."""
        smp = self.samples[first_in_region:] or self.samples[-1:]
        if not smp:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [],
                    "error": self.err or "no samples"}
        bits = 0
        for _, r in smp:
            bits |= r
        names = [n for b, n in self.REASONS.items() if bits & b and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(m for m, _ in smp), "sm_max_mhz": self.max_mhz,
                "reasons": names, "samples": len(smp), "source": self.source}


# ------------------------------------------------------------------ helpers

def source_sha() -> str:
    """Hash of the CUDA sources' code (comments and blank lines removed, so
    that a comment edit does not orphan the committed ncu records)."""
    import re
    csrc = os.path.join(ROOT, "bidirectional_selective_scan_vssm_b300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            text = open(os.path.join(csrc, f), encoding="utf-8").read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            text = re.sub(r"//[^\n]*", "", text)
            code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
            h.update(f.encode() + b"\0" + code.encode())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def ncu_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    path = os.path.join(PROFILES, "ncu_dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("source_sha") != source_sha():
        return None
    return e.get("dram_bytes_per_launch")


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# ------------------------------------------------------------------ CPU oracle leg

def oracle_sample_run(wl, inp, target_s, nthreads=0):
    """Time the fp64 oracle (as it stands) on a slice of the workload sized to
    about target_s seconds, on nthreads OpenMP threads (0: all cores).
    Returns (tokch, seconds, threads, description)."""
    import oracle
    threads = nthreads if nthreads > 0 else oracle.max_threads()

    def slice_inputs(nb, nd):
        s = (slice(0, nb), slice(0, nd))
        a = dict(x=np.asarray(inp.x[s], np.float64), delta=np.asarray(inp.delta[s], np.float64),
                 z=np.asarray(inp.z[s], np.float64), B=np.asarray(inp.B[:nb], np.float64),
                 C=np.asarray(inp.C[:nb], np.float64), A_fwd=inp.A_fwd[:nd].astype(np.float64),
                 A_bwd=inp.A_bwd[:nd].astype(np.float64), D_fwd=inp.D_fwd[:nd].astype(np.float64),
                 D_bwd=inp.D_bwd[:nd].astype(np.float64), step={})
        if wl.fused_step:
            a["step"] = dict(delta_bwd=np.asarray(inp.delta_bwd[s], np.float64),
                             delta_bias=inp.delta_bias[:nd].astype(np.float64),
                             delta_bias_bwd=inp.delta_bias_bwd[:nd].astype(np.float64),
                             delta_softplus=True)
        if wl.conv:
            a["step"].update({k: getattr(inp, k)[:nd].astype(np.float64)
                              for k in ("conv_w", "conv_b", "conv_w_bwd", "conv_b_bwd")})
        return a

    def run(a):
        t0 = time.perf_counter()
        oracle.scan(a["x"], a["delta"], a["A_fwd"], a["A_bwd"], a["B"], a["C"], a["D_fwd"],
                    a["D_bwd"], a["z"], dirs=wl.dirs, seg_len=wl.seg_len, nthreads=nthreads,
                    **a["step"])
        return time.perf_counter() - t0

    def shape(rows):
        nb = min(wl.batch, max(1, rows // wl.dim))
        nd = wl.dim if nb > 1 or rows >= wl.dim else min(wl.dim, rows)
        return nb, nd

    # calibrate on a few channels of one batch entry, then grow the sample
    # while it runs well under the target (a small calibration run is
    # dominated by thread start-up and overestimates the per-row time)
    rows = min(wl.dim, max(threads, 16))
    nb, nd = shape(rows)
    a = slice_inputs(nb, nd)
    secs = run(a)
    for _ in range(4):
        if secs >= 0.5 * target_s or nb * nd == wl.batch * wl.dim:
            break
        rows = max(rows + 1, int(nb * nd * target_s / max(secs, 1e-4)))
        nb, nd = shape(rows)
        a = slice_inputs(nb, nd)
        secs = run(a)
    reps = 1
    # a sample that covers the whole workload in well under the target is
    # repeated (at most 30 times) so that the time is not dominated by noise
    while secs < target_s and reps < 30 and nb * nd == wl.batch * wl.dim:
        secs += run(a)
        reps += 1
    desc = (f"{nb} of {wl.batch} batch entries x {nd} of {wl.dim} channels x {wl.seqlen} tokens "
            f"({nb * nd * wl.seqlen} token-channels), {reps} run(s), fp64, {threads} OpenMP threads")
    return reps * nb * nd * wl.seqlen, secs, threads, desc


def run_reference(args):
    rank, world = dist_init("gloo")
    if rank != 0:
        return
    wl = selected_workload(args)
    inp = make_inputs(wl, seed=0)
    # each step: a bounded oracle sample, so that the whole run stays within a
    # few minutes (at most --cpu-seconds per step)
    per_step = min(args.cpu_seconds, max(0.2, 150.0 / max(1, args.steps + args.warmup)))
    bpt = algorithmic_bytes(wl) / wl.tokch
    for _ in range(args.warmup):
        oracle_sample_run(wl, inp, per_step)
    tot_tok, tot_s, desc, threads = 0, 0.0, "", 0
    for _ in range(args.steps):
        tok, s, threads, desc = oracle_sample_run(wl, inp, per_step)
        tot_tok += tok
        tot_s += s
    gbs = tot_tok * bpt / tot_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_s / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, "n/a (CPU)"),
        "gtokch_per_s": round(tot_tok / tot_s / 1e9, 6),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": desc + " per step", "cpu": cpu_model()},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def workload_config(wl, l2_note):
    return {"workload": wl.name, "batch": wl.batch, "seqlen": wl.seqlen, "dim": wl.dim,
            "dstate": wl.dstate, "io_dtype": wl.dtype,
            "dirs": {DIR_FWD: "fwd", DIR_BWD: "bwd", DIR_BOTH: "both"}[wl.dirs],
            "seg_len": wl.seg_len or None, "gate": "silu(z)", "l2": l2_note,
            "step": ("softplus(delta + bias), own delta and bias per direction" if wl.fused_step
                     else "delta as given (post-softplus), shared by both directions"),
            "conv": (f"silu(depthwise conv, {wl.conv} taps), causal forward, reversed backward"
                     if wl.conv else None),
            "description": wl.description}


# ------------------------------------------------------------------ GPU leg

def run_ncssd(args):
    """The NC-SSD variant on the workload's shapes (x, z, B, C, D of the
    workload plus per-token weights m): HBM-bound, so its roofline is the
    measured copy bandwidth."""
    import torch
    import bidirectional_selective_scan_vssm_b300 as vssm

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU path)")
    torch.cuda.set_device(local)
    dist_init("nccl")
    dev = torch.device("cuda", local)
    wl = WORKLOADS[args.workload].scaled(ncssd=True)
    inp = make_inputs(wl, seed=rank)
    e = 4 if wl.dtype == "f32" else 2
    # bytes the variant must move: x, z read and out written once; B, C, m, D read
    step_bytes = (3 * wl.tokch * e + 2 * wl.batch * wl.seqlen * wl.dstate * e
                  + wl.batch * wl.seqlen * 4 + wl.dim * 4)

    def upload(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    base = {k: upload(inp.storage(k)) for k in ("x", "z", "B", "C")}
    base["m"] = torch.from_numpy(inp.m).to(dev)
    base["D"] = torch.from_numpy(inp.D_fwd).to(dev)
    nsets = int(min(64, max(2, math.ceil(3 * L2_BYTES / step_bytes))))
    sets = [base] + [{k: v.clone() for k, v in base.items()} for _ in range(nsets - 1)]
    outs = [torch.empty_like(base["x"]) for _ in range(nsets)]
    l2_note = (f"{nsets} rotating input/output sets, {nsets * step_bytes / 2**20:.0f} MiB "
               f"{'>' if nsets * step_bytes > L2_BYTES else '<='} 126 MiB L2")
    stream = torch.cuda.current_stream(dev)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    argsets, ws = [], None
    for s_, o in zip(sets, outs):
        a = vssm.NcssdArgs()
        a.x, a.z, a.B, a.C = (s_[k].data_ptr() for k in ("x", "z", "B", "C"))
        a.m, a.D, a.out = s_["m"].data_ptr(), s_["D"].data_ptr(), o.data_ptr()
        a.batch, a.dim, a.seqlen, a.dstate = wl.batch, wl.dim, wl.seqlen, wl.dstate
        a.dtype = vssm.VSSM_F32 if wl.dtype == "f32" else vssm.VSSM_BF16
        n = ctypes.c_size_t(0)
        vssm.lib.vssm_ncssd_workspace_size(ctypes.byref(a), ctypes.byref(n))
        if ws is None:
            ws = torch.empty(max(1, n.value), dtype=torch.uint8, device=dev)
        a.workspace, a.workspace_bytes = ws.data_ptr(), n.value
        argsets.append(a)

    def launch(i):
        st = vssm.lib.vssm_ncssd(ctypes.byref(argsets[i % nsets]), sptr)
        if st != 0:
            raise RuntimeError(vssm.lib.vssm_last_error().decode())

    for i in range(args.warmup):
        launch(i)
    torch.cuda.synchronize()
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(str(torch.cuda.get_device_properties(dev).uuid))
    sampler.start()
    barrier()
    torch.cuda.synchronize()
    first_sample = len(sampler.samples)
    start.record(stream)
    for i in range(args.steps):
        ev_b[i].record(stream)
        launch(i)
        ev_e[i].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    sampler.stop()
    region_s = reduce_max(start.elapsed_time(end) / 1e3)
    kern_avg_s = statistics.fmean(b.elapsed_time(e_) for b, e_ in zip(ev_b, ev_e)) / 1e3
    peaks, peaks_kind = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    gbs = aggregate(step_bytes * args.steps, world, region_s) / 1e9
    ach = step_bytes / kern_avg_s / 1e9
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(region_s / args.steps * 1e3, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if wl.dtype == "bf16" else "f32",
            "arithmetic": ("contractions as bf16 tensor-core MMAs on hi/lo operand splits, fp32 "
                           "accumulation and epilogue" if wl.dtype == "bf16" else "fp32 FMA pipe"),
            "data": "synthetic",
            "config": dict(workload_config(wl, l2_note), step="NC-SSD (vssm_ncssd)"),
            "gtokch_per_s": round(aggregate(wl.tokch * args.steps, world, region_s) / 1e9, 4),
            "roofline": {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(ach / hbm_peak, 4),
                         "traffic": ncu_traffic(wl.name + "+ncssd"),
                         "peak_kind": peaks_kind, "kernel_avg_us": round(kern_avg_s * 1e6, 3),
                         "launches_per_call": 1,
                         "algorithmic_bytes_per_launch": step_bytes},
            "cpu_baseline": None, "e2e": None, "clocks": sampler.summary(first_sample),
            "gpu_launches": args.steps, "kernel_source_sha": source_sha(),
        }
        print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    import bidirectional_selective_scan_vssm_b300 as vssm

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU path)")
    torch.cuda.set_device(local)
    dist_init("nccl")
    dev = torch.device("cuda", local)
    wl = selected_workload(args)
    inp = make_inputs(wl, seed=rank)
    set_bytes = algorithmic_bytes(wl)

    def upload(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    base = {k: upload(inp.storage(k)) for k in ("x", "delta", "z", "B", "C")}
    for k in ("A_fwd", "A_bwd", "D_fwd", "D_bwd"):
        base[k] = torch.from_numpy(getattr(inp, k)).to(dev)
    if wl.fused_step:
        base["delta_bwd"] = upload(inp.storage("delta_bwd"))
        base["delta_bias"] = torch.from_numpy(inp.delta_bias).to(dev)
        base["delta_bias_bwd"] = torch.from_numpy(inp.delta_bias_bwd).to(dev)
    if wl.conv:
        for k in ("conv_w", "conv_b", "conv_w_bwd", "conv_b_bwd"):
            base[k] = torch.from_numpy(getattr(inp, k)).to(dev)
    nsets = int(min(64, max(2, math.ceil(3 * L2_BYTES / set_bytes))))
    sets = [base] + [{k: v.clone() for k, v in base.items()} for _ in range(nsets - 1)]
    outs = [torch.empty_like(base["x"]) for _ in range(nsets)]
    total = nsets * set_bytes
    l2_note = (f"{nsets} rotating input/output sets, {total / 2**20:.0f} MiB "
               f"{'>' if total > L2_BYTES else '<='} 126 MiB L2")

    stream = torch.cuda.current_stream(dev)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    seg = wl.seg_len
    fn = vssm.lib.vssm_scan_folded if seg else vssm.lib.vssm_scan_bidir
    argsets = []
    ws = None
    for s, o in zip(sets, outs):
        a = vssm.make_args(s["x"], s["delta"], s["A_fwd"], s["A_bwd"], s["B"], s["C"],
                           s["D_fwd"], s["D_bwd"], s["z"], o, dirs=wl.dirs, **step_kwargs(s, wl))
        need = vssm.workspace_size(a, seg)
        if need and ws is None:
            ws = torch.empty(need, dtype=torch.uint8, device=dev)
        if need:
            a.workspace, a.workspace_bytes = ws.data_ptr(), need
        argsets.append(a)

    # token ranges per row and kernel launches per call (2 when few rows make
    # the library cut them and join the ranges by the carry)
    ranges, launches = vssm.plan(argsets[0], seg)

    grad_calls = []
    if args.grad:
        # the training step: the training forward (vssm_scan_train, which also
        # stores the state checkpoints) and the gradient of sum(dout * out)
        # from them, for a seeded dout; outputs, checkpoints and workspace
        # allocated once
        gen = torch.Generator(device=dev)
        gen.manual_seed(1234 + rank)
        dout = torch.randn(base["x"].shape, device=dev, generator=gen).to(base["x"].dtype)
        gws = None
        ckpt_bytes = vssm.ckpt_size(argsets[0])
        ckpts = [torch.empty(ckpt_bytes // 4, dtype=torch.float32, device=dev) for _ in range(nsets)]
        for s_, a, ck in zip(sets, argsets, ckpts):
            batch, dim, L = s_["x"].shape
            K = wl.conv
            f32 = dict(dtype=torch.float32, device=dev)
            outs_g = dict(dx=torch.empty_like(s_["x"]), ddelta=torch.empty_like(s_["x"]),
                          dz=torch.empty_like(s_["x"]), dB=torch.empty(batch, L, 16, **f32),
                          dC=torch.empty(batch, L, 16, **f32),
                          dA_fwd=torch.empty(dim, 16, **f32) if wl.dirs & 1 else None,
                          dA_bwd=torch.empty(dim, 16, **f32) if wl.dirs & 2 else None,
                          dD_fwd=torch.empty(dim, **f32) if wl.dirs & 1 else None,
                          dD_bwd=torch.empty(dim, **f32) if wl.dirs & 2 else None,
                          ddelta_bwd=torch.empty_like(s_["x"]) if wl.fused_step else None,
                          ddelta_bias=torch.empty(dim, **f32) if wl.fused_step else None,
                          ddelta_bias_bwd=torch.empty(dim, **f32) if wl.fused_step else None,
                          dconv_w=torch.empty(dim, K, **f32) if K else None,
                          dconv_b=torch.empty(dim, **f32) if K else None,
                          dconv_w_bwd=torch.empty(dim, K, **f32) if K else None,
                          dconv_b_bwd=torch.empty(dim, **f32) if K else None)
            g = vssm.GradArgs()
            g.dout = dout.data_ptr()
            for k, v in outs_g.items():
                setattr(g, k, v.data_ptr() if v is not None else None)
            g.ckpt, g.ckpt_bytes = ck.data_ptr(), ckpt_bytes
            ga = vssm.ScanArgs.from_buffer_copy(a)
            need = vssm.grad_workspace_size(ga, seg)
            if gws is None:
                gws = torch.empty(need, dtype=torch.uint8, device=dev)
            ga.workspace, ga.workspace_bytes = gws.data_ptr(), need
            grad_calls.append((ga, g, outs_g, ck))
        launches += vssm.grad_plan(grad_calls[0][0], grad_calls[0][1], seg)[1]

    def launch(i):
        a = ctypes.byref(argsets[i % nsets])
        if grad_calls:
            ga, g, _, ck = grad_calls[i % nsets]
            st = vssm.lib.vssm_scan_train(a, seg, ctypes.c_void_p(ck.data_ptr()), ck.numel() * 4, sptr)
            if st == 0:
                st = vssm.lib.vssm_scan_grad(ctypes.byref(ga), ctypes.byref(g), seg, sptr)
        else:
            st = fn(a, seg, sptr) if seg else fn(a, sptr)
        if st != 0:
            raise RuntimeError(vssm.lib.vssm_last_error().decode())

    for i in range(args.warmup):
        launch(i)
    torch.cuda.synchronize()

    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(str(torch.cuda.get_device_properties(dev).uuid))
    sampler.start()
    barrier()
    torch.cuda.synchronize()
    first_sample = len(sampler.samples)
    start.record(stream)
    for i in range(args.steps):
        ev_b[i].record(stream)
        launch(i)
        ev_e[i].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    sampler.stop()
    region_s = reduce_max(start.elapsed_time(end) / 1e3)
    kern_ms = [b.elapsed_time(e) for b, e in zip(ev_b, ev_e)]
    kern_avg_s = statistics.fmean(kern_ms) / 1e3

    # bytes a step must move: the forward's, plus with --grad the gradient's
    # (x, delta, z, dout read and dx, ddelta, dz written in the I/O dtype; B, C
    # read and dB, dC written in fp32; A, D read and dA, dD written)
    step_bytes = set_bytes
    if args.grad:
        e = 4 if wl.dtype == "f32" else 2
        ndir = 2 if wl.dirs == 3 else 1
        step_bytes += (7 * wl.tokch * e + 2 * wl.batch * wl.seqlen * wl.dstate * (e + 4)
                       + 2 * ndir * (wl.dim * wl.dstate + wl.dim) * 4)
    gbs = aggregate(step_bytes * args.steps, world, region_s) / 1e9
    gtok = aggregate(wl.tokch * args.steps, world, region_s) / 1e9
    peaks, peaks_kind = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    clocks = sampler.summary(first_sample)

    # Roofline of the scan kernel: the exp unit and the fp32 FMA pipe both
    # allow 32 state updates per clock per SM (1 ex2 + 4 fp32 ops each). When
    # the plan cuts rows (launches == 2) the events bracket the summary pass
    # and the scan together, and only the algorithmic updates are counted
    # (the summary pass's repeated ones are not credited).
    upd = exp_count(wl) * (2 if args.grad else 1)
    ach = upd / kern_avg_s / 1e9
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    max_mhz = float(clocks.get("sm_max_mhz") or FALLBACK_MAX_SM_MHZ)
    peak_upd = EX2_PER_CLK_SM * sms * max_mhz * 1e6 / 1e9
    kern_gbs = step_bytes / kern_avg_s / 1e9
    med = clocks.get("sm_mhz")
    roofline = {
        "bound": "alu", "achieved": round(ach, 2), "peak": round(peak_upd, 2),
        "unit": "Gupdate/s", "frac": round(ach / peak_upd, 4),
        "traffic": ncu_traffic(variant_key(wl) + ("+grad" if args.grad else "")),
        "update": "one (token, channel, state, direction) recurrence step: 1 MUFU ex2 + 4 fp32 FMA-pipe ops",
        "peak_basis": f"{EX2_PER_CLK_SM} ex2/clk/SM (and {FMA_PER_CLK_SM}/4 FMA-pipe updates/clk/SM) "
                      f"x {sms} SMs x {max_mhz:.0f} MHz max SM clock",
        "frac_at_median_clock": round(ach / (peak_upd * med / max_mhz), 4) if med else None,
        "kernel_avg_us": round(kern_avg_s * 1e6, 3),
        "launches_per_call": launches,
        "ranges_per_row": ranges,
        "kernel_hbm_gbs": round(kern_gbs, 1),
        "hbm_frac": round(kern_gbs / hbm_peak, 4),
        "hbm_peak_gbs": hbm_peak, "hbm_peak_kind": peaks_kind,
        "hbm_frac_spec_8tbs": round(kern_gbs / SPEC_HBM_GBS, 4),
        "algorithmic_bytes_per_launch": step_bytes,
    }

    # ---- end to end through the public API: pinned host -> device, scan, -> host
    e2e = None
    if args.e2e_steps > 0 and not args.grad:
        # end to end through the host-buffer entry point (vssm_scan_host):
        # page-locked host inputs in, the output back in page-locked host
        # memory; the copies and the scans of the slices overlap on three
        # streams inside the call, and the call ends when the output is home
        host = {k: v.cpu().pin_memory() for k, v in base.items()}
        out_h = torch.empty(base["x"].shape, dtype=base["x"].dtype).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = out_h.numel() * out_h.element_size()
        hkw = {k: host[k] for k in step_kwargs(host, wl)} if (wl.fused_step or wl.conv) else {}
        if hkw:
            raise SystemExit("the end-to-end leg covers the scan without step options or convolution")

        def e2e_step():
            vssm.scan_host(host["x"], host["delta"], host["A_fwd"], host["A_bwd"], host["B"],
                           host["C"], host["D_fwd"], host["D_bwd"], host["z"], out=out_h,
                           dirs=wl.dirs, seg_len=seg, device=dev, stream=stream, sync=False)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        e2e_s = reduce_max(e0.elapsed_time(e1) / 1e3)
        e2e = {"value": round(aggregate(set_bytes * args.e2e_steps, world, e2e_s) / 1e9, 3),
               "unit": "GB/s", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "steps": args.e2e_steps, "path": "vssm_scan_host (pinned host buffers, 8 slices)",
               "gtokch_per_s": round(aggregate(wl.tokch * args.e2e_steps, world, e2e_s) / 1e9, 4)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tok, secs, threads, desc = oracle_sample_run(wl, inp, args.cpu_seconds)
        cpu = {"value": round(tok * (set_bytes / wl.tokch) / secs / 1e9, 5), "unit": "GB/s",
               "cores": threads, "kind": "oracle", "sample": desc,
               "gtokch_per_s": round(tok / secs / 1e9, 6), "cpu": cpu_model()}
        tok1, secs1, _, desc1 = oracle_sample_run(wl, inp, min(5.0, args.cpu_seconds / 2), nthreads=1)
        cpu["single_thread"] = {"value": round(tok1 * (set_bytes / wl.tokch) / secs1 / 1e9, 5),
                                "unit": "GB/s", "gtokch_per_s": round(tok1 / secs1 / 1e9, 6),
                                "sample": desc1}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(region_s / args.steps * 1e3, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": dict(workload_config(wl, l2_note),
                           step="forward + gradient (training)" if args.grad else "forward"),
            "gtokch_per_s": round(gtok, 4),
            "hbm_frac_of_measured": round(gbs / world / hbm_peak, 4),
            "hbm_frac_of_spec_8tbs": round(gbs / world / SPEC_HBM_GBS, 4),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "clocks": clocks, "gpu_launches": args.steps * launches,
            "kernel_source_sha": source_sha(),
        }
        print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.ncssd:
        run_ncssd(args)
    else:
        run_ours(args)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
