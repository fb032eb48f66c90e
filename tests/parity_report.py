"""Parity report: the CUDA path against the fp64 oracle on every workload at
full size (needs a B300; run from the repository root):

    python tests/parity_report.py [--rows 48] [--out parity.json]

For each workload it runs the scan once on the seeded inputs (seed 0) through
the library and compares, with the oracle, every row of the small fp32
workload and a seeded sample of (batch, channel) rows of the others (the
oracle computes them one by one). It prints one JSON object: per workload the
normwise error max|g - r| / max|r| over the compared rows, the worst
elementwise relative error, the rows compared and the tolerance of the I/O
dtype (1e-4 float32, 2e-2 bfloat16). Not a test: the parity tests in this
directory are the gate; this gives the figures of the results table.
"""
import argparse
import json
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import oracle  # noqa: E402
from gpu_util import TOL, elementwise_rel, normwise_rel, to_device  # noqa: E402
from workloads import ORDER, WORKLOADS, make_inputs  # noqa: E402

import bidirectional_selective_scan_vssm_b300 as vssm  # noqa: E402


def run(wl, t):
    args = (t["x"], t["delta"], t["A_fwd"], t["A_bwd"], t["B"], t["C"], t["D_fwd"], t["D_bwd"],
            t["z"])
    if wl.seg_len:
        return vssm.scan_folded(*args, seg_len=wl.seg_len, dirs=wl.dirs)
    return vssm.scan_bidir(*args, dirs=wl.dirs)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--rows", type=int, default=48, help="sampled rows per large workload")
    ap.add_argument("--out", default=None)
    args = ap.parse_args()
    rep = {}
    for name in ORDER:
        wl = WORKLOADS[name]
        inp = make_inputs(wl, seed=0)
        got = run(wl, to_device(inp)).float().cpu().numpy()
        if wl.batch * wl.dim * wl.seqlen <= 1 << 20:
            ref = oracle.scan_inputs(inp)
            g, rows = got, wl.batch * wl.dim
        else:
            rng = np.random.default_rng(7)
            sel = [(int(rng.integers(0, wl.batch)), int(rng.integers(0, wl.dim)))
                   for _ in range(args.rows)]
            ref = oracle.scan_rows(inp, sel)
            g, rows = np.stack([got[b, d] for b, d in sel]), len(sel)
        rep[name] = {"normwise": float(normwise_rel(g, ref)),
                     "elementwise_max": float(elementwise_rel(g, ref)),
                     "rows": rows, "tolerance": TOL[wl.dtype], "dtype": wl.dtype}
    text = json.dumps(rep, indent=1)
    print(text)
    if args.out:
        with open(args.out, "w") as f:
            f.write(text + "\n")


if __name__ == "__main__":
    main()
