"""The fp64 oracle against its pins (CPU only)."""
import os
import shutil
import tempfile

import numpy as np
import pytest

import oracle
import oracle_pins as P
from workloads import WORKLOADS, make_inputs


@pytest.fixture(scope="module")
def lib():
    return oracle.load_library(oracle.build())


@pytest.mark.parametrize("pin", P.PINS, ids=lambda f: f.__name__)
def test_pin(lib, pin):
    assert pin(lib)


# Plausible mistakes, each planted in a copy of the C source. Every one must
# make at least one pin fail, which shows the pins can tell them apart from
# the correct recurrence.
MUTANTS = {
    "dropped_D_skip": ("acc[t] += y + Dd * xt;", "acc[t] += y;"),
    "exp_sign": ("exp(dt * Ad[n])", "exp(-dt * Ad[n])"),
    "B_C_swapped": ("dt * Bt[n] * xt", "dt * Ct[n] * xt"),
    "dropped_delta_in_input": ("dt * Bt[n] * xt", "Bt[n] * xt"),
    "output_before_update": (
        "h[n] = abar * h[n] + dt * Bt[n] * xt;\n            y += Ct[n] * h[n];",
        "y += Ct[n] * h[n];\n            h[n] = abar * h[n] + dt * Bt[n] * xt;"),
    "backward_not_reversed": ("rev ? (L - 1 - k) : k", "k"),
    "fwd_reset_off_by_one": ("(t % seg_len == 0)", "(t % seg_len == 1)"),
    "bwd_reset_at_fwd_start": ("(t % seg_len == seg_len - 1)", "(t % seg_len == 0)"),
    "gate_sign": ("return v / (1.0 + exp(-v));", "return v / (1.0 + exp(v));"),
    "bwd_uses_fwd_A": ("A_bwd + d * N", "A_fwd + d * N"),
    "state_not_reset_between_rows": ("for (long n = 0; n < N; ++n) h[n] = 0.0;", ""),
    "softplus_drops_log": ("log1p(exp(-fabs(v)))", "exp(-fabs(v))"),
    "softplus_wrong_branch": ("(v > 0.0 ? v : 0.0)", "(v > 0.0 ? 0.0 : v)"),
    "step_bias_not_added": ("softplus(raw[t] + bias)", "softplus(raw[t])"),
    "bwd_step_uses_fwd_bias": ("bias_bwd ? bias_bwd[d] : 0.0", "bias_fwd ? bias_fwd[d] : 0.0"),
    "bwd_uses_fwd_step": ("direction_step(delta_bwd + r * L", "direction_step(delta + r * L"),
    "conv_taps_reversed": ("t - (K - 1) + k;", "t - k;"),
    "conv_backward_is_causal": ("reverse ? t + (K - 1) - k", "reverse ? t - (K - 1) + k"),
    "conv_crosses_segments": ("if (seg_len > 0 && s / seg_len != t / seg_len) continue;", ""),
    "conv_without_silu": ("out[r * L + t] = silu(acc);", "out[r * L + t] = acc;"),
    "conv_bias_dropped": ("double acc = b ? b[d] : 0.0;", "double acc = 0.0;"),
    "bwd_reads_shared_input": ("scan_row_direction(x_bwd + r * L", "scan_row_direction(xr"),
    "grad_adjoint_not_carried": ("lam[n] = a * lam[n];", "lam[n] = 0.0;"),
    "grad_dB_without_step": ("dBk[t * N + n] += lam[n] * dtr[t] * xr[t];",
                             "dBk[t * N + n] += lam[n] * xr[t];"),
    "grad_ddelta_without_decay_term": ("+ Ak[n] * a * hp);", ");"),
    "grad_gate_derivative_sign": ("(1.0 + zt * (1.0 - sg))", "(1.0 - zt * (1.0 - sg))"),
    "grad_skip_dropped": ("double dxx = ds * Dk, ddt = 0.0;", "double dxx = 0.0, ddt = 0.0;"),
    "grad_dA_without_step": ("dAk[n] += lam[n] * a * hp * dtr[t];", "dAk[n] += lam[n] * a * hp;"),
    "grad_softplus_derivative_dropped": (
        "dst[k * L + t] * (use_softplus ? sigmoid(v[t] + bias) : 1.0)", "dst[k * L + t]"),
    "grad_softplus_derivative_without_bias": ("sigmoid(v[t] + bias) : 1.0", "sigmoid(v[t]) : 1.0"),
    "grad_bwd_bias_gradient_to_fwd": ("double *dbk = k && bias_bwd ? dbias_bwd : dbias_fwd;",
                                      "double *dbk = dbias_fwd;"),
    "grad_own_steps_swapped": ("double *dv = (k && delta_bwd ? ddelta_bwd : ddelta) + r * L;",
                               "double *dv = (delta_bwd ? ddelta_bwd : ddelta) + r * L;"),
    "grad_silu_derivative_is_sigmoid": ("return q + p * q * (1.0 - q);", "return q;"),
    "grad_conv_transpose_to_output_token": ("dx[r * L + sidx] += wk[d * K + j] * dp;",
                                            "dx[r * L + t] += wk[d * K + j] * dp;"),
    "grad_conv_taps_read_output_token": ("dwk[d * K + j] += dp * xraw[sidx];",
                                         "dwk[d * K + j] += dp * xraw[t];"),
    "grad_conv_bias_gradient_dropped": ("if (dcbk) dcbk[d] += dp;", ""),
    "grad_conv_recompute_without_bias": ("double a = cbk ? cbk[d] : 0.0;", "double a = 0.0;"),
    "ncssd_weight_dropped": ("h += mb[j] * Bb[j * N + n] * xb[d * L + j];",
                             "h += Bb[j * N + n] * xb[d * L + j];"),
    "ncssd_reads_C_for_B": ("h += mb[j] * Bb[j * N + n] * xb[d * L + j];",
                            "h += mb[j] * Cb[j * N + n] * xb[d * L + j];"),
    "ncssd_last_token_missed": ("for (long j = 0; j < L; ++j) h += mb[j]",
                                "for (long j = 0; j < L - 1; ++j) h += mb[j]"),
    "ncssd_skip_dropped": ("double y = D ? D[d] * xb[d * L + t] : 0.0;", "double y = 0.0;"),
    "ncssd_reads_state_of_next_channel": ("y += Cb[t * N + n] * H[n * dim + d];",
                                          "y += Cb[t * N + n] * H[n * dim + (d + 1) % dim];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name):
    old, new = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "vssm_oracle.c")).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    tmp = tempfile.mkdtemp(prefix="oracle_mutant_")
    try:
        path = os.path.join(tmp, "mutant.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        lib = oracle.load_library(oracle.compile_c(path, os.path.join(tmp, "libmutant.so")))
        assert P.failing_pins(lib), f"no pin caught the planted mistake {name}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


def test_thread_count_does_not_change_results(lib):
    inp = make_inputs(WORKLOADS["vim_ti_224"], seed=3)
    a = oracle.scan_inputs(inp, nthreads=1)
    b = oracle.scan_inputs(inp, nthreads=4)
    assert np.array_equal(a, b)


def test_rejects_bad_arguments(lib):
    x = np.zeros((1, 1, 6))
    A = -np.ones((1, 2))
    B = np.zeros((1, 6, 2))
    with pytest.raises(ValueError):   # backward folded needs L % seg_len == 0
        oracle.scan(x, x, A, A, B, B, dirs=3, seg_len=4)
    with pytest.raises(ValueError):
        oracle.scan(x, x, A, A, B, B, dirs=0)


def test_scan_rows_matches_full(lib):
    inp = make_inputs(WORKLOADS["vim_ti_224"].scaled(batch=2, dim=8, seqlen=19), seed=5)
    full = oracle.scan_inputs(inp)
    rows = [(0, 3), (1, 7), (1, 0)]
    sub = oracle.scan_rows(inp, rows)
    for i, (b, d) in enumerate(rows):
        assert np.array_equal(sub[i], full[b, d])
