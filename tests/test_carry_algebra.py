"""The algebra behind the carry join of token ranges (Vim page §3.1, parallel
scan), checked in fp64 on the CPU, independently of the oracle and the CUDA
path.

A range of the recurrence h_t = a_t * h_{t-1} + v_t (per state, a_t =
exp(delta_t * A)) maps an incoming state h to P * h + h_p, where
P = prod(a_t) over the range and h_p is the range's state from zero. These
maps compose associatively, (P1, h1) then (P2, h2) = (P1 * P2, P2 * h1 + h2);
the exclusive prefix of the ranges before a range, applied to h = 0, is the
state entering it. P also equals exp(A * sum(delta)) over the range, which
is what the summary pass stores; a forced-zero decay inside a range (folded
reset) makes P = 0 and cuts the carry.
"""
import numpy as np


def combine(m1, m2):
    P1, h1 = m1
    P2, h2 = m2
    return P1 * P2, P2 * h1 + h2


def recurrence(a, v, h0=0.0):
    h = np.full(a.shape[1:], h0, dtype=np.float64)
    out = []
    for t in range(a.shape[0]):
        h = a[t] * h + v[t]
        out.append(h.copy())
    return np.array(out)


def summary(a, v):
    return np.prod(a, axis=0), recurrence(a, v)[-1]


def test_combine_is_associative():
    rng = np.random.default_rng(0)
    for _ in range(200):
        ms = [(rng.uniform(0, 1, 16), rng.standard_normal(16)) for _ in range(3)]
        left = combine(combine(ms[0], ms[1]), ms[2])
        right = combine(ms[0], combine(ms[1], ms[2]))
        assert np.allclose(left[0], right[0], rtol=1e-14, atol=0)
        assert np.allclose(left[1], right[1], rtol=1e-13, atol=1e-15)


def test_folded_summaries_give_the_states_at_range_starts():
    rng = np.random.default_rng(1)
    L, N = 97, 16
    A = -np.exp(rng.uniform(np.log(0.5), np.log(16), N))
    delta = np.log1p(np.exp(rng.normal(-2, 0.5, L)))
    a = np.exp(delta[:, None] * A[None, :])
    v = rng.standard_normal((L, N))
    full = recurrence(a, v)
    cuts = [0, 13, 14, 40, 41, 77, L]                 # ranges of length 13, 1, 26, 1, 36, 20
    summ = [summary(a[s:e], v[s:e]) for s, e in zip(cuts[:-1], cuts[1:])]
    for k in range(1, len(cuts) - 1):
        state = (np.ones(N), np.zeros(N))
        for m in summ[:k]:
            state = combine(state, m)
        assert np.allclose(state[1], full[cuts[k] - 1], rtol=1e-12, atol=1e-14)
        # the range started from this state reproduces the full recurrence
        part = recurrence(a[cuts[k]:cuts[k + 1]], v[cuts[k]:cuts[k + 1]], 0.0)
        carried = part + np.cumprod(a[cuts[k]:cuts[k + 1]], axis=0) * state[1]
        assert np.allclose(carried, full[cuts[k]:cuts[k + 1]], rtol=1e-12, atol=1e-14)


def test_decay_product_is_exp_of_summed_step():
    rng = np.random.default_rng(2)
    A = -np.exp(rng.uniform(np.log(0.5), np.log(16), 16))
    delta = np.log1p(np.exp(rng.normal(-3, 0.5, 50)))
    prod = np.prod(np.exp(delta[:, None] * A[None, :]), axis=0)
    assert np.allclose(prod, np.exp(A * delta.sum()), rtol=1e-12)


def test_reset_inside_a_range_cuts_the_carry():
    rng = np.random.default_rng(3)
    a = rng.uniform(0.2, 1.0, (10, 4))
    v = rng.standard_normal((10, 4))
    a[6] = 0.0                                        # forced-zero decay at a segment start
    P, hp = summary(a, v)
    assert np.all(P == 0.0)
    # the state after the range does not depend on the incoming state
    h = rng.standard_normal(4)
    for t in range(10):
        h = a[t] * h + v[t]
    assert np.allclose(h, hp)
