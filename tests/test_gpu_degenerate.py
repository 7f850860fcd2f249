"""Degenerate parameters and flags of the method, on the device against the
float64 oracle: no discount (gamma = 0), one-step TD errors (lambda = 0), no
decay at all (gamma = lambda = 1: every tile's aggregate keeps beta = 1, so
each row is one long carry chain through the look-back), every step
terminated or truncated, and importance ratios at or beyond their clips
(V-trace log-ratios of +-50 and +-100, Retrace target probabilities of 0).

Tolerances: |gpu - ref| <= 1e-4 + 1e-5 |ref| for decaying recurrences.
With gamma = lambda = 1 and no flags every beta is 1: the recurrence is a
running sum within the episode, so it takes the prefix-sum bound
|gpu - ref| <= 1e-6 * S_t, with S_t the sum of |alpha| over the steps the
output at t accumulates, where each alpha counts every term that enters it
(GAE: |r_t| + |V_{t+1}| + |V_t|; a float32 sum is exact only to the rounding
of its addends, so a TD error that cancels to near zero still carries the
rounding of r and V); lambda-returns add |V_t| for their final A + V.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"

# packed rows, one look-back chain of three tiles, a long chain
SHAPES = [(8, 128), (4, 3000), (2, 20000)]
IDS = [f"{n}x{t}" for n, t in SHAPES]


@pytest.fixture(scope="module", autouse=True)
def built():
    from linear_recurrence_scan_gb300 import build
    build.build()


def L():
    import linear_recurrence_scan_gb300 as lib
    return lib


def dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def close(got, ref, what):
    g = got.double().cpu().numpy()
    err = np.abs(g - ref)
    bad = ~(err <= 1e-4 + 1e-5 * np.abs(ref))
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} off, first {i}: gpu {g[i]!r} ref {ref[i]!r}")


def close_chain(got, ref, terms, what, backward=True, extra=None):
    """beta = 1 chains: |gpu - ref| <= 1e-6 x the running sum (in scan order)
    of the magnitudes of every term that enters each alpha (`terms`: arrays
    summed element-wise), plus `extra` (|.| added at each step, not carried)."""
    a = sum(np.abs(np.asarray(t, dtype=np.float64)) for t in terms)
    S = np.flip(np.cumsum(np.flip(a, 1), 1), 1) if backward else np.cumsum(a, 1)
    if extra is not None:
        S = S + np.abs(np.asarray(extra, dtype=np.float64))
    g = got.double().cpu().numpy()
    err = np.abs(g - ref)
    bad = ~(err <= 1e-6 * S)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} off, first {i}: gpu {g[i]!r} ref {ref[i]!r} "
                             f"(S {S[i]!r})")


def batch(N, T, seed):
    rng = np.random.default_rng(seed)
    r = rng.standard_normal((N, T)).astype(np.float32)
    v = rng.standard_normal((N, T)).astype(np.float32)
    last = rng.standard_normal(N).astype(np.float32)
    return rng, r, v, last


@pytest.mark.parametrize("shape", SHAPES, ids=IDS)
@pytest.mark.parametrize("gl", [(0.0, 0.95), (0.99, 0.0), (0.0, 0.0)], ids=["gamma0", "lambda0", "both0"])
def test_gae_without_discount_or_trace(shape, gl):
    """gamma = 0 or lambda = 0: each advantage is the one-step TD error."""
    N, T = shape
    g, lam = gl
    rng, r, v, last = batch(N, T, 300 + T)
    term = (rng.random((N, T)) < 0.02).astype(np.float32)
    ref = oracle.gae(r, v, term, None, g, lam, None, last)
    close(L().compute_gae(dev(r), dev(v), dev(term), None, g, lam, None, dev(last)), ref, f"gae gamma {g} lambda {lam}")
    # beta = gamma lambda (1 - done) is 0 everywhere: the TD error itself
    np.testing.assert_array_equal(ref, oracle.gae(r, v, term, None, g, 0.0, None, last))


@pytest.mark.parametrize("shape", SHAPES, ids=IDS)
def test_no_decay_chains(shape):
    """gamma = lambda = 1 and no flags: GAE, TD(lambda), discounted returns and
    eligibility traces are plain running sums, carried across every tile."""
    N, T = shape
    rng, r, v, last = batch(N, T, 400 + T)
    zero = np.zeros((N, T), np.float32)
    adv, lret, disc = L().compute_gae_and_returns(dev(r), dev(v), dev(zero), None, 1.0, 1.0, None, dev(last))
    ref = oracle.gae(r, v, zero, None, 1.0, 1.0, None, last)
    # alpha_t = r_t + V_{t+1} - V_t (V_T = last_value)
    v_next = np.concatenate([v[:, 1:], last[:, None]], 1)
    close_chain(adv, ref, [r, v_next, v], "gae gamma = lambda = 1")
    close_chain(lret, ref + v.astype(np.float64), [r, v_next, v], "lambda returns gamma = lambda = 1",
                extra=v)
    # alpha_t = r_t, the window bootstrap enters at the last step
    carry = np.zeros((N, T), np.float64)
    carry[:, -1] = last
    close_chain(disc, oracle.discounted_returns(r, zero, None, 1.0, None, last), [r, carry],
                "discounted gamma = 1")
    z = L().compute_eligibility_traces(dev(r), dev(zero), 1.0, 1.0)
    close_chain(z, oracle.eligibility_traces(r, zero, 1.0, 1.0), [r], "eligibility gamma lambda = 1",
                backward=False)


@pytest.mark.parametrize("shape", SHAPES, ids=IDS)
@pytest.mark.parametrize("flag", ["terminated", "truncated"])
def test_every_step_flagged(shape, flag):
    """Every step terminated (or truncated, with a bootstrap value at every
    step): no recurrence survives a step."""
    N, T = shape
    rng, r, v, last = batch(N, T, 500 + T)
    ones, zero = np.ones((N, T), np.float32), np.zeros((N, T), np.float32)
    term, trunc = (ones, zero) if flag == "terminated" else (zero, ones)
    # bootstrap values where the contract reads them: truncated steps, and
    # the window end of a row that is not terminated there
    keep = trunc > 0
    keep[:, -1] |= term[:, -1] == 0
    bs = np.where(keep, rng.standard_normal((N, T)), 0.0).astype(np.float32)
    close(L().compute_gae(dev(r), dev(v), dev(term), dev(trunc), 0.99, 0.95, dev(bs)),
          oracle.gae(r, v, term, trunc, 0.99, 0.95, bs), f"gae, every step {flag}")
    close(L().compute_discounted_returns(dev(r), dev(term), dev(trunc), 0.99, dev(bs)),
          oracle.discounted_returns(r, term, trunc, 0.99, bs), f"discounted, every step {flag}")
    lpb = rng.standard_normal((N, T)).astype(np.float32)
    lpt = (lpb + 0.5 * rng.standard_normal((N, T))).astype(np.float32)
    vs, adv = L().compute_vtrace(dev(lpt), dev(lpb), dev(v), dev(r), dev(term), dev(trunc), 0.99, 1.0, 1.0, dev(bs))
    vs_ref, adv_ref = oracle.vtrace(lpt, lpb, v, r, term, trunc, 0.99, 1.0, 1.0, bs)
    close(vs, vs_ref, f"vtrace targets, every step {flag}")
    close(adv, adv_ref, f"vtrace advantages, every step {flag}")
    z = L().compute_eligibility_traces(dev(r), dev(ones), 0.99, 0.9)
    close(z, oracle.eligibility_traces(r, ones, 0.99, 0.9), "eligibility traces, every step done")


@pytest.mark.parametrize("shape", SHAPES, ids=IDS)
def test_ratios_at_and_beyond_their_clips(shape):
    """V-trace log-ratios of +-50 and +-100 (exp overflows to inf or underflows
    to 0 in float, and the clips take over) and Retrace target probabilities
    of 0 (the trace is cut) or ten times the behaviour probability."""
    N, T = shape
    rng, r, v, last = batch(N, T, 600 + T)
    term = (rng.random((N, T)) < 0.01).astype(np.float32)
    lpb = rng.standard_normal((N, T)).astype(np.float32)
    shift = rng.choice(np.array([-100.0, -50.0, 0.0, 50.0, 100.0], np.float32), (N, T))
    lpt = (lpb + shift).astype(np.float32)
    vs, adv = L().compute_vtrace(dev(lpt), dev(lpb), dev(v), dev(r), dev(term), None, 0.99, 1.0, 1.0, None,
                                 dev(last))
    vs_ref, adv_ref = oracle.vtrace(lpt, lpb, v, r, term, None, 0.99, 1.0, 1.0, None, last)
    close(vs, vs_ref, "vtrace targets, clipped ratios")
    close(adv, adv_ref, "vtrace advantages, clipped ratios")
    mu = rng.uniform(0.05, 1.0, (N, T)).astype(np.float32)
    pi = (mu * rng.choice(np.array([0.0, 1.0, 10.0], np.float32), (N, T))).astype(np.float32)
    q = rng.standard_normal((N, T)).astype(np.float32)
    eq = rng.standard_normal((N, T)).astype(np.float32)
    qret, radv = L().compute_retrace_from_probs(dev(pi), dev(mu), dev(q), dev(eq), dev(r), dev(term), None, 0.99,
                                                0.95, 1.0, 1.0)
    qret_ref, radv_ref = oracle.retrace(pi, mu, q, eq, r, term, None, 0.99, 0.95, 1.0, 1.0)
    close(qret, qret_ref, "retrace targets, cut and clipped traces")
    close(radv, radv_ref, "retrace advantages, cut and clipped traces")
