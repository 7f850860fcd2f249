"""Parity at the full benchmark workloads, in the launch configuration the
benchmark times: every estimator on its seeded synthetic workload, every row
compared with the float64 oracle (the oracle is a per-row loop, fast enough
in C to check all of them)."""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrence_scan_gb300 import synthetic

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from linear_recurrence_scan_gb300 import build
    build.build()


def L():
    import linear_recurrence_scan_gb300 as lib
    return lib


def dev(a):
    return None if a is None else torch.from_numpy(a).to(DEV)


def assert_disc(gpu, ref, what):
    g = gpu.double().cpu().numpy()
    err = np.abs(g - ref)
    bound = 1e-4 + 1e-5 * np.abs(ref)
    bad = ~(err <= bound)
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} off, max err {err.max()}"


def test_gae_8x128():
    c = synthetic.WORKLOADS["gae_8x128"]
    b = synthetic.workload_batch("gae_8x128")
    ref = oracle.gae(b["rewards"], b["values"], b["terminateds"], b["truncateds"], c["gamma"],
                     c["lambda_"], b["bootstrap_values"])
    got = L().compute_gae(dev(b["rewards"]), dev(b["values"]), dev(b["terminateds"]),
                          dev(b["truncateds"]), c["gamma"], c["lambda_"], dev(b["bootstrap_values"]))
    assert_disc(got, ref, "gae 8x128")


def test_gae_returns_4096x1024():
    c = synthetic.WORKLOADS["gae_returns_4096x1024"]
    b = synthetic.workload_batch("gae_returns_4096x1024")
    g, l = c["gamma"], c["lambda_"]
    r, v, term, last, nv = (dev(b[k]) for k in ("rewards", "values", "terminateds", "last_value",
                                                "next_values"))
    assert_disc(L().compute_gae(r, v, term, None, g, l, None, last),
                oracle.gae(b["rewards"], b["values"], b["terminateds"], None, g, l, None,
                           b["last_value"]), "gae 4096x1024")
    assert_disc(L().compute_discounted_returns(r, term, None, g, None, last),
                oracle.discounted_returns(b["rewards"], b["terminateds"], None, g, None,
                                          b["last_value"]), "discounted returns 4096x1024")
    assert_disc(L().compute_lambda_returns(r, nv, term, None, g, l, None, last),
                oracle.lambda_returns(b["rewards"], b["next_values"], b["terminateds"], None, g,
                                      l, None, b["last_value"]), "lambda returns 4096x1024")


def test_fused_gae_returns_4096x1024():
    """The fused kernel on the same workload matches all three oracles."""
    c = synthetic.WORKLOADS["gae_returns_4096x1024"]
    b = synthetic.workload_batch("gae_returns_4096x1024")
    g, l = c["gamma"], c["lambda_"]
    adv, lam, disc = L().compute_gae_and_returns(dev(b["rewards"]), dev(b["values"]),
                                                 dev(b["terminateds"]), None, g, l, None,
                                                 dev(b["last_value"]))
    assert_disc(adv, oracle.gae(b["rewards"], b["values"], b["terminateds"], None, g, l, None,
                                b["last_value"]), "fused gae")
    assert_disc(lam, oracle.lambda_returns(b["rewards"], b["next_values"], b["terminateds"], None,
                                           g, l, None, b["last_value"]), "fused lambda returns")
    assert_disc(disc, oracle.discounted_returns(b["rewards"], b["terminateds"], None, g, None,
                                                b["last_value"]), "fused discounted")


def _vtrace(b, c):
    args = (c["gamma"], c["rho_bar"], c["c_bar"])
    ref = oracle.vtrace(b["log_pi_target"], b["log_pi_behavior"], b["values"], b["rewards"],
                        b["terminateds"], b["truncateds"], *args, b["bootstrap_values"],
                        b["last_value"])
    got = L().compute_vtrace(dev(b["log_pi_target"]), dev(b["log_pi_behavior"]), dev(b["values"]),
                             dev(b["rewards"]), dev(b["terminateds"]), dev(b["truncateds"]), *args,
                             dev(b["bootstrap_values"]), dev(b["last_value"]))
    assert_disc(got[0], ref[0], "vtrace targets")
    assert_disc(got[1], ref[1], "vtrace advantages")


def _retrace(b, c):
    args = (c["gamma"], c["lambda_"], c["c_bar"], c["rho_bar"])
    keys = ("pi_taken", "mu_taken", "q_values", "expected_next_q", "rewards", "terminateds",
            "truncateds")
    ref = oracle.retrace(*(b[k] for k in keys), *args)
    got = L().compute_retrace_from_probs(*(dev(b[k]) for k in keys), *args)
    assert_disc(got[0], ref[0], "retrace targets")
    assert_disc(got[1], ref[1], "retrace advantages")


def test_vtrace_2048x4096():
    _vtrace(synthetic.workload_batch("vtrace_2048x4096"), synthetic.WORKLOADS["vtrace_2048x4096"])


def test_retrace_1024x16384():
    _retrace(synthetic.workload_batch("retrace_1024x16384"), synthetic.WORKLOADS["retrace_1024x16384"])


def test_long_rows_64x1m():
    c = synthetic.WORKLOADS["long_rows_64x1048576"]
    b = synthetic.workload_batch("long_rows_64x1048576")
    ref = oracle.episodic_prefix_sum(b["inputs"], b["prefix_dones"], None, "starts_at")
    got = L().compute_episodic_prefix_sum(dev(b["inputs"]), dev(b["prefix_dones"]), None,
                                          "starts_at")
    np.testing.assert_array_equal(got.double().cpu().numpy(), ref)
    ref = oracle.eligibility_traces(b["gradients"], b["trace_dones"], c["gamma"], c["lambda_"])
    got = L().compute_eligibility_traces(dev(b["gradients"]), dev(b["trace_dones"]), c["gamma"],
                                         c["lambda_"])
    assert_disc(got, ref, "eligibility traces 64x1M")


@pytest.mark.parametrize("kind", ["gae", "vtrace", "retrace"])
def test_million_step_rows(kind):
    """GAE / V-trace / Retrace on 64 rows of 2^20 steps with the distributions
    of their own workloads (the long-row regime of the throughput target)."""
    N, T = 64, 1 << 20
    if kind == "gae":
        c = synthetic.WORKLOADS["gae_returns_4096x1024"]
        b = synthetic.gae_batch(N, T, 0, 41, c["p_term"], 0.0, "last")
        ref = oracle.gae(b["rewards"], b["values"], b["terminateds"], None, c["gamma"],
                         c["lambda_"], None, b["last_value"])
        got = L().compute_gae(dev(b["rewards"]), dev(b["values"]), dev(b["terminateds"]), None,
                              c["gamma"], c["lambda_"], None, dev(b["last_value"]))
        assert_disc(got, ref, "gae 64x1M")
    elif kind == "vtrace":
        c = synthetic.WORKLOADS["vtrace_2048x4096"]
        _vtrace(synthetic.vtrace_batch(N, T, 0, 42, c["p_term"], c["p_trunc"], "2d"), c)
    else:
        c = synthetic.WORKLOADS["retrace_1024x16384"]
        _retrace(synthetic.retrace_batch(N, T, 0, 43, c["p_term"], 0.0), c)
