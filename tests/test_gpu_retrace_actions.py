"""Retrace from the full action-space inputs (compute_retrace with [N,T,A]
target probabilities and successor Q-values and int64 actions): the CUDA
path against the float64 oracle, element by element.

Cases cover packed tiles, one tile, rows split into many tiles (look-back,
with the step after each tile derived from the staged wide rows), ragged
tails, T not a multiple of 4 (element-wise staging, wide rows read from
global memory), widths that do not fit the staging ring (A = 12, 33), strided
float rows, [N,T,A] rows inside a longer buffer, with and without truncation
flags.  Tolerance: |gpu - ref| <= 1e-4 + 1e-5 |ref| per element.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from linear_recurrence_scan_gb300 import synthetic

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from linear_recurrence_scan_gb300 import build
    build.build()


def L():
    import linear_recurrence_scan_gb300 as lib
    return lib


def assert_disc(gpu, ref, what):
    g = gpu.double().cpu().numpy()
    assert g.shape == ref.shape, what
    err = np.abs(g - ref)
    bad = ~(err <= 1e-4 + 1e-5 * np.abs(ref))
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} off, first {i}: "
                             f"gpu {g[i]!r} ref {ref[i]!r}")


def batch(N, T, A, seed, p_trunc):
    b = synthetic.retrace_actions_batch(N, T, A, seed, 3, p_term=0.02, p_trunc=p_trunc)
    return b


def run_both(b, params, rs=None, wide_pad=0):
    """Oracle and CUDA results on one batch.  rs: row stride of the float
    [N,T] arrays (and actions); wide_pad: extra steps of room after each
    [N,T,A] row."""
    keys2 = ("action_probs_behavior", "q_values", "rewards", "terminateds", "truncateds")
    N, T, A = b["action_probs_target"].shape

    def dev2(a, dtype=None):
        if a is None:
            return None
        t = torch.from_numpy(np.ascontiguousarray(a))
        if rs is not None and rs != T:
            big = torch.zeros((N, rs), dtype=t.dtype)
            big[:, :T] = t
            return big.to(DEV)[:, :T]
        return t.to(DEV)

    def dev3(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if wide_pad:
            big = torch.full((N, T + wide_pad, A), float("nan"), dtype=torch.float32)
            big[:, :T] = t
            return big.to(DEV)[:, :T]
        return t.to(DEV)

    ref = oracle.retrace_actions(b["action_probs_target"], b["action_probs_behavior"],
                                 b["q_values"], b["next_q_values_all"], b["actions"],
                                 b["rewards"], b["terminateds"], b["truncateds"], *params)
    got = L().compute_retrace(dev3(b["action_probs_target"]), dev2(b["action_probs_behavior"]),
                              dev2(b["q_values"]), dev3(b["next_q_values_all"]),
                              dev2(b["actions"]), dev2(b["rewards"]), dev2(b["terminateds"]),
                              dev2(b["truncateds"]), *params)
    return ref, got


PARAMS = (0.97, 0.9, 1.0, 1.0)

# (N, T, A, row_stride or None, wide_pad)
CASES = [
    (8, 128, 4, None, 0),     # packed, staged
    (5, 37, 4, None, 0),      # T % 4 != 0: element-wise, wide rows from global memory
    (3, 1, 4, None, 0),
    (4, 2, 3, None, 0),
    (6, 1024, 4, None, 0),    # exactly one tile per row
    (3, 3000, 4, None, 0),    # look-back, ragged last tile
    (3, 2999, 4, None, 0),    # look-back, element-wise
    (2, 40000, 4, None, 0),   # many tiles per row
    (4, 5000, 1, None, 0),    # a single action
    (4, 5000, 2, None, 0),
    (4, 5000, 5, None, 0),    # odd width, still staged
    (4, 5000, 9, None, 0),    # widest staged width
    (3, 5000, 12, None, 0),   # too wide for the ring: wide rows from global memory
    (3, 700, 33, None, 0),
    (5, 100, 4, 104, 0),      # strided float rows, staged
    (5, 100, 4, 103, 0),      # strided float rows, element-wise
    (4, 3000, 4, None, 8),    # [N,T,A] rows inside a longer buffer (row stride (T+8) A)
    (4, 3000, 3, None, 3),    # same, row stride not a multiple of 4 words: from global
]
IDS = [f"{n}x{t}xA{a}" + (f"_rs{rs}" if rs else "") + (f"_pad{p}" if p else "")
       for n, t, a, rs, p in CASES]


@pytest.mark.parametrize("trunc", [0.0, 0.02], ids=["noflags", "trunc"])
@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_retrace_actions_parity(case, trunc):
    N, T, A, rs, pad = case
    b = batch(N, T, A, 101 + T + A, trunc)
    ref, got = run_both(b, PARAMS, rs, pad)
    assert_disc(got[0], ref[0], "retrace targets")
    assert_disc(got[1], ref[1], "retrace advantages")


def test_clips_and_lambda():
    """c_bar, rho_bar below the ratios and lambda < 1 on a look-back shape."""
    b = batch(3, 6000, 4, 7, 0.01)
    ref, got = run_both(b, (0.99, 0.8, 0.7, 0.6))
    assert_disc(got[0], ref[0], "targets")
    assert_disc(got[1], ref[1], "advantages")


def test_agrees_with_reduced_entry_point():
    """The in-kernel reduction gives what the per-step entry point gives on
    the reduced inputs, up to the rounding of E_pi[Q'] (summed in float32 in
    the kernel)."""
    b = batch(4, 4096, 4, 8, 0.0)
    probs = torch.from_numpy(b["action_probs_target"]).to(DEV)
    nq = torch.from_numpy(b["next_q_values_all"]).to(DEV)
    acts = torch.from_numpy(b["actions"]).to(DEV)
    d = {k: torch.from_numpy(b[k]).to(DEV) for k in ("action_probs_behavior", "q_values",
                                                     "rewards", "terminateds")}
    full = L().compute_retrace(probs, d["action_probs_behavior"], d["q_values"], nq, acts,
                               d["rewards"], d["terminateds"], None, *PARAMS)
    pi = probs.gather(-1, acts.unsqueeze(-1)).squeeze(-1).contiguous()
    eq = (probs.double() * nq.double()).sum(-1).float()
    red = L().compute_retrace_from_probs(pi, d["action_probs_behavior"], d["q_values"], eq,
                                         d["rewards"], d["terminateds"], None, *PARAMS)
    for x, y in zip(full, red):
        torch.testing.assert_close(x, y, rtol=1e-5, atol=1e-4)


def test_invalid_action_poisons_only_its_row():
    """An action outside [0, A) makes pi NaN: that row's advantage at the step
    and every target before it (in the row) are NaN; other rows are exact."""
    N, T, A = 3, 3000, 4
    b = batch(N, T, A, 9, 0.0)
    ref = oracle.retrace_actions(b["action_probs_target"], b["action_probs_behavior"],
                                 b["q_values"], b["next_q_values_all"], b["actions"],
                                 b["rewards"], b["terminateds"], None, *PARAMS)
    acts = b["actions"].copy()
    acts[1, 2000] = A
    got = L().compute_retrace(*(torch.from_numpy(x).to(DEV) for x in (
        b["action_probs_target"], b["action_probs_behavior"], b["q_values"],
        b["next_q_values_all"], acts, b["rewards"], b["terminateds"])), None, *PARAMS)
    qret, adv = (x.double().cpu().numpy() for x in got)
    assert np.isnan(adv[1, 2000])
    assert np.isnan(qret[1, :2000]).all()
    for r in (0, 2):
        np.testing.assert_allclose(qret[r], ref[0][r], rtol=1e-5, atol=1e-4)
        np.testing.assert_allclose(adv[r], ref[1][r], rtol=1e-5, atol=1e-4)


def test_full_size_1024x16384_a4():
    """The benchmark workload (1024 x 16384, A = 4), every element."""
    b = synthetic.retrace_actions_batch(1024, 16384, 4)
    c = synthetic.WORKLOADS["retrace_1024x16384"]
    params = (c["gamma"], c["lambda_"], c["c_bar"], c["rho_bar"])
    ref, got = run_both(b, params)
    assert_disc(got[0], ref[0], "targets 1024x16384")
    assert_disc(got[1], ref[1], "advantages 1024x16384")


CHECKS_CHILD = r"""
import json, sys
import torch
sys.path.insert(0, ROOT)
import linear_recurrence_scan_gb300 as L
from linear_recurrence_scan_gb300 import _native
N, T, A = 2, 64, 4
p = torch.full((N, T, A), 0.25, device="cuda")
z = torch.zeros(N, T, device="cuda")
one = torch.ones(N, T, device="cuda")
acts = torch.zeros(N, T, dtype=torch.int64, device="cuda")
def status(a):
    try:
        L.compute_retrace(p, one, z, p, a, z, z); torch.cuda.synchronize(); return "OK"
    except _native.RlscanError as e:
        return e.name
bad = acts.clone(); bad[1, 7] = -1
big = acts.clone(); big[0, 3] = A
print(json.dumps(dict(ok=status(acts), negative=status(bad), too_big=status(big))))
"""


def test_opt_in_action_range_check():
    env = dict(os.environ)
    env["RLSCAN_CHECKS"] = "1"
    r = subprocess.run([sys.executable, "-c", "ROOT = %r\n" % ROOT + CHECKS_CHILD], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res == dict(ok="OK", negative="RLSCAN_ERR_INVALID_INPUT",
                       too_big="RLSCAN_ERR_INVALID_INPUT"), res
