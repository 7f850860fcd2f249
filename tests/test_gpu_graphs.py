"""Calls captured into a CUDA graph and replayed with new inputs in the same
buffers.  Look-back tile states carry an epoch kept in the workspace header
and advanced by each launch, so a replay never mistakes the states of the
previous replay for its own.  Every replay is compared with the oracle."""
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


def close(got, ref, what):
    g = got.double().cpu().numpy()
    err = np.abs(g - ref)
    assert (err <= 1e-4 + 1e-5 * np.abs(ref)).all(), f"{what}: max err {err.max()}"


def test_graph_replays_with_new_inputs():
    N, T = 16, 20000   # rows of several tiles: look-back on every call
    b0 = synthetic.gae_batch(N, T, 0, 95, 0.01, 0.0, "last")
    r, v, term, last = (torch.from_numpy(b0[k]).to(DEV) for k in
                        ("rewards", "values", "terminateds", "last_value"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):   # warm-up on the capture's side stream (allocations, workspace)
        for _ in range(2):
            L().compute_gae(r, v, term, None, 0.99, 0.95, None, last)
            L().compute_gae_and_returns(r, v, term, None, 0.99, 0.95, None, last)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        adv = L().compute_gae(r, v, term, None, 0.99, 0.95, None, last)
        adv2, lam, disc = L().compute_gae_and_returns(r, v, term, None, 0.99, 0.95, None, last)
    for seed in (1, 2, 3, 1):
        b = synthetic.gae_batch(N, T, seed, 95, 0.01, 0.0, "last")
        for dst, k in ((r, "rewards"), (v, "values"), (term, "terminateds"), (last, "last_value")):
            dst.copy_(torch.from_numpy(b[k]))
        graph.replay()
        torch.cuda.synchronize()
        ref = oracle.gae(b["rewards"], b["values"], b["terminateds"], None, 0.99, 0.95, None,
                         b["last_value"])
        close(adv, ref, f"graph gae (seed {seed})")
        close(adv2, ref, f"graph fused gae (seed {seed})")
        close(disc, oracle.discounted_returns(b["rewards"], b["terminateds"], None, 0.99, None,
                                              b["last_value"]), f"graph discounted (seed {seed})")


def test_graph_replays_other_kernels():
    """Replays of the normalising path (scan with moment slots, then the
    normalising pass), masked GAE and the [N,T,A] Retrace front end."""
    N, T = 64, 3000
    def batches(seed):
        return (synthetic.gae_batch(N, T, seed, 96, 0.01, 0.0, "last"),
                synthetic.llm_tokens_batch(N, T, seed),
                synthetic.retrace_actions_batch(N, T, 4, seed, 97))
    b0 = batches(0)
    gkeys = ("rewards", "values", "terminateds", "last_value")
    mkeys = ("rewards", "values", "terminateds", "mask")
    rkeys = ("action_probs_target", "action_probs_behavior", "q_values", "next_q_values_all", "actions",
             "rewards", "terminateds")
    g = {k: torch.from_numpy(b0[0][k]).to(DEV) for k in gkeys}
    m = {k: torch.from_numpy(b0[1][k]).to(DEV) for k in mkeys}
    r = {k: torch.from_numpy(b0[2][k]).to(DEV) for k in rkeys}

    def calls():
        norm = L().compute_gae_normalized(g["rewards"], g["values"], g["terminateds"], None, 0.99, 0.95, None,
                                          g["last_value"], return_moments=True)
        masked = L().compute_gae(m["rewards"], m["values"], m["terminateds"], None, 1.0, 0.95, mask=m["mask"])
        ret = L().compute_retrace(*(r[k] for k in rkeys), None, 0.99, 0.95)
        return norm, masked, ret

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            calls()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        norm, masked, ret = calls()
    for seed in (1, 2, 1):
        b = batches(seed)
        for dst, src, keys in ((g, b[0], gkeys), (m, b[1], mkeys), (r, b[2], rkeys)):
            for k in keys:
                dst[k].copy_(torch.from_numpy(src[k]))
        graph.replay()
        torch.cuda.synchronize()
        bg, bm, br = b
        raw = oracle.gae(bg["rewards"], bg["values"], bg["terminateds"], None, 0.99, 0.95, None, bg["last_value"])
        want, (mean, sd) = oracle.normalize_advantages(raw, 1e-8)
        close(norm[0], want, f"graph normalized advantages (seed {seed})")
        mom = norm[-1].double().cpu().numpy()
        assert abs(mom[0] - mean) <= 1e-6 + 1e-5 * abs(mean) and abs(mom[1] - sd) <= 1e-5 * sd
        close(masked, oracle.gae_masked(bm["rewards"], bm["values"], bm["terminateds"], bm["mask"], None, 1.0,
                                        0.95), f"graph masked gae (seed {seed})")
        qret, adv = oracle.retrace_actions(*(br[k] for k in rkeys), None, 0.99, 0.95)
        close(ret[0], qret, f"graph retrace targets (seed {seed})")
        close(ret[1], adv, f"graph retrace advantages (seed {seed})")
