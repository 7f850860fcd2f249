"""A fixed set of seeded calls through every kernel family, for the bounds
test (test_gpu_bounds.py): packed tiles, ragged and unaligned rows
(element-wise staging), strided rows, look-back chains, deferred finishing,
wide [N,T,A] inputs, compact storage, masking, normalisation and the forward
scans.  ``run_all()`` returns every output as a numpy array; run as a script
it saves them to the .npz named on the command line and prints the library's
bounds-check report (used with RLSCAN_LIB pointing at the checked build).
"""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from linear_recurrence_scan_gb300 import synthetic  # noqa: E402

DEV = "cuda:0"
# (N, T, row stride or None)
SHAPES = [(8, 128, None), (5, 37, None), (4, 3000, None), (3, 2999, None), (2, 40000, None),
          (5, 100, 104), (5, 100, 103), (6, 1024, None)]


def _dev(a, rs=None, dtype=None):
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    if rs is not None and t.dim() == 2 and rs != t.shape[1]:
        big = torch.zeros((t.shape[0], rs), dtype=t.dtype)
        big[:, : t.shape[1]] = t
        return big.to(DEV)[:, : t.shape[1]]
    return t.to(DEV)


def run_all():
    import linear_recurrence_scan_gb300 as L
    out = {}

    def keep(name, *ts):
        for i, t in enumerate(ts):
            out[f"{name}.{i}"] = t.detach().float().cpu().numpy()

    for (N, T, rs) in SHAPES:
        tag = f"{N}x{T}" + (f"_rs{rs}" if rs else "")
        d = lambda a, dt=None: _dev(a, rs, dt)  # noqa: E731
        b = synthetic.gae_batch(N, T, 1, 61, 0.01, 0.01, "2d")
        keep(f"gae_trunc_bs.{tag}", L.compute_gae(d(b["rewards"]), d(b["values"]), d(b["terminateds"]),
                                                  d(b["truncateds"]), 0.99, 0.95, d(b["bootstrap_values"])))
        b = synthetic.gae_batch(N, T, 1, 62, 0.01, 0.0, "last")
        last = _dev(b["last_value"])
        keep(f"fused.{tag}", *L.compute_gae_and_returns(d(b["rewards"]), d(b["values"]), d(b["terminateds"]),
                                                        None, 0.99, 0.95, None, last))
        keep(f"normalized.{tag}", *L.compute_gae_normalized(d(b["rewards"]), d(b["values"]), d(b["terminateds"]),
                                                            None, 0.99, 0.95, None, last, return_moments=True))
        keep(f"gae_compact.{tag}", L.compute_gae(d(b["rewards"], torch.bfloat16), d(b["values"], torch.bfloat16),
                                                 d(b["terminateds"], torch.uint8), None, 0.99, 0.95, None, last,
                                                 out_dtype=torch.bfloat16))
        v = synthetic.vtrace_batch(N, T, 1, 63, 0.01, 0.01, "2d")
        keep(f"vtrace.{tag}", *L.compute_vtrace(d(v["log_pi_target"]), d(v["log_pi_behavior"]), d(v["values"]),
                                                d(v["rewards"]), d(v["terminateds"]), d(v["truncateds"]), 0.99,
                                                1.0, 1.0, d(v["bootstrap_values"])))
        bf = lambda k: d(v[k], torch.bfloat16)  # noqa: E731
        keep(f"vtrace_compact.{tag}", *L.compute_vtrace(bf("log_pi_target"), bf("log_pi_behavior"), bf("values"),
                                                        bf("rewards"), d(v["terminateds"], torch.uint8),
                                                        d(v["truncateds"], torch.uint8), 0.99, 1.0, 1.0,
                                                        bf("bootstrap_values")))
        r = synthetic.retrace_batch(N, T, 1, 64, 0.01, 0.01)
        keys = ("pi_taken", "mu_taken", "q_values", "expected_next_q", "rewards")
        keep(f"retrace.{tag}", *L.compute_retrace_from_probs(*(d(r[k]) for k in keys), d(r["terminateds"]),
                                                             d(r["truncateds"]), 0.99, 0.95))
        keep(f"retrace_compact.{tag}", *L.compute_retrace_from_probs(
            *(d(r[k], torch.bfloat16) for k in keys), d(r["terminateds"], torch.uint8),
            d(r["truncateds"], torch.uint8), 0.99, 0.95))
        m = synthetic.llm_tokens_batch(N, T, 1)
        keep(f"masked.{tag}", L.compute_gae(d(m["rewards"]), d(m["values"]), d(m["terminateds"]), None, 1.0, 0.95,
                                            mask=d(m["mask"])))
        lr = synthetic.long_rows_batch(N, T, 1)
        keep(f"elig.{tag}", L.compute_eligibility_traces(d(lr["gradients"]), d(lr["trace_dones"]), 0.99, 0.9))
        keep(f"prefix.{tag}", L.compute_episodic_prefix_sum(d(lr["inputs"]), d(lr["prefix_dones"]), None,
                                                            "starts_at"))
        if rs is None:  # the [N,T,A] arrays have their own strides
            a = synthetic.retrace_actions_batch(N, T, 4, 1, 65)
            akeys = ("action_probs_target", "action_probs_behavior", "q_values", "next_q_values_all", "actions",
                     "rewards", "terminateds")
            keep(f"retrace_actions.{tag}", *L.compute_retrace(*(_dev(a[k]) for k in akeys), None, 0.99, 0.95))
    torch.cuda.synchronize()
    L.workspace_status()
    return out


if __name__ == "__main__":
    from linear_recurrence_scan_gb300 import _native
    res = run_all()
    np.savez(sys.argv[1], **res)
    import ctypes
    viol, site = ctypes.c_ulonglong(0), ctypes.c_ulonglong(0)
    kind = _native.lib().rlscan_bounds_check(ctypes.addressof(viol), ctypes.addressof(site), 0)
    print(f"BOUNDS kind={kind} violations={viol.value} first_site={site.value}", flush=True)
