"""Throughput benchmark: env-steps/s and achieved HBM GB/s per estimator.

Default run (N=1): the headline workload is the largest single-GPU
configuration, eligibility traces + episodic prefix sums on 64 rows of 2^20
float32 steps (one "step" = both estimators over one batch); every other
named workload is measured in the same run with the same protocol and
reported under "workloads" (GAE + discounted returns + TD(lambda) on 4096 x
1024, V-trace 2048 x 4096, Retrace 1024 x 16384, GAE / V-trace / Retrace on
2^20-step rows, and the fused, masked, normalised, compact and [N,T,A]
variants).  --workload picks another headline (then alone).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--trials R]
                  [--impl ours|reference] [--workload NAME] [--suite auto|on|off]

Timing: W warm-up steps, then R trials of K back-to-back steps, one CUDA
event pair per trial; the reported time is the best trial's mean.  Prints
one JSON line (rank 0).  Under torchrun each rank runs its own batch (rows
are independent: weak scaling, no collective on the data path); times are
the max over ranks.
"""
from __future__ import annotations

import argparse
import concurrent.futures
import ctypes
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from linear_recurrence_scan_gb300 import synthetic  # noqa: E402
from linear_recurrence_scan_gb300.sharding import max_over_ranks  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# workloads: estimators, their inputs and algorithmic bytes per env-step
# (fp32 inputs read once + outputs written once; [N] vectors and the
# one-step halo are not counted)

_VTRACE_VALUES = ("log_pi_target", "log_pi_behavior", "values", "rewards", "bootstrap_values")
_RETRACE_VALUES = ("pi_taken", "mu_taken", "q_values", "expected_next_q", "rewards")


def _cfg_workloads():
    W = synthetic.WORKLOADS
    c1, c2, c3, c4 = (W[k] for k in ("gae_returns_4096x1024", "vtrace_2048x4096", "retrace_1024x16384",
                                      "long_rows_64x1048576"))
    return {
        "gae_returns_4096x1024": dict(
            desc="GAE + discounted returns + TD(lambda) returns, last_value bootstrap, no truncations",
            N=4096, T=1024, gen=lambda N, T: synthetic.workload_batch("gae_returns_4096x1024", N=N, T=T),
            estimators=[("gae", 16, c1), ("discounted_returns", 12, c1), ("lambda_returns", 16, c1)],
            # the step's three outputs from one kernel: r, v, term read once,
            # advantages, lambda-returns, discounted returns written
            fused=("gae_returns", 24, c1)),
        "gae_normalized_4096x1024": dict(
            desc="GAE advantages normalised over the batch (fused moments + in-place pass) "
                 "and TD(lambda) returns, last_value bootstrap, no truncations",
            N=4096, T=1024, gen=lambda N, T: synthetic.workload_batch("gae_returns_4096x1024", N=N, T=T),
            # r, v, term read once; normalised advantages and lambda-returns written
            estimators=[("gae_normalized", 20, c1)]),
        "gae_masked_4096x8192": dict(
            desc="token-level GAE with observation-skip masking on LLM rollouts (masked prompt, "
                 "tool observations and padding; outcome reward on the last response token)",
            N=4096, T=8192, gen=lambda N, T: synthetic.llm_tokens_batch(N, T),
            # r, v, term, mask read once; advantages written
            estimators=[("gae_masked", 20, dict(gamma=1.0, lambda_=0.95))]),
        "gae_compact_4096x1024": dict(
            desc="GAE on compact storage: bfloat16 rewards and values, uint8 flags, float32 "
                 "advantages (float32 arithmetic), last_value bootstrap",
            N=4096, T=1024, gen=lambda N, T: synthetic.compact(synthetic.workload_batch("gae_returns_4096x1024", N=N, T=T)),
            # 2 + 2 + 1 bytes read, 4 written
            estimators=[("gae_compact", 9, c1)]),
        "gae_returns_compact_4096x1024": dict(
            desc="GAE + discounted returns + TD(lambda) returns on compact storage: bfloat16 "
                 "values in and out, uint8 flags (float32 arithmetic), last_value bootstrap",
            N=4096, T=1024, gen=lambda N, T: synthetic.compact(synthetic.workload_batch("gae_returns_4096x1024", N=N, T=T)),
            # 2 + 2 + 1 bytes read, 3 x 2 written
            estimators=[("gae_returns_compact", 11, c1)]),
        "gae_8x128": dict(
            desc="GAE with truncations and 2-D bootstrap", N=8, T=128,
            gen=lambda N, T: synthetic.workload_batch("gae_8x128", N=N, T=T),
            estimators=[("gae_trunc_bs", 24, W["gae_8x128"])]),
        "vtrace_2048x4096": dict(
            desc="V-trace with truncations and 2-D bootstrap", N=2048, T=4096,
            gen=lambda N, T: synthetic.workload_batch("vtrace_2048x4096", N=N, T=T),
            estimators=[("vtrace", 36, c2)]),
        "vtrace_4096x1024": dict(
            desc="V-trace with truncations and 2-D bootstrap at the 4096 x 1024 shape "
                 "(like-for-like with the GAE step)", N=4096, T=1024,
            gen=lambda N, T: synthetic.vtrace_batch(N, T, 0, 2, c2["p_term"], c2["p_trunc"], "2d"),
            estimators=[("vtrace", 36, c2)]),
        "retrace_4096x1024": dict(
            desc="Retrace(lambda) on per-step inputs at the 4096 x 1024 shape (like-for-like)",
            N=4096, T=1024,
            gen=lambda N, T: synthetic.retrace_batch(N, T, 0, 3, c3["p_term"], 0.0),
            estimators=[("retrace", 32, c3)]),
        "retrace_1024x16384": dict(
            desc="Retrace(lambda) on per-step inputs, no truncations", N=1024, T=16384,
            gen=lambda N, T: synthetic.workload_batch("retrace_1024x16384", N=N, T=T),
            estimators=[("retrace", 32, c3)]),
        "vtrace_compact_2048x4096": dict(
            desc="V-trace with truncations and 2-D bootstrap on compact storage: bfloat16 "
                 "log-probabilities, values, rewards and bootstrap values, uint8 flags, bfloat16 "
                 "outputs (float32 arithmetic)", N=2048, T=4096,
            gen=lambda N, T: synthetic.compact(synthetic.workload_batch("vtrace_2048x4096", N=N, T=T), values=_VTRACE_VALUES),
            # 5 x 2 + 2 x 1 bytes read, 2 x 2 written
            estimators=[("vtrace_compact", 16, c2)]),
        "retrace_compact_1024x16384": dict(
            desc="Retrace(lambda) on per-step inputs in compact storage: bfloat16 probabilities, "
                 "Q-values and rewards, uint8 flags, bfloat16 outputs (float32 arithmetic)",
            N=1024, T=16384,
            gen=lambda N, T: synthetic.compact(synthetic.workload_batch("retrace_1024x16384", N=N, T=T), values=_RETRACE_VALUES),
            # 5 x 2 + 1 bytes read, 2 x 2 written
            estimators=[("retrace_compact", 15, c3)]),
        "retrace_actions_1024x16384x4": dict(
            desc="Retrace(lambda) from [N,T,A] target probabilities and successor Q-values with "
                 "int64 actions (A = 4), reduced in-kernel, no truncations",
            N=1024, T=16384,
            gen=lambda N, T: synthetic.retrace_actions_batch(N, T, 4, 0, 3, c3["p_term"], 0.0),
            # 2 x [N,T,4] f32 + int64 action + 4 [N,T] f32 in, 2 [N,T] f32 out
            estimators=[("retrace_actions", 64, c3)]),
        "long_rows_64x1048576": dict(
            desc="eligibility traces + episodic prefix sum (starts_at, integer inputs)",
            N=64, T=1 << 20, gen=lambda N, T: synthetic.workload_batch("long_rows_64x1048576", N=N, T=T),
            estimators=[("eligibility_traces", 12, c4), ("episodic_prefix_sum", 12, c4)]),
        "gae_64x1048576": dict(
            desc="GAE on 1M-step rows (last_value, no truncations)", N=64, T=1 << 20,
            gen=lambda N, T: synthetic.gae_batch(N, T, 0, 41, c1["p_term"], 0.0, "last"),
            estimators=[("gae", 16, c1)]),
        "vtrace_64x1048576": dict(
            desc="V-trace on 1M-step rows (truncations, 2-D bootstrap)", N=64, T=1 << 20,
            gen=lambda N, T: synthetic.vtrace_batch(N, T, 0, 42, c2["p_term"], c2["p_trunc"], "2d"),
            estimators=[("vtrace", 36, c2)]),
        "retrace_64x1048576": dict(
            desc="Retrace on 1M-step rows", N=64, T=1 << 20,
            gen=lambda N, T: synthetic.retrace_batch(N, T, 0, 43, c3["p_term"], 0.0),
            estimators=[("retrace", 32, c3)]),
    }


WORKLOADS = _cfg_workloads()

# inputs and outputs of each estimator (names in the synthetic batch)
IO = {
    "gae": (["rewards", "values", "terminateds"], ["last_value"], 1),
    "gae_trunc_bs": (["rewards", "values", "terminateds", "truncateds", "bootstrap_values"], [], 1),
    "discounted_returns": (["rewards", "terminateds"], ["last_value"], 1),
    "lambda_returns": (["rewards", "next_values", "terminateds"], ["last_value"], 1),
    "vtrace": (["log_pi_target", "log_pi_behavior", "values", "rewards", "terminateds",
                "truncateds", "bootstrap_values"], [], 2),
    "retrace": (["pi_taken", "mu_taken", "q_values", "expected_next_q", "rewards", "terminateds"],
                [], 2),
    "retrace_actions": (["action_probs_target", "action_probs_behavior", "q_values",
                         "next_q_values_all", "actions", "rewards", "terminateds"], [], 2),
    "eligibility_traces": (["gradients", "trace_dones"], [], 1),
    "episodic_prefix_sum": (["inputs", "prefix_dones"], [], 1),
    "gae_returns": (["rewards", "values", "terminateds"], ["last_value"], 3),
    "gae_normalized": (["rewards", "values", "terminateds"], ["last_value"], 2),
    "gae_masked": (["rewards", "values", "terminateds", "mask"], [], 1),
    "gae_compact": (["rewards", "values", "terminateds"], ["last_value"], 1),
    "gae_returns_compact": (["rewards", "values", "terminateds"], ["last_value"], 3),
    "vtrace_compact": (["log_pi_target", "log_pi_behavior", "values", "rewards", "terminateds",
                        "truncateds", "bootstrap_values"], [], 2),
    "retrace_compact": (["pi_taken", "mu_taken", "q_values", "expected_next_q", "rewards",
                         "terminateds"], [], 2),
}
# output element bytes (default 4)
OUT_BYTES = {"gae_returns_compact": 2, "vtrace_compact": 2, "retrace_compact": 2}
OUT_DTYPE = {"gae_returns_compact": "bf16", "vtrace_compact": "bf16", "retrace_compact": "bf16"}
# streams the end-to-end steps rotate over by default (copies of one step
# overlap another's compute)
E2E_STREAMS = 3

# kernels one call launches (default 1)
LAUNCHES = {"gae_normalized": 2}



METRIC = "env-steps/sec and achieved HBM GB/s (% of GB300 peak) per estimator, 1 GPU"

# The headline workload (the largest single-GPU configuration: 64 rows of
# 2^20 steps, eligibility traces + episodic prefix sums) and the workloads
# measured beside it in the same run (every estimator at its named shape,
# GAE / V-trace / Retrace on 2^20-step rows, and the fused, masked,
# normalised, compact and [N,T,A] variants).
HEADLINE = "long_rows_64x1048576"
SUITE = ["gae_8x128", "gae_returns_4096x1024", "vtrace_2048x4096", "retrace_1024x16384",
         "gae_64x1048576", "vtrace_64x1048576", "retrace_64x1048576",
         "vtrace_4096x1024", "retrace_4096x1024",
         "gae_normalized_4096x1024", "gae_masked_4096x8192", "gae_compact_4096x1024",
         "gae_returns_compact_4096x1024", "vtrace_compact_2048x4096",
         "retrace_compact_1024x16384", "retrace_actions_1024x16384x4"]


def step_kernels_of(wl_name):
    """Kernels of one step: the fused kernel when the workload has one, else
    one kernel per estimator."""
    wl = WORKLOADS[wl_name]
    return [wl["fused"]] if wl.get("fused") else list(wl["estimators"])


prep_kernels = step_kernels_of


def l2_plan(wl_name):
    """Rotating input sets so that consecutive steps never find their inputs
    in the 129 MB L2: one set when a step's inputs + outputs exceed 4x L2,
    else enough sets to cover 4x L2.  Returns (sets, bytes per set)."""
    wl = WORKLOADS[wl_name]
    N, T = wl["N"], wl["T"]
    batch = wl["gen"](min(N, 2), min(T, 256))
    kernels = step_kernels_of(wl_name)
    need_in = sorted({k for (n, _, _) in kernels for k in IO[n][0] + IO[n][1]})
    in_bytes = 0
    for k in need_in:
        v = batch[k]
        per_elem = v.itemsize * (int(np.prod(v.shape[2:])) if v.ndim > 2 else 1)
        in_bytes += per_elem * (N * T if v.ndim >= 2 else N)
    out_bytes = sum(IO[n][2] * N * T * OUT_BYTES.get(n, 4) for (n, _, _) in kernels)
    set_bytes = in_bytes + out_bytes
    n_sets = 1 if set_bytes > 4 * L2_BYTES else min(16, max(2, math.ceil(4 * L2_BYTES / set_bytes)))
    return n_sets, set_bytes


def workload_config(wl_name):
    """The `config` object of a workload: the same in both arms."""
    wl = WORKLOADS[wl_name]
    n_sets, set_bytes = l2_plan(wl_name)
    if n_sets == 1:
        l2 = f"inputs larger than L2: {set_bytes / 1e6:.0f} MB per step > 4 x 129 MB"
    else:
        l2 = (f"{n_sets} rotating input sets of {set_bytes / 1e6:.1f} MB "
              f"({n_sets * set_bytes / 1e6:.0f} MB > 129 MB L2)")
    return {"workload": wl_name, "description": wl["desc"], "num_envs": wl["N"],
            "seq_len": wl["T"], "estimators": [e[0] for e in wl["estimators"]],
            "parallelism": "rows: one independent batch per GPU (weak scaling, no collective)",
            "l2": l2}


def _csrc_hash():
    h = hashlib.sha256()
    d = os.path.join(ROOT, "linear_recurrence_scan_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def _measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _ncu_traffic(kernel, workload):
    """DRAM bytes per launch (read + write) that ncu recorded for this kernel
    and workload (profiles/traffic.json), if the capture was taken on the
    current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    e = rec.get("records", {}).get(f"{kernel}@{workload}")
    if not e or e.get("csrc_sha") != _csrc_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# clocks sampled during the run

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,utilization.gpu,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) >= 10:
                rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        loaded = [r for r in rows if (num(r[3]) or 0) > 0] or rows
        sm = [num(r[1]) for r in loaded if num(r[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in loaded:
            for name, val in zip(names, r[6:10]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": num(loaded[0][2]), "samples": len(rows),
                "samples_under_load": len(loaded), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# our arm

def _launcher(name, c, bufs, outs, N, T, ws, wsn, stream):
    """ABI call of one estimator on preallocated device buffers."""
    from linear_recurrence_scan_gb300 import _native
    lib = _native.lib()
    vp = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    b = {k: vp(v) for k, v in bufs.items()}
    o = [vp(t) for t in outs]
    g = float(c.get("gamma", 0.99))
    if name == "gae":
        return lambda: lib.rlscan_gae(b["rewards"], b["values"], b["terminateds"], None, None,
                                      b["last_value"], N, T, T, g, float(c["lambda_"]), o[0], ws,
                                      wsn, stream)
    if name == "gae_trunc_bs":
        return lambda: lib.rlscan_gae(b["rewards"], b["values"], b["terminateds"], b["truncateds"],
                                      b["bootstrap_values"], None, N, T, T, g, float(c["lambda_"]),
                                      o[0], ws, wsn, stream)
    if name == "discounted_returns":
        return lambda: lib.rlscan_discounted_returns(b["rewards"], b["terminateds"], None, None,
                                                     b["last_value"], N, T, T, g, o[0], ws, wsn,
                                                     stream)
    if name == "lambda_returns":
        return lambda: lib.rlscan_lambda_returns(b["rewards"], b["next_values"], b["terminateds"],
                                                 None, None, b["last_value"], N, T, T, g,
                                                 float(c["lambda_"]), o[0], ws, wsn, stream)
    if name == "vtrace":
        return lambda: lib.rlscan_vtrace(b["log_pi_target"], b["log_pi_behavior"], b["values"],
                                         b["rewards"], b["terminateds"], b["truncateds"],
                                         b["bootstrap_values"], None, N, T, T, g,
                                         float(c["rho_bar"]), float(c["c_bar"]), o[0], o[1], ws,
                                         wsn, stream)
    if name == "retrace":
        return lambda: lib.rlscan_retrace(b["pi_taken"], b["mu_taken"], b["q_values"],
                                          b["expected_next_q"], b["rewards"], b["terminateds"],
                                          None, N, T, T, g, float(c["lambda_"]), float(c["c_bar"]),
                                          float(c["rho_bar"]), o[0], o[1], ws, wsn, stream)
    if name == "retrace_actions":
        A = bufs["action_probs_target"].shape[2]
        return lambda: lib.rlscan_retrace_actions(
            b["action_probs_target"], b["action_probs_behavior"], b["q_values"],
            b["next_q_values_all"], b["actions"], b["rewards"], b["terminateds"], None, N, T, A, T,
            T * A, g, float(c["lambda_"]), float(c["c_bar"]), float(c["rho_bar"]), o[0], o[1], ws,
            wsn, stream)
    if name == "eligibility_traces":
        return lambda: lib.rlscan_eligibility_traces(b["gradients"], b["trace_dones"], None, N, T,
                                                     T, g, float(c["lambda_"]), o[0], ws, wsn,
                                                     stream)
    if name == "episodic_prefix_sum":
        return lambda: lib.rlscan_episodic_prefix_sum(b["inputs"], b["prefix_dones"], None, 1, N,
                                                      T, T, o[0], ws, wsn, stream)
    if name == "gae_compact":
        return lambda: lib.rlscan_gae_compact(b["rewards"], b["values"], b["terminateds"], None, None,
                                              b["last_value"], N, T, T, g, float(c["lambda_"]), 0,
                                              o[0], ws, wsn, stream)
    if name == "gae_returns_compact":
        return lambda: lib.rlscan_gae_returns_compact(b["rewards"], b["values"], b["terminateds"],
                                                      None, None, b["last_value"], N, T, T, g,
                                                      float(c["lambda_"]), 1, o[0], o[1], o[2], ws,
                                                      wsn, stream)
    if name == "vtrace_compact":
        return lambda: lib.rlscan_vtrace_compact(b["log_pi_target"], b["log_pi_behavior"], b["values"],
                                                 b["rewards"], b["terminateds"], b["truncateds"],
                                                 b["bootstrap_values"], None, N, T, T, g,
                                                 float(c["rho_bar"]), float(c["c_bar"]), 1, o[0], o[1],
                                                 ws, wsn, stream)
    if name == "retrace_compact":
        return lambda: lib.rlscan_retrace_compact(b["pi_taken"], b["mu_taken"], b["q_values"],
                                                  b["expected_next_q"], b["rewards"], b["terminateds"],
                                                  None, N, T, T, g, float(c["lambda_"]),
                                                  float(c["c_bar"]), float(c["rho_bar"]), 1, o[0],
                                                  o[1], ws, wsn, stream)
    if name == "gae_masked":
        return lambda: lib.rlscan_gae_masked(b["rewards"], b["values"], b["terminateds"], None, None,
                                             None, b["mask"], N, T, T, g, float(c["lambda_"]), o[0],
                                             ws, wsn, stream)
    if name == "gae_normalized":
        return lambda: lib.rlscan_gae_normalized(b["rewards"], b["values"], b["terminateds"], None,
                                                 None, b["last_value"], N, T, T, g,
                                                 float(c["lambda_"]), 1e-8, o[0], o[1], None, None,
                                                 ws, wsn, stream)
    if name == "gae_returns":
        return lambda: lib.rlscan_gae_returns(b["rewards"], b["values"], b["terminateds"], None,
                                              None, b["last_value"], N, T, T, g,
                                              float(c["lambda_"]), o[0], o[1], o[2], ws, wsn,
                                              stream)
    raise KeyError(name)


def _bf16(t):
    """A device tensor of bfloat16 bits (uint16 storage) viewed as bfloat16."""
    import torch
    return t.view(torch.bfloat16) if t.dtype == torch.uint16 else t


def _decode(a):
    """Compact host arrays as float32: bfloat16 bits -> float, uint8 -> float."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32)
    return a.astype(np.float32)


def _public_call(name, c, t):
    """The same estimator through the public PyTorch API (for e2e)."""
    import linear_recurrence_scan_gb300 as Lb
    g = float(c.get("gamma", 0.99))
    if name == "gae":
        return [Lb.compute_gae(t["rewards"], t["values"], t["terminateds"], None, g, c["lambda_"],
                               None, t["last_value"])]
    if name == "gae_trunc_bs":
        return [Lb.compute_gae(t["rewards"], t["values"], t["terminateds"], t["truncateds"], g,
                               c["lambda_"], t["bootstrap_values"])]
    if name == "discounted_returns":
        return [Lb.compute_discounted_returns(t["rewards"], t["terminateds"], None, g, None,
                                              t["last_value"])]
    if name == "lambda_returns":
        return [Lb.compute_lambda_returns(t["rewards"], t["next_values"], t["terminateds"], None, g,
                                          c["lambda_"], None, t["last_value"])]
    if name == "vtrace":
        return list(Lb.compute_vtrace(t["log_pi_target"], t["log_pi_behavior"], t["values"],
                                      t["rewards"], t["terminateds"], t["truncateds"], g,
                                      c["rho_bar"], c["c_bar"], t["bootstrap_values"]))
    if name == "retrace":
        return list(Lb.compute_retrace_from_probs(t["pi_taken"], t["mu_taken"], t["q_values"],
                                                  t["expected_next_q"], t["rewards"],
                                                  t["terminateds"], None, g, c["lambda_"],
                                                  c["c_bar"], c["rho_bar"]))
    if name == "retrace_actions":
        return list(Lb.compute_retrace(t["action_probs_target"], t["action_probs_behavior"],
                                       t["q_values"], t["next_q_values_all"], t["actions"],
                                       t["rewards"], t["terminateds"], None, g, c["lambda_"],
                                       c["c_bar"], c["rho_bar"]))
    if name == "eligibility_traces":
        return [Lb.compute_eligibility_traces(t["gradients"], t["trace_dones"], g, c["lambda_"])]
    if name == "episodic_prefix_sum":
        return [Lb.compute_episodic_prefix_sum(t["inputs"], t["prefix_dones"], None, "starts_at")]
    if name == "gae_masked":
        return [Lb.compute_gae(t["rewards"], t["values"], t["terminateds"], None, g, c["lambda_"],
                               mask=t["mask"])]
    if name == "gae_compact":
        return [Lb.compute_gae(_bf16(t["rewards"]), _bf16(t["values"]), t["terminateds"], None, g,
                               c["lambda_"], None, t["last_value"])]
    if name == "gae_returns_compact":
        import torch
        return list(Lb.compute_gae_and_returns(_bf16(t["rewards"]), _bf16(t["values"]),
                                               t["terminateds"], None, g, c["lambda_"], None,
                                               t["last_value"], out_dtype=torch.bfloat16))
    if name == "vtrace_compact":
        import torch
        return list(Lb.compute_vtrace(_bf16(t["log_pi_target"]), _bf16(t["log_pi_behavior"]),
                                      _bf16(t["values"]), _bf16(t["rewards"]), t["terminateds"],
                                      t["truncateds"], g, c["rho_bar"], c["c_bar"],
                                      _bf16(t["bootstrap_values"]), out_dtype=torch.bfloat16))
    if name == "retrace_compact":
        import torch
        return list(Lb.compute_retrace_from_probs(
            _bf16(t["pi_taken"]), _bf16(t["mu_taken"]), _bf16(t["q_values"]),
            _bf16(t["expected_next_q"]), _bf16(t["rewards"]), t["terminateds"], None, g, c["lambda_"],
            c["c_bar"], c["rho_bar"], out_dtype=torch.bfloat16))
    if name == "gae_normalized":
        return list(Lb.compute_gae_normalized(t["rewards"], t["values"], t["terminateds"], None, g,
                                              c["lambda_"], None, t["last_value"], 1e-8,
                                              outputs=("advantages", "lambda_returns")))
    if name == "gae_returns":
        return list(Lb.compute_gae_and_returns(t["rewards"], t["values"], t["terminateds"], None, g,
                                               c["lambda_"], None, t["last_value"]))
    raise KeyError(name)


class _Prepared:
    """One workload resident on the device: rotating input sets, outputs,
    workspace and one ABI launcher per kernel and set."""

    def __init__(self, wl_name, dev, stream):
        import torch
        from linear_recurrence_scan_gb300 import _native
        self.name = wl_name
        self.wl = wl = WORKLOADS[wl_name]
        self.N, self.T = N, T = wl["N"], wl["T"]
        self.step_kernels = step_kernels_of(wl_name)
        self.all_kernels = self.step_kernels + (list(wl["estimators"]) if wl.get("fused") else [])
        self.n_sets, self.set_bytes = l2_plan(wl_name)
        need_in = sorted({k for (n, _, _) in self.all_kernels for k in IO[n][0] + IO[n][1]})
        batch = wl["gen"](N, T)
        self.host = {k: batch[k] for k in need_in}
        del batch
        self.stream = stream
        sh = ctypes.c_void_p(stream.cuda_stream)
        lib = _native.lib()
        self.wsn = wsn = max(lib.rlscan_workspace_bytes(N, T), lib.rlscan_gae_normalized_workspace_bytes(N, T))
        ws = None
        self.keep = []  # every set's tensors stay allocated: the launchers hold raw pointers
        if wsn:
            ws_t = torch.empty(wsn, dtype=torch.uint8, device=dev)
            self.keep.append([ws_t])
            _native.check(lib.rlscan_workspace_init(ctypes.c_void_p(ws_t.data_ptr()), wsn, sh), "init")
            ws = ctypes.c_void_p(ws_t.data_ptr())
        self.sets = []
        for _ in range(self.n_sets):
            bufs = {k: torch.from_numpy(v).to(dev) for k, v in self.host.items()}
            self.keep.append(bufs)
            calls = {}
            for (name, _, c) in self.all_kernels:
                odt = torch.bfloat16 if OUT_DTYPE.get(name) == "bf16" else torch.float32
                outs = [torch.empty((N, T), dtype=odt, device=dev) for _ in range(IO[name][2])]
                self.keep.append(outs)
                calls[name] = _launcher(name, c, bufs, outs, N, T, ws, wsn, sh)
            self.sets.append(calls)
        ptrs = [t.data_ptr() for group in self.keep
                for t in (group.values() if isinstance(group, dict) else group)]
        assert len(ptrs) == len(set(ptrs)), "input sets must not share memory"
        torch.cuda.synchronize()

    def run(self, kernels, i):
        from linear_recurrence_scan_gb300 import _native
        calls = self.sets[i % self.n_sets]
        for (name, _, _) in kernels:
            st = calls[name]()
            if st != 0:
                raise _native.RlscanError(st, name)

    def region(self, kernels, K, offset, world):
        """K steps of `kernels` back to back on the stream, one CUDA event
        pair around the whole region (none between launches, which would
        serialise them); barrier + synchronize on both sides.  Returns ms
        per step (max over ranks) and the host wall time of the region."""
        import torch
        t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        t0e.record(self.stream)
        for i in range(K):
            self.run(kernels, offset + i)
        t1e.record(self.stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        return max_over_ranks(t0e.elapsed_time(t1e) / K), wall

    def trials(self, kernels, K, n_trials, offset, world):
        """`n_trials` regions of K steps; ms per step of each trial and the
        total host wall time."""
        out, wall = [], 0.0
        for r in range(n_trials):
            ms, w = self.region(kernels, K, offset + r * K, world)
            out.append(ms)
            wall += w
        return out, wall

    def free(self):
        import torch
        self.keep.clear()
        self.sets.clear()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


def _kernel_stats(name, bps, trial_ms, steps_per_call, peak, workload):
    """Per-launch figures of one kernel from its trials: the reported
    duration is the best trial's mean (the pages' minimum over trials)."""
    ts = np.array(trial_ms, dtype=np.float64)
    us = float(ts.min() * 1e3)
    gbs = bps * steps_per_call / (us * 1e-6) / 1e9
    alg = bps * steps_per_call
    traffic = _ncu_traffic(name, workload)
    return {"us_mean": round(us, 2), "us_trials": [round(float(t) * 1e3, 2) for t in ts],
            "env_steps_per_s": steps_per_call / (us * 1e-6), "bytes_per_env_step": bps,
            "algorithmic_bytes_per_launch": alg,
            "gb_per_s": round(gbs, 1), "frac_of_measured_hbm": round(gbs / peak, 4),
            "frac_of_nominal_8tbs": round(gbs / 8000.0, 4),
            "traffic": traffic, "traffic_over_algorithmic": (round(traffic / alg, 4)
                                                             if traffic else None)}


def _auto_steps(prep, kernels, world, target_ms=25.0, lo=20, hi=4000):
    """Steps per trial so that a trial of `kernels` lasts about `target_ms`."""
    ms, _ = prep.region(kernels, 3, 0, world)
    return int(min(hi, max(lo, math.ceil(target_ms / max(ms, 1e-4)))))


def measure_workload(prep, K, n_trials, warmup, world, peak):
    """Step timing and per-kernel / per-estimator figures of one prepared
    workload.  K steps per trial (None: sized to ~25 ms a trial)."""
    wl = prep.wl
    step_kernels = prep.step_kernels
    for i in range(warmup):
        prep.run(step_kernels, i)
    if K is None:
        K = _auto_steps(prep, step_kernels, world)
    trial_ms, wall = prep.trials(step_kernels, K, n_trials, warmup, world)
    ms_step = min(trial_ms)
    steps_per_call = prep.N * prep.T
    # per-launch durations of the step's kernels (the step itself when it is one kernel)
    if len(step_kernels) == 1:
        per_kernel = {step_kernels[0][0]: trial_ms}
    else:
        per_kernel = {e[0]: prep.trials([e], K, n_trials, warmup, world)[0] for e in step_kernels}
    per_est_times = per_kernel
    if wl.get("fused"):  # the estimators one kernel each, for the per-estimator figures
        for i in range(warmup):
            prep.run(wl["estimators"], i)
        per_est_times = {e[0]: prep.trials([e], K, n_trials, warmup, world)[0] for e in wl["estimators"]}
    step = {n: _kernel_stats(n, bps, per_kernel[n], steps_per_call, peak, prep.name)
            for (n, bps, _) in step_kernels}
    per_est = {n: _kernel_stats(n, bps, per_est_times[n], steps_per_call, peak, prep.name)
               for (n, bps, _) in wl["estimators"]}
    dominant = max(step_kernels, key=lambda e: min(per_kernel[e[0]]))[0]
    return {"K": K, "trials_ms": [round(t, 5) for t in trial_ms], "ms_per_step": ms_step,
            "wall": wall, "step": step, "per_estimator": per_est, "dominant": dominant,
            "env_steps_per_s": world * steps_per_call / (ms_step * 1e-3)}


def run_e2e(args, prep, dev, world):
    """End to end through the public API: pinned host inputs -> device, the
    step's call(s), results back to pinned host memory, every step.
    Consecutive steps go to E2E_STREAMS streams in turn (each with its own
    device and host buffers), so one step's upload, another's compute and a
    third's download overlap, as a pipeline of rollout batches would run."""
    import torch
    N, T = prep.N, prep.T
    step_kernels = prep.step_kernels
    e2e_in = sorted({k for (n, _, _) in step_kernels for k in IO[n][0] + IO[n][1]})
    pinned = {k: torch.from_numpy(prep.host[k]).pin_memory() for k in e2e_in}
    NS = max(1, args.e2e_streams)
    e2e_streams = [torch.cuda.Stream(dev) for _ in range(NS)]
    dsets = [{k: torch.empty(v.shape, dtype=v.dtype, device=dev) for k, v in pinned.items()}
             for _ in range(NS)]
    hsets = [[torch.empty((N, T), dtype=torch.bfloat16 if OUT_DTYPE.get(n) == "bf16"
                          else torch.float32).pin_memory()
              for (n, _, _) in step_kernels for _ in range(IO[n][2])] for _ in range(NS)]
    h2d = sum(v.numel() * v.element_size() for v in pinned.values())
    d2h = sum(o.numel() * o.element_size() for o in hsets[0])
    zero_copy = args.e2e_mode == "zerocopy"

    def e2e_step(i):
        j = i % NS
        with torch.cuda.stream(e2e_streams[j]):
            if zero_copy:
                # the public API on the pinned host tensors themselves: the
                # kernel reads the inputs and writes the (pinned) outputs over
                # the host link
                for (name, _, c) in step_kernels:
                    hsets[j] = _public_call(name, c, pinned)
                return
            for k in pinned:
                dsets[j][k].copy_(pinned[k], non_blocking=True)
            outs = []
            for (name, _, c) in step_kernels:
                outs += _public_call(name, c, dsets[j])
            for o, hbuf in zip(outs, hsets[j]):
                hbuf.copy_(o, non_blocking=True)
    for i in range(max(NS, min(args.warmup, 3))):
        e2e_step(i)
    torch.cuda.synchronize()
    K = args.e2e_steps if args.e2e_steps > 0 else args.steps
    e0 = time.perf_counter()
    for i in range(K):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks((time.perf_counter() - e0) / K)
    res = {"value": world * N * T / e2e_s, "unit": "env-steps/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K,
           "path": ("public compute_* API on pinned host tensors: the kernel reads the inputs "
                    "and writes the pinned outputs over the host link (zero copy)"
                    if zero_copy else
                    "pinned host -> device copies, public compute_* API, results -> pinned host")
                   + f"; steps round-robin over {NS} streams"}
    del pinned, dsets, hsets
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def capture_schedule(args, wl_name, warm=3, count=6):
    """A fixed launch schedule for DRAM-traffic captures: for each kernel of
    the workload (the step's and, for a fused step, each estimator's), `warm`
    launches then `count` more, back to back over the rotating input sets,
    with a synchronize between kernels.  Timing is not taken here; under
    `ncu --cache-control none` each launch's DRAM counters then include the
    write-back of its predecessor's outputs, so the mean over the `count`
    launches is one launch's read + write traffic.  Returns the schedule."""
    import torch
    from linear_recurrence_scan_gb300 import build
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    prep = _Prepared(wl_name, dev, torch.cuda.current_stream(dev))
    sched = []
    for e in prep.all_kernels:
        for i in range(warm + count):
            prep.run([e], i)
        torch.cuda.synchronize()
        sched.append({"kernel": e[0], "warm": warm, "count": count,
                      "algorithmic_bytes_per_launch": e[1] * prep.N * prep.T})
    prep.free()
    return {"workload": wl_name, "capture": sched}


def run_ours(args, wl_name, rank, world, local_rank, sub_workloads=()):
    import torch
    from linear_recurrence_scan_gb300 import build
    build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = _measured_peak()
    wl = WORKLOADS[wl_name]
    names = [e[0] for e in wl["estimators"]]

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    prep = _Prepared(wl_name, dev, stream)
    m = measure_workload(prep, args.steps, args.trials, args.warmup, world, peak)
    K = m["K"]
    e2e = run_e2e(args, prep, dev, world)
    prep.free()
    del prep

    # the other workloads: same protocol, steps per trial sized to ~25 ms
    subs = {}
    for sub in sub_workloads:
        if sub == wl_name:
            continue
        p = _Prepared(sub, dev, stream)
        sm = measure_workload(p, None, args.trials, args.warmup, world, peak)
        p.free()
        del p
        subs[sub] = {"config": workload_config(sub),
                     "steps": sm["K"], "trials": args.trials,
                     "ms_per_step": sm["ms_per_step"], "trials_ms": sm["trials_ms"],
                     "env_steps_per_s": sm["env_steps_per_s"],
                     "step": sm["step"], "per_estimator": sm["per_estimator"]}
    clocks = sampler.stop()

    d = m["step"][m["dominant"]]
    result = {
        "metric": METRIC,
        "value": m["env_steps_per_s"],
        "unit": "env-steps/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "trials": args.trials,
        "ms_per_step": m["ms_per_step"], "trials_ms": m["trials_ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if not any(n.endswith("_compact") for n in names) else
                 "f32 arithmetic on bf16 values / u8 flags", "data": "synthetic",
        "config": workload_config(wl_name),
        "step_kernels": [n for (n, _, _) in prep_kernels(wl_name)],
        "step": m["step"],
        "per_estimator": m["per_estimator"],
        "roofline": {"bound": "hbm", "kernel": m["dominant"], "achieved": d["gb_per_s"], "peak": peak,
                     "peak_source": peak_kind, "unit": "GB/s", "frac": d["frac_of_measured_hbm"],
                     "traffic": d["traffic"],
                     "algorithmic_bytes_per_launch": d["algorithmic_bytes_per_launch"]},
        "e2e": e2e,
        "gpu_launches": args.trials * K * sum(LAUNCHES.get(n, 1) for (n, _, _) in prep_kernels(wl_name)),
        "full_call_us": round(m["wall"] / (args.trials * K) * 1e6, 2),
        "timing": (f"{args.trials} trials of K back-to-back steps, one CUDA event pair per trial on "
                   "the launching stream (none between launches, which would serialise them), "
                   "barrier + synchronize around each trial; ms_per_step is the best trial's mean "
                   "(the pages' minimum over trials); per-kernel durations from trials of that "
                   "kernel alone; gpu_launches counts the step trials; full_call_us: host wall "
                   "time per step over the step trials"),
        "wall_s_timed": round(m["wall"], 4),
        "clocks": clocks,
    }
    if subs:
        result["workloads"] = subs
    return result


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline and reference arm)

def _oracle_call(name, c, b):
    import oracle
    g = float(c.get("gamma", 0.99))
    if name == "gae":
        return oracle.gae(b["rewards"], b["values"], b["terminateds"], None, g, c["lambda_"], None,
                          b["last_value"])
    if name == "gae_trunc_bs":
        return oracle.gae(b["rewards"], b["values"], b["terminateds"], b["truncateds"], g,
                          c["lambda_"], b["bootstrap_values"])
    if name == "discounted_returns":
        return oracle.discounted_returns(b["rewards"], b["terminateds"], None, g, None, b["last_value"])
    if name == "lambda_returns":
        return oracle.lambda_returns(b["rewards"], b["next_values"], b["terminateds"], None, g,
                                     c["lambda_"], None, b["last_value"])
    if name == "vtrace":
        return oracle.vtrace(b["log_pi_target"], b["log_pi_behavior"], b["values"], b["rewards"],
                             b["terminateds"], b["truncateds"], g, c["rho_bar"], c["c_bar"],
                             b["bootstrap_values"])
    if name == "retrace":
        return oracle.retrace(b["pi_taken"], b["mu_taken"], b["q_values"], b["expected_next_q"],
                              b["rewards"], b["terminateds"], None, g, c["lambda_"], c["c_bar"],
                              c["rho_bar"])
    if name == "retrace_actions":
        return oracle.retrace_actions(b["action_probs_target"], b["action_probs_behavior"],
                                      b["q_values"], b["next_q_values_all"], b["actions"],
                                      b["rewards"], b["terminateds"], None, g, c["lambda_"],
                                      c["c_bar"], c["rho_bar"])
    if name in ("gae_compact", "gae_returns_compact"):
        dec = {k: _decode(b[k]) for k in ("rewards", "values", "terminateds")}
        adv = oracle.gae(dec["rewards"], dec["values"], dec["terminateds"], None, g, c["lambda_"],
                         None, b["last_value"])
        if name == "gae_compact":
            return adv
        return adv, oracle.discounted_returns(dec["rewards"], dec["terminateds"], None, g, None,
                                              b["last_value"])
    if name == "vtrace_compact":
        dec = {k: _decode(b[k]) for k in _VTRACE_VALUES + ("terminateds", "truncateds")}
        return oracle.vtrace(dec["log_pi_target"], dec["log_pi_behavior"], dec["values"], dec["rewards"],
                             dec["terminateds"], dec["truncateds"], g, c["rho_bar"], c["c_bar"],
                             dec["bootstrap_values"])
    if name == "retrace_compact":
        dec = {k: _decode(b[k]) for k in _RETRACE_VALUES + ("terminateds",)}
        return oracle.retrace(dec["pi_taken"], dec["mu_taken"], dec["q_values"], dec["expected_next_q"],
                              dec["rewards"], dec["terminateds"], None, g, c["lambda_"], c["c_bar"],
                              c["rho_bar"])
    if name == "gae_masked":
        return oracle.gae_masked(b["rewards"], b["values"], b["terminateds"], b["mask"], None, g,
                                 c["lambda_"])
    if name == "gae_normalized":
        adv = oracle.gae(b["rewards"], b["values"], b["terminateds"], None, g, c["lambda_"], None,
                         b["last_value"])
        nv = np.zeros_like(b["values"])
        nv[:, :-1] = b["values"][:, 1:]
        nv[:, -1] = b["last_value"]
        return (oracle.normalize_advantages(adv, 1e-8)[0],
                oracle.lambda_returns(b["rewards"], nv, b["terminateds"], None, g, c["lambda_"],
                                      None, b["last_value"]))
    if name == "eligibility_traces":
        return oracle.eligibility_traces(b["gradients"], b["trace_dones"], g, c["lambda_"])
    if name == "episodic_prefix_sum":
        return oracle.episodic_prefix_sum(b["inputs"], b["prefix_dones"], None, "starts_at")
    raise KeyError(name)


def _slice(batch, r0, r1):
    out = {}
    for k, v in batch.items():
        if v is None:
            out[k] = None
        elif v.ndim == 2:
            out[k] = v[r0:r1]
        else:
            out[k] = v[r0:r1]
    return out


def oracle_time(wl_name, rows, threads, min_seconds=10.0, max_reps=10000, min_reps=3):
    """Time the oracle (as it is) on `rows` rows of the workload, rows split
    across `threads` host threads, for at least `min_reps` passes and
    `min_seconds`.  Returns the env-steps/s of the best pass and the
    description."""
    import oracle
    oracle.build()
    wl = WORKLOADS[wl_name]
    T = wl["T"]
    rows = min(rows, wl["N"])
    batch = wl["gen"](rows, T)
    chunks = [(i * rows // threads, (i + 1) * rows // threads) for i in range(threads)]
    chunks = [c for c in chunks if c[1] > c[0]]

    def one_pass():
        with concurrent.futures.ThreadPoolExecutor(max_workers=len(chunks)) as ex:
            futs = [ex.submit(lambda c: [_oracle_call(n, cfg, _slice(batch, *c))
                                         for (n, _, cfg) in wl["estimators"]], c) for c in chunks]
            for f in futs:
                f.result()
    one_pass()  # warm (page in, build)
    reps, t0, best = 0, time.perf_counter(), float("inf")
    while True:
        p0 = time.perf_counter()
        one_pass()
        best = min(best, time.perf_counter() - p0)
        reps += 1
        el = time.perf_counter() - t0
        if (el >= min_seconds and reps >= min_reps) or reps >= max_reps:
            break
    return rows * T / best, {"rows": rows, "seq_len": T, "passes": reps,
                             "seconds": round(el, 3)}


def _cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            txt = f.read()
        m = re.search(r"model name\s*:\s*(.+)", txt) or re.search(r"CPU part\s*:\s*(.+)", txt)
        return m.group(1).strip() if m else "unknown"
    except Exception:
        return "unknown"


def cpu_baseline(wl_name, seconds=8.0, one_core=True):
    """The oracle as it stands on the host cores, on a bounded sample of the
    workload (whole rows, every estimator of the workload)."""
    wl = WORKLOADS[wl_name]
    threads = os.cpu_count() or 1
    rows = min(wl["N"], max(threads, int(4_194_304 * 2 // wl["T"])))
    v, info = oracle_time(wl_name, rows, threads, min_seconds=seconds)
    out = {"value": v, "unit": "env-steps/s", "cores": threads, "kind": "oracle", "cpu": _cpu_model(),
           "sample": f"{info['rows']} of {wl['N']} rows x {info['seq_len']} steps, "
                     f"all estimators of the workload, best of {info['passes']} passes "
                     f"({info['seconds']} s), rows split over {threads} threads"}
    if one_core:
        rows1 = max(1, rows // threads)
        v1, info1 = oracle_time(wl_name, rows1, 1, min_seconds=seconds / 3)
        out["value_1core"] = v1
        out["sample"] += f"; 1-core figure: {info1['rows']} rows, best of {info1['passes']} passes"
    return out


def run_reference(args, wl_name):
    wl = WORKLOADS[wl_name]
    threads = os.cpu_count() or 1
    rows = min(wl["N"], max(threads, int(262_144 * 4 // wl["T"])))
    import oracle
    oracle.build()
    batch = wl["gen"](rows, wl["T"])
    chunks = [(i * rows // threads, (i + 1) * rows // threads) for i in range(threads)]
    chunks = [c for c in chunks if c[1] > c[0]]

    def step():
        with concurrent.futures.ThreadPoolExecutor(max_workers=len(chunks)) as ex:
            list(ex.map(lambda c: [_oracle_call(n, cfg, _slice(batch, *c))
                                   for (n, _, cfg) in wl["estimators"]], chunks))
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = (time.perf_counter() - t0) / args.steps
    v = rows * wl["T"] / el
    sample = (f"{rows} of {wl['N']} rows x {wl['T']} steps per step, all estimators, "
              f"rows split over {threads} threads")
    return {"impl": "reference", "metric": METRIC,
            "value": v, "unit": "env-steps/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": el * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl_name),
            "cpu_baseline": {"value": v, "unit": "env-steps/s", "cores": threads, "kind": "oracle",
                             "cpu": _cpu_model(), "sample": sample},
            "e2e": {"value": v, "unit": "env-steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200, help="steps per timed trial (headline)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--trials", type=int, default=5, help="timed trials of K steps each")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--suite", choices=["auto", "on", "off"], default="auto",
                    help="also measure the other workloads (auto: with the headline workload at N=1)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--capture-traffic", action="store_true",
                    help="run the fixed launch schedule of a DRAM-traffic capture (no timing)")
    ap.add_argument("--e2e-streams", type=int, default=E2E_STREAMS,
                    help="streams the end-to-end steps rotate over")
    ap.add_argument("--e2e-steps", type=int, default=0, help="end-to-end steps (0: --steps)")
    ap.add_argument("--e2e-mode", choices=["zerocopy", "copies"], default="copies",
                    help="end-to-end leg: kernels on the pinned host buffers, or explicit copies")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    args.trials = max(1, args.trials)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, args.workload)))
        return

    if args.capture_traffic:
        if rank == 0:
            print(json.dumps(capture_schedule(args, args.workload)))
        return

    suite = (args.suite == "on" or (args.suite == "auto" and args.workload == HEADLINE)) and world == 1
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    res = run_ours(args, args.workload, rank, world, local_rank, SUITE if suite else ())
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(args.workload)
            for sub, rec in res.get("workloads", {}).items():
                rec["cpu_baseline"] = cpu_baseline(sub, seconds=1.5, one_core=False)
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
