"""Throughput benchmark: env-steps/s and achieved HBM GB/s per estimator.

Default workload (N=1): GAE + discounted returns + TD(lambda) returns on a
4096 x 1024 float32 rollout buffer with a last_value bootstrap (one "step"
= the three estimators over one batch).  Other workloads: --workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload gae_returns_4096x1024|...]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own batch
(rows are independent: weak scaling, no collective on the data path); the
time is the max over ranks.
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
    """DRAM bytes per launch that an ncu capture recorded for this kernel and
    workload (profiles/traffic.md, a fenced JSON block), if the capture was
    taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    try:
        with open(path) as f:
            text = f.read()
        rec = json.loads(text.split("```json", 1)[1].split("```", 1)[0])
    except Exception:
        return None
    e = rec.get(f"{kernel}@{workload}")
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


def run_ours(args, wl_name, rank, world, local_rank):
    import torch
    from linear_recurrence_scan_gb300 import _native, build
    build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = WORKLOADS[wl_name]
    N, T = wl["N"], wl["T"]
    batch = wl["gen"](N, T)
    names = [e[0] for e in wl["estimators"]]
    fused = wl.get("fused")
    # the step: one fused kernel when the workload has one, else each estimator
    step_kernels = [fused] if fused else list(wl["estimators"])
    all_kernels = step_kernels + ([e for e in wl["estimators"]] if fused else [])
    need_in = sorted({k for (n, _, _) in all_kernels for k in IO[n][0] + IO[n][1]})
    host = {k: batch[k] for k in need_in}
    set_bytes = sum(v.nbytes for v in host.values()) + sum(
        IO[n][2] * N * T * OUT_BYTES.get(n, 4) for (n, _, _) in step_kernels)
    n_sets = 1 if set_bytes > 4 * L2_BYTES else min(16, max(2, math.ceil(4 * L2_BYTES / set_bytes)))
    stream = torch.cuda.current_stream(dev)
    sh = ctypes.c_void_p(stream.cuda_stream)
    lib = _native.lib()
    wsn = max(lib.rlscan_workspace_bytes(N, T), lib.rlscan_gae_normalized_workspace_bytes(N, T))
    ws = None
    if wsn:
        ws_t = torch.empty(wsn, dtype=torch.uint8, device=dev)
        _native.check(lib.rlscan_workspace_init(ctypes.c_void_p(ws_t.data_ptr()), wsn, sh), "init")
        ws = ctypes.c_void_p(ws_t.data_ptr())
    sets = []
    keep = []  # every set's tensors stay allocated: the launchers hold raw pointers
    for _ in range(n_sets):
        bufs = {k: torch.from_numpy(v).to(dev) for k, v in host.items()}
        keep.append(bufs)
        calls = {}
        for (name, bps, c) in all_kernels:
            odt = torch.bfloat16 if OUT_DTYPE.get(name) == "bf16" else torch.float32
            outs = [torch.empty((N, T), dtype=odt, device=dev) for _ in range(IO[name][2])]
            keep.append(outs)
            calls[name] = _launcher(name, c, bufs, outs, N, T, ws, wsn, sh)
        sets.append(calls)
    ptrs = [t.data_ptr() for group in keep for t in (group.values() if isinstance(group, dict) else group)]
    assert len(ptrs) == len(set(ptrs)), "input sets must not share memory"
    torch.cuda.synchronize()

    def run(kernels, i):
        calls = sets[i % n_sets]
        for (name, _, _) in kernels:
            st = calls[name]()
            if st != 0:
                raise _native.RlscanError(st, name)

    def region(kernels, K, offset):
        """K steps of `kernels` back to back on the stream, one CUDA event
        pair around the whole region (none between launches, which would
        serialise them); barrier + synchronize on both sides.  Returns ms
        per step and the host wall time of the region."""
        t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        t0e.record(stream)
        for i in range(K):
            run(kernels, offset + i)
        t1e.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        return t0e.elapsed_time(t1e) / K, wall

    def launch_durations(kernels, K):
        """Average device duration of each kernel: K launches of that kernel
        alone, back to back, timed as one region, three times."""
        out = {}
        for e in kernels:
            out[e[0]] = [region([e], K, args.warmup + r * K)[0] for r in range(3)]
        return out

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    for i in range(args.warmup):
        run(step_kernels, i)
    torch.cuda.synchronize()
    K = args.steps
    ms_step, wall = region(step_kernels, K, args.warmup)
    ms_step = max_over_ranks(ms_step)
    # per-launch durations of the step's kernels (the step itself when it is one kernel)
    per_kernel = ({step_kernels[0][0]: [ms_step]} if len(step_kernels) == 1
                  else launch_durations(step_kernels, K))
    per_est_times = per_kernel
    if fused:  # the estimators one kernel each, for the per-estimator figures
        for i in range(args.warmup):
            run(wl["estimators"], i)
        per_est_times = launch_durations(wl["estimators"], K)

    # e2e through the public API: pinned host inputs -> device, the step's
    # call(s), results back to pinned host memory, every step.  Consecutive
    # steps go to E2E_STREAMS streams in turn (each with its own device and
    # host buffers), so one step's upload, another's compute and a third's
    # download overlap, as a pipeline of rollout batches would run.
    e2e_in = sorted({k for (n, _, _) in step_kernels for k in IO[n][0] + IO[n][1]})
    pinned = {k: torch.from_numpy(host[k]).pin_memory() for k in e2e_in}
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
    e0 = time.perf_counter()
    for i in range(K):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks((time.perf_counter() - e0) / K)
    clocks = sampler.stop()

    steps_per_call = N * T
    peak, peak_kind = _measured_peak()

    def kernel_stats(name, bps, ts):
        ts = np.array(ts)
        avg_us = float(ts.mean() * 1e3)
        gbs = bps * steps_per_call / (avg_us * 1e-6) / 1e9
        return {"us_mean": round(avg_us, 2), "us_median": round(float(np.median(ts)) * 1e3, 2),
                "env_steps_per_s": steps_per_call / (avg_us * 1e-6), "bytes_per_env_step": bps,
                "gb_per_s": round(gbs, 1), "frac_of_measured_hbm": round(gbs / peak, 4),
                "frac_of_nominal_8tbs": round(gbs / 8000.0, 4)}
    per_est = {n: kernel_stats(n, bps, per_est_times[n]) for (n, bps, _) in wl["estimators"]}
    step_stats = {n: kernel_stats(n, bps, per_kernel[n]) for (n, bps, _) in step_kernels}
    dominant = max(step_kernels, key=lambda e: sum(per_kernel[e[0]]))[0]
    d = step_stats[dominant]
    result = {
        "metric": "env-steps/sec and achieved HBM GB/s (% of GB300 peak) per estimator, 1 GPU",
        "value": world * steps_per_call / (ms_step * 1e-3),
        "unit": "env-steps/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if not any(n.endswith("_compact") for n in names) else
                 "f32 arithmetic on bf16 values / u8 flags", "data": "synthetic",
        "config": {"workload": wl_name, "description": wl["desc"], "num_envs": N, "seq_len": T,
                   "estimators": names,
                   "step_kernels": [n for (n, _, _) in step_kernels],
                   "parallelism": f"rows, {world} independent batch(es)",
                   "l2": f"{n_sets} rotating input sets of {set_bytes / 1e6:.0f} MB "
                         f"({n_sets * set_bytes / 1e6:.0f} MB > 129 MB L2)"},
        "step": step_stats,
        "per_estimator": per_est,
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": d["gb_per_s"], "peak": peak,
                     "peak_source": peak_kind, "unit": "GB/s", "frac": d["frac_of_measured_hbm"],
                     "traffic": _ncu_traffic(dominant, wl_name),
                     "algorithmic_bytes_per_launch": d["bytes_per_env_step"] * steps_per_call},
        "e2e": {"value": world * steps_per_call / e2e_s, "unit": "env-steps/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "path": ("public compute_* API on pinned host tensors: the kernel reads the inputs "
                         "and writes the pinned outputs over the host link (zero copy)"
                         if zero_copy else
                         "pinned host -> device copies, public compute_* API, results -> pinned host")
                        + f"; steps round-robin over {NS} streams"},
        "gpu_launches": K * sum(LAUNCHES.get(n, 1) for (n, _, _) in step_kernels),
        "full_call_us": round(wall / K * 1e6, 2),
        "timing": "CUDA events around K back-to-back steps (no events between launches); "
                  "per-kernel durations from K back-to-back launches of that kernel alone; "
                  "full_call_us: host wall time of the timed region per step",
        "wall_s_timed": round(wall, 4),
        "clocks": clocks,
    }
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


def cpu_baseline(wl_name):
    wl = WORKLOADS[wl_name]
    threads = os.cpu_count() or 1
    rows = min(wl["N"], max(threads, int(4_194_304 * 2 // wl["T"])))
    v, info = oracle_time(wl_name, rows, threads, min_seconds=8.0)
    rows1 = max(1, rows // threads)
    v1, info1 = oracle_time(wl_name, rows1, 1, min_seconds=3.0)
    return {"value": v, "unit": "env-steps/s", "cores": threads, "kind": "oracle",
            "cpu": _cpu_model(), "value_1core": v1,
            "sample": f"{info['rows']} of {wl['N']} rows x {info['seq_len']} steps, "
                      f"all estimators of the step, best of {info['passes']} passes "
                      f"({info['seconds']} s), rows split over {threads} threads; 1-core figure: "
                      f"{info1['rows']} rows, best of {info1['passes']} passes"}


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
    return {"impl": "reference",
            "metric": "env-steps/sec and achieved HBM GB/s (% of GB300 peak) per estimator, 1 GPU",
            "value": v, "unit": "env-steps/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": el * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl_name, "description": wl["desc"], "num_envs": wl["N"],
                       "seq_len": wl["T"], "estimators": [e[0] for e in wl["estimators"]]},
            "cpu_baseline": {"value": v, "unit": "env-steps/s", "cores": threads, "kind": "oracle",
                             "cpu": _cpu_model(), "sample": sample},
            "e2e": {"value": v, "unit": "env-steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gae_returns_4096x1024", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-streams", type=int, default=E2E_STREAMS,
                    help="streams the end-to-end steps rotate over")
    ap.add_argument("--e2e-mode", choices=["zerocopy", "copies"], default="copies",
                    help="end-to-end leg: kernels on the pinned host buffers, or explicit copies")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, args.workload)))
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    res = run_ours(args, args.workload, rank, world, local_rank)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(args.workload)
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
