"""Plain float64 CPU oracle for the RL credit-assignment recurrences.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product (``linear_recurrence_scan_gb300``) never imports, links or executes
anything here, and nothing here imports the product: the two sides share no
code.  Inputs are numpy float32 arrays; outputs are numpy float64 arrays.

The arithmetic lives in ``rlscan_oracle.c`` (one sequential loop per
recurrence, each citing the page passage it writes out).  This module only
compiles that file with the host C compiler and marshals numpy arrays.

Parity of every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (brute-force summation, the pages' closed forms
and worked polynomials, the boundary-summary tables, and cross-estimator
identities).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rlscan_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

_default = None
_lock = threading.Lock()


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile an oracle source into a shared library with the host gcc.

    ``-ffp-contract=off`` keeps every multiply and add separately rounded, so
    the oracle gives the same bits on x86-64 and AArch64 hosts.  ``src`` and
    ``out`` let the pin tests build a deliberately broken copy in a temporary
    directory (mutation check); the default builds ``oracle/_build``.
    """
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-Wall", "-Wextra", "-shared", "-fPIC", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


_I64 = ctypes.c_int64
_D = ctypes.c_double
_P = ctypes.c_void_p

_SIGNATURES = {
    "oracle_gae": [_I64] * 5 + [_P] * 6 + [_D, _D, _P],
    "oracle_gae_masked": [_I64] * 5 + [_P] * 7 + [_D, _D, _P],
    "oracle_vtrace": [_I64] * 5 + [_P] * 8 + [_D, _D, _D, _P, _P],
    "oracle_retrace": [_I64] * 5 + [_P] * 7 + [_D, _D, _D, _D, _P, _P],
    "oracle_retrace_actions": [_I64] * 6 + [_P] * 8 + [_D, _D, _D, _D, _P, _P],
    "oracle_lambda_returns": [_I64] * 5 + [_P] * 6 + [_D, _D, _P],
    "oracle_discounted_returns": [_I64] * 5 + [_P] * 5 + [_D, _P],
    "oracle_eligibility_traces": [_I64] * 5 + [_P] * 3 + [_D, _D, _P],
    "oracle_episodic_prefix_sum": [_I64] * 5 + [_P] * 3 + [ctypes.c_int, _P],
    "oracle_linear_scan": [_I64] * 5 + [_P] * 3 + [ctypes.c_int, _P],
}


class _Rows:
    """Validates the [N,T] inputs of one call and converts them to float32."""

    def __init__(self, ref):
        ref = np.asarray(ref)
        if ref.ndim != 2:
            raise ValueError("expected a [num_envs, seq_len] array")
        self.N, self.T = ref.shape
        self.keep = []

    def mat(self, a, name):
        if a is None:
            return None
        a = np.ascontiguousarray(a, dtype=np.float32)
        if a.shape != (self.N, self.T):
            raise ValueError(f"{name}: shape {a.shape} != {(self.N, self.T)}")
        self.keep.append(a)
        return a.ctypes.data

    def vec(self, a, name):
        if a is None:
            return None
        a = np.ascontiguousarray(a, dtype=np.float32)
        if a.shape != (self.N,):
            raise ValueError(f"{name}: shape {a.shape} != {(self.N,)}")
        self.keep.append(a)
        return a.ctypes.data

    def out(self):
        o = np.empty((self.N, self.T), dtype=np.float64)
        self.keep.append(o)
        return o

    def head(self, rows):
        b, e = (0, self.N) if rows is None else rows
        return [self.N, self.T, self.T, b, e]


class Oracle:
    """One loaded oracle library.  The module-level functions use the default
    build (``oracle/_build/liboracle.so``)."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        for name, argtypes in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = argtypes
            fn.restype = _I64 if name == "oracle_retrace_actions" else None
        self._lib = lib

    def gae(self, rewards, values, terminateds, truncateds=None, gamma=0.99, lambda_=0.95,
            bootstrap_values=None, last_value=None, rows=None):
        """GAE advantages (float64)."""
        c = _Rows(rewards)
        out = c.out()
        self._lib.oracle_gae(*c.head(rows), c.mat(rewards, "rewards"), c.mat(values, "values"),
                           c.mat(terminateds, "terminateds"), c.mat(truncateds, "truncateds"),
                           c.mat(bootstrap_values, "bootstrap_values"),
                           c.vec(last_value, "last_value"), gamma, lambda_, out.ctypes.data)
        return out

    def gae_masked(self, rewards, values, terminateds, mask, truncateds=None, gamma=0.99,
                   lambda_=0.95, bootstrap_values=None, last_value=None, rows=None):
        """GAE with observation-skip masking (float64): masked steps carry
        the next step's advantage unchanged."""
        c = _Rows(rewards)
        out = c.out()
        self._lib.oracle_gae_masked(*c.head(rows), c.mat(rewards, "rewards"),
                                    c.mat(values, "values"), c.mat(terminateds, "terminateds"),
                                    c.mat(truncateds, "truncateds"),
                                    c.mat(bootstrap_values, "bootstrap_values"),
                                    c.vec(last_value, "last_value"), c.mat(mask, "mask"), gamma,
                                    lambda_, out.ctypes.data)
        return out

    def vtrace(self, log_pi_target, log_pi_behavior, values, rewards, terminateds, truncateds=None,
               gamma=0.99, rho_bar=1.0, c_bar=1.0, bootstrap_values=None, last_value=None,
               rows=None):
        """V-trace targets and advantages (float64, float64)."""
        c = _Rows(rewards)
        vs, adv = c.out(), c.out()
        self._lib.oracle_vtrace(*c.head(rows), c.mat(log_pi_target, "log_pi_target"),
                              c.mat(log_pi_behavior, "log_pi_behavior"), c.mat(values, "values"),
                              c.mat(rewards, "rewards"), c.mat(terminateds, "terminateds"),
                              c.mat(truncateds, "truncateds"),
                              c.mat(bootstrap_values, "bootstrap_values"),
                              c.vec(last_value, "last_value"), gamma, rho_bar, c_bar,
                              vs.ctypes.data, adv.ctypes.data)
        return vs, adv

    def retrace(self, pi_taken, mu_taken, q_values, expected_next_q, rewards, terminateds,
                truncateds=None, gamma=0.99, lambda_=1.0, c_bar=1.0, rho_bar=1.0, rows=None):
        """Retrace(lambda) targets and advantages from per-step inputs (float64)."""
        c = _Rows(rewards)
        qret, adv = c.out(), c.out()
        self._lib.oracle_retrace(*c.head(rows), c.mat(pi_taken, "pi_taken"),
                               c.mat(mu_taken, "mu_taken"), c.mat(q_values, "q_values"),
                               c.mat(expected_next_q, "expected_next_q"), c.mat(rewards, "rewards"),
                               c.mat(terminateds, "terminateds"), c.mat(truncateds, "truncateds"),
                               gamma, lambda_, c_bar, rho_bar, qret.ctypes.data, adv.ctypes.data)
        return qret, adv

    def retrace_actions(self, action_probs_target, action_probs_behavior, q_values,
                        next_q_values_all, actions, rewards, terminateds, truncateds=None,
                        gamma=0.99, lambda_=1.0, c_bar=1.0, rho_bar=1.0, rows=None):
        """Retrace(lambda) targets and advantages from the full action-space
        inputs ([N,T,A] target probabilities and successor Q-values, int64
        actions), in the argument order of the API's compute_retrace."""
        c = _Rows(rewards)
        probs = np.ascontiguousarray(action_probs_target, dtype=np.float32)
        nq = np.ascontiguousarray(next_q_values_all, dtype=np.float32)
        if probs.ndim != 3 or probs.shape[:2] != (c.N, c.T) or nq.shape != probs.shape:
            raise ValueError("action_probs_target and next_q_values_all must be [N, T, A]")
        acts = np.asarray(actions)
        if acts.shape != (c.N, c.T) or acts.dtype.kind not in "iu":
            raise ValueError("actions must be an integer [N, T] array")
        acts = np.ascontiguousarray(acts, dtype=np.int64)
        c.keep += [probs, nq, acts]
        qret, adv = c.out(), c.out()
        head = c.head(rows)
        bad = self._lib.oracle_retrace_actions(
            head[0], head[1], probs.shape[2], head[2], head[3], head[4], probs.ctypes.data,
            c.mat(action_probs_behavior, "action_probs_behavior"), c.mat(q_values, "q_values"),
            nq.ctypes.data, acts.ctypes.data, c.mat(rewards, "rewards"),
            c.mat(terminateds, "terminateds"), c.mat(truncateds, "truncateds"),
            gamma, lambda_, c_bar, rho_bar, qret.ctypes.data, adv.ctypes.data)
        if bad:
            raise ValueError(f"{bad} action indices outside [0, {probs.shape[2]})")
        return qret, adv

    def lambda_returns(self, rewards, next_values, terminateds, truncateds=None, gamma=0.99,
                       lambda_=0.95, bootstrap_values=None, last_value=None, rows=None):
        """TD(lambda) returns (float64)."""
        c = _Rows(rewards)
        out = c.out()
        self._lib.oracle_lambda_returns(*c.head(rows), c.mat(rewards, "rewards"),
                                      c.mat(next_values, "next_values"),
                                      c.mat(terminateds, "terminateds"),
                                      c.mat(truncateds, "truncateds"),
                                      c.mat(bootstrap_values, "bootstrap_values"),
                                      c.vec(last_value, "last_value"), gamma, lambda_,
                                      out.ctypes.data)
        return out

    def discounted_returns(self, rewards, terminateds, truncateds=None, gamma=0.99,
                           bootstrap_values=None, last_value=None, rows=None):
        """Discounted returns (float64)."""
        c = _Rows(rewards)
        out = c.out()
        self._lib.oracle_discounted_returns(*c.head(rows), c.mat(rewards, "rewards"),
                                          c.mat(terminateds, "terminateds"),
                                          c.mat(truncateds, "truncateds"),
                                          c.mat(bootstrap_values, "bootstrap_values"),
                                          c.vec(last_value, "last_value"), gamma, out.ctypes.data)
        return out

    def eligibility_traces(self, gradients, dones, gamma, lambda_, seed_values=None, rows=None):
        """Forward eligibility traces (float64)."""
        c = _Rows(gradients)
        out = c.out()
        self._lib.oracle_eligibility_traces(*c.head(rows), c.mat(gradients, "gradients"),
                                          c.mat(dones, "dones"), c.vec(seed_values, "seed_values"),
                                          gamma, lambda_, out.ctypes.data)
        return out

    def episodic_prefix_sum(self, inputs, dones, seed_values=None, boundary="ends_at", rows=None):
        """Episodic prefix sum (float64); boundary is "ends_at" or "starts_at"."""
        if boundary not in ("ends_at", "starts_at"):
            raise ValueError(f"boundary must be 'ends_at' or 'starts_at', got {boundary!r}")
        c = _Rows(inputs)
        out = c.out()
        self._lib.oracle_episodic_prefix_sum(*c.head(rows), c.mat(inputs, "inputs"),
                                           c.mat(dones, "dones"), c.vec(seed_values, "seed_values"),
                                           0 if boundary == "ends_at" else 1, out.ctypes.data)
        return out

    def linear_scan(self, alpha, beta, carry=None, direction="backward", rows=None):
        """Generic affine recurrence A_t = alpha_t + beta_t A_{t-+1} (float64)."""
        if direction not in ("backward", "forward"):
            raise ValueError(f"direction must be 'backward' or 'forward', got {direction!r}")
        c = _Rows(alpha)
        out = c.out()
        self._lib.oracle_linear_scan(*c.head(rows), c.mat(alpha, "alpha"), c.mat(beta, "beta"),
                                   c.vec(carry, "carry"), 0 if direction == "backward" else 1,
                                   out.ctypes.data)
        return out


def normalize_advantages(advantages, eps=1e-8):
    """Per-batch whitening of advantages (rl-triton paper Sec. 9.3, "fused
    advantage normalization", read as (A - mean) / (std + eps) over all N*T
    values with the unbiased standard deviation).  Two passes in float64:
    the mean, then the sum of squared deviations.  Returns the normalised
    array and (mean, std)."""
    a = np.asarray(advantages, dtype=np.float64)
    n = a.size
    mean = a.sum() / n
    dev = a - mean
    std = np.sqrt((dev * dev).sum() / (n - 1)) if n > 1 else float("nan")
    return dev / (std + eps), (float(mean), float(std))


def default() -> Oracle:
    """The oracle built from ``oracle/rlscan_oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def gae(*args, **kwargs):
    return default().gae(*args, **kwargs)


def gae_masked(*args, **kwargs):
    return default().gae_masked(*args, **kwargs)


def vtrace(*args, **kwargs):
    return default().vtrace(*args, **kwargs)


def retrace(*args, **kwargs):
    return default().retrace(*args, **kwargs)


def retrace_actions(*args, **kwargs):
    return default().retrace_actions(*args, **kwargs)


def lambda_returns(*args, **kwargs):
    return default().lambda_returns(*args, **kwargs)


def discounted_returns(*args, **kwargs):
    return default().discounted_returns(*args, **kwargs)


def eligibility_traces(*args, **kwargs):
    return default().eligibility_traces(*args, **kwargs)


def episodic_prefix_sum(*args, **kwargs):
    return default().episodic_prefix_sum(*args, **kwargs)


def linear_scan(*args, **kwargs):
    return default().linear_scan(*args, **kwargs)
