"""Seeded synthetic rollout buffers shaped like the pages' workloads.

This module draws random inputs and nothing else: it holds none of the
estimators' arithmetic.  The CUDA path (through the Python binding) and the
CPU oracle receive the very same arrays from here, bit for bit.

Every tensor has its own counter-based stream: numpy's Philox-4x64 generator
keyed by ``(seed, stream_id << 32 | tensor_id)``, so a tensor's values do not
depend on which other tensors were drawn, or in which order.

Recipes (num_envs x seq_len float32 buffers; the distributions follow the
workload descriptions of the rl-triton paper's benchmark regimes, Sec. 1 and
Sec. 7, and the caller-side conventions of the API reference):

* ``gae``       rewards, values ~ N(0,1); terminated ~ Bernoulli(p_term);
                truncated ~ Bernoulli(p_trunc) made exclusive with terminated;
                bootstrap_values ~ N(0,1) at truncated steps and at the last
                column when that step is not terminated, zero elsewhere; or a
                ``last_value`` [N] ~ N(0,1) when there are no truncations.
* ``returns``   the GAE recipe plus ``next_values``: values shifted one step
                left, the last column taken from the bootstrap (last_value or
                bootstrap_values[:, -1]), zeroed at truncated steps as the
                TD(lambda) API asks of its caller.
* ``vtrace``    rewards, values ~ N(0,1); log_pi_behavior ~ N(0,1);
                log_pi_target = log_pi_behavior + N(0, 0.5^2).
* ``retrace``   rewards, Q(s_t,a_t), E_pi[Q(s_{t+1},.)] ~ N(0,1);
                mu(a_t|s_t) ~ U(0.05, 1); pi(a_t|s_t) = mu * exp(N(0, 0.5^2)).
* ``retrace_actions``  the full action-space form of the retrace recipe with
                A actions (4 on the pages' Retrace benchmarks): target
                probabilities softmax(z), z ~ N(0,1)^A per step; behaviour
                probabilities softmax(z + N(0, 0.5^2)^A); the taken action
                drawn from the behaviour probabilities (inverse CDF of a
                uniform draw) as int64; action_probs_behavior = the behaviour
                probability of that action; Q(s_t,a_t), Q(s_{t+1},a) for
                every a, rewards ~ N(0,1); flags as for ``retrace``.
* ``llm_tokens``  token-level rollouts of an LLM policy, one response per
                row: a masked prompt of U[64, 512) tokens, a response whose
                length is U[T/4, T - prompt] tokens in which tool-call
                observations (masked) start with probability 1/256 per token
                and last U[16, 128) tokens, then masked padding; values
                ~ N(0,1) on response tokens (0 elsewhere); the outcome
                reward ~ N(0,1) on the last response token, which is also
                terminated; mask = 1 on the policy's response tokens.
* ``long_rows`` episode starts F ~ Bernoulli(p_start); prefix-sum inputs are
                integers uniform in [0, 9] stored as float32 with
                dones = F ("starts_at"); eligibility-trace dones mark the step
                before each start (dones[t] = F[t+1], dones[T-1] = 0) and
                gradients ~ N(0,1).
"""
from __future__ import annotations

import numpy as np

_TENSOR_IDS = {
    "rewards": 1, "values": 2, "terminateds": 3, "truncateds": 4,
    "bootstrap_values": 5, "last_value": 6, "log_pi_behavior": 7,
    "log_ratio": 8, "q_values": 9, "expected_next_q": 10, "mu_taken": 11,
    "pi_log_ratio": 12, "episode_starts": 13, "inputs": 14, "gradients": 15,
    "alpha": 16, "beta": 17, "carry": 18, "seed_values": 19, "beta_zero": 20,
    "action_logits": 21, "next_q_all": 22, "actions": 23, "behavior_logit_noise": 24,
    "prompt_len": 25, "response_len": 26, "obs_starts": 27, "obs_len": 28, "outcome": 29,
}

# The five workloads used by the tests and the benchmark, by name.  Shapes
# and distribution parameters are those of the benchmark regimes the
# rl-triton paper describes (massively parallel short rollouts through
# 1M-step rows); `stream` is the workload's component of the generator key.
WORKLOADS = {
    "gae_8x128": dict(stream=0, N=8, T=128, kind="gae", p_term=0.01, p_trunc=0.005,
                      bootstrap="2d", gamma=0.99, lambda_=0.95),
    "gae_returns_4096x1024": dict(stream=1, N=4096, T=1024, kind="returns", p_term=0.01,
                                  p_trunc=0.0, bootstrap="last", gamma=0.99, lambda_=0.95),
    "vtrace_2048x4096": dict(stream=2, N=2048, T=4096, kind="vtrace", p_term=0.002,
                             p_trunc=0.001, bootstrap="2d", gamma=0.99, rho_bar=1.0, c_bar=1.0),
    "retrace_1024x16384": dict(stream=3, N=1024, T=16384, kind="retrace", p_term=0.001,
                               p_trunc=0.0, gamma=0.99, lambda_=0.95, c_bar=1.0, rho_bar=1.0),
    "long_rows_64x1048576": dict(stream=4, N=64, T=1 << 20, kind="long_rows", p_start=1e-4,
                                 gamma=0.99, lambda_=0.9),
}


def stream(seed: int, stream_id: int, name: str) -> np.random.Generator:
    """Independent Philox stream for one named tensor of one workload."""
    tid = _TENSOR_IDS[name]
    key = np.array([seed & 0xFFFFFFFFFFFFFFFF,
                    ((stream_id & 0xFFFFFFFF) << 32) | (tid & 0xFFFFFFFF)], dtype=np.uint64)
    return np.random.Generator(np.random.Philox(key=key))


def normal(seed, stream_id, name, shape, std=1.0):
    x = stream(seed, stream_id, name).standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def bernoulli(seed, stream_id, name, shape, p):
    u = stream(seed, stream_id, name).random(shape, dtype=np.float32)
    return (u < np.float32(p)).astype(np.float32)


def uniform(seed, stream_id, name, shape, lo, hi):
    u = stream(seed, stream_id, name).random(shape, dtype=np.float32)
    return (np.float32(lo) + u * np.float32(hi - lo)).astype(np.float32)


def uniform_int(seed, stream_id, name, shape, lo, hi):
    """Integers uniform in [lo, hi] inclusive, stored as float32."""
    return stream(seed, stream_id, name).integers(lo, hi + 1, shape).astype(np.float32)


def _flags(N, T, seed, cid, p_term, p_trunc):
    term = bernoulli(seed, cid, "terminateds", (N, T), p_term)
    trunc = None
    if p_trunc > 0:
        trunc = bernoulli(seed, cid, "truncateds", (N, T), p_trunc)
        trunc[term > 0] = 0.0          # the two flags are mutually exclusive
    return term, trunc


def _bootstrap(N, T, seed, cid, term, trunc, mode):
    """bootstrap_values nonzero exactly where the episode continues past the
    step: truncated steps and the last column when it is not terminated."""
    if mode == "2d":
        draw = normal(seed, cid, "bootstrap_values", (N, T))
        where = np.zeros((N, T), dtype=bool)
        if trunc is not None:
            where |= trunc > 0
        where[:, T - 1] |= term[:, T - 1] == 0
        return np.where(where, draw, np.float32(0)).astype(np.float32), None
    if mode == "last":
        return None, normal(seed, cid, "last_value", (N,))
    return None, None


def gae_batch(N, T, seed=0, stream_id=0, p_term=0.01, p_trunc=0.005, bootstrap="2d"):
    term, trunc = _flags(N, T, seed, stream_id, p_term, p_trunc)
    bs, last = _bootstrap(N, T, seed, stream_id, term, trunc, bootstrap)
    return dict(rewards=normal(seed, stream_id, "rewards", (N, T)),
                values=normal(seed, stream_id, "values", (N, T)),
                terminateds=term, truncateds=trunc, bootstrap_values=bs, last_value=last)


def returns_batch(N, T, seed=0, stream_id=1, p_term=0.01, p_trunc=0.0, bootstrap="last"):
    """GAE inputs plus the TD(lambda) caller-side ``next_values``."""
    b = gae_batch(N, T, seed, stream_id, p_term, p_trunc, bootstrap)
    nv = np.empty((N, T), dtype=np.float32)
    nv[:, :-1] = b["values"][:, 1:]
    if b["last_value"] is not None:
        nv[:, -1] = b["last_value"]
    elif b["bootstrap_values"] is not None:
        nv[:, -1] = b["bootstrap_values"][:, -1]
    else:
        nv[:, -1] = 0.0
    if b["truncateds"] is not None:
        nv[b["truncateds"] > 0] = 0.0
    b["next_values"] = nv
    return b


def vtrace_batch(N, T, seed=0, stream_id=2, p_term=0.002, p_trunc=0.001, bootstrap="2d"):
    b = gae_batch(N, T, seed, stream_id, p_term, p_trunc, bootstrap)
    lpb = normal(seed, stream_id, "log_pi_behavior", (N, T))
    lpt = (lpb + normal(seed, stream_id, "log_ratio", (N, T), std=0.5)).astype(np.float32)
    b.update(log_pi_target=lpt, log_pi_behavior=lpb)
    return b


def retrace_batch(N, T, seed=0, stream_id=3, p_term=0.001, p_trunc=0.0):
    term, trunc = _flags(N, T, seed, stream_id, p_term, p_trunc)
    mu = uniform(seed, stream_id, "mu_taken", (N, T), 0.05, 1.0)
    eps = normal(seed, stream_id, "pi_log_ratio", (N, T), std=0.5)
    pi = (mu * np.exp(eps)).astype(np.float32)
    return dict(pi_taken=pi, mu_taken=mu,
                q_values=normal(seed, stream_id, "q_values", (N, T)),
                expected_next_q=normal(seed, stream_id, "expected_next_q", (N, T)),
                rewards=normal(seed, stream_id, "rewards", (N, T)),
                terminateds=term, truncateds=trunc)


def _softmax(z):
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)


def retrace_actions_batch(N, T, A=4, seed=0, stream_id=3, p_term=0.001, p_trunc=0.0):
    term, trunc = _flags(N, T, seed, stream_id, p_term, p_trunc)
    z = normal(seed, stream_id, "action_logits", (N, T, A))
    target = _softmax(z)
    z += normal(seed, stream_id, "behavior_logit_noise", (N, T, A), std=0.5)
    behavior = _softmax(z)
    del z
    u = stream(seed, stream_id, "actions").random((N, T), dtype=np.float32)
    cdf = np.cumsum(behavior, axis=-1)
    actions = np.minimum((u[..., None] >= cdf).sum(axis=-1), A - 1).astype(np.int64)
    del cdf
    mu = np.take_along_axis(behavior, actions[..., None], axis=-1)[..., 0]
    del behavior
    return dict(action_probs_target=target, action_probs_behavior=np.ascontiguousarray(mu),
                q_values=normal(seed, stream_id, "q_values", (N, T)),
                next_q_values_all=normal(seed, stream_id, "next_q_all", (N, T, A)),
                actions=actions,
                rewards=normal(seed, stream_id, "rewards", (N, T)),
                terminateds=term, truncateds=trunc)


def llm_tokens_batch(N, T, seed=0, stream_id=6):
    prompt = stream(seed, stream_id, "prompt_len").integers(64, 512, N)
    prompt = np.minimum(prompt, T // 2)
    lo = np.maximum(1, T // 4)
    resp = stream(seed, stream_id, "response_len").integers(0, 1 << 30, N)
    resp = lo + resp % np.maximum(1, T - prompt - lo + 1)
    end = np.minimum(prompt + resp, T)                     # first padding token
    t = np.arange(T)[None, :]
    response = (t >= prompt[:, None]) & (t < end[:, None])
    obs = np.zeros((N, T), dtype=bool)
    starts = stream(seed, stream_id, "obs_starts").random((N, T), dtype=np.float32) < 1.0 / 256
    lens = stream(seed, stream_id, "obs_len").integers(16, 128, (N, T))
    rows, cols = np.nonzero(starts & response)
    for r, c in zip(rows, cols):
        obs[r, c:c + lens[r, c]] = True
    mask = (response & ~obs).astype(np.float32)
    values = np.where(response, normal(seed, stream_id, "values", (N, T)), np.float32(0))
    rewards = np.zeros((N, T), np.float32)
    term = np.zeros((N, T), np.float32)
    last = np.maximum(end - 1, 0)
    outcome = normal(seed, stream_id, "outcome", (N,))
    rewards[np.arange(N), last] = outcome
    term[np.arange(N), last] = 1.0
    return dict(rewards=rewards, values=values.astype(np.float32), terminateds=term, mask=mask)


def compact(batch, values=("rewards", "values", "bootstrap_values"),
            flags=("terminateds", "truncateds")):
    """The same batch in compact storage: the named value arrays as the raw
    bits of bfloat16 (uint16, rounded to nearest even by torch), the flags
    as uint8; other arrays unchanged."""
    import torch
    out = {}
    for k, v in batch.items():
        if v is None:
            out[k] = None
        elif k in values:
            out[k] = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        elif k in flags:
            out[k] = v.astype(np.uint8)
        else:
            out[k] = v
    return out


def long_rows_batch(N, T, seed=0, stream_id=4, p_start=1e-4):
    starts = bernoulli(seed, stream_id, "episode_starts", (N, T), p_start)
    ends = np.zeros_like(starts)
    ends[:, :-1] = starts[:, 1:]
    return dict(inputs=uniform_int(seed, stream_id, "inputs", (N, T), 0, 9),
                prefix_dones=starts,
                gradients=normal(seed, stream_id, "gradients", (N, T)),
                trace_dones=ends)


def linear_scan_batch(N, T, seed=0, stream_id=5, p_zero=0.01, with_carry=True):
    """alpha ~ N(0,1); beta ~ U(0,1) with a fraction p_zero set to 0; carry ~ N(0,1)."""
    beta = uniform(seed, stream_id, "beta", (N, T), 0.0, 1.0)
    if p_zero > 0:
        beta[bernoulli(seed, stream_id, "beta_zero", (N, T), p_zero) > 0] = 0.0
    return dict(alpha=normal(seed, stream_id, "alpha", (N, T)), beta=beta,
                carry=normal(seed, stream_id, "carry", (N,)) if with_carry else None)


def workload_batch(name, seed=0, N=None, T=None):
    """Inputs of one of the five named workloads (optionally at a smaller shape)."""
    c = WORKLOADS[name]
    sid = c["stream"]
    N = c["N"] if N is None else N
    T = c["T"] if T is None else T
    kind = c["kind"]
    if kind == "gae":
        return gae_batch(N, T, seed, sid, c["p_term"], c["p_trunc"], c["bootstrap"])
    if kind == "returns":
        return returns_batch(N, T, seed, sid, c["p_term"], c["p_trunc"], c["bootstrap"])
    if kind == "vtrace":
        return vtrace_batch(N, T, seed, sid, c["p_term"], c["p_trunc"], c["bootstrap"])
    if kind == "retrace":
        return retrace_batch(N, T, seed, sid, c["p_term"], c["p_trunc"])
    if kind == "long_rows":
        return long_rows_batch(N, T, seed, sid, c["p_start"])
    raise KeyError(kind)
