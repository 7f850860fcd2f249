"""PyTorch-facing functions with the rl-triton API reference's names and
defaults.  Each one checks its arguments (residency, dtypes, shapes -- the
pages' always-on structural checks), allocates the outputs with torch, and
makes exactly one librlscan call on the current CUDA stream.  Tensors live
on the GPU, or in page-locked host memory, which the kernel reads and writes
in place over the host link (outputs are then page-locked host tensors,
ready once the stream has synchronised).  There is no CPU path: a missing
library or an ordinary CPU tensor raises.
"""
from __future__ import annotations

import collections
import ctypes
import threading

import torch

from . import _native

__all__ = [
    "compute_gae", "compute_gae_and_returns", "compute_gae_normalized", "compute_vtrace",
    "compute_retrace",
    "compute_retrace_from_probs", "compute_lambda_returns",
    "compute_discounted_returns", "compute_eligibility_traces", "compute_episodic_prefix_sum",
    "linear_scan", "workspace_status",
]


# ---------------------------------------------------------------------------
# marshalling helpers

def _vp(t):
    """Address of a tensor's data for a ctypes void* argument (None: NULL)."""
    return None if t is None else t.data_ptr()


def _check(name, t, shape, device=None, dtypes=(torch.float32,)):
    """CUDA tensors on `device`, or page-locked host tensors (the kernel then
    reads / writes them in place over the host link)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    cuda = t.is_cuda
    if not (cuda or t.is_pinned()):
        raise ValueError(f"{name} must be on CUDA or in page-locked (pinned) host memory")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: expected {' or '.join(str(d) for d in dtypes)}, got {t.dtype}")
    if t.shape != shape:
        raise ValueError(f"{name} shape {tuple(t.shape)} != {tuple(shape)}")
    if device is not None and cuda and t.get_device() != device.index:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _contiguous(t):
    """t with unit column stride and packed rows; a host copy stays
    page-locked (the kernel reads host tensors in place)."""
    c = t.contiguous()
    if c is not t and not c.is_cuda:
        c = c.pin_memory()
    return c


# Page-locked tensors a call reads or writes in place (its host arguments,
# outputs and copies) are referenced here until the stream has passed the
# call: torch's pinned-memory cache only tracks blocks used by its own
# copies, and could otherwise hand a block the caller has dropped to another
# tensor while the kernel still uses it.  (Device tensors need no such care:
# the caching allocator reuses them in stream order.)
_held_lock = threading.Lock()
_held = collections.deque()  # (event recorded after the call, tensors), in call order


def _release_finished():
    with _held_lock:
        while _held and _held[0][0].query():
            _held.popleft()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(device):
    """The current CUDA stream of `device` as an integer handle."""
    if _raw_stream is not None:
        return _raw_stream(device.index)
    return torch.cuda.current_stream(device).cuda_stream


class _Call:
    """Collects the [N,T] and [N] tensors of one call, finds a common row
    stride (making copies contiguous only when the strides differ), and
    allocates outputs with that stride."""

    def __init__(self, ref_name, ref, dtypes=(torch.float32,)):
        if not isinstance(ref, torch.Tensor) or ref.dim() != 2:
            raise ValueError(f"{ref_name} must be a [num_envs, seq_len] tensor")
        _check(ref_name, ref, ref.shape, dtypes=dtypes)
        self.N, self.T = ref.shape
        # pinned host inputs: outputs in pinned host memory too, the work on
        # the current CUDA device
        self.host = not ref.is_cuda
        self.device = (torch.device("cuda", torch.cuda.current_device()) if self.host
                       else ref.device)
        self.shape = ref.shape
        self.mats = {ref_name: ref}
        self.vecs = {}
        self.outs = []
        self.extra = []  # other tensors the call uses in place (wide inputs, actions)
        self.any_host = self.host

    def contiguous(self, t):
        return _contiguous(t)

    def keep(self, *ts):
        for t in ts:
            if t is not None:
                self.extra.append(t)
                self.any_host = self.any_host or not t.is_cuda

    def mat(self, name, t, required=True, dtypes=(torch.float32,)):
        if t is None:
            if required:
                raise ValueError(f"{name} is required")
            return
        _check(name, t, self.shape, self.device, dtypes)
        self.mats[name] = t
        self.any_host = self.any_host or not t.is_cuda

    def vec(self, name, t):
        if t is None:
            return
        _check(name, t, (self.N,), self.device)
        self.vecs[name] = self.contiguous(t)
        self.any_host = self.any_host or not t.is_cuda

    def finish(self, n_out, dtype=torch.float32):
        mats = self.mats.values()
        if all(t.is_contiguous() for t in mats):
            self.rs = self.T
        else:
            strides = {t.stride(0) if self.N > 1 else max(self.T, 1) for t in mats}
            ok = all(self.T <= 1 or t.stride(1) == 1 for t in mats) and len(strides) == 1
            rs = strides.pop() if ok else self.T
            if not ok or rs < self.T:
                self.mats = {k: self.contiguous(t) for k, t in self.mats.items()}
                rs = self.T
            self.rs = max(rs, self.T)
        where = dict(device="cpu", pin_memory=True) if self.host else dict(device=self.device)
        if self.rs == self.T:
            outs = [torch.empty((self.N, self.T), dtype=dtype, **where) for _ in range(n_out)]
        else:
            outs = [torch.empty_strided((self.N, self.T), (self.rs, 1), dtype=dtype, **where)
                    for _ in range(n_out)]
        self.outs = outs
        return outs

    def m(self, name):
        return _vp(self.mats.get(name))

    def v(self, name):
        return _vp(self.vecs.get(name))

    def stream(self):
        return _stream_handle(self.device)

    def launched(self, status, what):
        """Raise on an error status; otherwise keep the page-locked tensors
        of this call until the stream has passed it."""
        _native.check(status, what)
        if not (self.any_host or _held) or torch.cuda.is_current_stream_capturing():
            return  # a captured graph replays on memory its owner keeps alive
        if self.any_host:
            host = [t for t in (*self.mats.values(), *self.vecs.values(), *self.outs, *self.extra)
                    if not t.is_cuda]
            if host:
                ev = torch.cuda.Event()
                ev.record(torch.cuda.current_stream(self.device))
                with _held_lock:
                    _held.append((ev, host))
        if _held:
            _release_finished()


_ws_lock = threading.Lock()
_ws_cache = {}
_ws_bytes_cache = {}


def _workspace(device, stream_handle, nbytes):
    """A zero-initialised workspace for (device, stream), grown on demand.
    Calls on one stream are ordered, so they may share a workspace."""
    if nbytes == 0:
        return None, 0
    key = (device.index, stream_handle)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        with _ws_lock:
            ws = _ws_cache.get(key)
            if ws is None or ws.numel() < nbytes:
                size = max(nbytes, 0 if ws is None else 2 * ws.numel())
                size = (size + 255) // 256 * 256
                ws = torch.empty(size, dtype=torch.uint8, device=device)
                _native.check(_native.lib().rlscan_workspace_init(_vp(ws), size, stream_handle),
                              "rlscan_workspace_init")
                _ws_cache[key] = ws
    return ws.data_ptr(), ws.numel()


def _workspace_bytes(N, T):
    key = (N, T)
    n = _ws_bytes_cache.get(key)
    if n is None:
        n = _native.lib().rlscan_workspace_bytes(N, T)
        if len(_ws_bytes_cache) > 4096:
            _ws_bytes_cache.clear()
        _ws_bytes_cache[key] = n
    return n


def _ws_for(c):
    s = c.stream()
    p, n = _workspace(c.device, s, _workspace_bytes(c.N, c.T))
    return p, n, s


def workspace_status(device=None):
    """Synchronise the current stream and raise if a kernel recorded an
    error (a cross-block wait that timed out) in its workspace."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    s = _stream_handle(device)
    ws = _ws_cache.get((device.index, s))
    if ws is None:
        torch.cuda.current_stream(device).synchronize()
        return
    _native.check(_native.lib().rlscan_workspace_status(_vp(ws), ws.numel(), s),
                  "rlscan_workspace_status")


# ---------------------------------------------------------------------------
# estimators (rl-triton API reference signatures)

_BF16 = (torch.bfloat16,)
_FLAG8 = (torch.uint8, torch.bool)
_OUT_DTYPES = {torch.float32: 0, torch.bfloat16: 1}


def _compact_call(rewards, values, terminateds, truncateds, bootstrap_values, last_value, n_out,
                  out_dtype):
    """Arguments of the compact-storage entry points: bf16 values, uint8 /
    bool flags, float32 last_value; outputs of ``out_dtype``."""
    if out_dtype not in _OUT_DTYPES:
        raise ValueError("out_dtype must be torch.float32 or torch.bfloat16")
    c = _Call("rewards", rewards, _BF16)
    c.mat("values", values, dtypes=_BF16)
    c.mat("terminateds", terminateds, dtypes=_FLAG8)
    c.mat("truncateds", truncateds, False, _FLAG8)
    c.mat("bootstrap_values", bootstrap_values, False, _BF16)
    c.vec("last_value", last_value)
    if last_value is not None and bootstrap_values is not None:
        raise ValueError("pass either last_value or bootstrap_values, not both")
    if last_value is not None and truncateds is not None:
        raise ValueError("last_value cannot be combined with truncateds; use bootstrap_values")
    if bootstrap_values is not None and truncateds is None:
        raise ValueError("compact storage: the window bootstrap is last_value (float32 [N])")
    outs = c.finish(n_out, out_dtype)
    return c, outs


def compute_gae(rewards, values, terminateds, truncateds=None, gamma=0.99, lambda_=0.95,
                bootstrap_values=None, last_value=None, mask=None, out_dtype=None):
    """GAE advantages [num_envs, seq_len] (rl-triton API reference, compute_gae).
    ``mask`` (an addition, float 0/1 [num_envs, seq_len]) selects
    observation-skip masking: masked steps carry the next step's advantage
    unchanged (beta = 1), unmasked steps are plain GAE steps.
    bfloat16 rewards select compact storage: values and bootstrap_values
    bfloat16, flags uint8 or bool, last_value float32; ``out_dtype``
    (float32 by default, or bfloat16) sets the output type."""
    if isinstance(rewards, torch.Tensor) and rewards.dtype == torch.bfloat16:
        if mask is not None:
            raise ValueError("mask is not available with compact storage")
        c, (out,) = _compact_call(rewards, values, terminateds, truncateds, bootstrap_values,
                                  last_value, 1, out_dtype or torch.float32)
        ws, wsn, s = _ws_for(c)
        c.launched(_native.lib().rlscan_gae_compact(
            c.m("rewards"), c.m("values"), c.m("terminateds"), c.m("truncateds"),
            c.m("bootstrap_values"), c.v("last_value"), c.N, c.T, c.rs, float(gamma),
            float(lambda_), _OUT_DTYPES[out_dtype or torch.float32], _vp(out), ws, wsn, s),
            "rlscan_gae_compact")
        return out
    c = _Call("rewards", rewards)
    c.mat("values", values)
    c.mat("terminateds", terminateds)
    c.mat("truncateds", truncateds, False)
    c.mat("bootstrap_values", bootstrap_values, False)
    c.mat("mask", mask, False)
    c.vec("last_value", last_value)
    if last_value is not None and bootstrap_values is not None:
        raise ValueError("pass either last_value or bootstrap_values, not both")
    if last_value is not None and truncateds is not None:
        raise ValueError("last_value cannot be combined with truncateds; use bootstrap_values")
    (out,) = c.finish(1)
    ws, wsn, s = _ws_for(c)
    if mask is not None:
        c.launched(_native.lib().rlscan_gae_masked(
            c.m("rewards"), c.m("values"), c.m("terminateds"), c.m("truncateds"),
            c.m("bootstrap_values"), c.v("last_value"), c.m("mask"), c.N, c.T, c.rs,
            float(gamma), float(lambda_), _vp(out), ws, wsn, s), "rlscan_gae_masked")
        return out
    c.launched(_native.lib().rlscan_gae(
        c.m("rewards"), c.m("values"), c.m("terminateds"), c.m("truncateds"),
        c.m("bootstrap_values"), c.v("last_value"), c.N, c.T, c.rs, float(gamma), float(lambda_),
        _vp(out), ws, wsn, s), "rlscan_gae")
    return out


def compute_gae_and_returns(rewards, values, terminateds, truncateds=None, gamma=0.99,
                            lambda_=0.95, bootstrap_values=None, last_value=None,
                            outputs=("advantages", "lambda_returns", "discounted_returns"),
                            out_dtype=None):
    """GAE advantages, lambda-returns (= advantages + values) and discounted
    returns from one pass over the inputs (one fused kernel).  ``outputs``
    selects which are produced; returns them as a tuple in that order.
    bfloat16 rewards select compact storage (see compute_gae)."""
    known = ("advantages", "lambda_returns", "discounted_returns")
    if not outputs or any(o not in known for o in outputs):
        raise ValueError(f"outputs must be a non-empty subset of {known}")
    if isinstance(rewards, torch.Tensor) and rewards.dtype == torch.bfloat16:
        c, outs = _compact_call(rewards, values, terminateds, truncateds, bootstrap_values,
                                last_value, len(outputs), out_dtype or torch.float32)
        by_name = dict(zip(outputs, outs))
        ws, wsn, s = _ws_for(c)
        c.launched(_native.lib().rlscan_gae_returns_compact(
            c.m("rewards"), c.m("values"), c.m("terminateds"), c.m("truncateds"),
            c.m("bootstrap_values"), c.v("last_value"), c.N, c.T, c.rs, float(gamma),
            float(lambda_), _OUT_DTYPES[out_dtype or torch.float32],
            _vp(by_name.get("advantages")), _vp(by_name.get("lambda_returns")),
            _vp(by_name.get("discounted_returns")), ws, wsn, s), "rlscan_gae_returns_compact")
        return tuple(outs)
    c = _Call("rewards", rewards)
    c.mat("values", values)
    c.mat("terminateds", terminateds)
    c.mat("truncateds", truncateds, False)
    c.mat("bootstrap_values", bootstrap_values, False)
    c.vec("last_value", last_value)
    if last_value is not None and bootstrap_values is not None:
        raise ValueError("pass either last_value or bootstrap_values, not both")
    if last_value is not None and truncateds is not None:
        raise ValueError("last_value cannot be combined with truncateds; use bootstrap_values")
    outs = c.finish(len(outputs))
    by_name = dict(zip(outputs, outs))
    ws, wsn, s = _ws_for(c)
    c.launched(_native.lib().rlscan_gae_returns(
        c.m("rewards"), c.m("values"), c.m("terminateds"), c.m("truncateds"),
        c.m("bootstrap_values"), c.v("last_value"), c.N, c.T, c.rs, float(gamma), float(lambda_),
        _vp(by_name.get("advantages")), _vp(by_name.get("lambda_returns")),
        _vp(by_name.get("discounted_returns")), ws, wsn, s), "rlscan_gae_returns")
    return tuple(outs)


def compute_gae_normalized(rewards, values, terminateds, truncateds=None, gamma=0.99,
                           lambda_=0.95, bootstrap_values=None, last_value=None, eps=1e-8,
                           outputs=("advantages", "lambda_returns"), return_moments=False):
    """GAE advantages normalised over the whole batch, (A - mean) / (std + eps)
    with the unbiased standard deviation, fused with the returns (which use
    the raw advantages).  ``outputs`` selects from "advantages" (normalised,
    always produced), "lambda_returns" and "discounted_returns"; returns them
    as a tuple in that order, followed by a CUDA float tensor (mean, std) of
    the raw advantages when ``return_moments``."""
    known = ("advantages", "lambda_returns", "discounted_returns")
    if "advantages" not in outputs or any(o not in known for o in outputs):
        raise ValueError(f"outputs must include 'advantages' and be a subset of {known}")
    c = _Call("rewards", rewards)
    c.mat("values", values)
    c.mat("terminateds", terminateds)
    c.mat("truncateds", truncateds, False)
    c.mat("bootstrap_values", bootstrap_values, False)
    c.vec("last_value", last_value)
    if last_value is not None and bootstrap_values is not None:
        raise ValueError("pass either last_value or bootstrap_values, not both")
    if last_value is not None and truncateds is not None:
        raise ValueError("last_value cannot be combined with truncateds; use bootstrap_values")
    outs = c.finish(len(outputs))
    by_name = dict(zip(outputs, outs))
    moments = torch.empty(2, dtype=torch.float32, device=c.device) if return_moments else None
    s = c.stream()
    need = _native.lib().rlscan_gae_normalized_workspace_bytes(c.N, c.T)
    ws, wsn = _workspace(c.device, s, need)
    c.launched(_native.lib().rlscan_gae_normalized(
        c.m("rewards"), c.m("values"), c.m("terminateds"), c.m("truncateds"),
        c.m("bootstrap_values"), c.v("last_value"), c.N, c.T, c.rs, float(gamma), float(lambda_),
        float(eps), _vp(by_name["advantages"]), _vp(by_name.get("lambda_returns")),
        _vp(by_name.get("discounted_returns")), _vp(moments), ws, wsn, s),
        "rlscan_gae_normalized")
    return tuple(outs) + ((moments,) if return_moments else ())


def compute_vtrace(log_pi_target, log_pi_behavior, values, rewards, terminateds, truncateds=None,
                   gamma=0.99, rho_bar=1.0, c_bar=1.0, bootstrap_values=None, last_value=None,
                   out_dtype=None):
    """V-trace (targets, advantages) (rl-triton API reference, compute_vtrace).
    bfloat16 rewards select compact storage: the log-probabilities, values
    and bootstrap_values bfloat16 too, flags uint8 or bool, last_value
    float32; ``out_dtype`` (float32 by default, or bfloat16) sets the output
    type."""
    if isinstance(rewards, torch.Tensor) and rewards.dtype == torch.bfloat16:
        out_dtype = out_dtype or torch.float32
        if out_dtype not in _OUT_DTYPES:
            raise ValueError("out_dtype must be torch.float32 or torch.bfloat16")
        c = _Call("rewards", rewards, _BF16)
        for name, t in (("log_pi_target", log_pi_target), ("log_pi_behavior", log_pi_behavior),
                        ("values", values)):
            c.mat(name, t, dtypes=_BF16)
        c.mat("terminateds", terminateds, dtypes=_FLAG8)
        c.mat("truncateds", truncateds, False, _FLAG8)
        c.mat("bootstrap_values", bootstrap_values, False, _BF16)
        c.vec("last_value", last_value)
        if last_value is not None and bootstrap_values is not None:
            raise ValueError("pass either last_value or bootstrap_values, not both")
        if bootstrap_values is not None and truncateds is None:
            raise ValueError("compact storage: the window bootstrap is last_value (float32 [N])")
        vs, adv = c.finish(2, out_dtype)
        ws, wsn, s = _ws_for(c)
        c.launched(_native.lib().rlscan_vtrace_compact(
            c.m("log_pi_target"), c.m("log_pi_behavior"), c.m("values"), c.m("rewards"),
            c.m("terminateds"), c.m("truncateds"), c.m("bootstrap_values"), c.v("last_value"),
            c.N, c.T, c.rs, float(gamma), float(rho_bar), float(c_bar), _OUT_DTYPES[out_dtype],
            _vp(vs), _vp(adv), ws, wsn, s), "rlscan_vtrace_compact")
        return vs, adv
    if out_dtype not in (None, torch.float32):
        raise ValueError("bfloat16 outputs need compact (bfloat16) inputs")
    c = _Call("rewards", rewards)
    c.mat("log_pi_target", log_pi_target)
    c.mat("log_pi_behavior", log_pi_behavior)
    c.mat("values", values)
    c.mat("rewards", rewards)
    c.mat("terminateds", terminateds)
    c.mat("truncateds", truncateds, False)
    c.mat("bootstrap_values", bootstrap_values, False)
    c.vec("last_value", last_value)
    if last_value is not None and bootstrap_values is not None:
        raise ValueError("pass either last_value or bootstrap_values, not both")
    vs, adv = c.finish(2)
    ws, wsn, s = _ws_for(c)
    c.launched(_native.lib().rlscan_vtrace(
        c.m("log_pi_target"), c.m("log_pi_behavior"), c.m("values"), c.m("rewards"),
        c.m("terminateds"), c.m("truncateds"), c.m("bootstrap_values"), c.v("last_value"),
        c.N, c.T, c.rs, float(gamma), float(rho_bar), float(c_bar), _vp(vs), _vp(adv),
        ws, wsn, s), "rlscan_vtrace")
    return vs, adv


def compute_retrace(action_probs_target, action_probs_behavior, q_values, next_q_values_all,
                    actions, rewards, terminateds, truncateds=None, gamma=0.99, lambda_=1.0,
                    c_bar=1.0, rho_bar=1.0):
    """Retrace(lambda) (targets, advantages) from the full action-space inputs
    (rl-triton API reference, compute_retrace): action_probs_target and
    next_q_values_all [N,T,A] float32, actions [N,T] int64, the other
    arguments [N,T] float32.  The action dimension is reduced inside the
    kernel: E_pi[Q'] with the target probabilities of the same step, and
    pi(a_t|s_t) gathered at ``actions``."""
    c = _Call("rewards", rewards)
    for name, t in (("action_probs_behavior", action_probs_behavior), ("q_values", q_values),
                    ("rewards", rewards), ("terminateds", terminateds)):
        c.mat(name, t)
    c.mat("truncateds", truncateds, False)
    if not isinstance(actions, torch.Tensor) or actions.dtype != torch.int64:
        raise TypeError("actions must be an int64 torch.Tensor")
    if not (actions.is_pinned() or (actions.is_cuda and actions.device == c.device)):
        raise ValueError(f"actions must be on {c.device} or in pinned host memory")
    if tuple(actions.shape) != (c.N, c.T):
        raise ValueError(f"actions shape {tuple(actions.shape)} != {(c.N, c.T)}")
    wide = []
    for name, t in (("action_probs_target", action_probs_target),
                    ("next_q_values_all", next_q_values_all)):
        if not isinstance(t, torch.Tensor) or t.dim() != 3:
            raise ValueError(f"{name} must be a [num_envs, seq_len, num_actions] tensor")
        _check(name, t, (c.N, c.T, t.shape[2]), c.device)
        wide.append(t)
    A = wide[0].shape[2]
    if wide[1].shape[2] != A:
        raise ValueError("action_probs_target and next_q_values_all differ in num_actions")
    qret, adv = c.finish(2)
    # actions share the float arrays' row stride; the [N,T,A] pair shares one
    # row stride of its own with unit inner strides
    acts = actions
    if c.N > 1 and acts.stride(0) != c.rs or (c.T > 1 and acts.stride(1) != 1):
        acts = torch.empty_strided((c.N, c.T), (c.rs, 1), dtype=torch.int64, device=c.device)
        acts.copy_(actions, non_blocking=True)

    def inner_ok(t):
        return (A <= 1 or t.stride(2) == 1) and (c.T <= 1 or t.stride(1) == A)
    ars = c.T * A
    if all(inner_ok(t) for t in wide) and (c.N <= 1 or len({t.stride(0) for t in wide}) == 1):
        if c.N > 1:
            ars = wide[0].stride(0)
    else:
        ars = -1
    if ars < c.T * A:
        wide = [c.contiguous(t) for t in wide]
        ars = c.T * A
    c.keep(*wide, acts)
    ws, wsn, s = _ws_for(c)
    c.launched(_native.lib().rlscan_retrace_actions(
        _vp(wide[0]), c.m("action_probs_behavior"), c.m("q_values"), _vp(wide[1]), _vp(acts),
        c.m("rewards"), c.m("terminateds"), c.m("truncateds"), c.N, c.T, A, c.rs, ars,
        float(gamma), float(lambda_), float(c_bar), float(rho_bar), _vp(qret), _vp(adv),
        ws, wsn, s), "rlscan_retrace_actions")
    return qret, adv


def compute_retrace_from_probs(pi_taken, mu_taken, q_values, expected_next_q, rewards,
                               terminateds, truncateds=None, gamma=0.99, lambda_=1.0, c_bar=1.0,
                               rho_bar=1.0, out_dtype=None):
    """Retrace(lambda) (targets, advantages) from per-step inputs:
    pi(a_t|s_t), mu(a_t|s_t), Q(s_t,a_t), E_pi[Q(s_{t+1},.)] (rl-triton API
    reference, compute_retrace, after its action-dimension reduction).
    bfloat16 rewards select compact storage: the other value inputs
    bfloat16 too, flags uint8 or bool; ``out_dtype`` (float32 by default, or
    bfloat16) sets the output type."""
    if isinstance(rewards, torch.Tensor) and rewards.dtype == torch.bfloat16:
        out_dtype = out_dtype or torch.float32
        if out_dtype not in _OUT_DTYPES:
            raise ValueError("out_dtype must be torch.float32 or torch.bfloat16")
        c = _Call("rewards", rewards, _BF16)
        for name, t in (("pi_taken", pi_taken), ("mu_taken", mu_taken), ("q_values", q_values),
                        ("expected_next_q", expected_next_q)):
            c.mat(name, t, dtypes=_BF16)
        c.mat("terminateds", terminateds, dtypes=_FLAG8)
        c.mat("truncateds", truncateds, False, _FLAG8)
        qret, adv = c.finish(2, out_dtype)
        ws, wsn, s = _ws_for(c)
        c.launched(_native.lib().rlscan_retrace_compact(
            c.m("pi_taken"), c.m("mu_taken"), c.m("q_values"), c.m("expected_next_q"),
            c.m("rewards"), c.m("terminateds"), c.m("truncateds"), c.N, c.T, c.rs,
            float(gamma), float(lambda_), float(c_bar), float(rho_bar), _OUT_DTYPES[out_dtype],
            _vp(qret), _vp(adv), ws, wsn, s), "rlscan_retrace_compact")
        return qret, adv
    if out_dtype not in (None, torch.float32):
        raise ValueError("bfloat16 outputs need compact (bfloat16) inputs")
    c = _Call("rewards", rewards)
    for name, t in (("pi_taken", pi_taken), ("mu_taken", mu_taken), ("q_values", q_values),
                    ("expected_next_q", expected_next_q), ("rewards", rewards),
                    ("terminateds", terminateds)):
        c.mat(name, t)
    c.mat("truncateds", truncateds, False)
    qret, adv = c.finish(2)
    ws, wsn, s = _ws_for(c)
    c.launched(_native.lib().rlscan_retrace(
        c.m("pi_taken"), c.m("mu_taken"), c.m("q_values"), c.m("expected_next_q"),
        c.m("rewards"), c.m("terminateds"), c.m("truncateds"), c.N, c.T, c.rs,
        float(gamma), float(lambda_), float(c_bar), float(rho_bar), _vp(qret), _vp(adv),
        ws, wsn, s), "rlscan_retrace")
    return qret, adv


def compute_lambda_returns(rewards, next_values, terminateds, truncateds=None, gamma=0.99,
                           lambda_=0.95, bootstrap_values=None, last_value=None):
    """TD(lambda) returns (rl-triton API reference, compute_lambda_returns;
    ``last_value`` is an addition: the window bootstrap as an [N] vector)."""
    c = _Call("rewards", rewards)
    c.mat("next_values", next_values)
    c.mat("terminateds", terminateds)
    c.mat("truncateds", truncateds, False)
    c.mat("bootstrap_values", bootstrap_values, False)
    c.vec("last_value", last_value)
    if last_value is not None and bootstrap_values is not None:
        raise ValueError("pass either last_value or bootstrap_values, not both")
    (out,) = c.finish(1)
    ws, wsn, s = _ws_for(c)
    c.launched(_native.lib().rlscan_lambda_returns(
        c.m("rewards"), c.m("next_values"), c.m("terminateds"), c.m("truncateds"),
        c.m("bootstrap_values"), c.v("last_value"), c.N, c.T, c.rs, float(gamma), float(lambda_),
        _vp(out), ws, wsn, s), "rlscan_lambda_returns")
    return out


def compute_discounted_returns(rewards, terminateds, truncateds=None, gamma=0.99,
                               bootstrap_values=None, last_value=None):
    """Discounted returns (rl-triton API reference, compute_discounted_returns)."""
    c = _Call("rewards", rewards)
    c.mat("terminateds", terminateds)
    c.mat("truncateds", truncateds, False)
    c.mat("bootstrap_values", bootstrap_values, False)
    c.vec("last_value", last_value)
    if last_value is not None and bootstrap_values is not None:
        raise ValueError("pass either last_value or bootstrap_values, not both")
    (out,) = c.finish(1)
    ws, wsn, s = _ws_for(c)
    c.launched(_native.lib().rlscan_discounted_returns(
        c.m("rewards"), c.m("terminateds"), c.m("truncateds"), c.m("bootstrap_values"),
        c.v("last_value"), c.N, c.T, c.rs, float(gamma), _vp(out), ws, wsn, s),
        "rlscan_discounted_returns")
    return out


def compute_eligibility_traces(gradients, dones, gamma, lambda_, seed_values=None):
    """Forward eligibility traces (rl-triton API reference, compute_eligibility_traces)."""
    c = _Call("gradients", gradients)
    c.mat("gradients", gradients)
    c.mat("dones", dones)
    c.vec("seed_values", seed_values)
    (out,) = c.finish(1)
    ws, wsn, s = _ws_for(c)
    c.launched(_native.lib().rlscan_eligibility_traces(
        c.m("gradients"), c.m("dones"), c.v("seed_values"), c.N, c.T, c.rs, float(gamma),
        float(lambda_), _vp(out), ws, wsn, s), "rlscan_eligibility_traces")
    return out


def compute_episodic_prefix_sum(inputs, dones, seed_values=None, boundary="ends_at"):
    """Episodic prefix sum (rl-triton API reference, compute_episodic_prefix_sum)."""
    if boundary not in ("ends_at", "starts_at"):
        raise ValueError(f"boundary must be 'ends_at' or 'starts_at', got {boundary!r}")
    c = _Call("inputs", inputs)
    c.mat("inputs", inputs)
    c.mat("dones", dones)
    c.vec("seed_values", seed_values)
    (out,) = c.finish(1)
    ws, wsn, s = _ws_for(c)
    c.launched(_native.lib().rlscan_episodic_prefix_sum(
        c.m("inputs"), c.m("dones"), c.v("seed_values"),
        _native.ENDS_AT if boundary == "ends_at" else _native.STARTS_AT,
        c.N, c.T, c.rs, _vp(out), ws, wsn, s), "rlscan_episodic_prefix_sum")
    return out


def linear_scan(alpha, beta, carry=None, direction="backward"):
    """Generic affine recurrence (rl-triton paper Eq. 1 and its forward mirror)."""
    if direction not in ("backward", "forward"):
        raise ValueError(f"direction must be 'backward' or 'forward', got {direction!r}")
    c = _Call("alpha", alpha)
    c.mat("alpha", alpha)
    c.mat("beta", beta)
    c.vec("carry", carry)
    (out,) = c.finish(1)
    ws, wsn, s = _ws_for(c)
    c.launched(_native.lib().rlscan_linear_scan(
        c.m("alpha"), c.m("beta"), c.v("carry"),
        _native.BACKWARD if direction == "backward" else _native.FORWARD,
        c.N, c.T, c.rs, _vp(out), ws, wsn, s), "rlscan_linear_scan")
    return out
