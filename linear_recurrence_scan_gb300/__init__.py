"""GB300-native batched linear-recurrence scans for RL credit assignment.

The compute path is the CUDA library ``librlscan.so`` (hand-written sm_103a
kernels behind the C ABI in ``include/rlscan.h``); ``api`` binds it for
PyTorch tensors.  ``synthetic`` draws seeded rollout buffers.  Importing the
package does not load the library; the first estimator call does (and raises
if it has not been built).
"""
__version__ = "0.1.0"

_API = {
    "compute_gae", "compute_gae_and_returns", "compute_gae_normalized", "compute_vtrace",
    "compute_retrace",
    "compute_retrace_from_probs", "compute_lambda_returns",
    "compute_discounted_returns", "compute_eligibility_traces", "compute_episodic_prefix_sum",
    "linear_scan", "workspace_status",
}


def __getattr__(name):
    if name in _API:
        from . import api
        value = getattr(api, name)
        globals()[name] = value  # later lookups skip this hook
        return value
    raise AttributeError(name)


def __dir__():
    return sorted(set(globals()) | _API)
