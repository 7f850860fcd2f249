"""ctypes binding of librlscan (the C ABI declared in include/rlscan.h).

Marshalling only: every computation happens in the CUDA kernels of the
library.  If the library has not been built, loading fails with an error
(there is no CPU fallback).
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
# RLSCAN_LIB selects another build of the library (e.g. the checked build)
LIB_PATH = os.environ.get("RLSCAN_LIB") or os.path.join(HERE, "_build", "librlscan.so")

STATUS = {
    0: "RLSCAN_OK", 1: "RLSCAN_ERR_NULL", 2: "RLSCAN_ERR_SHAPE", 3: "RLSCAN_ERR_ARG_CONFLICT",
    4: "RLSCAN_ERR_ARG_VALUE", 5: "RLSCAN_ERR_WORKSPACE", 6: "RLSCAN_ERR_CUDA",
    7: "RLSCAN_ERR_INVALID_INPUT", 8: "RLSCAN_ERR_TIMEOUT", 9: "RLSCAN_ERR_SCRATCH_LIMIT",
    10: "RLSCAN_ERR_MEMORY",
}
ENDS_AT, STARTS_AT = 0, 1
BACKWARD, FORWARD = 0, 1


class RlscanError(RuntimeError):
    """A librlscan call returned a non-zero status."""

    def __init__(self, status: int, where: str):
        self.status = status
        self.name = STATUS.get(status, f"status {status}")
        msg = lib().rlscan_status_string(status).decode()
        super().__init__(f"{where}: {self.name} ({msg})")


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_I = ctypes.c_int

# argument types of every entry point, in declaration order
SIGNATURES = {
    "rlscan_version": ([], _I),
    "rlscan_status_string": ([_I], ctypes.c_char_p),
    "rlscan_bounds_check": ([_P, _P, _I], _I),
    "rlscan_workspace_bytes": ([_I64, _I64], _SZ),
    "rlscan_workspace_init": ([_P, _SZ, _P], _I),
    "rlscan_workspace_status": ([_P, _SZ, _P], _I),
    "rlscan_gae": ([_P] * 6 + [_I64] * 3 + [_F, _F, _P, _P, _SZ, _P], _I),
    "rlscan_gae_noalloc": ([_P] * 6 + [_I64] * 3 + [_F, _F, _P, _P], _I),
    "rlscan_gae_normalized_workspace_bytes": ([_I64, _I64], _SZ),
    "rlscan_gae_normalized": ([_P] * 6 + [_I64] * 3 + [_F, _F, _F, _P, _P, _P, _P, _P, _SZ, _P], _I),
    "rlscan_gae_compact": ([_P] * 6 + [_I64] * 3 + [_F, _F, _I, _P, _P, _SZ, _P], _I),
    "rlscan_gae_returns_compact": ([_P] * 6 + [_I64] * 3 + [_F, _F, _I, _P, _P, _P, _P, _SZ, _P], _I),
    "rlscan_vtrace_compact": ([_P] * 8 + [_I64] * 3 + [_F, _F, _F, _I, _P, _P, _P, _SZ, _P], _I),
    "rlscan_retrace_compact": ([_P] * 7 + [_I64] * 3 + [_F, _F, _F, _F, _I, _P, _P, _P, _SZ, _P], _I),
    "rlscan_gae_masked": ([_P] * 7 + [_I64] * 3 + [_F, _F, _P, _P, _SZ, _P], _I),
    "rlscan_gae_returns": ([_P] * 6 + [_I64] * 3 + [_F, _F, _P, _P, _P, _P, _SZ, _P], _I),
    "rlscan_vtrace": ([_P] * 8 + [_I64] * 3 + [_F, _F, _F, _P, _P, _P, _SZ, _P], _I),
    "rlscan_retrace": ([_P] * 7 + [_I64] * 3 + [_F] * 4 + [_P, _P, _P, _SZ, _P], _I),
    "rlscan_retrace_actions": ([_P] * 8 + [_I64] * 5 + [_F] * 4 + [_P, _P, _P, _SZ, _P], _I),
    "rlscan_lambda_returns": ([_P] * 6 + [_I64] * 3 + [_F, _F, _P, _P, _SZ, _P], _I),
    "rlscan_discounted_returns": ([_P] * 5 + [_I64] * 3 + [_F, _P, _P, _SZ, _P], _I),
    "rlscan_eligibility_traces": ([_P] * 3 + [_I64] * 3 + [_F, _F, _P, _P, _SZ, _P], _I),
    "rlscan_episodic_prefix_sum": ([_P] * 3 + [_I] + [_I64] * 3 + [_P, _P, _SZ, _P], _I),
    "rlscan_linear_scan": ([_P] * 3 + [_I] + [_I64] * 3 + [_P, _P, _SZ, _P], _I),
}

_lib = None
_lock = threading.Lock()


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -m linear_recurrence_scan_gb300.build)")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (argtypes, restype) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.argtypes = argtypes
                fn.restype = restype
            _lib = handle
    return _lib


def check(status: int, where: str) -> None:
    if status != 0:
        raise RlscanError(status, where)
