"""The C ABI without a GPU: the library builds, loads, exports every function
include/rlscan.h declares, and rejects bad arguments before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rlscan.h")


@pytest.fixture(scope="module")
def lib():
    from linear_recurrence_scan_gb300 import _native, build
    build.build()
    return _native.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rlscan_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["rlscan_gae", "rlscan_vtrace", "rlscan_retrace", "rlscan_lambda_returns",
                     "rlscan_discounted_returns", "rlscan_eligibility_traces",
                     "rlscan_episodic_prefix_sum", "rlscan_linear_scan",
                     "rlscan_workspace_bytes", "rlscan_workspace_init", "rlscan_workspace_status"]:
        assert required in names


def test_library_exports_every_declared_function(lib):
    from linear_recurrence_scan_gb300 import _native
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in rlscan.h but not exported"
        assert name in _native.SIGNATURES, f"{name} has no Python binding signature"


def test_version_and_status_strings(lib):
    assert lib.rlscan_version() == (0 << 16) | (1 << 8) | 0
    for code in range(11):
        assert lib.rlscan_status_string(code) and lib.rlscan_status_string(code) != b"unknown status"
    assert lib.rlscan_status_string(99) == b"unknown status"


def test_normal_build_has_no_bounds_checking(lib):
    """Only the checked build counts bounds violations; the normal build
    reports 0 (not checked) and zeroes both values, without a device."""
    v, site = ctypes.c_ulonglong(7), ctypes.c_ulonglong(7)
    assert lib.rlscan_bounds_check(ctypes.addressof(v), ctypes.addressof(site), 1) == 0
    assert v.value == 0 and site.value == 0
    assert lib.rlscan_bounds_check(None, None, 0) == 0


def test_workspace_bytes(lib):
    assert lib.rlscan_workspace_bytes(0, 100) == 0
    assert lib.rlscan_workspace_bytes(10, 0) == 0
    assert lib.rlscan_workspace_bytes(4096, 512) == 0             # one tile per row for every kernel
    assert lib.rlscan_workspace_bytes(4096, 1024) == 64 + 16 * 2 * 4096
    # header + 16 bytes per (1024-step tile, scan), two scans at most
    assert lib.rlscan_workspace_bytes(2, 1025) == 64 + 16 * 2 * 2 * 2
    assert lib.rlscan_workspace_bytes(64, 1 << 20) == 64 + 16 * 2 * 64 * 1024


P = None  # NULL pointer


def gae(lib, **kw):
    a = dict(r=1, v=2, term=3, trunc=P, bs=P, last=P, N=2, T=4, rs=4, out=10)
    a.update(kw)
    vp = lambda x: None if x is None else ctypes.c_void_p(x * 256)
    return lib.rlscan_gae(vp(a["r"]), vp(a["v"]), vp(a["term"]), vp(a["trunc"]), vp(a["bs"]),
                          vp(a["last"]), a["N"], a["T"], a["rs"], 0.99, 0.95, vp(a["out"]),
                          None, 0, None)


def test_gae_validation(lib):
    assert gae(lib, N=-1) == 2
    assert gae(lib, T=-1) == 2
    assert gae(lib, rs=3) == 2
    assert gae(lib, N=0) == 0 and gae(lib, T=0, rs=0) == 0     # no-ops, no CUDA call
    assert gae(lib, r=None) == 1
    assert gae(lib, out=None) == 1
    assert gae(lib, bs=5, last=6) == 3                           # exclusive bootstraps
    assert gae(lib, trunc=5, last=6) == 3                        # last_value with truncateds
    assert gae(lib, out=2) == 3                                  # output aliases an input


def test_enum_and_null_validation(lib):
    vp = lambda x: ctypes.c_void_p(x * 256)
    assert lib.rlscan_episodic_prefix_sum(vp(1), vp(2), None, 7, 2, 4, 4, vp(3), None, 0, None) == 4
    assert lib.rlscan_linear_scan(vp(1), vp(2), None, 5, 2, 4, 4, vp(3), None, 0, None) == 4
    assert lib.rlscan_linear_scan(None, vp(2), None, 0, 2, 4, 4, vp(3), None, 0, None) == 1
    assert lib.rlscan_linear_scan(vp(1), vp(2), None, 0, 2, 4, 4, vp(1), None, 0, None) == 3
    assert lib.rlscan_vtrace(*[vp(i) for i in range(1, 6)], None, None, None, 2, 4, 4,
                             0.99, 1.0, 1.0, vp(9), vp(9), None, 0, None) == 3
    assert lib.rlscan_retrace(*[vp(i) for i in range(1, 7)], None, 2, 4, 4, 0.99, 0.95, 1.0, 1.0,
                              vp(8), None, None, 0, None) == 1
    assert lib.rlscan_discounted_returns(vp(1), vp(2), None, vp(3), vp(4), 2, 4, 4, 0.99, vp(5),
                                         None, 0, None) == 3
    assert lib.rlscan_lambda_returns(vp(1), vp(2), vp(3), None, None, None, 2, 4, 3, 0.99, 0.9,
                                     vp(5), None, 0, None) == 2
    assert lib.rlscan_eligibility_traces(vp(1), vp(2), None, 2, 4, 4, 0.99, 0.9, vp(2),
                                         None, 0, None) == 3
    assert lib.rlscan_workspace_init(None, 64, None) == 1
    assert lib.rlscan_workspace_init(ctypes.c_void_p(8), 64, None) == 5


def retrace_actions(lib, **kw):
    a = dict(probs=1, mu=2, q=3, nq=4, acts=5, r=6, term=7, trunc=P, N=2, T=4, A=4, rs=4, ars=16,
             qret=10, adv=11)
    a.update(kw)
    vp = lambda x: None if x is None else ctypes.c_void_p(x * 256)
    return lib.rlscan_retrace_actions(vp(a["probs"]), vp(a["mu"]), vp(a["q"]), vp(a["nq"]),
                                      vp(a["acts"]), vp(a["r"]), vp(a["term"]), vp(a["trunc"]),
                                      a["N"], a["T"], a["A"], a["rs"], a["ars"], 0.99, 1.0, 1.0,
                                      1.0, vp(a["qret"]), vp(a["adv"]), None, 0, None)


def test_retrace_actions_validation(lib):
    assert retrace_actions(lib, A=0) == 4
    assert retrace_actions(lib, A=65537, ars=4 * 65537) == 4
    assert retrace_actions(lib, ars=15) == 2                     # [N,T,A] rows overlap
    assert retrace_actions(lib, rs=3) == 2
    assert retrace_actions(lib, N=0) == 0                        # no-op, no CUDA call
    assert retrace_actions(lib, acts=None) == 1
    assert retrace_actions(lib, nq=None) == 1
    assert retrace_actions(lib, adv=None) == 1
    assert retrace_actions(lib, adv=10) == 3                     # outputs alias
    assert retrace_actions(lib, qret=4) == 3                     # output aliases an input
    assert retrace_actions(lib, adv=5) == 3


def test_gae_normalized_validation(lib):
    vp = lambda x: None if x is None else ctypes.c_void_p(x * 256)
    need = lib.rlscan_gae_normalized_workspace_bytes(2, 4)
    assert need >= 64 + 16 * 4096 and lib.rlscan_gae_normalized_workspace_bytes(0, 4) == 0
    # look-back part of the workspace (rounded to 256 bytes) before the moments region
    assert (lib.rlscan_gae_normalized_workspace_bytes(64, 1 << 20) - need
            == (lib.rlscan_workspace_bytes(64, 1 << 20) + 255) // 256 * 256 - 256)

    def call(adv=10, eps=1e-8, ws=20, wsn=None, moments=None):
        return lib.rlscan_gae_normalized(vp(1), vp(2), vp(3), None, None, None, 2, 4, 4, 0.99,
                                         0.95, eps, vp(adv), None, None, vp(moments), vp(ws),
                                         need if wsn is None else wsn, None)
    assert call(adv=None) == 1
    assert call(eps=-1.0) == 4
    assert call(eps=float("nan")) == 4
    assert call(ws=None) == 5
    assert call(wsn=need - 1) == 5
    assert call(moments=10) == 3                                  # moments alias the advantages
    assert call(adv=2) == 3                                       # output aliases an input


def test_python_layer_rejects_cpu_and_wrong_dtype():
    import torch
    import linear_recurrence_scan_gb300 as L
    x = torch.zeros(2, 4)
    with pytest.raises(ValueError, match="CUDA"):
        L.compute_gae(x, x, x)
    with pytest.raises(ValueError, match="boundary"):
        L.compute_episodic_prefix_sum(x, x, boundary="middle")
    with pytest.raises(ValueError, match="direction"):
        L.linear_scan(x, x, direction="sideways")
    with pytest.raises(ValueError, match="CUDA"):
        L.compute_retrace(torch.zeros(2, 4, 3), x, x, torch.zeros(2, 4, 3),
                          torch.zeros(2, 4, dtype=torch.int64), x, x)
