"""rlscan_gae_noalloc: GAE for callers that cannot allocate device memory.

Some callers may not call cudaMalloc when they run (a plugin inside a
framework that owns all device memory, a loop whose policy forbids
allocation because it can synchronise the device, a runtime with a fixed
budget).  For them the library keeps the cross-block scratch in a buffer
built into its own image.  This test drives that entry point through the C
ABI, twice in a row on different shapes and data, and checks each result
against rlscan_gae (which takes a caller workspace) within the parity
tolerance used everywhere else (|a - b| <= 1e-4 + 1e-5 |b|).  It also checks
that a shape needing more scratch than the buffer holds is refused before
any device work.  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _vp(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@pytest.fixture(scope="module")
def lib():
    from linear_recurrence_scan_gb300 import _native, build
    build.build()
    return _native.lib()


def _inputs(seed, N, T, trunc):
    rng = np.random.default_rng(seed)
    term = (rng.random((N, T)) < 0.01).astype(np.float32)
    tr = None
    bs = None
    last = None
    if trunc:
        tr = (rng.random((N, T)) < 0.005).astype(np.float32)
        tr[term > 0] = 0
        keep = tr > 0
        keep[:, -1] = True
        bs = np.where(keep, rng.standard_normal((N, T)), 0).astype(np.float32)
    else:
        last = rng.standard_normal(N).astype(np.float32)
    r = rng.standard_normal((N, T)).astype(np.float32)
    v = rng.standard_normal((N, T)).astype(np.float32)
    d = lambda a: None if a is None else torch.from_numpy(a).cuda()
    return [d(x) for x in (r, v, term, tr, bs, last)]


def _with_workspace(lib, args, N, T, stream):
    out = torch.empty((N, T), device="cuda")
    wsn = lib.rlscan_workspace_bytes(N, T)
    ws = torch.empty(max(wsn, 16), dtype=torch.uint8, device="cuda")
    assert lib.rlscan_workspace_init(_vp(ws), ws.numel(), stream) == 0
    st = lib.rlscan_gae(*[_vp(a) for a in args], N, T, T, 0.99, 0.95, _vp(out), _vp(ws),
                        ws.numel(), stream)
    assert st == 0
    return out


def _no_alloc(lib, args, N, T, stream):
    out = torch.empty((N, T), device="cuda")
    st = lib.rlscan_gae_noalloc(*[_vp(a) for a in args], N, T, T, 0.99, 0.95, _vp(out), stream)
    assert st == 0, lib.rlscan_status_string(st)
    return out


def test_no_alloc_gae_matches_workspace_gae_on_two_calls(lib):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # two calls in a row: different shapes, specialisations and data, both
    # long enough (T > 1024) that the cross-block scratch is used
    for seed, (N, T, trunc) in enumerate([(64, 20000, True), (33, 70001, False)]):
        args = _inputs(seed, N, T, trunc)
        got = _no_alloc(lib, args, N, T, stream)
        ref = _with_workspace(lib, args, N, T, stream)
        torch.cuda.synchronize()
        g, r = got.double().cpu().numpy(), ref.double().cpu().numpy()
        assert np.isfinite(g).all()
        assert (np.abs(g - r) <= 1e-4 + 1e-5 * np.abs(r)).all(), float(np.abs(g - r).max())


def test_no_alloc_refuses_shapes_beyond_its_buffer(lib):
    fake = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    st = lib.rlscan_gae_noalloc(fake, fake, fake, None, None, None, 262141, 1025, 1025, 0.99,
                                0.95, ctypes.c_void_p(512), None)
    assert st == 9  # RLSCAN_ERR_SCRATCH_LIMIT
    assert b"scratch" in lib.rlscan_status_string(st)
