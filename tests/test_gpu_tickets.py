"""The workspace ticket across calls of different kinds, through the C ABI.

A workspace's header holds the tile ticket, the exit count and the call
epoch.  Rows split across tiles draw every tile from the ticket (look-back);
whole rows packed into tiles draw each thread block's last tile from it when
a workspace is given, and none without one.  Each thread block counts itself
out after its last draw, and the last one re-arms the ticket and advances the
epoch.  These tests run long interleaved sequences of such calls on one
workspace and one stream -- packed rows with and without the workspace,
split rows with immediate and deferred finishing, forward and backward
scans, several estimators -- and compare every result with the float64
oracle (|gpu - ref| <= 1e-4 + 1e-5 |ref|; integer prefix sums bit-exact), so
a ticket left armed, a stale epoch or a tile drawn twice would show as a
wrong or NaN element.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from linear_recurrence_scan_gb300 import _native, build
    build.build()
    return _native.lib()


def _vp(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _close(got, ref, what):
    g = got.double().cpu().numpy()
    err = np.abs(g - ref)
    bad = ~(err <= 1e-4 + 1e-5 * np.abs(ref))
    assert not bad.any(), f"{what}: {bad.sum()} elements off, max err {float(np.nanmax(err))}"


def test_interleaved_packed_and_split_calls_share_one_workspace(lib):
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    big = lib.rlscan_workspace_bytes(64, 1 << 16)
    ws = torch.empty(big, dtype=torch.uint8, device="cuda")
    assert lib.rlscan_workspace_init(_vp(ws), big, s) == 0
    rng = np.random.default_rng(21)
    # (N, T) shapes: packed short rows (one tile per row or several rows per
    # tile), split rows finished at once, and many tiles per row in flight
    # (deferred finishing)
    shapes = [(4096, 1024), (1000, 300), (256, 5000), (64, 1 << 16), (3000, 1024), (8, 20000)]
    for rep in range(3):
        for N, T in shapes:
            r = rng.standard_normal((N, T)).astype(np.float32)
            v = rng.standard_normal((N, T)).astype(np.float32)
            term = (rng.random((N, T)) < 0.01).astype(np.float32)
            last = rng.standard_normal(N).astype(np.float32)
            d = {k: torch.from_numpy(a).cuda() for k, a in dict(r=r, v=v, term=term, last=last).items()}
            adv = torch.empty((N, T), device="cuda")
            for use_ws in (True, False):
                if not use_ws and lib.rlscan_workspace_bytes(N, T) > 0 and T > 1024:
                    continue  # split rows need the workspace
                w, wn = (_vp(ws), big) if use_ws else (None, 0)
                st = lib.rlscan_gae(_vp(d["r"]), _vp(d["v"]), _vp(d["term"]), None, None, _vp(d["last"]), N, T,
                                    T, 0.99, 0.95, _vp(adv), w, wn, s)
                assert st == 0, (N, T, st)
                _close(adv, oracle.gae(r, v, term, None, 0.99, 0.95, None, last),
                       f"gae {N}x{T} rep {rep} workspace {use_ws}")
            # a forward scan on the same workspace: integer prefix sums, bit-exact
            x = rng.integers(0, 10, (N, T)).astype(np.float32)
            dn = (rng.random((N, T)) < 1e-3).astype(np.float32)
            dx, ddn = torch.from_numpy(x).cuda(), torch.from_numpy(dn).cuda()
            out = torch.empty((N, T), device="cuda")
            assert lib.rlscan_episodic_prefix_sum(_vp(dx), _vp(ddn), None, 1, N, T, T, _vp(out), _vp(ws), big,
                                                  s) == 0
            np.testing.assert_array_equal(out.double().cpu().numpy(),
                                          oracle.episodic_prefix_sum(x, dn, None, "starts_at"),
                                          err_msg=f"prefix {N}x{T} rep {rep}")
    assert lib.rlscan_workspace_status(_vp(ws), big, s) == 0


def test_back_to_back_packed_calls_without_sync(lib):
    """Many packed calls queued back to back (the next kernel's blocks start
    while the previous one drains), each on its own output, checked after."""
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    N, T = 4096, 1024
    wsn = lib.rlscan_workspace_bytes(N, T)
    ws = torch.empty(wsn, dtype=torch.uint8, device="cuda")
    assert lib.rlscan_workspace_init(_vp(ws), wsn, s) == 0
    rng = np.random.default_rng(22)
    r = rng.standard_normal((N, T)).astype(np.float32)
    term = (rng.random((N, T)) < 0.01).astype(np.float32)
    last = rng.standard_normal(N).astype(np.float32)
    dr, dt, dl = (torch.from_numpy(a).cuda() for a in (r, term, last))
    outs = [torch.empty((N, T), device="cuda") for _ in range(12)]
    gammas = [0.9 + 0.008 * i for i in range(12)]
    for o, g in zip(outs, gammas):
        assert lib.rlscan_discounted_returns(_vp(dr), _vp(dt), None, None, _vp(dl), N, T, T, g, _vp(o),
                                             _vp(ws), wsn, s) == 0
    torch.cuda.synchronize()
    for o, g in zip(outs, gammas):
        _close(o, oracle.discounted_returns(r, term, None, g, None, last), f"discounted gamma {g}")
    assert lib.rlscan_workspace_status(_vp(ws), wsn, s) == 0
