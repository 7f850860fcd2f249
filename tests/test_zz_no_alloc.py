"""rlscan_gae_noalloc: GAE for callers that cannot allocate device memory.

Some callers may not call cudaMalloc when they run (a plugin inside a
framework that owns all device memory, a loop whose policy forbids
allocation because it can synchronise the device, a runtime with a fixed
budget).  For them the library keeps the cross-block scratch in a buffer
built into its own image.  These tests drive that entry point through the C
ABI:

* twice in a row on different shapes and data, each result checked element
  by element against the float64 oracle and against rlscan_gae (which takes
  a caller workspace), within the parity tolerance used everywhere else
  (|a - b| <= 1e-4 + 1e-5 |b|);
* at exactly the largest shape the buffer holds (131,070 tiles), against
  rlscan_gae and, on sampled rows, the oracle;
* shapes one tile beyond the limit, and argument conflicts, are refused
  before any device work (fake pointers that are never dereferenced);
* a cross-block wait that runs out (a child process withholds one tile's
  state) gives NaN where the missing carry was needed, exact values
  elsewhere, and the next call on the same buffer is exact again.

The file is named to be collected last.
"""
import ctypes
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SCRATCH_LIMIT = 9   # RLSCAN_ERR_SCRATCH_LIMIT
ARG_CONFLICT = 3    # RLSCAN_ERR_ARG_CONFLICT
MAX_TILES = ((4 << 20) - 64) // 32   # 131,070 states of 32 bytes after the 64-byte header


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
    return r, v, term, tr, bs, last


def _dev(arrays):
    return [None if a is None else torch.from_numpy(a).cuda() for a in arrays]


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


def _close(got, ref, what):
    err = np.abs(got - ref)
    bad = ~(err <= 1e-4 + 1e-5 * np.abs(ref))
    assert not bad.any(), f"{what}: {bad.sum()} elements off, max err {float(err.max())}"


def test_no_alloc_gae_matches_oracle_on_two_calls(lib):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # two calls in a row: different shapes, specialisations and data, both
    # long enough (T > 2048) that the cross-block scratch is used
    for seed, (N, T, trunc) in enumerate([(64, 20000, True), (33, 70001, False)]):
        host = _inputs(seed, N, T, trunc)
        args = _dev(host)
        got = _no_alloc(lib, args, N, T, stream)
        with_ws = _with_workspace(lib, args, N, T, stream)
        torch.cuda.synchronize()
        g = got.double().cpu().numpy()
        r, v, term, tr, bs, last = host
        _close(g, oracle.gae(r, v, term, tr, 0.99, 0.95, bs, last), f"oracle, call {seed + 1}")
        _close(g, with_ws.double().cpu().numpy(), f"rlscan_gae, call {seed + 1}")


def test_no_alloc_at_the_largest_shape_its_buffer_holds(lib):
    # 43,690 rows of 2,049 steps: the workspace counts 32 bytes per started
    # 1024 steps of a row, so 131,070 of them and the header fill exactly
    # 4 MiB (the rows are split across tiles, so the scratch is used)
    N, T = 43690, 2049
    assert N * -(-T // 1024) == MAX_TILES
    assert lib.rlscan_workspace_bytes(N, T) == 4 << 20
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    host = _inputs(7, N, T, False)
    args = _dev(host)
    got = _no_alloc(lib, args, N, T, stream)
    with_ws = _with_workspace(lib, args, N, T, stream)
    torch.cuda.synchronize()
    g = got.double().cpu().numpy()
    _close(g, with_ws.double().cpu().numpy(), "rlscan_gae at the limit")
    rows = np.random.default_rng(8).choice(N, 64, replace=False)
    rows.sort()
    r, v, term, _, _, last = host
    _close(g[rows], oracle.gae(r[rows], v[rows], term[rows], None, 0.99, 0.95, None, last[rows]),
           "oracle on sampled rows at the limit")


def test_no_alloc_refuses_shapes_beyond_its_buffer(lib):
    fake = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    out = ctypes.c_void_p(512)
    for N, T in [(MAX_TILES + 1, 1024), (43691, 2049), (262141, 1025)]:
        st = lib.rlscan_gae_noalloc(fake, fake, fake, None, None, None, N, T, T, 0.99, 0.95, out, None)
        assert st == SCRATCH_LIMIT, (N, T, st)
    assert b"scratch" in lib.rlscan_status_string(SCRATCH_LIMIT)


def test_no_alloc_refuses_argument_conflicts_before_any_device_work(lib):
    fake = ctypes.c_void_p(256)  # never dereferenced: the conflicts are found on the host
    other = ctypes.c_void_p(4096)
    out = ctypes.c_void_p(512)
    N, T = 4, 5000
    # bootstrap_values together with last_value; last_value with truncateds;
    # the output aliasing an input
    assert lib.rlscan_gae_noalloc(fake, fake, fake, None, other, other, N, T, T, 0.99, 0.95, out,
                                  None) == ARG_CONFLICT
    assert lib.rlscan_gae_noalloc(fake, fake, fake, other, None, other, N, T, T, 0.99, 0.95, out,
                                  None) == ARG_CONFLICT
    assert lib.rlscan_gae_noalloc(fake, fake, fake, None, None, None, N, T, T, 0.99, 0.95, fake,
                                  None) == ARG_CONFLICT


CHILD = r"""
import ctypes, json, sys
import numpy as np, torch
sys.path.insert(0, ROOT)
import oracle
from linear_recurrence_scan_gb300 import _native
lib = _native.lib()
vp = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

def call(r, v, term, last, gamma, lam):
    N, T = r.shape
    out = torch.empty((N, T), device="cuda")
    d = [torch.from_numpy(a).cuda() for a in (r, v, term, last)]
    st = lib.rlscan_gae_noalloc(vp(d[0]), vp(d[1]), vp(d[2]), None, None, vp(d[3]), N, T, T,
                                gamma, lam, vp(out), s)
    assert st == 0, st
    torch.cuda.synchronize()
    return out.double().cpu().numpy()

# gamma = lambda = 1 and no terminations: every tile's aggregate keeps b = 1,
# so each row is one carry chain; small integers keep every sum exact
N, T = 2, 5 * 4096
rng = np.random.default_rng(0)
r = rng.integers(0, 4, (N, T)).astype(np.float32)
v = rng.integers(0, 4, (N, T)).astype(np.float32)
term = np.zeros((N, T), np.float32)
last = rng.integers(0, 4, N).astype(np.float32)
got = call(r, v, term, last, 1.0, 1.0)
ref = oracle.gae(r, v, term, None, 1.0, 1.0, None, last)
# scan order runs backward: row 0's NaN part lies before (in time) the withheld tile
nan0 = np.isnan(got[0])
k = int(np.argmin(nan0)) if nan0.any() else 0
# the next call on the same buffer: two tiles (tickets 0 and 1, below the withheld one)
r2, v2 = r[:1, :4096].copy(), v[:1, :4096].copy()
t2, l2 = term[:1, :4096].copy(), last[:1].copy()
again = call(r2, v2, t2, l2, 0.99, 0.95)
ref2 = oracle.gae(r2, v2, t2, None, 0.99, 0.95, None, l2)
print(json.dumps(dict(
    row1_exact=bool(np.array_equal(got[1], ref[1])),
    row0_nan_prefix=k, row0_head_nan=bool(k > 0 and nan0[:k].all()),
    row0_tail_exact=bool(k < T and np.array_equal(got[0, k:], ref[0, k:])),
    again_close=bool((np.abs(again - ref2) <= 1e-4 + 1e-5 * np.abs(ref2)).all()))))
"""


def test_no_alloc_wait_that_runs_out_gives_nan_and_later_calls_are_exact():
    env = dict(os.environ)
    # ticket order is (position in row, row): tile 1*N + 0 is row 0's second
    # tile in scan order; the chain to the row's start must pass through it
    env["RLSCAN_TEST_WITHHOLD_TILE"] = str(1 * 2 + 0)
    env["RLSCAN_SPIN_LIMIT_NS"] = str(20_000_000)
    r = subprocess.run([sys.executable, "-c", "ROOT = %r\n" % ROOT + CHILD], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["row1_exact"] and res["row0_tail_exact"], res
    assert res["row0_head_nan"], res
    assert res["again_close"], res
