"""Failure detection without a GPU fault: a cross-block wait that runs out.

A child process sets RLSCAN_TEST_WITHHOLD_TILE so that one look-back tile
never publishes its state, and a 20 ms look-back bound.  Its successors in
the same row must give up after the bound, record RLSCAN_ERR_TIMEOUT in the
workspace, write NaN for the values that depended on the missing carry, and
the kernel must finish: row 0 is NaN before the withheld tile's region and
exact from it on (whatever the tile size), the other row is exact, the
stream stays usable, and
rlscan_workspace_status reports the timeout.  Nothing traps, asserts or
hangs on the device.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys, time
import numpy as np, torch
sys.path.insert(0, ROOT)
import oracle
import linear_recurrence_scan_gb300 as L
from linear_recurrence_scan_gb300 import _native
N, T = 2, 5 * 4096
rng = np.random.default_rng(0)
a = rng.integers(0, 4, (N, T)).astype(np.float32)
b = np.ones((N, T), np.float32)              # every aggregate keeps b = 1: a real chain
t0 = time.time()
out = L.linear_scan(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), None, "backward")
status = "OK"
try:
    L.workspace_status()
except _native.RlscanError as e:
    status = e.name
elapsed = time.time() - t0
got = out.double().cpu().numpy()
ref = oracle.linear_scan(a, b, None, "backward")
# after the timeout the same stream still works (a single-tile shape: the
# hook, still set in this process, only affects multi-tile rows)
a2, b2 = a[1:, :1000].copy(), b[1:, :1000].copy()
again = L.linear_scan(torch.from_numpy(a2).cuda(), torch.from_numpy(b2).cuda(), None, "backward")
torch.cuda.synchronize()
nan0 = np.isnan(got[0])
k = int(np.argmin(nan0)) if nan0.any() else 0     # first exact position of row 0
print(json.dumps(dict(
    status=status, elapsed=elapsed,
    row1_exact=bool(np.array_equal(got[1], ref[1])),
    row0_nan_prefix=int(k), row0_head_nan=bool(k > 0 and nan0[:k].all()),
    row0_tail_exact=bool(k < T and np.array_equal(got[0, k:], ref[0, k:])),
    again_exact=bool(np.array_equal(again.double().cpu().numpy(),
                                    oracle.linear_scan(a2, b2, None, "backward"))))))
"""


def test_withheld_tile_times_out_and_reports():
    env = dict(os.environ)
    # ticket order is (position in row, row): tile 1*N + 0 is row 0's second
    # tile in scan order; the chain to the row's start must pass through it
    env["RLSCAN_TEST_WITHHOLD_TILE"] = str(1 * 2 + 0)
    env["RLSCAN_SPIN_LIMIT_NS"] = str(20_000_000)
    code = "ROOT = %r\n" % ROOT + CHILD
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["status"] == "RLSCAN_ERR_TIMEOUT", res
    assert res["row1_exact"] and res["row0_tail_exact"], res
    assert res["row0_head_nan"], res
    assert res["again_exact"], res
    assert res["elapsed"] < 30, res


CHECKS_CHILD = r"""
import json, sys
import numpy as np, torch
sys.path.insert(0, ROOT)
import linear_recurrence_scan_gb300 as L
from linear_recurrence_scan_gb300 import _native
N, T = 3, 64
z = torch.zeros(N, T, device="cuda")
r = torch.randn(N, T, device="cuda")
term = z.clone(); term[0, 5] = 1
trunc = z.clone(); trunc[1, 7] = 1
bs = z.clone(); bs[1, 7] = 2.0; bs[:, -1] = 1.0
def status(fn):
    try:
        fn(); torch.cuda.synchronize(); return "OK"
    except _native.RlscanError as e:
        return e.name
both = trunc.clone(); both[0, 5] = 1          # a step both terminated and truncated
stray = bs.clone(); stray[2, 10] = 3.0        # bootstrap at an interior non-truncated step
print(json.dumps(dict(
    clean=status(lambda: L.compute_gae(r, r, term, trunc, 0.99, 0.95, bs)),
    overlap=status(lambda: L.compute_gae(r, r, term, both, 0.99, 0.95, bs)),
    stray=status(lambda: L.compute_gae(r, r, term, trunc, 0.99, 0.95, stray)),
    overlap_disc=status(lambda: L.compute_discounted_returns(r, term, both, 0.99, bs)),
    no_trunc=status(lambda: L.compute_gae(r, r, term, None, 0.99, 0.95, stray)))))
"""


def test_opt_in_content_checks():
    """RLSCAN_CHECKS=1: the pages' correctness-warning checks (exclusive
    flags, zero bootstrap at interior non-truncated steps) reject bad inputs
    with RLSCAN_ERR_INVALID_INPUT and pass conforming ones."""
    env = dict(os.environ)
    env["RLSCAN_CHECKS"] = "1"
    r = subprocess.run([sys.executable, "-c", "ROOT = %r\n" % ROOT + CHECKS_CHILD], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res == dict(clean="OK", overlap="RLSCAN_ERR_INVALID_INPUT",
                       stray="RLSCAN_ERR_INVALID_INPUT", overlap_disc="RLSCAN_ERR_INVALID_INPUT",
                       no_trunc="OK"), res
