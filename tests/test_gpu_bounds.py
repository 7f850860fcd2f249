"""Bounds-checked build.  compute-sanitizer is not available on these GPUs,
so the library is also built with RLSCAN_CHECK_BOUNDS=1: every global
access of the scan kernels and every bulk copy's source and shared-memory
destination is tested against the extent of its argument, and a failed test
is counted (and the access skipped).  A child process runs the calls of
bounds_calls.py through that build; the test requires zero violations and
outputs bit-identical to the normal build's on the same calls (the checks
change no arithmetic)."""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_checked_build_finds_no_violation_and_matches(tmp_path):
    from linear_recurrence_scan_gb300 import build
    build.build()
    checked = build.build_checked()
    out = tmp_path / "checked.npz"
    env = dict(os.environ, RLSCAN_LIB=checked)
    r = subprocess.run([sys.executable, os.path.join(HERE, "bounds_calls.py"), str(out)], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    report = [line for line in r.stdout.splitlines() if line.startswith("BOUNDS")]
    assert report == ["BOUNDS kind=1 violations=0 first_site=0"], (report, r.stdout[-2000:])
    import bounds_calls
    mine = bounds_calls.run_all()
    theirs = np.load(out)
    assert sorted(mine) == sorted(theirs.files)
    for k in mine:
        assert np.array_equal(mine[k], theirs[k], equal_nan=True), k


def test_normal_build_reports_no_checking():
    import ctypes
    from linear_recurrence_scan_gb300 import _native
    v, s = ctypes.c_ulonglong(7), ctypes.c_ulonglong(7)
    assert _native.lib().rlscan_bounds_check(ctypes.addressof(v), ctypes.addressof(s), 0) == 0
    assert v.value == 0 and s.value == 0


def test_checked_build_reports_planted_short_extents(tmp_path):
    """Positive control: with RLSCAN_TEST_CHECK_SHORT=1 the checked build
    takes every [N,T] argument to end one row early.  Every real access stays
    inside the real arrays (nothing can fault); the accesses to the last row
    must be reported as violations (and skipped)."""
    from linear_recurrence_scan_gb300 import build
    checked = build.build_checked()
    env = dict(os.environ, RLSCAN_LIB=checked, RLSCAN_TEST_CHECK_SHORT="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "bounds_calls.py"), str(tmp_path / "short.npz")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    report = [line for line in r.stdout.splitlines() if line.startswith("BOUNDS")]
    assert len(report) == 1 and report[0].startswith("BOUNDS kind=1 "), report
    fields = dict(kv.split("=") for kv in report[0].split()[1:])
    assert int(fields["violations"]) > 0 and int(fields["first_site"]) in range(1, 10), report
