"""Parity of every benchmark workload at its full size, in the launch
configuration bench.py times.

For each named workload and each kernel it times, the test builds the same
seeded inputs, makes the same C-ABI call through bench.py's own launcher
(same shapes, workspace, output dtypes, shape and staging choice), and
compares the outputs with the float64 oracle on three blocks of rows (the
first, a middle and the last rows; rows are independent, so the oracle on a
block is the oracle of those rows).  The normalised step, whose whitening
couples all rows, is compared on every element.  Compact-storage kernels are
compared against the oracle on the decoded (bfloat16 / uint8) inputs.

Tolerances: float32 outputs |gpu - ref| <= 1e-4 + 1e-5 |ref|; bfloat16
outputs add one bfloat16 rounding (2^-8 |ref|); integer prefix sums are
bit-exact.
"""
import ctypes
import os
import sys

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402

DEV = "cuda:0"
BLOCK = 8  # rows per compared block


def _blocks(N):
    starts = sorted({0, max(0, N // 2 - BLOCK // 2), max(0, N - BLOCK)})
    return [(r, min(N, r + BLOCK)) for r in starts]


def _kernels():
    out = []
    for wl_name, wl in bench.WORKLOADS.items():
        seen = set()
        for (name, _, c) in bench.step_kernels_of(wl_name) + list(wl["estimators"]):
            if name in seen:
                continue
            seen.add(name)
            out.append((wl_name, name))
    return out


KERNELS = _kernels()


def _refs(name, ref, rows):
    """The oracle's outputs in the order of the kernel's output buffers."""
    if name == "gae_returns_compact":  # advantages, lambda-returns (A + V), discounted returns
        adv, disc = ref
        return [adv, adv + bench._decode(rows["values"]).astype(np.float64), disc]
    return list(ref) if isinstance(ref, tuple) else [ref]


def _check(got, ref, what, bf16, exact):
    g = got.double().cpu().numpy()
    if exact:
        np.testing.assert_array_equal(g, ref, err_msg=what)
        return
    err = np.abs(g - ref)
    bound = 1e-4 + (1e-5 + (2.0 ** -8 if bf16 else 0.0)) * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} off, first {i}: gpu {g[i]!r} ref {ref[i]!r}")


@pytest.fixture(scope="module")
def lib():
    from linear_recurrence_scan_gb300 import _native, build
    build.build()
    return _native.lib()


@pytest.mark.parametrize("wl_name,name", KERNELS, ids=[f"{w}-{n}" for w, n in KERNELS])
def test_bench_workload_parity(lib, wl_name, name):
    wl = bench.WORKLOADS[wl_name]
    N, T = wl["N"], wl["T"]
    c = next(cc for (n, _, cc) in bench.step_kernels_of(wl_name) + list(wl["estimators"]) if n == name)
    batch = wl["gen"](N, T)
    ins, row_ins, nout = bench.IO[name]
    bufs = {k: torch.from_numpy(np.ascontiguousarray(batch[k])).to(DEV) for k in ins + row_ins}
    odt = torch.bfloat16 if bench.OUT_DTYPE.get(name) == "bf16" else torch.float32
    outs = [torch.empty((N, T), dtype=odt, device=DEV) for _ in range(nout)]
    stream = torch.cuda.current_stream()
    sh = ctypes.c_void_p(stream.cuda_stream)
    wsn = max(lib.rlscan_workspace_bytes(N, T), lib.rlscan_gae_normalized_workspace_bytes(N, T))
    ws_t = torch.empty(max(wsn, 16), dtype=torch.uint8, device=DEV)
    assert lib.rlscan_workspace_init(ctypes.c_void_p(ws_t.data_ptr()), ws_t.numel(), sh) == 0
    call = bench._launcher(name, c, bufs, outs, N, T, ctypes.c_void_p(ws_t.data_ptr()), wsn, sh)
    for _ in range(2):  # twice: the second call runs on a used workspace, as in the timed steps
        st = call()
        assert st == 0, (wl_name, name, st)
    torch.cuda.synchronize()
    assert lib.rlscan_workspace_status(ctypes.c_void_p(ws_t.data_ptr()), ws_t.numel(), sh) == 0
    bf16 = odt == torch.bfloat16
    exact = name == "episodic_prefix_sum"
    if name == "gae_normalized":
        refs = _refs(name, bench._oracle_call(name, c, batch), batch)
        for q, ref in enumerate(refs):
            _check(outs[q], ref, f"{wl_name} {name} output {q}", bf16, exact)
        return
    if name == "gae_returns":
        import oracle
        g, lam = float(c.get("gamma", 0.99)), float(c["lambda_"])
    for r0, r1 in _blocks(N):
        sub = bench._slice(batch, r0, r1)
        if name == "gae_returns":
            adv = oracle.gae(sub["rewards"], sub["values"], sub["terminateds"], None, g, lam, None,
                             sub["last_value"])
            disc = oracle.discounted_returns(sub["rewards"], sub["terminateds"], None, g, None,
                                             sub["last_value"])
            refs = [adv, adv + sub["values"].astype(np.float64), disc]
        else:
            refs = _refs(name, bench._oracle_call(name, c, sub), sub)
        for q, ref in enumerate(refs):
            _check(outs[q][r0:r1], ref, f"{wl_name} {name} output {q} rows {r0}:{r1}", bf16, exact)
