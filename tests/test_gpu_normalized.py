"""GAE with batch-normalised advantages against the float64 oracle: gae()
then normalize_advantages().  The returns are compared with their own
oracles (they use the raw advantages).  The device path is the scan with
per-CTA moment slots followed by the normalising pass (every block of which
combines the slots); the shapes cover its flat
(vector) walk, its strided and unaligned walks, packed and long-row scans,
each with the discounted returns requested (two scans per step) and
without them (one scan).

Tolerances: normalised advantages and returns |gpu - ref| <= 1e-4 + 1e-5 |ref|;
the reported (mean, std) within 1e-5 relative (+1e-6 absolute for the mean).
"""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrence_scan_gb300 import synthetic

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from linear_recurrence_scan_gb300 import build
    build.build()


def L():
    import linear_recurrence_scan_gb300 as lib
    return lib


def dev(a, rs=None):
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if rs is not None and a.ndim == 2 and rs != a.shape[1]:
        big = torch.zeros((a.shape[0], rs), dtype=torch.float32)
        big[:, : a.shape[1]] = t
        return big.to(DEV)[:, : a.shape[1]]
    return t.to(DEV)


def assert_disc(gpu, ref, what):
    g = gpu.double().cpu().numpy()
    err = np.abs(g - ref)
    bad = ~(err <= 1e-4 + 1e-5 * np.abs(ref))
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} off, first {i}: "
                             f"gpu {g[i]!r} ref {ref[i]!r}")


# (N, T, row stride or None, mode): packed (one tile, many tiles,
# truncations with a 2-D bootstrap, strided rows, a large batch), one tile
# per row, look-back and deferred look-back, element-wise staging
CASES = [
    (8, 128, None, "last"), (5, 37, None, "last"), (6, 1024, None, "last"),
    (3, 3000, None, "last"), (2, 40000, None, "2d"), (64, 1 << 16, None, "last"),
    (5, 100, 104, "2d"), (5, 100, 103, "last"), (4096, 1024, None, "last"),
    (512, 256, None, "2d"), (20000, 512, None, "last"),
]
IDS = [f"{n}x{t}" + (f"_rs{rs}" if rs else "") + f"_{m}" for n, t, rs, m in CASES]


@pytest.mark.parametrize("with_disc", [True, False], ids=["two_scans", "one_scan"])
@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_normalized_parity(case, with_disc):
    N, T, rs, mode = case
    b = synthetic.gae_batch(N, T, 3, 51, 0.01, 0.005 if mode == "2d" else 0.0, mode)
    g, lam, eps = 0.99, 0.95, 1e-8
    trunc = b["truncateds"]
    bs, last = b["bootstrap_values"], b["last_value"]
    raw = oracle.gae(b["rewards"], b["values"], b["terminateds"], trunc, g, lam, bs, last)
    want, (mean, sd) = oracle.normalize_advantages(raw, eps)
    outputs = ("advantages", "lambda_returns") + (("discounted_returns",) if with_disc else ())
    got = L().compute_gae_normalized(
        dev(b["rewards"], rs), dev(b["values"], rs), dev(b["terminateds"], rs), dev(trunc, rs), g,
        lam, dev(bs, rs), dev(last), eps, outputs=outputs, return_moments=True)
    adv, lret, mom = got[0], got[1], got[-1]
    disc = got[2] if with_disc else None
    assert_disc(adv, want, "normalized advantages")
    m = mom.double().cpu().numpy()
    assert abs(m[0] - mean) <= 1e-6 + 1e-5 * abs(mean), (m, mean)
    assert abs(m[1] - sd) <= 1e-5 * sd, (m, sd)
    nv = np.zeros_like(b["values"])
    nv[:, :-1] = b["values"][:, 1:]
    if mode == "last":
        nv[:, -1] = b["last_value"]
        lam_ref = oracle.lambda_returns(b["rewards"], nv, b["terminateds"], None, g, lam, None, last)
        disc_ref = oracle.discounted_returns(b["rewards"], b["terminateds"], None, g, None, last)
        assert_disc(lret, lam_ref, "lambda returns")
    else:
        assert_disc(lret, raw + b["values"].astype(np.float64), "lambda returns = raw A + V")
        disc_ref = oracle.discounted_returns(b["rewards"], b["terminateds"], trunc, g, bs, None)
    if with_disc:
        assert_disc(disc, disc_ref, "discounted returns")


def test_repeated_and_interleaved_calls():
    """Repeated calls, and calls interleaved with other entry points on the
    same workspace, agree (long rows: look-back tile states and moment slots
    share the workspace)."""
    N, T = 64, 1 << 14
    b = synthetic.gae_batch(N, T, 4, 52, 0.01, 0.0, "last")
    args = [dev(b[k]) for k in ("rewards", "values", "terminateds")]
    first = L().compute_gae_normalized(*args, None, 0.99, 0.95, None, dev(b["last_value"]))[0]
    for _ in range(3):
        L().compute_gae(*args, None, 0.99, 0.95, None, dev(b["last_value"]))
        again = L().compute_gae_normalized(*args, None, 0.99, 0.95, None, dev(b["last_value"]))[0]
        torch.testing.assert_close(again, first, rtol=1e-6, atol=1e-6)


def test_packed_repeated_and_interleaved_calls():
    """Packed tiles are assigned to CTAs statically, so the moment slots are
    summed in the same order every time: repeated calls, interleaved with
    other entry points and other shapes on the same workspace, give the same
    bits."""
    N, T = 4096, 1024
    b = synthetic.gae_batch(N, T, 5, 53, 0.01, 0.0, "last")
    args = [dev(b[k]) for k in ("rewards", "values", "terminateds")]
    first = L().compute_gae_normalized(*args, None, 0.99, 0.95, None, dev(b["last_value"]),
                                       return_moments=True)
    for _ in range(3):
        L().compute_gae(*args, None, 0.99, 0.95, None, dev(b["last_value"]))
        L().compute_gae_normalized(dev(b["rewards"][:64]), dev(b["values"][:64]), dev(b["terminateds"][:64]),
                                   None, 0.99, 0.95, None, dev(b["last_value"][:64]))
        again = L().compute_gae_normalized(*args, None, 0.99, 0.95, None, dev(b["last_value"]),
                                           return_moments=True)
        for x, y in zip(first, again):
            assert torch.equal(x, y)
    raw = oracle.gae(b["rewards"], b["values"], b["terminateds"], None, 0.99, 0.95, None, b["last_value"])
    assert_disc(first[0], oracle.normalize_advantages(raw, 1e-8)[0], "normalized advantages")
    L().workspace_status()  # raises if any wait timed out


def test_moments_region_over_stale_tile_states():
    """The moments region of a small normalising call lies where a larger
    call on the same workspace left its look-back tile states; the scan
    writes every slot the pass combines, so stale words there change
    nothing (one- and two-scan kernels)."""
    import ctypes
    from linear_recurrence_scan_gb300 import _native
    lib = _native.lib()
    vp = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    big = lib.rlscan_workspace_bytes(64, 1 << 16)
    N, T = 256, 1024
    need = lib.rlscan_gae_normalized_workspace_bytes(N, T)
    assert need < big
    ws = torch.empty(big, dtype=torch.uint8, device=DEV)
    assert lib.rlscan_workspace_init(vp(ws), big, s) == 0
    b = synthetic.gae_batch(64, 1 << 16, 6, 54, 0.01, 0.0, "last")
    d = {k: dev(b[k]) for k in ("rewards", "values", "terminateds", "last_value")}
    out = torch.empty((64, 1 << 16), device=DEV)
    for _ in range(2):  # tile states of two calls (two epochs) over the region
        assert lib.rlscan_gae(vp(d["rewards"]), vp(d["values"]), vp(d["terminateds"]), None, None,
                              vp(d["last_value"]), 64, 1 << 16, 1 << 16, 0.99, 0.95, vp(out), vp(ws), big, s) == 0
    c = synthetic.gae_batch(N, T, 7, 55, 0.01, 0.0, "last")
    e = {k: dev(c[k]) for k in ("rewards", "values", "terminateds", "last_value")}
    raw = oracle.gae(c["rewards"], c["values"], c["terminateds"], None, 0.99, 0.95, None, c["last_value"])
    want, (mean, sd) = oracle.normalize_advantages(raw, 1e-8)
    for disc in (None, torch.empty((N, T), device=DEV)):
        adv = torch.empty((N, T), device=DEV)
        mom = torch.empty(2, device=DEV)
        assert lib.rlscan_gae_normalized(vp(e["rewards"]), vp(e["values"]), vp(e["terminateds"]), None, None,
                                         vp(e["last_value"]), N, T, T, 0.99, 0.95, 1e-8, vp(adv), None, vp(disc),
                                         vp(mom), vp(ws), need, s) == 0
        assert_disc(adv, want, "normalized advantages over stale states")
        m = mom.double().cpu().numpy()
        assert abs(m[0] - mean) <= 1e-6 + 1e-5 * abs(mean) and abs(m[1] - sd) <= 1e-5 * sd, (m, mean, sd)
    assert lib.rlscan_workspace_status(vp(ws), big, s) == 0


def test_single_value_gives_nan():
    x = torch.ones(1, 1, device=DEV)
    adv, = L().compute_gae_normalized(x, x, torch.zeros(1, 1, device=DEV), outputs=("advantages",))
    assert torch.isnan(adv).all()


def test_eps_must_be_non_negative():
    from linear_recurrence_scan_gb300 import _native
    x = torch.ones(2, 4, device=DEV)
    with pytest.raises(_native.RlscanError):
        L().compute_gae_normalized(x, x, torch.zeros(2, 4, device=DEV), eps=-1.0)
