"""Size limits: one 2^26-step row (a look-back chain of 32768 tiles), millions
of very short rows (packed tiles), and a buffer of 2^31 elements per array
(64-bit indexing).  The largest case is generated on the device with a
seeded torch generator and compared with the oracle on sampled rows (rows
are independent, so the oracle computes each sampled row exactly).
Tolerance: |gpu - ref| <= 1e-4 + 1e-5 |ref|.
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


def assert_disc(got, ref, what):
    err = np.abs(got - ref)
    bad = ~(err <= 1e-4 + 1e-5 * np.abs(ref))
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} off, first {i}: "
                             f"gpu {got[i]!r} ref {ref[i]!r}")


def test_one_row_of_2p26_steps():
    T = 1 << 26
    b = synthetic.gae_batch(1, T, 2, 91, 0.001, 0.0, "last")
    keys = ("rewards", "values", "terminateds")
    got = L().compute_gae(*(torch.from_numpy(b[k]).to(DEV) for k in keys), None, 0.99, 0.95,
                          None, torch.from_numpy(b["last_value"]).to(DEV))
    ref = oracle.gae(b["rewards"], b["values"], b["terminateds"], None, 0.99, 0.95, None,
                     b["last_value"])
    assert_disc(got.double().cpu().numpy(), ref, "gae 1 x 2^26")


@pytest.mark.parametrize("shape", [(1 << 22, 4), (1 << 24, 1)], ids=["4Mx4", "16Mx1"])
def test_millions_of_short_rows(shape):
    N, T = shape
    b = synthetic.returns_batch(N, T, 2, 92)
    keys = ("rewards", "values", "terminateds")
    adv, lam, disc = L().compute_gae_and_returns(
        *(torch.from_numpy(b[k]).to(DEV) for k in keys), None, 0.99, 0.95, None,
        torch.from_numpy(b["last_value"]).to(DEV))
    ref = oracle.gae(b["rewards"], b["values"], b["terminateds"], None, 0.99, 0.95, None,
                     b["last_value"])
    assert_disc(adv.double().cpu().numpy(), ref, f"gae {N}x{T}")
    ref = oracle.discounted_returns(b["rewards"], b["terminateds"], None, 0.99, None,
                                    b["last_value"])
    assert_disc(disc.double().cpu().numpy(), ref, f"discounted {N}x{T}")


def test_two_to_the_31_elements_per_array():
    """65536 x 32768: every [N,T] array has 2^31 elements (8.6 GB), beyond
    32-bit indexing; the rows checked are spread over the buffer."""
    N, T = 1 << 16, 1 << 15
    if torch.cuda.get_device_properties(0).total_memory < 48 * (1 << 30):
        pytest.skip("needs about 40 GB of device memory")
    g = torch.Generator(device=DEV)
    g.manual_seed(1234)
    r = torch.randn((N, T), device=DEV, generator=g)
    v = torch.randn((N, T), device=DEV, generator=g)
    term = (torch.rand((N, T), device=DEV, generator=g) < 0.01).float()
    last = torch.randn((N,), device=DEV, generator=g)
    adv = L().compute_gae(r, v, term, None, 0.99, 0.95, None, last)
    rows = [0, 1, 4097, 32768, 40000, N - 2, N - 1]
    sel = torch.tensor(rows, device=DEV)
    host = {k: t.index_select(0, sel).cpu().numpy() for k, t in
            (("r", r), ("v", v), ("term", term))}
    ref = oracle.gae(host["r"], host["v"], host["term"], None, 0.99, 0.95, None,
                     last.index_select(0, sel).cpu().numpy())
    assert_disc(adv.index_select(0, sel).double().cpu().numpy(), ref, "gae 65536 x 32768")
    del r, v, term, adv
    torch.cuda.empty_cache()
