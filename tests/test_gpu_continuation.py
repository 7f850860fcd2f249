"""Streaming continuation and offset views, on the device against the
float64 oracle.

A row scanned in two calls: the forward scans of the second part are seeded
with the first part's last output, and the backward scans of the first part
take the second part's first output as their carry.  Pieced together, the
two calls must match the oracle on the whole row, as one call does.  The two
calls compose tiles differently from one call, so the comparison is against
the oracle at its tolerance, |gpu - ref| <= 1e-4 + 1e-5 |ref|; integer prefix
sums are bit-exact.  The seed enters a forward recurrence ungated (d_{-1} = 0
in the API reference's eligibility traces and "ends_at" prefix sums), so for
those the caller gates it with the first part's last done flag.

The split falls at T1 = 2999, so the second part's base is not 16-byte
aligned, and views into a wider buffer at a column offset are checked
directly too.  Both take the element-wise staging path, and their outputs
must equal those of the aligned, contiguous call bit for bit (the
arithmetic does not depend on the staging).
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
N, T, T1 = 6, 5000, 2999


@pytest.fixture(scope="module", autouse=True)
def built():
    from linear_recurrence_scan_gb300 import build
    build.build()


def L():
    import linear_recurrence_scan_gb300 as lib
    return lib


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def close(got, ref, what):
    g = got.double().cpu().numpy()
    err = np.abs(g - ref)
    bad = ~(err <= 1e-4 + 1e-5 * np.abs(ref))
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} off, first {i}: gpu {g[i]!r} ref {ref[i]!r}")


def inputs(seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((N, T)).astype(np.float32)
    d = (rng.random((N, T)) < 1e-3).astype(np.float32)
    return rng, x, d


def test_eligibility_traces_continue_from_a_gated_seed():
    _, g, d = inputs(700)
    gd, dd = dev(g), dev(d)
    z1 = L().compute_eligibility_traces(gd[:, :T1], dd[:, :T1], 0.99, 0.9)
    seed = z1[:, -1] * (1.0 - dd[:, T1 - 1])
    z2 = L().compute_eligibility_traces(gd[:, T1:], dd[:, T1:], 0.99, 0.9, seed)
    close(torch.cat([z1, z2], 1), oracle.eligibility_traces(g, d, 0.99, 0.9), "eligibility traces in two calls")


@pytest.mark.parametrize("boundary", ["ends_at", "starts_at"])
def test_integer_prefix_sums_continue_bit_exactly(boundary):
    rng, _, d = inputs(701)
    x = rng.integers(0, 10, (N, T)).astype(np.float32)
    xd, dd = dev(x), dev(d)
    c1 = L().compute_episodic_prefix_sum(xd[:, :T1], dd[:, :T1], None, boundary)
    seed = c1[:, -1] * (1.0 - dd[:, T1 - 1]) if boundary == "ends_at" else c1[:, -1]
    c2 = L().compute_episodic_prefix_sum(xd[:, T1:], dd[:, T1:], seed, boundary)
    ref = oracle.episodic_prefix_sum(x, d, None, boundary)
    np.testing.assert_array_equal(torch.cat([c1, c2], 1).double().cpu().numpy(), ref)


@pytest.mark.parametrize("direction", ["forward", "backward"])
def test_linear_scan_continues_through_its_carry(direction):
    rng, a, _ = inputs(702)
    b = rng.uniform(0, 1, (N, T)).astype(np.float32)
    carry = rng.standard_normal(N).astype(np.float32)
    ad, bd = dev(a), dev(b)
    if direction == "forward":
        p1 = L().linear_scan(ad[:, :T1], bd[:, :T1], dev(carry), "forward")
        p2 = L().linear_scan(ad[:, T1:], bd[:, T1:], p1[:, -1], "forward")
    else:
        p2 = L().linear_scan(ad[:, T1:], bd[:, T1:], dev(carry), "backward")
        p1 = L().linear_scan(ad[:, :T1], bd[:, :T1], p2[:, 0], "backward")
    close(torch.cat([p1, p2], 1), oracle.linear_scan(a, b, carry, direction), f"{direction} scan in two calls")


def test_discounted_returns_continue_through_last_value():
    rng, r, term = inputs(703)
    last = rng.standard_normal(N).astype(np.float32)
    rd, td = dev(r), dev(term)
    g2 = L().compute_discounted_returns(rd[:, T1:], td[:, T1:], None, 0.99, None, dev(last))
    g1 = L().compute_discounted_returns(rd[:, :T1], td[:, :T1], None, 0.99, None, g2[:, 0])
    close(torch.cat([g1, g2], 1), oracle.discounted_returns(r, term, None, 0.99, None, last),
          "discounted returns in two calls")


def _offset_view(a):
    """a inside a wider buffer, one column in: the base is 4 bytes off a
    16-byte boundary, the row stride T + 4 a whole number of 16-byte units."""
    big = torch.full((a.shape[0], a.shape[1] + 4), float("nan"), dtype=torch.float32, device=DEV)
    big[:, 1:a.shape[1] + 1] = dev(a)
    v = big[:, 1:a.shape[1] + 1]
    assert v.data_ptr() % 16 == 4
    return v


def test_offset_views_match_the_aligned_call():
    rng, r, term = inputs(704)
    v = rng.standard_normal((N, T)).astype(np.float32)
    last = rng.standard_normal(N).astype(np.float32)
    got = L().compute_gae(_offset_view(r), _offset_view(v), _offset_view(term), None, 0.99, 0.95, None, dev(last))
    close(got, oracle.gae(r, v, term, None, 0.99, 0.95, None, last), "gae on offset views")
    aligned = L().compute_gae(dev(r), dev(v), dev(term), None, 0.99, 0.95, None, dev(last))
    assert torch.equal(got, aligned)
    g, d = r, term
    z = L().compute_eligibility_traces(_offset_view(g), _offset_view(d), 0.99, 0.9)
    assert torch.equal(z, L().compute_eligibility_traces(dev(g), dev(d), 0.99, 0.9))
