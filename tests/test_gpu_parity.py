"""CUDA path vs the float64 oracle, element by element, on seeded inputs.

Shapes span packed tiles (several rows per CTA tile), exactly one tile,
rows split across many tiles (decoupled look-back), ragged tails, T not a
multiple of 4 and row strides that are not (element-wise staging), and
strided rows.  Tolerances (floating point):
  * discounted estimators: |gpu - ref| <= 1e-4 + 1e-5 |ref| per element;
  * beta = 1 prefix sums on real inputs: <= 1e-6 * (running sum of |x| in
    the episode, the seed included);
  * prefix sums of integer-valued inputs (partial sums < 2^24): bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from linear_recurrence_scan_gb300 import build
    build.build()


def L():
    import linear_recurrence_scan_gb300 as lib
    return lib


def to_dev(a, rs=None):
    """numpy [N,T] -> CUDA tensor, optionally inside a wider row stride."""
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if rs is not None and a.ndim == 2 and rs != a.shape[1]:
        big = torch.full((a.shape[0], rs), float("nan"), dtype=torch.float32)
        big[:, : a.shape[1]] = t
        return big.to(DEV)[:, : a.shape[1]]
    return t.to(DEV)


def host(t):
    return t.double().cpu().numpy()


def assert_disc(gpu, ref, what):
    g = host(gpu)
    assert g.shape == ref.shape, what
    err = np.abs(g - ref)
    bound = 1e-4 + 1e-5 * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements off, first {tuple(i)}: "
                             f"gpu {g[tuple(i)]!r} ref {ref[tuple(i)]!r}")


# shapes: (N, T, row_stride or None)
SHAPES = [
    (8, 128, None),      # the pages' small PPO shape, packed
    (5, 37, None),       # T % 4 != 0: element-wise staging, packed
    (3, 1, None),
    (4, 2, None),
    (6, 1024, None),     # one row per heavy tile, two per light tile
    (3, 2048, None),     # exactly one light tile; two heavy tiles
    (4, 3000, None),     # look-back, ragged last tile
    (3, 2999, None),     # look-back with element-wise staging
    (2, 40000, None),    # many tiles per row
    (5, 100, 104),       # strided rows, bulk-copy path
    (5, 100, 103),       # strided rows, element-wise path
]
IDS = [f"{n}x{t}" + (f"_rs{rs}" if rs else "") for n, t, rs in SHAPES]


def flags(rng, N, T, p_term, p_trunc):
    term = (rng.random((N, T)) < p_term).astype(np.float32)
    trunc = (rng.random((N, T)) < p_trunc).astype(np.float32)
    trunc[term > 0] = 0
    return term, trunc


def bootstrap(rng, term, trunc):
    N, T = term.shape
    bs = rng.standard_normal((N, T)).astype(np.float32)
    keep = np.zeros((N, T), bool)
    if trunc is not None:
        keep |= trunc > 0
    keep[:, -1] |= term[:, -1] == 0
    return np.where(keep, bs, 0).astype(np.float32)


VARIANTS = ["plain", "last_value", "bs_column", "trunc", "trunc_bs"]


def make_case(seed, N, T, variant):
    rng = np.random.default_rng(seed)
    term, trunc = flags(rng, N, T, 0.02, 0.02)
    d = dict(r=rng.standard_normal((N, T)).astype(np.float32),
             v=rng.standard_normal((N, T)).astype(np.float32), term=term,
             trunc=None, bs=None, last=None)
    if variant == "last_value":
        d["last"] = rng.standard_normal(N).astype(np.float32)
    elif variant == "bs_column":
        d["bs"] = bootstrap(rng, term, None)
    elif variant == "trunc":
        d["trunc"] = trunc
    elif variant == "trunc_bs":
        d["trunc"] = trunc
        d["bs"] = bootstrap(rng, term, trunc)
    return d, rng


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("N,T,rs", SHAPES, ids=IDS)
def test_gae(N, T, rs, variant):
    c, _ = make_case(1, N, T, variant)
    ref = oracle.gae(c["r"], c["v"], c["term"], c["trunc"], 0.99, 0.95, c["bs"], c["last"])
    got = L().compute_gae(to_dev(c["r"], rs), to_dev(c["v"], rs), to_dev(c["term"], rs),
                          to_dev(c["trunc"], rs), 0.99, 0.95, to_dev(c["bs"], rs), to_dev(c["last"]))
    assert_disc(got, ref, "gae")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("N,T,rs", SHAPES, ids=IDS)
def test_gae_and_returns_fused(N, T, rs, variant):
    """One kernel, three outputs: GAE, lambda-returns = GAE + V, discounted
    returns on the same rewards, flags and bootstrap."""
    c, _ = make_case(11, N, T, variant)
    adv = oracle.gae(c["r"], c["v"], c["term"], c["trunc"], 0.99, 0.95, c["bs"], c["last"])
    disc = oracle.discounted_returns(c["r"], c["term"], c["trunc"], 0.99, c["bs"], c["last"])
    got = L().compute_gae_and_returns(to_dev(c["r"], rs), to_dev(c["v"], rs), to_dev(c["term"], rs),
                                      to_dev(c["trunc"], rs), 0.99, 0.95, to_dev(c["bs"], rs),
                                      to_dev(c["last"]))
    assert_disc(got[0], adv, "fused advantages")
    assert_disc(got[1], adv + c["v"].astype(np.float64), "fused lambda returns")
    assert_disc(got[2], disc, "fused discounted returns")


@pytest.mark.parametrize("outputs", [("discounted_returns",), ("lambda_returns", "advantages")])
def test_gae_and_returns_output_subsets(outputs):
    c, _ = make_case(12, 5, 3000, "last_value")
    ref = {"advantages": oracle.gae(c["r"], c["v"], c["term"], None, 0.99, 0.95, None, c["last"])}
    ref["lambda_returns"] = ref["advantages"] + c["v"].astype(np.float64)
    ref["discounted_returns"] = oracle.discounted_returns(c["r"], c["term"], None, 0.99, None,
                                                          c["last"])
    got = L().compute_gae_and_returns(to_dev(c["r"]), to_dev(c["v"]), to_dev(c["term"]), None,
                                      0.99, 0.95, None, to_dev(c["last"]), outputs=outputs)
    assert len(got) == len(outputs)
    for name, t in zip(outputs, got):
        assert_disc(t, ref[name], name)


@pytest.mark.parametrize("variant", VARIANTS + ["trunc_last"])
@pytest.mark.parametrize("N,T,rs", SHAPES, ids=IDS)
def test_vtrace(N, T, rs, variant):
    c, rng = make_case(2, N, T, "trunc" if variant == "trunc_last" else variant)
    if variant == "trunc_last":
        c["last"] = rng.standard_normal(N).astype(np.float32)
    lpb = rng.standard_normal((N, T)).astype(np.float32)
    lpt = (lpb + 0.5 * rng.standard_normal((N, T))).astype(np.float32)
    args = (0.99, 1.0, 0.9)
    vs, adv = oracle.vtrace(lpt, lpb, c["v"], c["r"], c["term"], c["trunc"], *args, c["bs"], c["last"])
    gvs, gadv = L().compute_vtrace(to_dev(lpt, rs), to_dev(lpb, rs), to_dev(c["v"], rs),
                                   to_dev(c["r"], rs), to_dev(c["term"], rs), to_dev(c["trunc"], rs),
                                   *args, to_dev(c["bs"], rs), to_dev(c["last"]))
    assert_disc(gvs, vs, "vtrace targets")
    assert_disc(gadv, adv, "vtrace advantages")


@pytest.mark.parametrize("trunc", [False, True])
@pytest.mark.parametrize("N,T,rs", SHAPES, ids=IDS)
def test_retrace(N, T, rs, trunc):
    rng = np.random.default_rng(3)
    term, tr = flags(rng, N, T, 0.02, 0.02)
    tr = tr if trunc else None
    mu = rng.uniform(0.05, 1, (N, T)).astype(np.float32)
    pi = (mu * np.exp(0.5 * rng.standard_normal((N, T)))).astype(np.float32)
    q, eq, r = (rng.standard_normal((N, T)).astype(np.float32) for _ in range(3))
    args = (0.99, 0.95, 1.0, 1.0)
    qret, adv = oracle.retrace(pi, mu, q, eq, r, term, tr, *args)
    gq, ga = L().compute_retrace_from_probs(*(to_dev(x, rs) for x in (pi, mu, q, eq, r, term, tr)),
                                            *args)
    assert_disc(gq, qret, "retrace targets")
    assert_disc(ga, adv, "retrace advantages")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("N,T,rs", SHAPES, ids=IDS)
def test_lambda_returns(N, T, rs, variant):
    c, rng = make_case(4, N, T, variant)
    nv = rng.standard_normal((N, T)).astype(np.float32)
    if c["trunc"] is not None:
        nv[c["trunc"] > 0] = 0
    ref = oracle.lambda_returns(c["r"], nv, c["term"], c["trunc"], 0.99, 0.9, c["bs"], c["last"])
    got = L().compute_lambda_returns(to_dev(c["r"], rs), to_dev(nv, rs), to_dev(c["term"], rs),
                                     to_dev(c["trunc"], rs), 0.99, 0.9, to_dev(c["bs"], rs),
                                     to_dev(c["last"]))
    assert_disc(got, ref, "lambda returns")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("N,T,rs", SHAPES, ids=IDS)
def test_discounted_returns(N, T, rs, variant):
    c, _ = make_case(5, N, T, variant)
    ref = oracle.discounted_returns(c["r"], c["term"], c["trunc"], 0.99, c["bs"], c["last"])
    got = L().compute_discounted_returns(to_dev(c["r"], rs), to_dev(c["term"], rs),
                                         to_dev(c["trunc"], rs), 0.99, to_dev(c["bs"], rs),
                                         to_dev(c["last"]))
    assert_disc(got, ref, "discounted returns")


@pytest.mark.parametrize("seeded", [False, True])
@pytest.mark.parametrize("N,T,rs", SHAPES, ids=IDS)
def test_eligibility_traces(N, T, rs, seeded):
    rng = np.random.default_rng(6)
    g = rng.standard_normal((N, T)).astype(np.float32)
    d = (rng.random((N, T)) < 0.02).astype(np.float32)
    seed = rng.standard_normal(N).astype(np.float32) if seeded else None
    ref = oracle.eligibility_traces(g, d, 0.99, 0.9, seed)
    got = L().compute_eligibility_traces(to_dev(g, rs), to_dev(d, rs), 0.99, 0.9, to_dev(seed))
    assert_disc(got, ref, "eligibility traces")


@pytest.mark.parametrize("boundary", ["ends_at", "starts_at"])
@pytest.mark.parametrize("N,T,rs", SHAPES, ids=IDS)
def test_prefix_sum_integers_bit_exact(N, T, rs, boundary):
    rng = np.random.default_rng(7)
    x = rng.integers(0, 10, (N, T)).astype(np.float32)
    d = (rng.random((N, T)) < 0.001).astype(np.float32)
    seed = rng.integers(0, 100, N).astype(np.float32)
    ref = oracle.episodic_prefix_sum(x, d, seed, boundary)
    got = L().compute_episodic_prefix_sum(to_dev(x, rs), to_dev(d, rs), to_dev(seed), boundary)
    np.testing.assert_array_equal(host(got), ref)


@pytest.mark.parametrize("boundary", ["ends_at", "starts_at"])
@pytest.mark.parametrize("N,T,rs", SHAPES, ids=IDS)
def test_prefix_sum_real_inputs(N, T, rs, boundary):
    rng = np.random.default_rng(8)
    x = rng.standard_normal((N, T)).astype(np.float32)
    d = (rng.random((N, T)) < 0.0005).astype(np.float32)
    seed = rng.standard_normal(N).astype(np.float32)
    ref = oracle.episodic_prefix_sum(x, d, seed, boundary)
    scale = oracle.episodic_prefix_sum(np.abs(x), d, np.abs(seed), boundary)
    got = host(L().compute_episodic_prefix_sum(to_dev(x, rs), to_dev(d, rs), to_dev(seed), boundary))
    err = np.abs(got - ref)
    # the beta = 1 bound: 1e-6 x the running sum of |alpha| within the episode
    assert (err <= 1e-6 * scale).all(), float((err / scale).max())


@pytest.mark.parametrize("direction", ["backward", "forward"])
@pytest.mark.parametrize("N,T,rs", SHAPES, ids=IDS)
def test_linear_scan(N, T, rs, direction):
    rng = np.random.default_rng(9)
    a = rng.standard_normal((N, T)).astype(np.float32)
    b = rng.uniform(0, 1, (N, T)).astype(np.float32)
    b[rng.random((N, T)) < 0.01] = 0
    carry = rng.standard_normal(N).astype(np.float32)
    ref = oracle.linear_scan(a, b, carry, direction)
    got = L().linear_scan(to_dev(a, rs), to_dev(b, rs), to_dev(carry), direction)
    assert_disc(got, ref, "linear scan")


def test_unit_beta_long_chain_carries_across_tiles():
    """beta = 1 everywhere: every tile's aggregate has b = 1, so the look-back
    must walk back to the row's first tile; integer inputs keep it exact."""
    rng = np.random.default_rng(10)
    N, T = 3, 9000
    x = rng.integers(0, 4, (N, T)).astype(np.float32)
    ones = np.ones((N, T), np.float32)
    carry = np.array([1, 2, 3], np.float32)
    for direction in ("forward", "backward"):
        ref = oracle.linear_scan(x, ones, carry, direction)
        got = L().linear_scan(to_dev(x), to_dev(ones), to_dev(carry), direction)
        np.testing.assert_array_equal(host(got), ref)


def test_empty_shapes_are_noops():
    lib = L()
    z = torch.zeros((0, 5), device=DEV)
    assert lib.compute_gae(z, z, z).shape == (0, 5)
    z = torch.zeros((3, 0), device=DEV)
    assert lib.compute_discounted_returns(z, z).shape == (3, 0)


def test_repeat_calls_reuse_workspace_without_clearing():
    """Epoch-tagged tile states: back-to-back calls on one workspace, with
    different data, each match the oracle (no stale state is consumed)."""
    lib = L()
    for seed in range(4):
        rng = np.random.default_rng(100 + seed)
        N, T = 4, 5000
        a = rng.standard_normal((N, T)).astype(np.float32)
        b = rng.uniform(0.5, 1, (N, T)).astype(np.float32)
        ref = oracle.linear_scan(a, b, None, "backward")
        assert_disc(lib.linear_scan(to_dev(a), to_dev(b)), ref, f"repeat {seed}")
    lib.workspace_status()
