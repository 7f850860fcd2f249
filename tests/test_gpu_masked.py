"""GAE with observation-skip masking: the CUDA path against the float64
oracle, element by element, over the shapes of the parity suite (packed
tiles, one tile, look-back, deferred look-back on few long rows, ragged
tails, element-wise staging, strided rows), every bootstrap variant, random
masks and token-level LLM rollouts (prompt, tool observations, padding).
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


def dev(a, rs=None):
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if rs is not None and a.ndim == 2 and rs != a.shape[1]:
        big = torch.full((a.shape[0], rs), float("nan"), dtype=torch.float32)
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


SHAPES = [(8, 128, None), (5, 37, None), (3, 1, None), (6, 1024, None), (3, 3000, None),
          (3, 2999, None), (2, 40000, None), (64, 1 << 15, None), (5, 100, 104), (5, 100, 103)]
SIDS = [f"{n}x{t}" + (f"_rs{rs}" if rs else "") for n, t, rs in SHAPES]
VARIANTS = ["plain", "last_value", "bs_column", "trunc", "trunc_bs"]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", SHAPES, ids=SIDS)
def test_masked_gae_parity(shape, variant):
    N, T, rs = shape
    rng = np.random.default_rng(N * 7919 + T)
    b = synthetic.gae_batch(N, T, 5, 61, 0.02, 0.02 if variant.startswith("trunc") else 0.0,
                            "2d" if variant in ("bs_column", "trunc_bs") else "last")
    trunc = b["truncateds"] if variant.startswith("trunc") else None
    bs = b["bootstrap_values"] if variant in ("bs_column", "trunc_bs") else None
    last = b["last_value"] if variant == "last_value" else None
    if bs is not None and trunc is None:   # window bootstrap column only
        bs = bs.copy()
        bs[:, :-1] = 0.0
    mask = (rng.random((N, T)) < 0.7).astype(np.float32)
    ref = oracle.gae_masked(b["rewards"], b["values"], b["terminateds"], mask, trunc, 0.99, 0.95,
                            bs, last)
    got = L().compute_gae(dev(b["rewards"], rs), dev(b["values"], rs), dev(b["terminateds"], rs),
                          dev(trunc, rs), 0.99, 0.95, dev(bs, rs), dev(last), mask=dev(mask, rs))
    assert_disc(got, ref, f"masked gae {variant}")


def test_all_ones_mask_equals_gae():
    b = synthetic.gae_batch(16, 3000, 6, 62, 0.01, 0.01, "2d")
    args = [dev(b[k]) for k in ("rewards", "values", "terminateds", "truncateds")]
    plain = L().compute_gae(*args, 0.99, 0.95, dev(b["bootstrap_values"]))
    masked = L().compute_gae(*args, 0.99, 0.95, dev(b["bootstrap_values"]),
                             mask=torch.ones_like(args[0]))
    torch.testing.assert_close(masked, plain, rtol=0, atol=0)


@pytest.mark.parametrize("shape", [(64, 8192), (4096, 8192)], ids=["64x8192", "4096x8192"])
def test_llm_token_rollouts(shape):
    """Token-level LLM rollouts (the long-response regime of the paper's
    Sec. 9.1: up to 8192-token responses, 4096 rollouts per update)."""
    N, T = shape
    b = synthetic.llm_tokens_batch(N, T)
    ref = oracle.gae_masked(b["rewards"], b["values"], b["terminateds"], b["mask"], None, 1.0,
                            0.95, None, None)
    got = L().compute_gae(dev(b["rewards"]), dev(b["values"]), dev(b["terminateds"]), None, 1.0,
                          0.95, mask=dev(b["mask"]))
    assert_disc(got, ref, "llm token gae")
