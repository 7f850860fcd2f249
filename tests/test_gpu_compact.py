"""Compact storage (bfloat16 values, uint8 / bool flags, float32 or
bfloat16 outputs) for GAE and fused GAE + returns.

The oracle runs on the decoded inputs (bfloat16 -> float is exact, so both
sides see the same numbers).  Float32 outputs: |gpu - ref| <= 1e-4 + 1e-5
|ref|.  Bfloat16 outputs: the same bound plus the output rounding (at most
2^-9 relative, taken as 2^-8), and bit equality with the float32 outputs
rounded to nearest even by torch.
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


def place(t, rs):
    """CUDA copy of t, inside rows of stride rs when given."""
    if t is None:
        return None
    if rs is None or t.dim() != 2 or rs == t.shape[1]:
        return t.to(DEV)
    big = torch.zeros((t.shape[0], rs), dtype=t.dtype)
    big[:, : t.shape[1]] = t
    return big.to(DEV)[:, : t.shape[1]]


def compact_batch(N, T, variant, seed, flag_dtype=torch.uint8):
    trunc = variant.startswith("trunc")
    b = synthetic.gae_batch(N, T, seed, 71, 0.02, 0.02 if trunc else 0.0,
                            "2d" if variant == "trunc_bs" else "last")
    bf = {k: torch.from_numpy(b[k]).to(torch.bfloat16) for k in ("rewards", "values")}
    fl = {"terminateds": torch.from_numpy(b["terminateds"]).to(flag_dtype)}
    if trunc:
        fl["truncateds"] = torch.from_numpy(b["truncateds"]).to(flag_dtype)
    if variant == "trunc_bs":
        bf["bootstrap_values"] = torch.from_numpy(b["bootstrap_values"]).to(torch.bfloat16)
    last = torch.from_numpy(b["last_value"]) if variant == "last_value" else None
    dec = {k: v.float().numpy() for k, v in {**bf, **fl}.items()}
    return bf, fl, last, dec


def assert_close(got, ref, what, bf16):
    g = got.double().cpu().numpy()
    err = np.abs(g - ref)
    bound = 1e-4 + (1e-5 + (2.0 ** -8 if bf16 else 0.0)) * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} off, first {i}: "
                             f"gpu {g[i]!r} ref {ref[i]!r}")


SHAPES = [(8, 128, None), (5, 37, None), (4096, 1024, None), (3, 3000, None), (2, 40000, None),
          (64, 1 << 16, None), (5, 96, 112), (5, 96, 104)]
SIDS = [f"{n}x{t}" + (f"_rs{rs}" if rs else "") for n, t, rs in SHAPES]
VARIANTS = ["plain", "last_value", "trunc", "trunc_bs"]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", SHAPES, ids=SIDS)
def test_compact_gae(shape, variant):
    N, T, rs = shape
    bf, fl, last, dec = compact_batch(N, T, variant, 11 + T, torch.uint8)
    ref = oracle.gae(dec["rewards"], dec["values"], dec["terminateds"], dec.get("truncateds"),
                     0.99, 0.95, dec.get("bootstrap_values"), None if last is None else last.numpy())
    args = (place(bf["rewards"], rs), place(bf["values"], rs), place(fl["terminateds"], rs),
            place(fl.get("truncateds"), rs), 0.99, 0.95, place(bf.get("bootstrap_values"), rs),
            place(last, None))
    f32 = L().compute_gae(*args)
    assert f32.dtype == torch.float32
    assert_close(f32, ref, f"compact gae {variant} (float32 out)", False)
    b16 = L().compute_gae(*args, out_dtype=torch.bfloat16)
    assert b16.dtype == torch.bfloat16
    assert_close(b16, ref, f"compact gae {variant} (bf16 out)", True)
    assert torch.equal(b16.view(torch.int16), f32.to(torch.bfloat16).view(torch.int16))


@pytest.mark.parametrize("variant", ["last_value", "trunc_bs"])
@pytest.mark.parametrize("shape", [(8, 128, None), (4096, 1024, None), (3, 5000, None),
                                   (64, 1 << 16, None)], ids=["8x128", "4096x1024", "3x5000",
                                                              "64x65536"])
def test_compact_gae_returns(shape, variant):
    N, T, rs = shape
    bf, fl, last, dec = compact_batch(N, T, variant, 12 + T, torch.bool)
    lv = None if last is None else last.numpy()
    trunc, bs = dec.get("truncateds"), dec.get("bootstrap_values")
    adv_ref = oracle.gae(dec["rewards"], dec["values"], dec["terminateds"], trunc, 0.99, 0.95, bs, lv)
    disc_ref = oracle.discounted_returns(dec["rewards"], dec["terminateds"], trunc, 0.99, bs, lv)
    for out_dtype in (torch.float32, torch.bfloat16):
        adv, lam, disc = L().compute_gae_and_returns(
            place(bf["rewards"], rs), place(bf["values"], rs), place(fl["terminateds"], rs),
            place(fl.get("truncateds"), rs), 0.99, 0.95, place(bf.get("bootstrap_values"), rs),
            place(last, None), out_dtype=out_dtype)
        b = out_dtype == torch.bfloat16
        assert_close(adv, adv_ref, "compact fused advantages", b)
        assert_close(lam, adv_ref + dec["values"].astype(np.float64), "compact fused lambda returns", b)
        assert_close(disc, disc_ref, "compact fused discounted returns", b)


def test_compact_rejects_mixed_storage():
    bf, fl, last, dec = compact_batch(4, 64, "last_value", 3)
    with pytest.raises(TypeError):
        L().compute_gae(place(bf["rewards"], None), place(bf["values"], None).float(),
                        place(fl["terminateds"], None), None, 0.99, 0.95, None,
                        place(last, None))
    with pytest.raises(ValueError):
        L().compute_gae(place(bf["rewards"], None), place(bf["values"], None),
                        place(fl["terminateds"], None), None, 0.99, 0.95,
                        place(bf["values"], None), None)
