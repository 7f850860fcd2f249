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


# (N, T, row stride): packed rows, split rows on few rows (the regular shape,
# deferred finishing on the longest), split rows on 512 or more rows (the
# short-row shape with look-back), strided and unaligned rows
SHAPES = [(8, 128, None), (5, 37, None), (4096, 1024, None), (3, 3000, None), (2, 40000, None),
          (64, 1 << 16, None), (600, 5000, None), (520, 2100, 2104), (5, 96, 112), (5, 96, 104)]
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
                                   (64, 1 << 16, None), (600, 5000, None)],
                         ids=["8x128", "4096x1024", "3x5000", "64x65536", "600x5000"])
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


def _bf(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16)


def _u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.uint8)


OFF_SHAPES = [(8, 128, None), (5, 37, None), (4096, 1024, None), (3, 5000, None), (64, 1 << 16, None),
              (600, 5000, None), (520, 2100, 2104), (5, 96, 112)]
OFF_IDS = [f"{n}x{t}" + (f"_rs{rs}" if rs else "") for n, t, rs in OFF_SHAPES]


@pytest.mark.parametrize("variant", ["last_value", "trunc_bs"])
@pytest.mark.parametrize("shape", OFF_SHAPES, ids=OFF_IDS)
def test_compact_vtrace(shape, variant):
    """bf16 log-probabilities, values, rewards and bootstrap values, u8 flags;
    the oracle runs on the decoded inputs."""
    N, T, rs = shape
    trunc = variant == "trunc_bs"
    b = synthetic.vtrace_batch(N, T, 13 + T, 72, 0.01, 0.01 if trunc else 0.0, "2d" if trunc else "last")
    vals = {k: _bf(b[k]) for k in ("log_pi_target", "log_pi_behavior", "values", "rewards")}
    if trunc:
        vals["bootstrap_values"] = _bf(b["bootstrap_values"])
    fl = {"terminateds": _u8(b["terminateds"])}
    if trunc:
        fl["truncateds"] = _u8(b["truncateds"])
    last = None if trunc else torch.from_numpy(b["last_value"])
    dec = {k: v.float().numpy() for k, v in {**vals, **fl}.items()}
    vs_ref, adv_ref = oracle.vtrace(dec["log_pi_target"], dec["log_pi_behavior"], dec["values"], dec["rewards"],
                                    dec["terminateds"], dec.get("truncateds"), 0.99, 1.0, 1.0,
                                    dec.get("bootstrap_values"), None if last is None else last.numpy())
    args = [place(vals[k], rs) for k in ("log_pi_target", "log_pi_behavior", "values", "rewards")]
    args += [place(fl["terminateds"], rs), place(fl.get("truncateds"), rs), 0.99, 1.0, 1.0,
             place(vals.get("bootstrap_values"), rs), place(last, None)]
    vs32, adv32 = L().compute_vtrace(*args)
    assert vs32.dtype == torch.float32
    assert_close(vs32, vs_ref, f"compact vtrace targets {variant}", False)
    assert_close(adv32, adv_ref, f"compact vtrace advantages {variant}", False)
    vs16, adv16 = L().compute_vtrace(*args, out_dtype=torch.bfloat16)
    assert vs16.dtype == torch.bfloat16
    assert_close(vs16, vs_ref, f"compact vtrace targets {variant} (bf16 out)", True)
    assert_close(adv16, adv_ref, f"compact vtrace advantages {variant} (bf16 out)", True)
    assert torch.equal(vs16.view(torch.int16), vs32.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(adv16.view(torch.int16), adv32.to(torch.bfloat16).view(torch.int16))


@pytest.mark.parametrize("variant", ["plain", "trunc"])
@pytest.mark.parametrize("shape", OFF_SHAPES, ids=OFF_IDS)
def test_compact_retrace(shape, variant):
    """bf16 probabilities, Q-values and rewards, u8 flags."""
    N, T, rs = shape
    trunc = variant == "trunc"
    b = synthetic.retrace_batch(N, T, 14 + T, 73, 0.01, 0.01 if trunc else 0.0)
    vals = {k: _bf(b[k]) for k in ("pi_taken", "mu_taken", "q_values", "expected_next_q", "rewards")}
    fl = {"terminateds": _u8(b["terminateds"])}
    if trunc:
        fl["truncateds"] = _u8(b["truncateds"])
    dec = {k: v.float().numpy() for k, v in {**vals, **fl}.items()}
    q_ref, adv_ref = oracle.retrace(dec["pi_taken"], dec["mu_taken"], dec["q_values"], dec["expected_next_q"],
                                    dec["rewards"], dec["terminateds"], dec.get("truncateds"), 0.99, 0.95, 1.0, 1.0)
    args = [place(vals[k], rs) for k in ("pi_taken", "mu_taken", "q_values", "expected_next_q", "rewards")]
    args += [place(fl["terminateds"], rs), place(fl.get("truncateds"), rs), 0.99, 0.95, 1.0, 1.0]
    q32, adv32 = L().compute_retrace_from_probs(*args)
    assert_close(q32, q_ref, f"compact retrace targets {variant}", False)
    assert_close(adv32, adv_ref, f"compact retrace advantages {variant}", False)
    q16, adv16 = L().compute_retrace_from_probs(*args, out_dtype=torch.bfloat16)
    assert_close(q16, q_ref, f"compact retrace targets {variant} (bf16 out)", True)
    assert_close(adv16, adv_ref, f"compact retrace advantages {variant} (bf16 out)", True)
    assert torch.equal(q16.view(torch.int16), q32.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(adv16.view(torch.int16), adv32.to(torch.bfloat16).view(torch.int16))


def test_compact_offpolicy_rejects_mixed_storage():
    b = synthetic.vtrace_batch(4, 64, 3, 74, 0.01, 0.01, "2d")
    lpt, lpb, v, r = (_bf(b[k]).to(DEV) for k in ("log_pi_target", "log_pi_behavior", "values", "rewards"))
    term, trunc = _u8(b["terminateds"]).to(DEV), _u8(b["truncateds"]).to(DEV)
    with pytest.raises(TypeError):
        L().compute_vtrace(lpt, lpb, v.float(), r, term, trunc)
    with pytest.raises(ValueError):  # 2-D bootstrap without truncation flags
        L().compute_vtrace(lpt, lpb, v, r, term, None, bootstrap_values=_bf(b["bootstrap_values"]).to(DEV))
    with pytest.raises(ValueError):  # bf16 outputs from float32 inputs
        L().compute_retrace_from_probs(*(torch.ones(2, 8, device=DEV) for _ in range(6)),
                                       out_dtype=torch.bfloat16)
