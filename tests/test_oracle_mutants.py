"""Sensitivity of the oracle pins: plant one plausible mistake at a time in a
temporary copy of the oracle's C source (never in the repository file),
build it on the CPU, and require that at least one pin catches it.

The mistakes are the kinds a transcription of the pages could make: a
dropped gate, a wrong sign, an off-by-one index, a swapped clip, a seeded
carry that should be zero, a boundary convention keyed to the wrong step.
"""
import os

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "rlscan_oracle.c")

MUTANTS = {
    # GAE: bootstrap not gated by termination
    "gae_drop_term_gate": (
        "double delta = AT(r, row, t, rs) + gamma * (1.0 - te) * vn - vrow[t];",
        "double delta = AT(r, row, t, rs) + gamma * vn - vrow[t];"),
    # GAE: baseline added instead of subtracted
    "gae_sign_of_V": (
        "double delta = AT(r, row, t, rs) + gamma * (1.0 - te) * vn - vrow[t];",
        "double delta = AT(r, row, t, rs) + gamma * (1.0 - te) * vn + vrow[t];"),
    # GAE: window carry seeded with the bootstrap (double counting)
    "gae_seeded_carry": (
        "        double A_next = 0.0;\n",
        "        double A_next = last_value ? (double)last_value[row] : 0.0;\n"),
    # successor value taken at t instead of t+1
    "continuation_index": (
        "    return (t < T - 1) ? x[t + 1] : bs_last;",
        "    return (t < T - 1) ? x[t] : bs_last;"),
    # truncation does not mask the stored successor value
    "continuation_trunc_mask": (
        "(1.0 - AT(trunc, row, t, rs)) * x[t + 1] : 0.0;",
        "x[t + 1] : 0.0;"),
    # done ignores truncation
    "done_ignores_trunc": (
        "    double d = term + trunc;",
        "    double d = term + 0.0 * trunc;"),
    # V-trace: rho and c swapped in the decay
    "vtrace_c_rho_swap": (
        "+ gamma * c * (1.0 - done_flag(te, tr)) * D_next;",
        "+ gamma * rho * (1.0 - done_flag(te, tr)) * D_next;"),
    # V-trace: advantage bootstraps from V instead of vs
    "vtrace_adv_uses_V": (
        "double nvs = continuation(vs, t, T, trunc, bs, last_value, row, rs);",
        "double nvs = continuation(vrow, t, T, trunc, bs, last_value, row, rs);"),
    # Retrace: trace weight c_t instead of c_{t+1}
    "retrace_no_index_shift": (
        "c_next = lam * min2(c_bar, pi[t + 1] / AT(mu, row, t + 1, rs));",
        "c_next = lam * min2(c_bar, pi[t] / AT(mu, row, t, rs));"),
    # Retrace: lambda dropped from c
    "retrace_drop_lambda": (
        "c_next = lam * min2(c_bar, pi[t + 1] / AT(mu, row, t + 1, rs));",
        "c_next = min2(c_bar, pi[t + 1] / AT(mu, row, t + 1, rs));"),
    # Retrace: advantage not gated by termination
    "retrace_adv_gate": (
        "adv[t] = rho * (AT(r, row, t, rs) + gamma * (1.0 - te) * qn - AT(q, row, t, rs));",
        "adv[t] = rho * (AT(r, row, t, rs) + gamma * qn - AT(q, row, t, rs));"),
    # Retrace front end: successor Q weighted with the next step's probabilities
    "retrace_actions_next_step_weights": (
        "for (int64_t a = 0; a < A; ++a) s += (double)pt[a] * (double)qt[a];",
        "for (int64_t a = 0; a < A; ++a) s += (double)(t + 1 < T ? pt + A : pt)[a] * (double)qt[a];"),
    # Retrace front end: taken-action probability gathered from the Q-values
    "retrace_actions_gather_q": (
        "pi_d[t] = (double)pt[at];",
        "pi_d[t] = (double)qt[at];"),
    # Retrace front end: action index mirrored
    "retrace_actions_gather_index": (
        "pi_d[t] = (double)pt[at];",
        "pi_d[t] = (double)pt[A - 1 - at];"),
    # masked GAE: a masked step resets instead of carrying
    "masked_reset": (
        "            if (AT(mask, row, t, rs) == 0.0) {\n                A = carry;",
        "            if (AT(mask, row, t, rs) == 0.0) {\n                A = 0.0;"),
    # masked GAE: the carry across a masked step is discounted
    "masked_discounted_carry": (
        "            if (AT(mask, row, t, rs) == 0.0) {\n                A = carry;",
        "            if (AT(mask, row, t, rs) == 0.0) {\n                A = gamma * lam * carry;"),
    # masked GAE: mask ignored
    "masked_ignored": (
        "            if (AT(mask, row, t, rs) == 0.0) {\n                A = carry;",
        "            if (AT(mask, row, t, rs) == 2.0) {\n                A = carry;"),
    # TD(lambda): (1 - lambda) weight replaced by lambda
    "td_value_weight": (
        "double G = AT(r, row, t, rs) + gamma * (1.0 - lam) * nd * AT(nv, row, t, rs)",
        "double G = AT(r, row, t, rs) + gamma * lam * nd * AT(nv, row, t, rs)"),
    # TD(lambda): carry G_T dropped
    "td_zero_carry": (
        "        double G_next = returns_bs(bs, last_value, row, T - 1, T, rs);\n"
        "        for (int64_t t = T - 1; t >= 0; --t) {\n"
        "            double te = AT(term, row, t, rs);\n"
        "            double tr = trunc ? AT(trunc, row, t, rs) : 0.0;\n"
        "            double nd",
        "        double G_next = 0.0;\n"
        "        for (int64_t t = T - 1; t >= 0; --t) {\n"
        "            double te = AT(term, row, t, rs);\n"
        "            double tr = trunc ? AT(trunc, row, t, rs) : 0.0;\n"
        "            double nd"),
    # discounted returns: truncation bootstrap dropped
    "disc_drop_trunc_bootstrap": (
        "double G = AT(r, row, t, rs) + gamma * tr * returns_bs(bs, last_value, row, t, T, rs)",
        "double G = AT(r, row, t, rs)"),
    # eligibility traces gated on d_t instead of d_{t-1}
    "elig_gate_current_step": (
        "double z = AT(g, row, t, rs) + gamma * lam * (1.0 - d_prev) * z_prev;",
        "double z = AT(g, row, t, rs) + gamma * lam * (1.0 - AT(dones, row, t, rs)) * z_prev;"),
    # prefix sum: the two boundary conventions swapped
    "prefix_conventions_swapped": (
        "double gate = (boundary == 0) ? (1.0 - d_prev) : (1.0 - d_t);",
        "double gate = (boundary == 0) ? (1.0 - d_t) : (1.0 - d_prev);"),
    # generic scan: operands of the affine map transposed (beta added, alpha scaled)
    "linear_operands_swapped": (
        "                A = AT(alpha, row, t, rs) + AT(beta, row, t, rs) * A;\n"
        "                out[t] = A;\n"
        "            }\n"
        "        } else {",
        "                A = AT(beta, row, t, rs) + AT(alpha, row, t, rs) * A;\n"
        "                out[t] = A;\n"
        "            }\n"
        "        } else {"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name} not unique/absent"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(mutated), out=str(tmp_path / "libmutant.so"))
    failing = pins.failing_checks(oracle.Oracle(lib))
    assert failing, f"no pin caught the planted mistake {name}"


# The normalisation is numpy code in oracle/__init__.py: plant mistakes in a
# copy of that function's source and run the normalisation pins on it.
NORMALIZE_MUTANTS = {
    "biased_std": ("/ (n - 1)", "/ n"),
    "eps_in_variance": ("return dev / (std + eps)", "return dev / np.sqrt(std * std + eps)"),
    "mean_not_removed": ("return dev / (std + eps)", "return a / (std + eps)"),
}


@pytest.mark.parametrize("name", sorted(NORMALIZE_MUTANTS))
def test_normalize_pins_catch_planted_mistake(name):
    import inspect
    import numpy as np
    old, new = NORMALIZE_MUTANTS[name]
    src = inspect.getsource(oracle.normalize_advantages)
    assert src.count(old) == 1, f"mutation site for {name} not unique/absent"
    ns = {"np": np}
    exec(src.replace(old, new), ns)
    fn = ns["normalize_advantages"]
    caught = False
    for chk in (pins.check_normalize_against_stdlib, pins.check_normalize_invariants):
        try:
            chk(None, fn)
        except AssertionError:
            caught = True
    assert caught, f"no pin caught the planted mistake {name}"
