"""Pins of the float64 oracle against facts the pages and the mathematics fix.

Each ``check_*`` function takes an oracle instance and raises AssertionError
when the oracle disagrees with:

* the hand-derived boundary-table cases in ``golden/boundary_tables.json``;
* brute-force O(T^2) direct summation of A_t = sum_k (prod beta) alpha_k
  (+ prod beta * carry), with alpha/beta built from the rl-triton paper's
  Table 1 and Sec. 3.2 -- a different algorithm from the oracle's loop;
* closed forms the pages state (GAE's exponentially weighted TD sum, the
  Retrace telescoped sum and its four-step polynomial, Appendix A's four-step
  polynomial, the TD(lambda) window-edge identity, the forward-view
  lambda-return, the Monte Carlo return at lambda = 1);
* special cases and cross-estimator identities (TD(1) = discounted returns,
  lambda-returns = GAE targets, on-policy V-trace = GAE(1), Retrace with
  pi = mu = GAE on Q, eligibility traces at lambda = 0, prefix-sum counters,
  starts_at vs shifted ends_at, severing at flags, split-row continuation).

The functions are shared by ``test_oracle_pins.py`` (the real oracle must
pass all of them) and ``test_oracle_mutants.py`` (every planted mistake must
fail at least one of them).
"""
from __future__ import annotations

import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "boundary_tables.json")

TOL = 1e-10


def _close(a, b, tol=TOL, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = np.abs(a - b)
    bound = tol * (1.0 + np.abs(b))
    if not np.all(err <= bound):
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: mismatch at {i}: {a[i]!r} vs {b[i]!r}")


def _f32(x):
    return np.asarray(x, dtype=np.float32)


# --------------------------------------------------------------------------
# random small inputs (test-local, seeded)
# --------------------------------------------------------------------------

def _flags(rng, N, T, p_term=0.12, p_trunc=0.1):
    term = (rng.random((N, T)) < p_term).astype(np.float32)
    trunc = (rng.random((N, T)) < p_trunc).astype(np.float32)
    trunc[term > 0] = 0
    return term, trunc


def _conforming_bs(rng, term, trunc):
    """bootstrap_values nonzero only at truncated steps and the last column."""
    N, T = term.shape
    bs = rng.standard_normal((N, T)).astype(np.float32)
    keep = np.zeros((N, T), dtype=bool)
    if trunc is not None:
        keep |= trunc > 0
    keep[:, -1] = True
    return np.where(keep, bs, 0).astype(np.float32)


# --------------------------------------------------------------------------
# brute force: direct summation
# --------------------------------------------------------------------------

def _direct_backward(alpha, beta, carry):
    alpha = np.asarray(alpha, np.float64)
    beta = np.asarray(beta, np.float64)
    N, T = alpha.shape
    out = np.zeros((N, T))
    for n in range(N):
        for t in range(T):
            acc, prod = 0.0, 1.0
            for k in range(t, T):
                acc += prod * alpha[n, k]
                prod *= beta[n, k]
            out[n, t] = acc + prod * carry[n]
    return out


def _direct_forward(alpha, beta, carry):
    alpha = np.asarray(alpha, np.float64)
    beta = np.asarray(beta, np.float64)
    N, T = alpha.shape
    out = np.zeros((N, T))
    for n in range(N):
        for t in range(T):
            acc, prod = 0.0, 1.0
            for k in range(t, -1, -1):
                acc += prod * alpha[n, k]
                prod *= beta[n, k]
            out[n, t] = acc + prod * carry[n]
    return out


def _d64(x, shape=None):
    if x is None:
        return np.zeros(shape)
    return np.asarray(x, np.float64)


def _table1_next(x, trunc, bs, last, T):
    """Successor value per the paper Sec. 3.2 and the API bootstrap rule
    (second transcription, vectorised)."""
    N = x.shape[0]
    bs = _d64(bs, (N, T)).copy()
    if last is not None:
        bs[:, -1] = np.asarray(last, np.float64)
    nxt = np.zeros((N, T))
    if trunc is not None:
        nxt[:, :-1] = x[:, 1:] * (1 - _d64(trunc)[:, :-1])
        return nxt + bs
    nxt[:, :-1] = x[:, 1:]
    nxt[:, -1] = bs[:, -1]
    return nxt


def check_brute_force(orc):
    rng = np.random.default_rng(1234)
    N, T = 4, 37
    g, l = 0.9, 0.8
    for trial in range(5):
        r = _f32(rng.standard_normal((N, T)))
        v = _f32(rng.standard_normal((N, T)))
        term, trunc = _flags(rng, N, T)
        use_trunc = trial in (2, 3)
        tr = trunc if use_trunc else None
        bs = _conforming_bs(rng, term, tr) if trial in (1, 2) else None
        last = _f32(rng.standard_normal(N)) if trial in (0, 4) else None
        d = np.minimum(1, _d64(term) + _d64(tr, (N, T)))

        # GAE (Table 1 row GAE, carry A_T = 0)
        vn = _table1_next(_d64(v), tr, bs, last, T)
        alpha = _d64(r) + g * (1 - _d64(term)) * vn - _d64(v)
        beta = g * l * (1 - d)
        _close(orc.gae(r, v, term, tr, g, l, bs, last),
               _direct_backward(alpha, beta, np.zeros(N)), what=f"gae brute {trial}")

        # V-trace (Table 1 row V-Trace)
        lpb = _f32(rng.standard_normal((N, T)))
        lpt = _f32(lpb + 0.5 * rng.standard_normal((N, T)))
        rb, cb = 1.1, 0.9
        ratio = np.exp(_d64(lpt) - _d64(lpb))
        rho, c = np.minimum(rb, ratio), np.minimum(cb, ratio)
        alpha = rho * (_d64(r) + g * (1 - _d64(term)) * vn - _d64(v))
        beta = g * c * (1 - d)
        delta = _direct_backward(alpha, beta, np.zeros(N))
        vs_ref = delta + _d64(v)
        nvs = _table1_next(vs_ref, tr, bs, last, T)
        adv_ref = rho * (_d64(r) + g * (1 - _d64(term)) * nvs - _d64(v))
        vs, adv = orc.vtrace(lpt, lpb, v, r, term, tr, g, rb, cb, bs, last)
        _close(vs, vs_ref, what=f"vtrace vs brute {trial}")
        _close(adv, adv_ref, what=f"vtrace adv brute {trial}")

        # Retrace (Table 1 row Retrace, c_T = 0)
        mu = _f32(rng.uniform(0.05, 1, (N, T)))
        pi = _f32(mu * np.exp(0.5 * rng.standard_normal((N, T))))
        q = _f32(rng.standard_normal((N, T)))
        eq = _f32(rng.standard_normal((N, T)))
        lr, cr, rr = 0.95, 1.2, 0.8
        ratio = _d64(pi) / _d64(mu)
        cc = lr * np.minimum(cr, ratio)
        cnext = np.zeros((N, T))
        cnext[:, :-1] = cc[:, 1:]
        alpha = _d64(r) + g * (1 - _d64(term)) * _d64(eq) - _d64(q)
        beta = g * cnext * (1 - d)
        qret_ref = _direct_backward(alpha, beta, np.zeros(N)) + _d64(q)
        qn = np.zeros((N, T))
        qn[:, :-1] = qret_ref[:, 1:]
        adv_ref = np.minimum(rr, ratio) * (_d64(r) + g * (1 - _d64(term)) * qn - _d64(q))
        qret, adv = orc.retrace(pi, mu, q, eq, r, term, tr, g, lr, cr, rr)
        _close(qret, qret_ref, what=f"retrace qret brute {trial}")
        _close(adv, adv_ref, what=f"retrace adv brute {trial}")

        # TD(lambda) and discounted returns (Table 1 rows, carry = bs[T-1])
        nv = _f32(rng.standard_normal((N, T)))
        bsf = _d64(bs, (N, T)).copy()
        if last is not None:
            bsf[:, -1] = _d64(last)
        trf = _d64(tr, (N, T))
        alpha = _d64(r) + g * (1 - l) * (1 - d) * _d64(nv) + g * trf * bsf
        beta = g * l * (1 - d)
        _close(orc.lambda_returns(r, nv, term, tr, g, l, bs, last),
               _direct_backward(alpha, beta, bsf[:, -1]), what=f"td brute {trial}")
        alpha = _d64(r) + g * trf * bsf
        beta = g * (1 - d)
        _close(orc.discounted_returns(r, term, tr, g, bs, last),
               _direct_backward(alpha, beta, bsf[:, -1]), what=f"disc brute {trial}")

        # forward scans (Table 1 rows Elig. Traces and Prefix Sum)
        dn = np.maximum(_d64(term), trf).astype(np.float32)
        seed = _f32(rng.standard_normal(N)) if trial % 2 else None
        sd = _d64(seed, (N,))
        dprev = np.zeros((N, T))
        dprev[:, 1:] = _d64(dn)[:, :-1]
        _close(orc.eligibility_traces(r, dn, g, l, seed),
               _direct_forward(_d64(r), g * l * (1 - dprev), sd), what=f"elig brute {trial}")
        _close(orc.episodic_prefix_sum(r, dn, seed, "ends_at"),
               _direct_forward(_d64(r), 1 - dprev, sd), what=f"prefix ends brute {trial}")
        _close(orc.episodic_prefix_sum(r, dn, seed, "starts_at"),
               _direct_forward(_d64(r), 1 - _d64(dn), sd), what=f"prefix starts brute {trial}")

        # generic scan (Eq. 1 and its forward mirror)
        b = _f32(rng.uniform(-1.2, 1.2, (N, T)))
        _close(orc.linear_scan(r, b, seed, "backward"), _direct_backward(r, b, sd),
               what=f"linear bwd brute {trial}")
        _close(orc.linear_scan(r, b, seed, "forward"), _direct_forward(r, b, sd),
               what=f"linear fwd brute {trial}")


# --------------------------------------------------------------------------
# golden boundary-table cases
# --------------------------------------------------------------------------

def check_golden(orc):
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    assert len(cases) >= 20
    for c in cases:
        inp = {k: np.asarray(v, np.float32) for k, v in c["inputs"].items()}
        p = c["params"]
        e = c["estimator"]
        if e == "gae":
            got = {"out": orc.gae(inp["rewards"], inp["values"], inp["terminateds"],
                                  inp.get("truncateds"), p["gamma"], p["lambda_"],
                                  inp.get("bootstrap_values"), inp.get("last_value"))}
        elif e == "vtrace":
            vs, adv = orc.vtrace(inp["log_pi_target"], inp["log_pi_behavior"], inp["values"],
                                 inp["rewards"], inp["terminateds"], inp.get("truncateds"),
                                 p["gamma"], p["rho_bar"], p["c_bar"],
                                 inp.get("bootstrap_values"), inp.get("last_value"))
            got = {"vs": vs, "adv": adv}
        elif e == "retrace":
            qret, adv = orc.retrace(inp["pi_taken"], inp["mu_taken"], inp["q_values"],
                                    inp["expected_next_q"], inp["rewards"], inp["terminateds"],
                                    inp.get("truncateds"), p["gamma"], p["lambda_"],
                                    p["c_bar"], p["rho_bar"])
            got = {"qret": qret, "adv": adv}
        elif e == "lambda_returns":
            got = {"out": orc.lambda_returns(inp["rewards"], inp["next_values"],
                                             inp["terminateds"], inp.get("truncateds"),
                                             p["gamma"], p["lambda_"],
                                             inp.get("bootstrap_values"), inp.get("last_value"))}
        elif e == "discounted_returns":
            got = {"out": orc.discounted_returns(inp["rewards"], inp["terminateds"],
                                                 inp.get("truncateds"), p["gamma"],
                                                 inp.get("bootstrap_values"),
                                                 inp.get("last_value"))}
        elif e == "eligibility_traces":
            got = {"out": orc.eligibility_traces(inp["gradients"], inp["dones"], p["gamma"],
                                                 p["lambda_"], inp.get("seed_values"))}
        elif e == "episodic_prefix_sum":
            got = {"out": orc.episodic_prefix_sum(inp["inputs"], inp["dones"],
                                                  inp.get("seed_values"), p["boundary"])}
        elif e == "linear_scan":
            got = {"out": orc.linear_scan(inp["alpha"], inp["beta"], inp.get("carry"),
                                          p["direction"])}
        else:
            raise AssertionError(f"unknown estimator {e}")
        for k, want in c["expected"].items():
            _close(got[k], np.asarray(want, np.float64), tol=0.0, what=c["id"] + ":" + k)


# --------------------------------------------------------------------------
# closed forms stated on the pages
# --------------------------------------------------------------------------

def check_gae_closed_forms(orc):
    """GAE: A_t = sum_k (gamma lambda)^k delta_{t+k} (paper Sec. 3.3.1; GAE
    tutorial Sec. 1); lambda = 0 gives delta; lambda = 1 gives the Monte Carlo
    return minus the baseline."""
    rng = np.random.default_rng(7)
    N, T, g, l = 3, 29, 0.97, 0.9
    r = _f32(rng.standard_normal((N, T)))
    v = _f32(rng.standard_normal((N, T)))
    last = _f32(rng.standard_normal(N))
    zero = np.zeros((N, T), np.float32)
    V = np.concatenate([_d64(v), _d64(last)[:, None]], axis=1)       # V(s_0..s_T)
    delta = _d64(r) + g * V[:, 1:] - V[:, :-1]
    want = np.array([[sum((g * l) ** k * delta[n, t + k] for k in range(T - t))
                      for t in range(T)] for n in range(N)])
    _close(orc.gae(r, v, zero, None, g, l, None, last), want, what="gae sum of (gl)^k delta")
    _close(orc.gae(r, v, zero, None, g, 0.0, None, last), delta, what="gae lambda=0")
    mc = np.array([[sum(g ** (k - t) * _d64(r)[n, k] for k in range(t, T))
                    + g ** (T - t) * V[n, T] for t in range(T)] for n in range(N)])
    _close(orc.gae(r, v, zero, None, g, 1.0, None, last), mc - V[:, :-1],
           what="gae lambda=1 Monte Carlo")
    # With flags: the exponentially weighted sum stops at the end of the
    # episode; terminated steps drop V(s_{t+1}); truncated ones take bs.
    term, trunc = _flags(rng, N, T, 0.1, 0.1)
    bs = _conforming_bs(rng, term, trunc)
    nxt = np.zeros((N, T))
    for n in range(N):
        for t in range(T):
            if trunc[n, t] > 0 or t == T - 1:
                nxt[n, t] = bs[n, t]
            elif term[n, t] == 0:
                nxt[n, t] = v[n, t + 1]
    delta = _d64(r) + g * nxt - _d64(v)
    want = np.zeros((N, T))
    for n in range(N):
        for t in range(T):
            acc = 0.0
            for k in range(t, T):
                acc += (g * l) ** (k - t) * delta[n, k]
                if term[n, k] > 0 or trunc[n, k] > 0:
                    break
            want[n, t] = acc
    _close(orc.gae(r, v, term, trunc, g, l, bs, None), want, what="gae episodic sum")


def check_vtrace_on_policy(orc):
    """On-policy V-trace (log ratios 0, rho_bar = c_bar = 1): the target is the
    n-step Monte Carlo return bootstrapped at the window end, i.e. GAE(1)+V,
    and the advantage equals target minus V (paper Sec. 3.3.2)."""
    rng = np.random.default_rng(8)
    N, T, g = 3, 31, 0.95
    r = _f32(rng.standard_normal((N, T)))
    v = _f32(rng.standard_normal((N, T)))
    last = _f32(rng.standard_normal(N))
    z = np.zeros((N, T), np.float32)
    V = np.concatenate([_d64(v), _d64(last)[:, None]], axis=1)
    mc = np.array([[sum(g ** (k - t) * _d64(r)[n, k] for k in range(t, T))
                    + g ** (T - t) * V[n, T] for t in range(T)] for n in range(N)])
    vs, adv = orc.vtrace(z, z, v, r, z, None, g, 1.0, 1.0, None, last)
    _close(vs, mc, what="vtrace on-policy target")
    _close(adv, mc - _d64(v), what="vtrace on-policy advantage")
    # with flags: targets equal GAE(lambda=1) + V on the same inputs
    term, trunc = _flags(rng, N, T, 0.1, 0.1)
    bs = _conforming_bs(rng, term, trunc)
    vs, _ = orc.vtrace(z, z, v, r, term, trunc, g, 1.0, 1.0, bs, None)
    _close(vs, orc.gae(r, v, term, trunc, g, 1.0, bs, None) + _d64(v),
           what="vtrace = gae(1) + V with flags")


def check_retrace_closed_forms(orc):
    """Retrace: Delta_t = sum_{k>=t} gamma^{k-t} (prod_{i=t+1}^k c_i) delta_k,
    truncated at the window end (Retrace tutorial Sec. 2), its four-step
    polynomial in which c_0 never appears (Sec. 5), and the two-step
    telescoping with EQ_0 = Q_1 (Sec. 1)."""
    rng = np.random.default_rng(9)
    N, T, g, l = 3, 23, 0.9, 0.8
    mu = _f32(rng.uniform(0.05, 1, (N, T)))
    pi = _f32(mu * np.exp(0.5 * rng.standard_normal((N, T))))
    q = _f32(rng.standard_normal((N, T)))
    eq = _f32(rng.standard_normal((N, T)))
    r = _f32(rng.standard_normal((N, T)))
    z = np.zeros((N, T), np.float32)
    c = l * np.minimum(1.0, _d64(pi) / _d64(mu))
    delta = _d64(r) + g * _d64(eq) - _d64(q)
    want = np.zeros((N, T))
    for n in range(N):
        for t in range(T):
            acc, prod = 0.0, 1.0
            for k in range(t, T):
                if k > t:
                    prod *= c[n, k]
                acc += g ** (k - t) * prod * delta[n, k]
            want[n, t] = acc
    qret, _ = orc.retrace(pi, mu, q, eq, r, z, None, g, l, 1.0, 1.0)
    _close(qret - _d64(q), want, what="retrace telescoped sum")
    # four-step polynomial: Delta_0 = d0 + g c1 d1 + g^2 c1 c2 d2 + g^3 c1 c2 c3 d3
    s = slice(0, 4)
    qret4, _ = orc.retrace(pi[:, s], mu[:, s], q[:, s], eq[:, s], r[:, s], z[:, s], None,
                           g, l, 1.0, 1.0)
    d, cc = delta[:, s], c[:, s]
    poly = (d[:, 0] + g * cc[:, 1] * d[:, 1] + g ** 2 * cc[:, 1] * cc[:, 2] * d[:, 2]
            + g ** 3 * cc[:, 1] * cc[:, 2] * cc[:, 3] * d[:, 3])
    _close(qret4[:, 0] - _d64(q)[:, 0], poly, what="retrace 4-step polynomial")
    # telescoping over two steps with full traces (c = 1) and EQ_0 = Q_1
    pi2 = np.ones((N, 2), np.float32)
    mu2 = np.full((N, 2), 0.5, np.float32)
    eq2 = eq[:, :2].copy()
    eq2[:, 0] = q[:, 1]
    qr2, _ = orc.retrace(pi2, mu2, q[:, :2], eq2, r[:, :2], z[:, :2], None, g, 1.0, 1.0, 1.0)
    _close(qr2[:, 0], _d64(r)[:, 0] + g * _d64(r)[:, 1] + g * g * _d64(eq2)[:, 1],
           what="retrace two-step telescoping")


def check_retrace_matches_gae_on_policy(orc):
    """With pi = mu and c_bar = 1 the traces are c = lambda, so Retrace on Q
    with EQ_t set to the successor value GAE would use is GAE on Q (the
    carries agree because both are zero at the window end)."""
    rng = np.random.default_rng(10)
    N, T, g, l = 3, 27, 0.93, 0.7
    q = _f32(rng.standard_normal((N, T)))
    r = _f32(rng.standard_normal((N, T)))
    term, trunc = _flags(rng, N, T, 0.1, 0.1)
    bs = _conforming_bs(rng, term, trunc)
    nxt = _table1_next(_d64(q), trunc, bs, None, T)
    p = _f32(rng.uniform(0.1, 1, (N, T)))
    qret, _ = orc.retrace(p, p, q, _f32(nxt), r, term, trunc, g, l, 1.0, 1.0)
    _close(qret - _d64(q), orc.gae(r, q, term, trunc, g, l, bs, None), tol=1e-9,
           what="retrace(pi=mu) = gae on Q")


def check_returns_closed_forms(orc):
    """TD(lambda): window edge G_{T-1} = r + gamma V(s_T) (paper Sec. 3.3.4);
    lambda = 0 is one-step TD and lambda = 1 is the discounted return
    (returns tutorial Sec. 2); the forward view is the lambda-weighted mixture
    of n-step returns (returns tutorial Sec. 4).  Discounted returns: each
    r_k discounted by gamma^{k-t} and cut at the first boundary flag, with the
    continuation value at truncations and at the window end (Sec. 1)."""
    rng = np.random.default_rng(11)
    N, T, g, l = 3, 21, 0.95, 0.75
    r = _f32(rng.standard_normal((N, T)))
    vnext = _f32(rng.standard_normal((N, T)))       # V(s_{t+1}) for t = 0..T-1
    z = np.zeros((N, T), np.float32)
    last = vnext[:, -1].copy()
    G = orc.lambda_returns(r, vnext, z, None, g, l, None, last)
    _close(G[:, -1], _d64(r)[:, -1] + g * _d64(last), what="td window edge")
    _close(orc.lambda_returns(r, vnext, z, None, g, 0.0, None, last),
           _d64(r) + g * _d64(vnext), what="td lambda=0")
    # forward view: G^l_t = (1-l) sum_{n=1}^{H-1} l^{n-1} G^(n)_t + l^{H-1} G^(H)_t
    want = np.zeros((N, T))
    for m in range(N):
        for t in range(T):
            H = T - t
            def nstep(n):
                return (sum(g ** k * float(r[m, t + k]) for k in range(n))
                        + g ** n * float(vnext[m, t + n - 1]))
            want[m, t] = ((1 - l) * sum(l ** (n - 1) * nstep(n) for n in range(1, H))
                          + l ** (H - 1) * nstep(H))
    _close(G, want, what="td forward view")
    # discounted returns with flags, written as the masked discounted sum
    term, trunc = _flags(rng, N, T, 0.1, 0.1)
    bs = _conforming_bs(rng, term, trunc)
    want = np.zeros((N, T))
    for m in range(N):
        for t in range(T):
            acc = 0.0
            for k in range(t, T):
                acc += g ** (k - t) * float(r[m, k])
                if term[m, k] > 0:
                    break
                if trunc[m, k] > 0 or k == T - 1:
                    acc += g ** (k - t + 1) * float(bs[m, k])
                    break
            want[m, t] = acc
    _close(orc.discounted_returns(r, term, trunc, g, bs, None), want, what="disc masked sum")
    # lambda = 1 reproduces discounted returns (with every flag kind)
    nv = _f32(rng.standard_normal((N, T)))
    nv[trunc > 0] = 0
    _close(orc.lambda_returns(r, nv, term, trunc, g, 1.0, bs, None),
           orc.discounted_returns(r, term, trunc, g, bs, None), what="td(1) = disc")


def check_lambda_returns_equal_gae_targets(orc):
    """lambda-returns equal GAE targets A + V when next_values are the
    successor values (returns tutorial Sec. 6), flags included."""
    rng = np.random.default_rng(12)
    N, T, g, l = 4, 33, 0.97, 0.9
    r = _f32(rng.standard_normal((N, T)))
    v = _f32(rng.standard_normal((N, T)))
    term, trunc = _flags(rng, N, T, 0.1, 0.1)
    bs = _conforming_bs(rng, term, trunc)
    nv = np.zeros((N, T), np.float32)
    nv[:, :-1] = v[:, 1:]
    nv[:, -1] = bs[:, -1]
    nv[trunc > 0] = 0
    _close(orc.lambda_returns(r, nv, term, trunc, g, l, bs, None),
           orc.gae(r, v, term, trunc, g, l, bs, None) + _d64(v), tol=1e-9,
           what="lambda returns = gae + V")
    last = _f32(rng.standard_normal(N))
    nv[:, -1] = last
    nv[:, :-1] = v[:, 1:]
    _close(orc.lambda_returns(r, nv, term, None, g, l, None, last),
           orc.gae(r, v, term, None, g, l, None, last) + _d64(v), tol=1e-9,
           what="lambda returns = gae + V (last_value)")


def check_forward_scans(orc):
    """Eligibility traces: within an episode z_t = sum (gamma lambda)^{t-k} g_k
    plus the decayed seed while no reset has happened (returns tutorial
    Sec. 3-4); lambda = 0 gives z = g.  Prefix sums: x = 1 counts steps within
    the episode; starts_at on flags shifted right equals ends_at."""
    rng = np.random.default_rng(13)
    N, T, g, l = 3, 40, 0.9, 0.8
    gr = _f32(rng.standard_normal((N, T)))
    dn = (rng.random((N, T)) < 0.12).astype(np.float32)
    seed = _f32(rng.standard_normal(N))
    want = np.zeros((N, T))
    for m in range(N):
        for t in range(T):
            acc, k = 0.0, t
            while True:
                acc += (g * l) ** (t - k) * float(gr[m, k])
                if k == 0:
                    acc += (g * l) ** (t + 1) * float(seed[m])
                    break
                if dn[m, k - 1] > 0:
                    break
                k -= 1
            want[m, t] = acc
    _close(orc.eligibility_traces(gr, dn, g, l, seed), want, what="elig episodic sum")
    _close(orc.eligibility_traces(gr, dn, g, 0.0, seed), _d64(gr), what="elig lambda=0")
    ones = np.ones((N, T), np.float32)
    cnt = np.zeros((N, T))
    for m in range(N):
        c = 0
        for t in range(T):
            c = c + 1 if (t == 0 or dn[m, t - 1] == 0) else 1
            cnt[m, t] = c
    _close(orc.episodic_prefix_sum(ones, dn, None, "ends_at"), cnt, tol=0.0,
           what="prefix counter")
    x = _f32(rng.integers(0, 10, (N, T)))
    shifted = np.zeros_like(dn)
    shifted[:, 1:] = dn[:, :-1]
    _close(orc.episodic_prefix_sum(x, shifted, seed, "starts_at"),
           orc.episodic_prefix_sum(x, dn, seed, "ends_at"), tol=0.0,
           what="starts_at(shift) = ends_at")


def check_appendix_a_polynomial(orc):
    """Generic scan, T = 4 (paper Sec. 5.1 / Appendix A):
    A_0 = a0 + b0 (a1 + b1 (a2 + b2 a3)); the forward mirror likewise."""
    rng = np.random.default_rng(14)
    a = _f32(rng.standard_normal((5, 4)))
    b = _f32(rng.standard_normal((5, 4)))
    A, B = _d64(a), _d64(b)
    got = orc.linear_scan(a, b, None, "backward")
    _close(got[:, 0], A[:, 0] + B[:, 0] * (A[:, 1] + B[:, 1] * (A[:, 2] + B[:, 2] * A[:, 3])),
           what="appendix A polynomial")
    got = orc.linear_scan(a, b, None, "forward")
    _close(got[:, 3], A[:, 3] + B[:, 3] * (A[:, 2] + B[:, 2] * (A[:, 1] + B[:, 1] * A[:, 0])),
           what="forward polynomial")


def check_severing_and_continuation(orc):
    """Paper Sec. 5.2: nothing crosses a done flag -- perturbing every input
    after a flag leaves the outputs up to the flag unchanged (backward), and
    perturbing inputs before a flag leaves outputs after it unchanged
    (forward).  Streaming continuation: a row split in two, the second part
    seeded (forward) or carried (backward) with the first part's boundary
    output, equals one call."""
    rng = np.random.default_rng(15)
    N, T, g, l, k = 2, 30, 0.9, 0.8, 13
    r = _f32(rng.standard_normal((N, T)))
    v = _f32(rng.standard_normal((N, T)))
    term = np.zeros((N, T), np.float32)
    term[:, k] = 1
    r2, v2 = r.copy(), v.copy()
    r2[:, k + 1:] += 1.5
    v2[:, k + 1:] -= 2.0
    last = _f32(rng.standard_normal(N))
    a = orc.gae(r, v, term, None, g, l, None, last)
    b = orc.gae(r2, v2, term, None, g, l, None, last)
    _close(a[:, :k + 1], b[:, :k + 1], tol=0.0, what="gae severing")
    a = orc.discounted_returns(r, term, None, g, None, last)
    b = orc.discounted_returns(r2, term, None, g, None, last + 1)
    _close(a[:, :k + 1], b[:, :k + 1], tol=0.0, what="disc severing")
    a = orc.eligibility_traces(r, term, g, l, None)
    r3 = r.copy()
    r3[:, :k + 1] += 3.0
    b = orc.eligibility_traces(r3, term, g, l, last)
    _close(a[:, k + 1:], b[:, k + 1:], tol=0.0, what="elig severing")
    # continuation
    al = _f32(rng.standard_normal((N, T)))
    be = _f32(rng.uniform(0, 1, (N, T)))
    full = orc.linear_scan(al, be, last, "forward")
    part = orc.linear_scan(al[:, k:].copy(), be[:, k:].copy(), _f32(full[:, k - 1]), "forward")
    _close(part, full[:, k:], tol=1e-6, what="forward continuation")
    full = orc.linear_scan(al, be, last, "backward")
    part = orc.linear_scan(al[:, :k].copy(), be[:, :k].copy(), _f32(full[:, k]), "backward")
    _close(part, full[:, :k], tol=1e-6, what="backward continuation")
    full = orc.discounted_returns(r, np.zeros((N, T), np.float32), None, g, None, last)
    part = orc.discounted_returns(r[:, :k].copy(), np.zeros((N, k), np.float32), None, g,
                                  None, _f32(full[:, k]))
    _close(part, full[:, :k], tol=1e-6, what="disc continuation")
    x = _f32(rng.integers(0, 10, (N, T)))
    dn = (rng.random((N, T)) < 0.1).astype(np.float32)
    full = orc.episodic_prefix_sum(x, dn, None, "ends_at")
    # the carry into step k is severed when dn[k-1] = 1; emulate with the seed
    seed2 = _f32(np.where(dn[:, k - 1] > 0, 0.0, full[:, k - 1]))
    dn2 = dn[:, k:].copy()
    part = orc.episodic_prefix_sum(x[:, k:].copy(), dn2, seed2, "ends_at")
    _close(part, full[:, k:], tol=0.0, what="prefix continuation")


# --------------------------------------------------------------------------
# Retrace from the full action-space inputs ([N,T,A] probabilities and
# successor Q-values, int64 actions)
# --------------------------------------------------------------------------

GOLDEN_RETRACE_ACTIONS = os.path.join(os.path.dirname(__file__), "golden",
                                      "retrace_actions_worked.json")


def _retrace_actions_inputs(rng, N, T, A, dyadic):
    if dyadic:  # every product and sum below is exact in float32 and float64
        probs = _f32(rng.integers(0, 9, (N, T, A)) / 8.0)
        nq = _f32(rng.integers(-8, 9, (N, T, A)))
    else:
        w = rng.random((N, T, A)) + 0.05
        probs = _f32(w / w.sum(-1, keepdims=True))
        nq = _f32(rng.standard_normal((N, T, A)))
    acts = rng.integers(0, A, (N, T)).astype(np.int64)
    mu = _f32(rng.uniform(0.1, 1.0, (N, T)))
    q = _f32(rng.standard_normal((N, T)))
    r = _f32(rng.standard_normal((N, T)))
    term, trunc = _flags(rng, N, T, 0.1, 0.1)
    return probs, nq, acts, mu, q, r, term, trunc


def check_retrace_actions_golden(orc):
    """The hand-worked two-action example (API reference, compute_retrace)."""
    with open(GOLDEN_RETRACE_ACTIONS) as f:
        c = json.load(f)
    i, p = c["inputs"], c["params"]
    qret, adv = orc.retrace_actions(
        _f32(i["action_probs_target"]), _f32(i["action_probs_behavior"]), _f32(i["q_values"]),
        _f32(i["next_q_values_all"]), np.asarray(i["actions"], np.int64), _f32(i["rewards"]),
        _f32(i["terminateds"]), None, p["gamma"], p["lambda_"], p["c_bar"], p["rho_bar"])
    _close(qret, c["expected"]["retrace_targets"], tol=0.0, what="retrace actions golden Q_ret")
    _close(adv, c["expected"]["advantages"], tol=0.0, what="retrace actions golden advantages")


def check_retrace_actions_reduction(orc):
    """The action dimension enters only through the library gather
    pi_t = take_along_axis(pi_target, actions) and the library contraction
    EQ_t = einsum(pi_target[t,:], Qnext[t,:]) at the same step: with
    binary-fraction inputs both are exact, and the result must equal Retrace
    on those per-step values bit for bit."""
    rng = np.random.default_rng(21)
    N, T, A, g, l = 4, 37, 5, 0.9, 0.8
    probs, nq, acts, mu, q, r, term, trunc = _retrace_actions_inputs(rng, N, T, A, True)
    pi = np.take_along_axis(probs, acts[..., None], axis=-1)[..., 0]
    eq = np.einsum("nta,nta->nt", probs.astype(np.float64), nq.astype(np.float64))
    assert np.array_equal(_f32(eq).astype(np.float64), eq)
    for tr in (None, trunc):
        want = orc.retrace(pi, mu, q, _f32(eq), r, term, tr, g, l, 1.0, 0.9)
        got = orc.retrace_actions(probs, mu, q, nq, acts, r, term, tr, g, l, 1.0, 0.9)
        _close(got[0], want[0], tol=0.0, what="retrace actions targets vs gathered inputs")
        _close(got[1], want[1], tol=0.0, what="retrace actions advantages vs gathered inputs")


def check_retrace_actions_relabelling(orc):
    """Renaming the actions by a permutation (columns of both [N,T,A] arrays
    and the action indices together) leaves every output unchanged."""
    rng = np.random.default_rng(22)
    N, T, A, g, l = 3, 29, 4, 0.95, 0.9
    probs, nq, acts, mu, q, r, term, trunc = _retrace_actions_inputs(rng, N, T, A, False)
    sigma = np.array([2, 0, 3, 1])
    inv = np.argsort(sigma)
    base = orc.retrace_actions(probs, mu, q, nq, acts, r, term, trunc, g, l, 1.0, 1.0)
    perm = orc.retrace_actions(np.ascontiguousarray(probs[..., inv]), mu, q,
                               np.ascontiguousarray(nq[..., inv]), sigma[acts], r, term, trunc,
                               g, l, 1.0, 1.0)
    _close(perm[0], base[0], tol=1e-12, what="retrace actions relabelled targets")
    _close(perm[1], base[1], tol=1e-12, what="retrace actions relabelled advantages")


def check_retrace_actions_one_hot(orc):
    """A deterministic target policy (one-hot on action b_t) with mu = 1:
    EQ_t = Qnext[t, b_t], the traces are c_t = lambda [a_t = b_t] and rho_t =
    [a_t = b_t], and Delta_t is the telescoped sum
    sum_{k>=t} gamma^{k-t} prod_{i=t+1}^{k} c_i (1 - done_{i-1}) delta_k
    (Retrace tutorial Sec. 2) with delta_k = r_k + gamma (1-term_k) EQ_k - Q_k."""
    rng = np.random.default_rng(23)
    N, T, A, g, l = 3, 19, 3, 0.9, 0.7
    b = rng.integers(0, A, (N, T))
    acts = np.where(rng.random((N, T)) < 0.7, b, rng.integers(0, A, (N, T))).astype(np.int64)
    probs = _f32(np.eye(A)[b])
    nq = _f32(rng.standard_normal((N, T, A)))
    mu = np.ones((N, T), np.float32)
    q = _f32(rng.standard_normal((N, T)))
    r = _f32(rng.standard_normal((N, T)))
    term, trunc = _flags(rng, N, T, 0.1, 0.1)
    qret, adv = orc.retrace_actions(probs, mu, q, nq, acts, r, term, trunc, g, l, 1.0, 1.0)
    hit = (acts == b).astype(np.float64)
    eqv = np.take_along_axis(_d64(nq), b[..., None], axis=-1)[..., 0]
    delta = _d64(r) + g * (1.0 - _d64(term)) * eqv - _d64(q)
    done = np.minimum(1.0, _d64(term) + _d64(trunc))
    want = np.zeros((N, T))
    for n in range(N):
        for t in range(T):
            acc, prod = 0.0, 1.0
            for k in range(t, T):
                if k > t:
                    prod *= l * hit[n, k] * (1.0 - done[n, k - 1])
                acc += g ** (k - t) * prod * delta[n, k]
            want[n, t] = acc
    _close(qret - _d64(q), want, what="retrace one-hot telescoped sum")
    qn = np.concatenate([qret[:, 1:], np.zeros((N, 1))], axis=1)
    _close(adv, hit * (_d64(r) + g * (1.0 - _d64(term)) * qn - _d64(q)),
           what="retrace one-hot advantages")


# --------------------------------------------------------------------------
# observation-skip masking (GAE)
# --------------------------------------------------------------------------

def check_gae_masked(orc):
    """Observation-skip GAE (paper Sec. 9.3: the recurrence is carried across
    masked tokens, beta = 1): an all-ones mask is plain GAE; an all-zeros
    mask gives zero; a hand-worked case; and brute force -- for an unmasked
    step, A_t = sum over unmasked k >= t of (prod over unmasked j in [t, k)
    of gamma lambda (1 - done_j)) delta_k, with delta from the paper's
    successor rule; a masked step holds the next unmasked step's value (0
    past the last one)."""
    rng = np.random.default_rng(41)
    N, T, g, l = 4, 29, 0.93, 0.8
    r = _f32(rng.standard_normal((N, T)))
    v = _f32(rng.standard_normal((N, T)))
    term, trunc = _flags(rng, N, T, 0.1, 0.1)
    bs = _conforming_bs(rng, term, trunc)
    ones = np.ones((N, T), np.float32)
    _close(orc.gae_masked(r, v, term, ones, trunc, g, l, bs), orc.gae(r, v, term, trunc, g, l, bs),
           tol=0.0, what="all-ones mask = GAE")
    _close(orc.gae_masked(r, v, term, 0 * ones, trunc, g, l, bs), np.zeros((N, T)), tol=0.0,
           what="all-zeros mask")
    # hand-worked: r = (1,2,3,4), V = 0, no flags, mask (1,0,1,0), gamma 0.5,
    # lambda 1: A_3 = 0 (masked, past the end), A_2 = 3, A_1 = A_2 = 3,
    # A_0 = 1 + 0.5 * 3 = 2.5
    hw = orc.gae_masked(_f32([[1, 2, 3, 4]]), _f32([[0, 0, 0, 0]]), _f32([[0, 0, 0, 0]]),
                        _f32([[1, 0, 1, 0]]), None, 0.5, 1.0)
    _close(hw, [[2.5, 3.0, 3.0, 0.0]], tol=0.0, what="masked hand-worked")
    for tr, b, last in ((None, None, _f32(rng.standard_normal(N))), (trunc, bs, None)):
        mask = (rng.random((N, T)) < 0.6).astype(np.float32)
        got = orc.gae_masked(r, v, term, mask, tr, g, l, b, last)
        nxt = _table1_next(_d64(v), tr, b, last, T)
        delta = _d64(r) + g * (1 - _d64(term)) * nxt - _d64(v)
        done = np.minimum(1.0, _d64(term) + _d64(tr, (N, T)))
        want = np.zeros((N, T))
        for n in range(N):
            for t in range(T):
                t0 = t
                while t0 < T and mask[n, t0] == 0:
                    t0 += 1
                acc, prod = 0.0, 1.0
                for k in range(t0, T):
                    if mask[n, k] == 0:
                        continue
                    acc += prod * delta[n, k]
                    prod *= g * l * (1 - done[n, k])
                want[n, t] = acc
        _close(got, want, what="masked GAE brute force")


# --------------------------------------------------------------------------
# advantage normalisation (per-batch whitening)
# --------------------------------------------------------------------------

def check_normalize_against_stdlib(orc, normalize=None):
    """(A - mean) / (std + eps) with the unbiased standard deviation, against
    Python's statistics.fmean / statistics.stdev (an independent
    implementation), for several shapes and eps."""
    import statistics
    normalize = normalize or _normalize_of(orc)
    rng = np.random.default_rng(31)
    for shape, eps in (((1, 2), 0.0), ((3, 7), 1e-8), ((4, 33), 0.5), ((2, 100), 1e-3)):
        x = rng.standard_normal(shape) * 3.0 + 1.5
        vals = [float(v) for v in x.ravel()]
        mean, sd = statistics.fmean(vals), statistics.stdev(vals)
        got, (gm, gs) = normalize(x, eps)
        _close(gm, mean, tol=1e-12, what="normalize mean")
        _close(gs, sd, tol=1e-12, what="normalize std")
        _close(got, (x - mean) / (sd + eps), tol=1e-12, what="normalized values")


def check_normalize_invariants(orc, normalize=None):
    """With eps = 0 the result has mean 0 and unbiased standard deviation 1,
    and is unchanged by a positive affine map of the inputs."""
    normalize = normalize or _normalize_of(orc)
    rng = np.random.default_rng(32)
    x = rng.standard_normal((5, 40))
    y, _ = normalize(x, 0.0)
    _close(y.mean(), 0.0, tol=1e-12, what="normalized mean")
    _close(y.std(ddof=1), 1.0, tol=1e-12, what="normalized std")
    z, _ = normalize(2.5 * x - 7.0, 0.0)
    _close(z, y, tol=1e-10, what="normalization affine invariance")


def _normalize_of(orc):
    import oracle
    return getattr(orc, "normalize_advantages", oracle.normalize_advantages)


ALL_CHECKS = [
    check_golden,
    check_brute_force,
    check_gae_closed_forms,
    check_vtrace_on_policy,
    check_retrace_closed_forms,
    check_retrace_matches_gae_on_policy,
    check_returns_closed_forms,
    check_lambda_returns_equal_gae_targets,
    check_forward_scans,
    check_appendix_a_polynomial,
    check_severing_and_continuation,
    check_retrace_actions_golden,
    check_retrace_actions_reduction,
    check_retrace_actions_relabelling,
    check_retrace_actions_one_hot,
    check_gae_masked,
    check_normalize_against_stdlib,
    check_normalize_invariants,
]


def failing_checks(orc):
    """Names of the checks the given oracle fails (used by the mutation test)."""
    bad = []
    for chk in ALL_CHECKS:
        try:
            chk(orc)
        except AssertionError:
            bad.append(chk.__name__)
    return bad
