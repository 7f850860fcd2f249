/*
 * rlscan_oracle.c -- plain, sequential, float64 reference for the batched
 * first-order linear recurrences of RL credit assignment.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library,
 * its Python binding) may include, link, import or execute this file.  The
 * only callers are the tests, the smoke check and the CPU-baseline leg of the
 * benchmark.  It shares no code, header, table or constant with the CUDA
 * sources.
 *
 * Every function is the definition written out: one row at a time, one time
 * step at a time, in the direction the recurrence runs, in double precision.
 * No blocking, no reordering, no associative scan.  Inputs are the float32
 * arrays both sides receive; each element is widened to double on read.
 *
 * Sources (page title, section):
 *   [API]     "rl-triton kernels -- API reference" (simonsays1980.github.io/
 *             rl-triton/kernels/), the docstring and the unfused long-sequence
 *             branch of each compute_* function.
 *   [PAPER]   "rl-triton: High-Performance Triton GPU Kernels for
 *             Reinforcement Learning Credit Assignment" (arXiv 2608.17641),
 *             Eq. 1, Table 1, Sec. 3.2 and Sec. 3.3.x.
 *   [RETURNS] "Returns and Eligibility Traces with Triton Associative Scans".
 *   [RETRACE] "Retrace(lambda) with Triton Associative Scans".
 *   [GAE]     "Technical Deep Dive into the GAE Triton Kernel".
 *
 * Layout: every [N,T] input is row-major float32 with row stride `rs`
 * elements (rs >= T); every [N] input is dense float32; every output is dense
 * row-major float64 [N,T] (row stride T).  Rows [row_begin, row_end) are
 * processed, so a caller may split rows across host threads.  Nullable
 * inputs are passed as NULL.
 *
 * Flags are float 0/1.  "done" is min(1, terminated + truncated) as in the
 * [API] unfused branches; values outside {0,1} are outside the contract and
 * are used in the arithmetic as given.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

#define AT(p, row, t, rs) ((double)(p)[(int64_t)(row) * (rs) + (t)])

static double done_flag(double term, double trunc)
{
    double d = term + trunc;
    return d > 1.0 ? 1.0 : d;
}

static double min2(double a, double b) { return a < b ? a : b; }

/*
 * Continuation value of the successor state at step t, shared by GAE and
 * V-trace ([API] compute_gae / compute_vtrace docstrings, "bootstrap_values
 * supplies the true continuation value"; [PAPER] Sec. 3.2).
 *
 *   bs_t = bootstrap_values[t] (0 when absent); last_value, when given,
 *          replaces bs_{T-1}.
 *   with truncation flags:    next_t = (t<T-1 ? (1-trunc_t) x_{t+1} : 0) + bs_t
 *   without truncation flags: next_t = (t<T-1 ? x_{t+1} : bs_{T-1})
 *
 * The second form is the fused no-truncation path, which reads only the
 * final bootstrap column; on inputs that follow the documented rule (zero
 * bootstrap at interior non-truncated steps) both forms agree.
 * `x` is the per-step value being continued (V for the TD error, the
 * V-trace target vs for the advantage).
 */
static double continuation(const double *x, int64_t t, int64_t T,
                           const float *trunc, const float *bs,
                           const float *last_value, int64_t row, int64_t rs)
{
    double bs_t = 0.0, bs_last = 0.0;
    if (bs) {
        bs_t = AT(bs, row, t, rs);
        bs_last = AT(bs, row, T - 1, rs);
    }
    if (last_value) {
        bs_last = (double)last_value[row];
        if (t == T - 1) bs_t = bs_last;
    }
    if (trunc) {
        double nx = (t < T - 1) ? (1.0 - AT(trunc, row, t, rs)) * x[t + 1] : 0.0;
        return nx + bs_t;
    }
    return (t < T - 1) ? x[t + 1] : bs_last;
}

/*
 * GAE -- [API] compute_gae; [PAPER] Table 1 row "GAE", Sec. 3.3.1;
 * [GAE] Sec. 1 and Sec. 5.
 *   delta_t = r_t + gamma (1-term_t) V_next_t - V_t
 *   A_t     = delta_t + gamma lambda (1-done_t) A_{t+1},   A_T = 0
 */
void oracle_gae(int64_t N, int64_t T, int64_t rs, int64_t row_begin, int64_t row_end,
                const float *r, const float *v, const float *term, const float *trunc,
                const float *bs, const float *last_value,
                double gamma, double lam, double *adv)
{
    (void)N;
    double *vrow = (double *)malloc((size_t)(T > 0 ? T : 1) * sizeof(double));
    if (!vrow) return;
    for (int64_t row = row_begin; row < row_end; ++row) {
        double *out = adv + row * T;
        for (int64_t t = 0; t < T; ++t) vrow[t] = AT(v, row, t, rs);
        double A_next = 0.0;
        for (int64_t t = T - 1; t >= 0; --t) {
            double vn = continuation(vrow, t, T, trunc, bs, last_value, row, rs);
            double te = AT(term, row, t, rs);
            double tr = trunc ? AT(trunc, row, t, rs) : 0.0;
            double delta = AT(r, row, t, rs) + gamma * (1.0 - te) * vn - vrow[t];
            double A = delta + gamma * lam * (1.0 - done_flag(te, tr)) * A_next;
            out[t] = A;
            A_next = A;
        }
    }
    free(vrow);
}

/*
 * GAE with observation-skip masking -- [PAPER] Sec. 9.3 (planned extension:
 * "observation-skip masking that carries the recurrence across masked
 * tokens (beta_t = 1)").  Reading: a masked step (mask_t = 0) contributes
 * nothing and hands the value through, A_t = A_{t+1}; an unmasked step is
 * the GAE step of oracle_gae, unchanged (its successor value is V_next_t as
 * defined there).  mask is float 0/1.
 */
void oracle_gae_masked(int64_t N, int64_t T, int64_t rs, int64_t row_begin, int64_t row_end,
                       const float *r, const float *v, const float *term, const float *trunc,
                       const float *bs, const float *last_value, const float *mask,
                       double gamma, double lam, double *adv)
{
    (void)N;
    double *vrow = (double *)malloc((size_t)(T > 0 ? T : 1) * sizeof(double));
    if (!vrow) return;
    for (int64_t row = row_begin; row < row_end; ++row) {
        double *out = adv + row * T;
        for (int64_t t = 0; t < T; ++t) vrow[t] = AT(v, row, t, rs);
        double carry = 0.0;  /* A_{t+1} */
        for (int64_t t = T - 1; t >= 0; --t) {
            double A;
            if (AT(mask, row, t, rs) == 0.0) {
                A = carry;
            } else {
                double vnext = continuation(vrow, t, T, trunc, bs, last_value, row, rs);
                double te = AT(term, row, t, rs);
                double tr = trunc ? AT(trunc, row, t, rs) : 0.0;
                double td = AT(r, row, t, rs) + gamma * (1.0 - te) * vnext - vrow[t];
                A = td + gamma * lam * (1.0 - done_flag(te, tr)) * carry;
            }
            out[t] = A;
            carry = A;
        }
    }
    free(vrow);
}

/*
 * V-trace -- [API] compute_vtrace (docstring and unfused branch);
 * [PAPER] Table 1 row "V-Trace", Sec. 3.3.2.
 *   ratio_t = exp(log_pi_target_t - log_pi_behavior_t)
 *   rho_t = min(rho_bar, ratio_t),  c_t = min(c_bar, ratio_t)
 *   Delta_t = rho_t (r_t + gamma (1-term_t) V_next_t - V_t)
 *             + gamma c_t (1-done_t) Delta_{t+1},          Delta_T = 0
 *   vs_t  = Delta_t + V_t
 *   adv_t = rho_t (r_t + gamma (1-term_t) vs_next_t - V_t)
 * V_next and vs_next use the same continuation rule (see continuation()).
 */
void oracle_vtrace(int64_t N, int64_t T, int64_t rs, int64_t row_begin, int64_t row_end,
                   const float *lpt, const float *lpb, const float *v, const float *r,
                   const float *term, const float *trunc, const float *bs,
                   const float *last_value, double gamma, double rho_bar, double c_bar,
                   double *vs_out, double *adv_out)
{
    (void)N;
    double *vrow = (double *)malloc((size_t)(T > 0 ? T : 1) * sizeof(double));
    if (!vrow) return;
    for (int64_t row = row_begin; row < row_end; ++row) {
        double *vs = vs_out + row * T;
        double *adv = adv_out + row * T;
        for (int64_t t = 0; t < T; ++t) vrow[t] = AT(v, row, t, rs);

        double D_next = 0.0;
        for (int64_t t = T - 1; t >= 0; --t) {
            double ratio = exp(AT(lpt, row, t, rs) - AT(lpb, row, t, rs));
            double rho = min2(rho_bar, ratio);
            double c = min2(c_bar, ratio);
            double te = AT(term, row, t, rs);
            double tr = trunc ? AT(trunc, row, t, rs) : 0.0;
            double vn = continuation(vrow, t, T, trunc, bs, last_value, row, rs);
            double D = rho * (AT(r, row, t, rs) + gamma * (1.0 - te) * vn - vrow[t])
                       + gamma * c * (1.0 - done_flag(te, tr)) * D_next;
            vs[t] = D + vrow[t];
            D_next = D;
        }
        for (int64_t t = 0; t < T; ++t) {
            double ratio = exp(AT(lpt, row, t, rs) - AT(lpb, row, t, rs));
            double rho = min2(rho_bar, ratio);
            double te = AT(term, row, t, rs);
            double nvs = continuation(vs, t, T, trunc, bs, last_value, row, rs);
            adv[t] = rho * (AT(r, row, t, rs) + gamma * (1.0 - te) * nvs - vrow[t]);
        }
    }
    free(vrow);
}

/*
 * Retrace(lambda) on per-step (reduced) inputs -- [API] compute_retrace
 * (docstring and unfused branch); [PAPER] Table 1 row "Retrace", Sec. 3.3.3;
 * [RETRACE] Sec. 2, 3, 4 and 6.
 *   ratio_t = pi_t / mu_t                  (pi, mu: probabilities of a_t)
 *   c_t   = lambda min(c_bar, ratio_t),   rho_t = min(rho_bar, ratio_t)
 *   delta_t = r_t + gamma (1-term_t) EQ_t - Q_t     (EQ_t = E_pi[Q(s_{t+1},.)])
 *   Delta_t = delta_t + gamma c_{t+1} (1-done_t) Delta_{t+1},  c_T = 0, Delta_T = 0
 *   Qret_t = Q_t + Delta_t
 *   adv_t  = rho_t (r_t + gamma (1-term_t) Qret_{t+1} - Q_t),  Qret_T = 0
 * truncateds may be NULL (all zero).
 */
/*
 * One row of the Retrace recurrence above, with the taken action's target
 * probability pi_t and the expected successor value EQ_t given in double.
 */
static void retrace_row(int64_t T, int64_t row, int64_t rs, const double *pi, const double *eq,
                        const float *mu, const float *q, const float *r, const float *term,
                        const float *trunc, double gamma, double lam, double c_bar,
                        double rho_bar, double *qret, double *adv)
{
    double D_next = 0.0;
    for (int64_t t = T - 1; t >= 0; --t) {
        double c_next = 0.0;
        if (t < T - 1)
            c_next = lam * min2(c_bar, pi[t + 1] / AT(mu, row, t + 1, rs));
        double te = AT(term, row, t, rs);
        double tr = trunc ? AT(trunc, row, t, rs) : 0.0;
        double delta = AT(r, row, t, rs) + gamma * (1.0 - te) * eq[t] - AT(q, row, t, rs);
        double D = delta + gamma * c_next * (1.0 - done_flag(te, tr)) * D_next;
        qret[t] = AT(q, row, t, rs) + D;
        D_next = D;
    }
    for (int64_t t = 0; t < T; ++t) {
        double rho = min2(rho_bar, pi[t] / AT(mu, row, t, rs));
        double te = AT(term, row, t, rs);
        double qn = (t < T - 1) ? qret[t + 1] : 0.0;
        adv[t] = rho * (AT(r, row, t, rs) + gamma * (1.0 - te) * qn - AT(q, row, t, rs));
    }
}

void oracle_retrace(int64_t N, int64_t T, int64_t rs, int64_t row_begin, int64_t row_end,
                    const float *pi, const float *mu, const float *q, const float *eq,
                    const float *r, const float *term, const float *trunc,
                    double gamma, double lam, double c_bar, double rho_bar,
                    double *qret_out, double *adv_out)
{
    (void)N;
    double *pi_d = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double *eq_d = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    for (int64_t row = row_begin; row < row_end; ++row) {
        for (int64_t t = 0; t < T; ++t) {
            pi_d[t] = AT(pi, row, t, rs);
            eq_d[t] = AT(eq, row, t, rs);
        }
        retrace_row(T, row, rs, pi_d, eq_d, mu, q, r, term, trunc, gamma, lam, c_bar, rho_bar,
                    qret_out + row * T, adv_out + row * T);
    }
    free(pi_d);
    free(eq_d);
}

/*
 * Retrace(lambda) from the full action-space inputs -- [API] compute_retrace
 * (its signature: action_probs_target and next_q_values_all [N,T,A],
 * actions int64 [N,T], action_probs_behavior the behaviour probability of
 * the taken action; its unfused branch reduces the action dimension first).
 *   EQ_t = sum_a pi_target[t,a] * Qnext[t,a]     (a = 0 .. A-1 in order;
 *          the target weights are those stored at the same step t, as the
 *          API's reduction multiplies the two [N,T,A] tensors element-wise)
 *   pi_t = pi_target[t, actions[t]]
 * then the recurrence of oracle_retrace with mu_t = action_probs_behavior[t].
 * The [N,T,A] arrays are dense (row stride T*A); actions and the [N,T] arrays
 * have row stride rs.  Returns the number of steps whose action index lies
 * outside [0, A); their rows are left unwritten.
 */
int64_t oracle_retrace_actions(int64_t N, int64_t T, int64_t A, int64_t rs, int64_t row_begin,
                               int64_t row_end, const float *probs, const float *mu,
                               const float *q, const float *next_q_all, const int64_t *actions,
                               const float *r, const float *term, const float *trunc,
                               double gamma, double lam, double c_bar, double rho_bar,
                               double *qret_out, double *adv_out)
{
    (void)N;
    int64_t bad = 0;
    double *pi_d = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double *eq_d = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    for (int64_t row = row_begin; row < row_end; ++row) {
        int64_t row_bad = 0;
        for (int64_t t = 0; t < T; ++t) {
            const float *pt = probs + (row * T + t) * A;
            const float *qt = next_q_all + (row * T + t) * A;
            double s = 0.0;
            for (int64_t a = 0; a < A; ++a) s += (double)pt[a] * (double)qt[a];
            eq_d[t] = s;
            int64_t at = actions[row * rs + t];
            if (at < 0 || at >= A) {
                ++row_bad;
                pi_d[t] = 0.0;
            } else {
                pi_d[t] = (double)pt[at];
            }
        }
        bad += row_bad;
        if (row_bad == 0)
            retrace_row(T, row, rs, pi_d, eq_d, mu, q, r, term, trunc, gamma, lam, c_bar,
                        rho_bar, qret_out + row * T, adv_out + row * T);
    }
    free(pi_d);
    free(eq_d);
    return bad;
}

/*
 * Bootstrap column and carry shared by TD(lambda) and discounted returns:
 * bs_t = bootstrap_values[t] (0 when absent), last_value replaces bs_{T-1};
 * the scan carry G_T is bs_{T-1} ([API] unfused branches of
 * compute_lambda_returns / compute_discounted_returns; [PAPER] Sec. 3.3.4).
 */
static double returns_bs(const float *bs, const float *last_value, int64_t row,
                         int64_t t, int64_t T, int64_t rs)
{
    if (last_value && t == T - 1) return (double)last_value[row];
    return bs ? AT(bs, row, t, rs) : 0.0;
}

/*
 * TD(lambda) returns -- [API] compute_lambda_returns; [PAPER] Table 1 row
 * "TD(lambda)", Sec. 3.3.4; [RETURNS] Sec. 2.
 *   G_t = r_t + gamma (1-lambda)(1-done_t) nv_t + gamma trunc_t bs_t
 *         + gamma lambda (1-done_t) G_{t+1},        G_T = bs_{T-1}
 * nv_t = next_values[t] (the caller zeroes it at truncated steps).
 */
void oracle_lambda_returns(int64_t N, int64_t T, int64_t rs, int64_t row_begin, int64_t row_end,
                           const float *r, const float *nv, const float *term,
                           const float *trunc, const float *bs, const float *last_value,
                           double gamma, double lam, double *out_all)
{
    (void)N;
    for (int64_t row = row_begin; row < row_end; ++row) {
        double *out = out_all + row * T;
        double G_next = returns_bs(bs, last_value, row, T - 1, T, rs);
        for (int64_t t = T - 1; t >= 0; --t) {
            double te = AT(term, row, t, rs);
            double tr = trunc ? AT(trunc, row, t, rs) : 0.0;
            double nd = 1.0 - done_flag(te, tr);
            double G = AT(r, row, t, rs) + gamma * (1.0 - lam) * nd * AT(nv, row, t, rs)
                       + gamma * tr * returns_bs(bs, last_value, row, t, T, rs)
                       + gamma * lam * nd * G_next;
            out[t] = G;
            G_next = G;
        }
    }
}

/*
 * Discounted returns -- [API] compute_discounted_returns; [PAPER] Table 1
 * row "Disc. Returns", Sec. 3.3.4; [RETURNS] Sec. 1.
 *   G_t = r_t + gamma trunc_t bs_t + gamma (1-done_t) G_{t+1},   G_T = bs_{T-1}
 */
void oracle_discounted_returns(int64_t N, int64_t T, int64_t rs, int64_t row_begin, int64_t row_end,
                               const float *r, const float *term, const float *trunc,
                               const float *bs, const float *last_value,
                               double gamma, double *out_all)
{
    (void)N;
    for (int64_t row = row_begin; row < row_end; ++row) {
        double *out = out_all + row * T;
        double G_next = returns_bs(bs, last_value, row, T - 1, T, rs);
        for (int64_t t = T - 1; t >= 0; --t) {
            double te = AT(term, row, t, rs);
            double tr = trunc ? AT(trunc, row, t, rs) : 0.0;
            double G = AT(r, row, t, rs) + gamma * tr * returns_bs(bs, last_value, row, t, T, rs)
                       + gamma * (1.0 - done_flag(te, tr)) * G_next;
            out[t] = G;
            G_next = G;
        }
    }
}

/*
 * Eligibility traces (forward in time) -- [API] compute_eligibility_traces;
 * [PAPER] Table 1 row "Elig. Traces", Sec. 3.3.5; [RETURNS] Sec. 3.
 *   z_t = g_t + gamma lambda (1 - d_{t-1}) z_{t-1},   d_{-1} = 0,  z_{-1} = seed
 * seed_values may be NULL (zero seed).
 */
void oracle_eligibility_traces(int64_t N, int64_t T, int64_t rs, int64_t row_begin, int64_t row_end,
                               const float *g, const float *dones, const float *seed,
                               double gamma, double lam, double *out_all)
{
    (void)N;
    for (int64_t row = row_begin; row < row_end; ++row) {
        double *out = out_all + row * T;
        double z_prev = seed ? (double)seed[row] : 0.0;
        double d_prev = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            double z = AT(g, row, t, rs) + gamma * lam * (1.0 - d_prev) * z_prev;
            out[t] = z;
            z_prev = z;
            d_prev = AT(dones, row, t, rs);
        }
    }
}

/*
 * Episodic prefix sum (forward in time) -- [API] compute_episodic_prefix_sum;
 * [PAPER] Table 1 row "Prefix Sum", Sec. 3.3.6.
 *   boundary 0 ("ends_at"):   C_t = x_t + (1 - d_{t-1}) C_{t-1},  d_{-1} = 0
 *   boundary 1 ("starts_at"): C_t = x_t + (1 - d_t)     C_{t-1}
 *   C_{-1} = seed (0 when seed_values is NULL)
 */
void oracle_episodic_prefix_sum(int64_t N, int64_t T, int64_t rs, int64_t row_begin, int64_t row_end,
                                const float *x, const float *dones, const float *seed,
                                int boundary, double *out_all)
{
    (void)N;
    for (int64_t row = row_begin; row < row_end; ++row) {
        double *out = out_all + row * T;
        double C_prev = seed ? (double)seed[row] : 0.0;
        double d_prev = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            double d_t = AT(dones, row, t, rs);
            double gate = (boundary == 0) ? (1.0 - d_prev) : (1.0 - d_t);
            double C = AT(x, row, t, rs) + gate * C_prev;
            out[t] = C;
            C_prev = C;
            d_prev = d_t;
        }
    }
}

/*
 * Generic affine recurrence on given coefficients -- [PAPER] Eq. 1 and its
 * forward mirror (Sec. 1), boundary carry as in Sec. 4.1 step 4.
 *   direction 0 (backward): A_t = alpha_t + beta_t A_{t+1},  A_T    = carry
 *   direction 1 (forward):  A_t = alpha_t + beta_t A_{t-1},  A_{-1} = carry
 * carry may be NULL (zero).
 */
void oracle_linear_scan(int64_t N, int64_t T, int64_t rs, int64_t row_begin, int64_t row_end,
                        const float *alpha, const float *beta, const float *carry,
                        int direction, double *out_all)
{
    (void)N;
    for (int64_t row = row_begin; row < row_end; ++row) {
        double *out = out_all + row * T;
        double A = carry ? (double)carry[row] : 0.0;
        if (direction == 0) {
            for (int64_t t = T - 1; t >= 0; --t) {
                A = AT(alpha, row, t, rs) + AT(beta, row, t, rs) * A;
                out[t] = A;
            }
        } else {
            for (int64_t t = 0; t < T; ++t) {
                A = AT(alpha, row, t, rs) + AT(beta, row, t, rs) * A;
                out[t] = A;
            }
        }
    }
}
