// estimators.cuh -- per-estimator coefficient and output functors.
//
// Each estimator turns the raw rollout inputs of one thread's ITEMS
// consecutive time steps into the affine-scan coefficients (alpha_t, beta_t)
// in registers, names the boundary value folded into the scan at the row
// end (backward) or row start (forward), and turns the scan result A_t into
// the outputs.  Sources: rl-triton paper Table 1 and Sec. 3.2-3.3; rl-triton
// API reference (compute_* docstrings); "Retrace(lambda) with Triton
// Associative Scans" Sec. 3-6.
//
// Interface (all static, I = items per thread):
//   NIN, NOUT       number of [N,T] inputs and outputs
//   K               affine recurrences solved per step (1, or 2 for the
//                   fused GAE + returns estimator)
//   FWD             true for forward-in-time recurrences
//   HALO            bit j set: input j is also read one step outside the
//                   thread's range (t+1 backward, t-1 forward)
//   ROWSCALAR       the per-row scalar argument is used
//   Keep<I>         values saved from coeffs() for post()
//   coeffs<I, EDGE>(x, xn, kb, p, rsc, a, b, keep)
//       x[j][k] = input j at the thread's k-th step; xn[j] = input j at the
//       neighbouring step outside the range (only meaningful for HALO
//       inputs); EDGE: the row's boundary step (t = T-1 backward, t = 0
//       forward) is element kb of the range (otherwise kb is ignored and the
//       boundary tests compile away); rsc = this row's scalar (only
//       meaningful when EDGE).  Writes a[s][k], b[s][k] for each scan s < K.
//   boundary(x, k, rsc, p, bv)
//       values folded in at the row boundary element k, one per scan: A_T
//       (backward) or A_{-1} (forward); the kernel sets a += b * bv, b = 0.
//   post<I, EDGE>(x, xn, kb, p, rsc, A, A_after, keep, o)
//       A[s][k] = scan s at the k-th step; A_after[s] = scan s at the step
//       after the range (backward only; used for successor targets).
#pragma once

#include "checks.cuh"
#include "params.cuh"
#include "ptx.cuh"

namespace rlscan {
namespace est {

// done_t = min(1, terminated_t + truncated_t)
__device__ __forceinline__ float done_of(float term, float trunc) { return fminf(1.f, term + trunc); }

// min(clip, x) that keeps a NaN x (fminf would return the clip), so an
// undefined ratio such as 0/0 shows in the outputs instead of being clipped:
// the NaN-propagating form of the minimum (PTX min.NaN.f32, one instruction)
__device__ __forceinline__ float clip_above(float clip, float x)
{
    float r;
    asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(clip), "f"(x));
    return r;
}

// Importance ratios.  RLSCAN_FAST_RATIO=1 (default) takes CUDA's fast
// intrinsics __expf and __fdividef (relative error of a few 1e-7 for the
// log-ratios and probabilities of these estimators) instead of the
// correctly rounded expf and IEEE division; the ratio is clipped and
// multiplies terms whose own float32 rounding is of that size, so the
// outputs stay far inside the parity bound.  Measured: compact Retrace
// 1024 x 16384 55.2 -> 48.4 us, compact V-trace 33.4 -> 32.4 us; the
// float32 kernels, bandwidth-bound, unchanged.
#ifndef RLSCAN_FAST_RATIO
#define RLSCAN_FAST_RATIO 1
#endif
__device__ __forceinline__ float ratio_exp(float log_ratio) { return RLSCAN_FAST_RATIO ? __expf(log_ratio) : expf(log_ratio); }
__device__ __forceinline__ float ratio_div(float num, float den) { return RLSCAN_FAST_RATIO ? __fdividef(num, den) : num / den; }

// ---------------------------------------------------------------------------
// GAE: alpha = r + gamma (1-term) Vn - V, beta = gamma lambda (1-done), A_T = 0.
// Inputs: 0 rewards, 1 values, 2 terminateds, [3 truncateds], [3+TRUNC bootstrap].
// Vn at T-1 is the bootstrap (bootstrap column or last_value / scalar column).
template <bool TRUNC, bool BS2D>
struct GAE {
    static_assert(TRUNC || !BS2D, "2-D bootstrap is read only with truncation flags");
    static constexpr int NIN = 3 + TRUNC + BS2D, NOUT = 1;
    static constexpr unsigned FLAGS = (1u << 2) | (TRUNC ? (1u << 3) : 0u);  // 0/1 inputs
    static constexpr int K = 1;  // affine recurrences per step
    static constexpr bool FWD = false, ROWSCALAR = !BS2D;
    static constexpr unsigned HALO = 1u << 1;
    static constexpr int TR = 3, BS = 3 + TRUNC;
    template <int I> struct Keep {};

    template <int I, bool EDGE>
    __device__ static void coeffs(const float (&x)[NIN][I], const float (&xn)[NIN], int kb,
                                  const Params &p, float rsc, float (&a)[K][I], float (&b)[K][I], Keep<I> &)
    {
        const float g = p.c0, gl = p.c0 * p.c1;
#pragma unroll
        for (int k = 0; k < I; ++k) {
            const bool last = (EDGE && k == kb);
            const float vnext = (k + 1 < I) ? x[1][k + 1] : xn[1];
            const float term = x[2][k];
            float vn, done;
            if constexpr (TRUNC) {
                const float tr = x[TR][k];
                float bs;
                if constexpr (BS2D) bs = x[BS][k];
                else bs = last ? rsc : 0.f;
                vn = last ? bs : fmaf(1.f - tr, vnext, bs);
                done = done_of(term, tr);
            } else {
                vn = last ? rsc : vnext;
                done = term;
            }
            a[0][k] = fmaf(g * (1.f - term), vn, x[0][k]) - x[1][k];
            b[0][k] = gl * (1.f - done);
        }
    }
    template <int I>
    __device__ static void boundary(const float (&)[NIN][I], int, float, const Params &, float (&bv)[K]) { bv[0] = 0.f; }
    template <int I, bool EDGE>
    __device__ static void post(const float (&)[NIN][I], const float (&)[NIN], int, const Params &,
                                float, const float (&A)[K][I], const float (&)[K], const Keep<I> &, float (&o)[NOUT][I])
    {
#pragma unroll
        for (int k = 0; k < I; ++k) o[0][k] = A[0][k];
    }
};

// ---------------------------------------------------------------------------
// GAE with observation-skip masking (rl-triton paper Sec. 9.3: the
// recurrence is carried across masked tokens, beta = 1): the GAE map of an
// unmasked step, and the identity map (alpha = 0, beta = 1) at a masked one:
//   alpha = m alpha_GAE,  beta = m beta_GAE + (1 - m),  m = mask_t in {0, 1}.
// Inputs: those of GAE<TRUNC, BS2D>, then the mask.
template <bool TRUNC, bool BS2D>
struct GAEMasked : GAE<TRUNC, BS2D> {
    using Base = GAE<TRUNC, BS2D>;
    static constexpr int NIN = Base::NIN + 1, MASK = Base::NIN;
    template <int I> struct Keep {};

    template <int I, bool EDGE>
    __device__ static void coeffs(const float (&x)[NIN][I], const float (&xn)[NIN], int kb,
                                  const Params &p, float rsc, float (&a)[1][I], float (&b)[1][I], Keep<I> &)
    {
        const float(&xb)[Base::NIN][I] = reinterpret_cast<const float(&)[Base::NIN][I]>(x);
        const float(&xnb)[Base::NIN] = reinterpret_cast<const float(&)[Base::NIN]>(xn);
        typename Base::template Keep<I> kb_unused;
        Base::template coeffs<I, EDGE>(xb, xnb, kb, p, rsc, a, b, kb_unused);
#pragma unroll
        for (int k = 0; k < I; ++k) {
            const float m = x[MASK][k];
            a[0][k] *= m;
            b[0][k] = fmaf(m, b[0][k], 1.f - m);
        }
    }
    template <int I>
    __device__ static void boundary(const float (&)[NIN][I], int, float, const Params &, float (&bv)[1]) { bv[0] = 0.f; }
    template <int I, bool EDGE>
    __device__ static void post(const float (&)[NIN][I], const float (&)[NIN], int, const Params &,
                                float, const float (&A)[1][I], const float (&)[1], const Keep<I> &, float (&o)[1][I])
    {
#pragma unroll
        for (int k = 0; k < I; ++k) o[0][k] = A[0][k];
    }
};

// ---------------------------------------------------------------------------
// V-trace: ratio = exp(lpt - lpb), rho = min(rho_bar, ratio), c = min(c_bar, ratio);
// alpha = rho (r + gamma (1-term) Vn - V), beta = gamma c (1-done), D_T = 0;
// vs = D + V, adv = rho (r + gamma (1-term) vsn - V).
// Inputs: 0 lpt, 1 lpb, 2 values, 3 rewards, 4 terminateds, [5 truncateds], [5+TRUNC bootstrap].
// Constants: c0 gamma, c1 rho_bar, c2 c_bar.
template <bool TRUNC, bool BS2D>
struct VTrace {
    static_assert(TRUNC || !BS2D, "2-D bootstrap is read only with truncation flags");
    static constexpr int NIN = 5 + TRUNC + BS2D, NOUT = 2;
    static constexpr unsigned FLAGS = (1u << 4) | (TRUNC ? (1u << 5) : 0u);  // 0/1 inputs
    static constexpr int K = 1;  // affine recurrences per step
    static constexpr bool FWD = false, ROWSCALAR = !BS2D;
    static constexpr bool LB_ROW_MAJOR = true;  // measured faster on 2^20-step rows
    static constexpr int LB_NAP_MAX = 0;        // polls without pausing (likewise)
    static constexpr unsigned HALO = 1u << 2;
    static constexpr int TR = 5, BS = 5 + TRUNC;
    // alpha and the weight w = rho gamma (1-term) (1-trunc) of the successor:
    // adv_t = rho (r + gamma (1-term) vs_{t+1} - V) is alpha_t + w_t D_{t+1}
    // (vs_{t+1} = D_{t+1} + V_{t+1}, and alpha_t holds the V_{t+1} and
    // bootstrap terms), alpha_t itself at the row's last step
    template <int I> struct Keep { float a[I], w[I]; };

    // successor of x at element k: the next value, or the bootstrap at a
    // truncation and at the row's last step
    template <int I>
    __device__ static float successor(const float (&x)[NIN][I], int k, bool last, float nxt, float rsc)
    {
        if constexpr (TRUNC) {
            float bs;
            if constexpr (BS2D) bs = x[BS][k];
            else bs = last ? rsc : 0.f;
            return last ? bs : fmaf(1.f - x[TR][k], nxt, bs);
        } else {
            return last ? rsc : nxt;
        }
    }

    template <int I, bool EDGE>
    __device__ static void coeffs(const float (&x)[NIN][I], const float (&xn)[NIN], int kb,
                                  const Params &p, float rsc, float (&a)[K][I], float (&b)[K][I], Keep<I> &keep)
    {
        const float g = p.c0;
#pragma unroll
        for (int k = 0; k < I; ++k) {
            const bool last = (EDGE && k == kb);
            const float ratio = ratio_exp(x[0][k] - x[1][k]);
            const float rho = clip_above(p.c1, ratio), c = clip_above(p.c2, ratio);
            const float term = x[4][k];
            const float vn = successor<I>(x, k, last, (k + 1 < I) ? x[2][k + 1] : xn[2], rsc);
            float done;
            if constexpr (TRUNC) done = done_of(term, x[TR][k]);
            else done = term;
            const float gt = g * (1.f - term);
            const float gc = g * c;
            a[0][k] = rho * (fmaf(gt, vn, x[3][k]) - x[2][k]);
            b[0][k] = fmaf(-gc, done, gc);  // gamma c (1 - done)
            keep.a[k] = a[0][k];
            if constexpr (TRUNC) keep.w[k] = rho * gt * (1.f - x[TR][k]);
            else keep.w[k] = rho * gt;
        }
    }
    template <int I>
    __device__ static void boundary(const float (&)[NIN][I], int, float, const Params &, float (&bv)[K]) { bv[0] = 0.f; }
    template <int I, bool EDGE>
    __device__ static void post(const float (&x)[NIN][I], const float (&xn)[NIN], int kb,
                                const Params &p, float rsc, const float (&A)[K][I], const float (&A_after)[K],
                                const Keep<I> &keep, float (&o)[NOUT][I])
    {
#pragma unroll
        for (int k = 0; k < I; ++k) {
            const bool last = (EDGE && k == kb);
            const float d_next = (k + 1 < I) ? A[0][k + 1] : A_after[0];
            o[0][k] = A[0][k] + x[2][k];
            o[1][k] = last ? keep.a[k] : fmaf(keep.w[k], d_next, keep.a[k]);
        }
    }
};

// ---------------------------------------------------------------------------
// Retrace on per-step inputs: ratio = pi/mu, c = lambda min(c_bar, ratio),
// rho = min(rho_bar, ratio); alpha = r + gamma (1-term) EQ - Q,
// beta = gamma c_{t+1} (1-done) with c_T = 0; Qret = D + Q;
// adv = rho (r + gamma (1-term) Qret_{t+1} - Q), Qret_T = 0.
// Inputs: 0 pi, 1 mu, 2 q, 3 eq, 4 rewards, 5 terminateds, [6 truncateds].
// Constants: c0 gamma, c1 lambda, c2 c_bar, c3 rho_bar.
template <bool TRUNC>
struct Retrace {
    static constexpr int NIN = 6 + TRUNC, NOUT = 2;
    static constexpr unsigned FLAGS = (1u << 5) | (TRUNC ? (1u << 6) : 0u);  // 0/1 inputs
    static constexpr int K = 1;  // affine recurrences per step
    static constexpr bool FWD = false, ROWSCALAR = false;
    static constexpr unsigned HALO = (1u << 0) | (1u << 1) | (1u << 2);
    // adv_t = rho (r + gamma (1-term) Qret_{t+1} - Q) with Qret_{t+1} =
    // D_{t+1} + Q_{t+1} (0 after the row's last step) is u_t + w_t D_{t+1}:
    // u = rho (r + gamma (1-term) Q_{t+1} - Q), w = rho gamma (1-term)
    template <int I> struct Keep { float u[I], w[I]; };

    template <int I, bool EDGE>
    __device__ static void coeffs(const float (&x)[NIN][I], const float (&xn)[NIN], int kb,
                                  const Params &p, float, float (&a)[K][I], float (&b)[K][I], Keep<I> &keep)
    {
        const float g = p.c0, gl = p.c0 * p.c1;
        float c[I + 1];  // min(c_bar, ratio); the trace coefficient is lambda times it
#pragma unroll
        for (int k = 0; k < I; ++k) {
            const float ratio = ratio_div(x[0][k], x[1][k]);
            c[k] = clip_above(p.c2, ratio);
            keep.w[k] = clip_above(p.c3, ratio);  // rho, until the second loop
        }
        c[I] = clip_above(p.c2, ratio_div(xn[0], xn[1]));
#pragma unroll
        for (int k = 0; k < I; ++k) {
            const bool last = (EDGE && k == kb);
            const float term = x[5][k];
            float done;
            if constexpr (TRUNC) done = done_of(term, x[6][k]);
            else done = term;
            const float gcn = last ? 0.f : gl * c[k + 1];
            const float gt = g * (1.f - term);
            a[0][k] = fmaf(gt, x[3][k], x[4][k]) - x[2][k];
            b[0][k] = fmaf(-gcn, done, gcn);  // gamma lambda min(c_bar, ratio_{t+1}) (1 - done)
            const float qn = last ? 0.f : ((k + 1 < I) ? x[2][k + 1] : xn[2]);
            keep.u[k] = keep.w[k] * (fmaf(gt, qn, x[4][k]) - x[2][k]);
            keep.w[k] *= gt;
        }
    }
    template <int I>
    __device__ static void boundary(const float (&)[NIN][I], int, float, const Params &, float (&bv)[K]) { bv[0] = 0.f; }
    template <int I, bool EDGE>
    __device__ static void post(const float (&x)[NIN][I], const float (&xn)[NIN], int kb,
                                const Params &p, float, const float (&A)[K][I], const float (&A_after)[K],
                                const Keep<I> &keep, float (&o)[NOUT][I])
    {
#pragma unroll
        for (int k = 0; k < I; ++k) {
            const bool last = (EDGE && k == kb);
            const float d_next = (k + 1 < I) ? A[0][k + 1] : A_after[0];
            o[0][k] = A[0][k] + x[2][k];
            o[1][k] = last ? keep.u[k] : fmaf(keep.w[k], d_next, keep.u[k]);
        }
    }
};

// ---------------------------------------------------------------------------
// Retrace from the full action-space inputs (API reference, compute_retrace
// signature): the narrow inputs of Retrace above, except that pi (0) and
// EQ (3) are not read from global memory.  prepass() derives them per step
// from three wide arrays staged beside the narrow ones:
//   wide 0  target probabilities pi(.|s_t)     A words per step
//   wide 1  successor values Q(s_{t+1}, .)     A words per step
//   wide 2  int64 action a_t                   2 words per step
//   EQ_t = sum_a pi(a|s_t) Q(s_{t+1}, a)   (weights of the same step t, as
//          the API's reduction multiplies the two [N,T,A] tensors)
//   pi_t = pi(a_t|s_t), NaN when a_t lies outside [0, A)
// Inputs (narrow): 1 mu, 2 q, 4 rewards, 5 terminateds, [6 truncateds].
template <bool TRUNC>
struct RetraceActions : Retrace<TRUNC> {
    static constexpr int NWIDE = 3;
    // with truncation flags a 1024-step stage leaves room for one CTA per SM:
    // 512-step tiles keep three
    static constexpr int WIDE_TILE = TRUNC ? 512 : 1024;
    static constexpr unsigned DERIVED = (1u << 0) | (1u << 3);
    static constexpr int PI = 0, EQ = 3;

    __host__ __device__ static int wide_words(int w, int A) { return w < 2 ? A : 2; }

    // Fill the derived arrays of one tile (pi_out / eq_out: their stage
    // slots, data from offset 4).  Step e of the tile (packed: row e / C,
    // column e % C; long rows: e < len, plus e = len for the step after the
    // tile) is read from the stage's wide region `wsm` when `staged`, else
    // from global memory.  Consecutive threads take consecutive steps, so
    // the wide rows are read without bank conflicts (shared) or coalesced
    // (global).  The derived slots overlay the wide region, so when staged
    // every thread reads all its steps before any thread writes (named
    // barrier BAR of the THREADS compute threads).
    template <int TILE, int AST, int THREADS, int BAR, class Geo>
    __device__ static void prepass(const Params &p, const Geo &tg, float *pi_out, float *eq_out,
                                   const float *wsm, bool staged, int tid)
    {
        constexpr int MAXK = TILE / THREADS + 1;
        const int A = p.A;
        const int total = p.packed ? tg.nrows * p.C : tg.len + ((tg.t0 + tg.len < p.T) ? 1 : 0);
        const float *sp = wsm;
        const float *sq = wsm + (TILE + 4) * A;
        const long long *sa = reinterpret_cast<const long long *>(wsm + 2 * (TILE + 4) * A);
        const float nan = __int_as_float(0x7fc00000);
        float pv[MAXK], ev[MAXK];
#pragma unroll
        for (int k = 0; k < MAXK; ++k) {
            const int e = tid + k * THREADS;
            pv[k] = 0.f;
            ev[k] = 0.f;
            if (e >= total) continue;
            int i = 0, c = e;
            if (p.packed) {
                i = e / p.C;
                c = e - i * p.C;
                if (c >= tg.len) continue;
            }
            if (staged && A == 4) {
                const float4 u = *reinterpret_cast<const float4 *>(sp + 4 * e);
                const float4 v = *reinterpret_cast<const float4 *>(sq + 4 * e);
                const long long a = sa[e];
                const int ai = static_cast<int>(a);
                ev[k] = fmaf(u.w, v.w, fmaf(u.z, v.z, fmaf(u.y, v.y, u.x * v.x)));
                const float pk = ai == 0 ? u.x : (ai == 1 ? u.y : (ai == 2 ? u.z : u.w));
                pv[k] = static_cast<unsigned long long>(a) < 4ull ? pk : nan;
                continue;
            }
            const float *pr, *nq;
            long long a;
            if (staged) {
                pr = sp + e * A;
                nq = sq + e * A;
                a = sa[e];
            } else {
                const int64_t row = tg.row0 + i, t = tg.t0 + c;
                pr = static_cast<const float *>(p.wide[0]) + row * p.wide_rs[0] + t * A;
                nq = static_cast<const float *>(p.wide[1]) + row * p.wide_rs[1] + t * A;
                const long long *ap = reinterpret_cast<const long long *>(p.wide[2]) + (row * p.wide_rs[2] >> 1) + t;
                if (!(span_ok(p, p.wide[0], wide_extent(p, 0), pr, 4u * A, kSiteWide) &&
                      span_ok(p, p.wide[1], wide_extent(p, 1), nq, 4u * A, kSiteWide) &&
                      span_ok(p, p.wide[2], wide_extent(p, 2), ap, 8, kSiteWide))) {
                    ev[k] = 0.f;
                    pv[k] = nan;
                    continue;
                }
                a = __ldg(ap);
            }
            float eq = 0.f;
            for (int q = 0; q < A; ++q) eq = fmaf(pr[q], nq[q], eq);
            ev[k] = eq;
            pv[k] = (a >= 0 && a < A) ? pr[a] : nan;
        }
        if (staged) ptx::named_barrier(BAR, THREADS);
#pragma unroll
        for (int k = 0; k < MAXK; ++k) {
            const int e = tid + k * THREADS;
            if (e < total) {
                pi_out[4 + e] = pv[k];
                eq_out[4 + e] = ev[k];
            }
        }
    }
};

// ---------------------------------------------------------------------------
// TD(lambda): alpha = r + gamma (1-lambda)(1-done) nv + gamma trunc bs,
// beta = gamma lambda (1-done), A_T = bs_{T-1}.
// Inputs: 0 rewards, 1 next_values, 2 terminateds, [3 truncateds], [3+TRUNC bootstrap].
// Row scalar: bs_{T-1} (last_value, or the bootstrap column) when no 2-D bootstrap.
template <bool TRUNC, bool BS2D>
struct LambdaReturns {
    static_assert(TRUNC || !BS2D, "2-D bootstrap is read only with truncation flags");
    static constexpr int NIN = 3 + TRUNC + BS2D, NOUT = 1;
    static constexpr int K = 1;  // affine recurrences per step
    static constexpr bool FWD = false, ROWSCALAR = !BS2D;
    static constexpr unsigned HALO = 0;
    static constexpr int TR = 3, BS = 3 + TRUNC;
    template <int I> struct Keep {};

    template <int I, bool EDGE>
    __device__ static void coeffs(const float (&x)[NIN][I], const float (&)[NIN], int kb,
                                  const Params &p, float rsc, float (&a)[K][I], float (&b)[K][I], Keep<I> &)
    {
        const float g = p.c0, gl = p.c0 * p.c1, g1l = p.c0 * (1.f - p.c1);
#pragma unroll
        for (int k = 0; k < I; ++k) {
            const float term = x[2][k];
            if constexpr (TRUNC) {
                const bool last = (EDGE && k == kb);
                const float tr = x[TR][k];
                float bs;
                if constexpr (BS2D) bs = x[BS][k];
                else bs = last ? rsc : 0.f;
                const float nd = 1.f - done_of(term, tr);
                a[0][k] = fmaf(g * tr, bs, fmaf(g1l * nd, x[1][k], x[0][k]));
                b[0][k] = gl * nd;
            } else {
                const float nd = 1.f - term;
                a[0][k] = fmaf(g1l * nd, x[1][k], x[0][k]);
                b[0][k] = gl * nd;
            }
        }
    }
    template <int I>
    __device__ static void boundary(const float (&x)[NIN][I], int k, float rsc, const Params &, float (&bv)[K])
    {
        if constexpr (BS2D) bv[0] = x[BS][k];
        else bv[0] = rsc;
    }
    template <int I, bool EDGE>
    __device__ static void post(const float (&)[NIN][I], const float (&)[NIN], int, const Params &,
                                float, const float (&A)[K][I], const float (&)[K], const Keep<I> &, float (&o)[NOUT][I])
    {
#pragma unroll
        for (int k = 0; k < I; ++k) o[0][k] = A[0][k];
    }
};

// ---------------------------------------------------------------------------
// Discounted returns: alpha = r + gamma trunc bs, beta = gamma (1-done), A_T = bs_{T-1}.
// Inputs: 0 rewards, 1 terminateds, [2 truncateds], [2+TRUNC bootstrap].
template <bool TRUNC, bool BS2D>
struct Discounted {
    static_assert(TRUNC || !BS2D, "2-D bootstrap is read only with truncation flags");
    static constexpr int NIN = 2 + TRUNC + BS2D, NOUT = 1;
    static constexpr int K = 1;  // affine recurrences per step
    static constexpr bool FWD = false, ROWSCALAR = !BS2D;
    static constexpr unsigned HALO = 0;
    static constexpr int TR = 2, BS = 2 + TRUNC;
    template <int I> struct Keep {};

    template <int I, bool EDGE>
    __device__ static void coeffs(const float (&x)[NIN][I], const float (&)[NIN], int kb,
                                  const Params &p, float rsc, float (&a)[K][I], float (&b)[K][I], Keep<I> &)
    {
        const float g = p.c0;
#pragma unroll
        for (int k = 0; k < I; ++k) {
            const float term = x[1][k];
            if constexpr (TRUNC) {
                const bool last = (EDGE && k == kb);
                const float tr = x[TR][k];
                float bs;
                if constexpr (BS2D) bs = x[BS][k];
                else bs = last ? rsc : 0.f;
                a[0][k] = fmaf(g * tr, bs, x[0][k]);
                b[0][k] = g * (1.f - done_of(term, tr));
            } else {
                a[0][k] = x[0][k];
                b[0][k] = g * (1.f - term);
            }
        }
    }
    template <int I>
    __device__ static void boundary(const float (&x)[NIN][I], int k, float rsc, const Params &, float (&bv)[K])
    {
        if constexpr (BS2D) bv[0] = x[BS][k];
        else bv[0] = rsc;
    }
    template <int I, bool EDGE>
    __device__ static void post(const float (&)[NIN][I], const float (&)[NIN], int, const Params &,
                                float, const float (&A)[K][I], const float (&)[K], const Keep<I> &, float (&o)[NOUT][I])
    {
#pragma unroll
        for (int k = 0; k < I; ++k) o[0][k] = A[0][k];
    }
};

// ---------------------------------------------------------------------------
// Eligibility traces (forward): alpha = g_t, beta = gamma lambda (1 - d_{t-1}),
// d_{-1} = 0, A_{-1} = seed.  Inputs: 0 gradients, 1 dones.
struct Eligibility {
    static constexpr int NIN = 2, NOUT = 1;
    static constexpr int K = 1;  // affine recurrences per step
    static constexpr bool FWD = true, ROWSCALAR = true;
    static constexpr int DEFER_RING = 4;  // long rows: a fourth stage measured faster
    static constexpr bool LB_LATE = true;  // ... and a later predecessor fetch
    static constexpr unsigned HALO = 1u << 1;
    template <int I> struct Keep {};

    template <int I, bool EDGE>
    __device__ static void coeffs(const float (&x)[NIN][I], const float (&xn)[NIN], int kb,
                                  const Params &p, float, float (&a)[K][I], float (&b)[K][I], Keep<I> &)
    {
        const float gl = p.c0 * p.c1;
#pragma unroll
        for (int k = 0; k < I; ++k) {
            float dprev = (k > 0) ? x[1][k - 1] : xn[1];
            if (EDGE && k == kb) dprev = 0.f;
            a[0][k] = x[0][k];
            b[0][k] = gl * (1.f - dprev);
        }
    }
    template <int I>
    __device__ static void boundary(const float (&)[NIN][I], int, float rsc, const Params &, float (&bv)[K]) { bv[0] = rsc; }
    template <int I, bool EDGE>
    __device__ static void post(const float (&)[NIN][I], const float (&)[NIN], int, const Params &,
                                float, const float (&A)[K][I], const float (&)[K], const Keep<I> &, float (&o)[NOUT][I])
    {
#pragma unroll
        for (int k = 0; k < I; ++k) o[0][k] = A[0][k];
    }
};

// ---------------------------------------------------------------------------
// Episodic prefix sum (forward): alpha = x_t; beta = 1 - d_{t-1} (ends_at,
// d_{-1} = 0) or 1 - d_t (starts_at); A_{-1} = seed.  Inputs: 0 inputs, 1 dones.
template <bool STARTS_AT>
struct Prefix {
    static constexpr int NIN = 2, NOUT = 1;
    static constexpr int K = 1;  // affine recurrences per step
    static constexpr bool FWD = true, ROWSCALAR = true;
    static constexpr bool LB_CHAIN = true;  // beta = 1 within episodes
    static constexpr unsigned HALO = STARTS_AT ? 0u : (1u << 1);
    template <int I> struct Keep {};

    template <int I, bool EDGE>
    __device__ static void coeffs(const float (&x)[NIN][I], const float (&xn)[NIN], int kb,
                                  const Params &, float, float (&a)[K][I], float (&b)[K][I], Keep<I> &)
    {
#pragma unroll
        for (int k = 0; k < I; ++k) {
            float d;
            if constexpr (STARTS_AT) {
                d = x[1][k];
            } else {
                d = (k > 0) ? x[1][k - 1] : xn[1];
                if (EDGE && k == kb) d = 0.f;
            }
            a[0][k] = x[0][k];
            b[0][k] = 1.f - d;
        }
    }
    template <int I>
    __device__ static void boundary(const float (&)[NIN][I], int, float rsc, const Params &, float (&bv)[K]) { bv[0] = rsc; }
    template <int I, bool EDGE>
    __device__ static void post(const float (&)[NIN][I], const float (&)[NIN], int, const Params &,
                                float, const float (&A)[K][I], const float (&)[K], const Keep<I> &, float (&o)[NOUT][I])
    {
#pragma unroll
        for (int k = 0; k < I; ++k) o[0][k] = A[0][k];
    }
};

// ---------------------------------------------------------------------------
// Generic affine scan on given alpha, beta; boundary = carry.  Inputs: 0 alpha, 1 beta.
template <bool FORWARD>
struct Linear {
    static constexpr int NIN = 2, NOUT = 1;
    static constexpr int K = 1;  // affine recurrences per step
    static constexpr bool FWD = FORWARD, ROWSCALAR = true;
    static constexpr bool LB_CHAIN = true;  // beta is the caller's: often 1
    static constexpr unsigned HALO = 0;
    template <int I> struct Keep {};

    template <int I, bool EDGE>
    __device__ static void coeffs(const float (&x)[NIN][I], const float (&)[NIN], int,
                                  const Params &, float, float (&a)[K][I], float (&b)[K][I], Keep<I> &)
    {
#pragma unroll
        for (int k = 0; k < I; ++k) {
            a[0][k] = x[0][k];
            b[0][k] = x[1][k];
        }
    }
    template <int I>
    __device__ static void boundary(const float (&)[NIN][I], int, float rsc, const Params &, float (&bv)[K]) { bv[0] = rsc; }
    template <int I, bool EDGE>
    __device__ static void post(const float (&)[NIN][I], const float (&)[NIN], int, const Params &,
                                float, const float (&A)[K][I], const float (&)[K], const Keep<I> &, float (&o)[NOUT][I])
    {
#pragma unroll
        for (int k = 0; k < I; ++k) o[0][k] = A[0][k];
    }
};

// ---------------------------------------------------------------------------
// GAE together with lambda-returns and discounted returns from one read.
// Scan 0 is GAE (alpha = r + gamma (1-term) Vn - V, beta = gamma lambda
// (1-done), A_T = 0); lambda-returns are A + V (the identity the returns
// tutorial states for lambda-returns as GAE targets, Sec. 6; it equals the
// TD(lambda) recurrence with V(s_{t+1}) taken from `values` and the
// bootstrap); scan 1 is the discounted return (alpha = r + gamma trunc bs,
// beta = gamma (1-done), G_T = bs_{T-1}).
// Inputs as GAE: 0 rewards, 1 values, 2 terminateds, [3 truncateds], [3+TRUNC bootstrap].
// Outputs: 0 advantages, 1 lambda-returns, 2 discounted returns (each may be null).
template <bool TRUNC, bool BS2D>
struct GAEReturns {
    static_assert(TRUNC || !BS2D, "2-D bootstrap is read only with truncation flags");
    static constexpr int NIN = 3 + TRUNC + BS2D, NOUT = 3;
    static constexpr unsigned FLAGS = (1u << 2) | (TRUNC ? (1u << 3) : 0u);  // 0/1 inputs
    static constexpr int K = 2;
    static constexpr bool FWD = false, ROWSCALAR = !BS2D;
    static constexpr unsigned HALO = 1u << 1;
    static constexpr int TR = 3, BS = 3 + TRUNC;
    template <int I> struct Keep {};

    template <int I, bool EDGE>
    __device__ static void coeffs(const float (&x)[NIN][I], const float (&xn)[NIN], int kb,
                                  const Params &p, float rsc, float (&a)[K][I], float (&b)[K][I], Keep<I> &)
    {
        const float g = p.c0, gl = p.c0 * p.c1;
#pragma unroll
        for (int k = 0; k < I; ++k) {
            const bool last = (EDGE && k == kb);
            const float vnext = (k + 1 < I) ? x[1][k + 1] : xn[1];
            const float term = x[2][k];
            float vn, done, ret_alpha;
            if constexpr (TRUNC) {
                const float tr = x[TR][k];
                float bs;
                if constexpr (BS2D) bs = x[BS][k];
                else bs = last ? rsc : 0.f;
                vn = last ? bs : fmaf(1.f - tr, vnext, bs);
                done = done_of(term, tr);
                ret_alpha = fmaf(g * tr, bs, x[0][k]);
            } else {
                vn = last ? rsc : vnext;
                done = term;
                ret_alpha = x[0][k];
            }
            a[0][k] = fmaf(g * (1.f - term), vn, x[0][k]) - x[1][k];
            b[0][k] = gl * (1.f - done);
            a[1][k] = ret_alpha;
            b[1][k] = g * (1.f - done);
        }
    }
    template <int I>
    __device__ static void boundary(const float (&x)[NIN][I], int k, float rsc, const Params &, float (&bv)[K])
    {
        bv[0] = 0.f;
        if constexpr (BS2D) bv[1] = x[BS][k];
        else bv[1] = rsc;
    }
    template <int I, bool EDGE>
    __device__ static void post(const float (&x)[NIN][I], const float (&)[NIN], int, const Params &,
                                float, const float (&A)[K][I], const float (&)[K], const Keep<I> &,
                                float (&o)[NOUT][I])
    {
#pragma unroll
        for (int k = 0; k < I; ++k) {
            o[0][k] = A[0][k];
            o[1][k] = A[0][k] + x[1][k];
            o[2][k] = A[1][k];
        }
    }
};

// GAE + returns whose kernel also accumulates the batch moments (sum and
// sum of squares) of the advantages, output 0, for their normalisation.
template <bool TRUNC, bool BS2D>
struct GAEReturnsMoments : GAEReturns<TRUNC, BS2D> {
    static constexpr bool MOMENTS = true;
};

// The same without the discounted returns: one scan (GAE), outputs 0
// advantages and 1 lambda-returns (A + V), and the batch moments of the
// advantages.
template <bool TRUNC, bool BS2D>
struct GAELambdaMoments : GAE<TRUNC, BS2D> {
    using Base = GAE<TRUNC, BS2D>;
    static constexpr int NOUT = 2;
    static constexpr bool MOMENTS = true;

    template <int I, bool EDGE>
    __device__ static void post(const float (&x)[Base::NIN][I], const float (&)[Base::NIN], int, const Params &,
                                float, const float (&A)[1][I], const float (&)[1],
                                const typename Base::template Keep<I> &, float (&o)[NOUT][I])
    {
#pragma unroll
        for (int k = 0; k < I; ++k) {
            o[0][k] = A[0][k];
            o[1][k] = A[0][k] + x[1][k];
        }
    }
};

// Compact storage of an estimator's inputs and outputs: value inputs in
// VB-byte elements (2: bfloat16), flag inputs (Base::FLAGS) in FB-byte
// elements (1: uint8 0/1), outputs in OB-byte elements (4: float,
// 2: bfloat16 rounded to nearest even).  The arithmetic is the base
// estimator's, in float: a bf16 value is the float with the same upper 16
// bits, so every stored input is read exactly.
template <class Base, int VB, int FB, int OB>
struct Compact : Base {
    static constexpr int OUT_BYTES = OB;
    __host__ __device__ static constexpr int in_bytes(int j) { return ((Base::FLAGS >> j) & 1u) ? FB : VB; }
};

}  // namespace est
}  // namespace rlscan
