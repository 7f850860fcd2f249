/*
 * rlscan.h -- C ABI of librlscan, batched first-order linear recurrences for
 * reinforcement-learning credit assignment on NVIDIA GB300 (sm_103a).
 *
 * Every estimator solves, for each row (environment) of a [N, T] rollout
 * buffer, the affine recurrence
 *
 *     backward:  A_t = alpha_t + beta_t * A_{t+1}      (t = T-1 .. 0)
 *     forward:   A_t = alpha_t + beta_t * A_{t-1}      (t = 0 .. T-1)
 *
 * ("rl-triton: High-Performance Triton GPU Kernels for Reinforcement Learning
 * Credit Assignment", Eq. 1 and its forward mirror in Sec. 1), with the
 * per-step coefficients alpha_t, beta_t built inside the kernel from the raw
 * rollout tensors (same paper, Table 1 and Sec. 3.3).  The recurrence is
 * evaluated as an associative scan under (a1,b1) o (a2,b2) = (a1 + b1 a2,
 * b1 b2) (Eq. 2, Prop. 1).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers are owned by the caller: device memory, or page-locked host
 *    memory (cudaHostAlloc / cudaHostRegister), which the kernel reads and
 *    writes in place over the host link with plain loads and stores (zero
 *    copy; bulk asynchronous copies are used for device memory only).
 *    Pageable host memory is read the same way on a device that reports
 *    cudaDevAttrPageableMemoryAccess, and refused (RLSCAN_ERR_MEMORY, before
 *    any work is enqueued) on one that does not.  The workspace must be
 *    device memory.  The library never allocates, frees or retains them.
 *  - [N,T] arrays are float32, row-major, element stride 1, row stride
 *    `row_stride` elements (row_stride >= T), the same stride for every
 *    [N,T] argument of a call, inputs and outputs alike.  [N] arrays are
 *    dense float32.
 *  - Flags (terminateds, truncateds, dones) are float32 0.0 / 1.0.  The
 *    combined boundary flag is done_t = min(1, terminated_t + truncated_t).
 *    terminated and truncated are mutually exclusive; other flag values are
 *    outside the contract.
 *  - Outputs must not overlap any input or each other.  Passing the same
 *    pointer for an output and an input returns RLSCAN_ERR_ARG_CONFLICT;
 *    partial overlaps are not detected.
 *  - Nullable arguments are marked; NULL selects the documented default.
 *  - Every call only enqueues work on `stream` and returns; nothing is
 *    synchronised except in rlscan_workspace_status().
 *  - N == 0 or T == 0 is a no-op returning RLSCAN_OK.
 *  - Alignment: when T and row_stride are multiples of 4 and every [N,T]
 *    pointer is 16-byte aligned, rows are staged into shared memory with
 *    bulk asynchronous copies (TMA); otherwise an element-wise path is used.
 *    Both give the same results.
 *  - Workspace: rows longer than one kernel tile are scanned by several
 *    thread blocks that pass carries through a caller-provided workspace
 *    (decoupled look-back).  rlscan_workspace_bytes(N, T) gives the size
 *    that suffices for every entry point at that shape except the
 *    normalising one (rlscan_gae_normalized_workspace_bytes); it is 0 for
 *    T <= 512, where none needs one and `ws` may be NULL (when one is given
 *    for shorter rows, its ticket spreads the last tiles over the thread
 *    blocks as they become free).  A workspace must be zeroed once
 *    with rlscan_workspace_init() before its first use; afterwards it needs
 *    no clearing between calls (the kernels keep a call counter in it, so
 *    calls captured into a CUDA graph may be replayed).  One workspace serves one call at a time:
 *    calls that use the same workspace must be ordered (same stream, or
 *    synchronised).  Calls on different workspaces may run concurrently.
 *  - Arithmetic is float32; the importance ratios of V-trace and Retrace use
 *    CUDA's fast exponential and division (__expf, __fdividef: relative
 *    error of a few 1e-7 on these inputs).
 */
#ifndef RLSCAN_H
#define RLSCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA runtime headers. */
typedef struct CUstream_st *rlscan_stream_t;

typedef enum rlscan_status {
    RLSCAN_OK = 0,
    RLSCAN_ERR_NULL = 1,          /* a required pointer is NULL */
    RLSCAN_ERR_SHAPE = 2,         /* N < 0, T < 0 or row_stride < T */
    RLSCAN_ERR_ARG_CONFLICT = 3,  /* mutually exclusive arguments, or an output equals an input */
    RLSCAN_ERR_ARG_VALUE = 4,     /* enum or scalar argument out of range */
    RLSCAN_ERR_WORKSPACE = 5,     /* workspace needed but NULL, too small or misaligned */
    RLSCAN_ERR_CUDA = 6,          /* the CUDA runtime refused the launch */
    RLSCAN_ERR_INVALID_INPUT = 7, /* content check failed (only with RLSCAN_CHECKS=1) */
    RLSCAN_ERR_TIMEOUT = 8,       /* a cross-block wait gave up (reported by rlscan_workspace_status) */
    RLSCAN_ERR_SCRATCH_LIMIT = 9, /* shape needs more scratch than rlscan_gae_noalloc's built-in buffer */
    RLSCAN_ERR_MEMORY = 10        /* a pointer the GPU cannot reach: neither device (or managed) memory nor
                                     page-locked host memory, nor pageable memory on a device that
                                     reads pageable memory */
} rlscan_status;

typedef enum rlscan_dtype {
    RLSCAN_F32 = 0,   /* float32 */
    RLSCAN_BF16 = 1,  /* bfloat16 */
    RLSCAN_U8 = 2     /* uint8 */
} rlscan_dtype;

typedef enum rlscan_boundary {
    RLSCAN_ENDS_AT = 0,   /* done[t] = 1: the segment ends at t, reset lands at t+1 */
    RLSCAN_STARTS_AT = 1  /* done[t] = 1: the segment starts at t, reset lands at t  */
} rlscan_boundary;

typedef enum rlscan_direction {
    RLSCAN_BACKWARD = 0,  /* A_t = alpha_t + beta_t A_{t+1}, A_T    = carry */
    RLSCAN_FORWARD = 1    /* A_t = alpha_t + beta_t A_{t-1}, A_{-1} = carry */
} rlscan_direction;

/* Library version, (major << 16) | (minor << 8) | patch. */
int rlscan_version(void);

/* Static description of a status code.  Never NULL. */
const char *rlscan_status_string(rlscan_status status);

/* Bytes of workspace that suffice for every entry point on an [N, T] buffer
 * (except rlscan_gae_normalized, which has its own query): a 64-byte header
 * and 32 bytes per 1024 steps of every row.  0 for T <= 512, where no entry
 * point needs one, and for N <= 0 or T <= 0. */
size_t rlscan_workspace_bytes(int64_t N, int64_t T);

/* Zero a workspace of `ws_bytes` bytes (asynchronously on `stream`).  Call
 * once after allocating it.  ws must be 16-byte aligned.
 * Errors: RLSCAN_ERR_NULL, RLSCAN_ERR_WORKSPACE (misaligned), RLSCAN_ERR_CUDA. */
rlscan_status rlscan_workspace_init(void *ws, size_t ws_bytes, rlscan_stream_t stream);

/* Synchronise `stream`, then return and clear the error recorded in the
 * workspace by earlier calls (RLSCAN_OK if none; RLSCAN_ERR_TIMEOUT if a
 * cross-block wait gave up, in which case the affected outputs hold NaN).
 * A CUDA error raised by the synchronisation is returned as RLSCAN_ERR_CUDA. */
rlscan_status rlscan_workspace_status(void *ws, size_t ws_bytes, rlscan_stream_t stream);

/*
 * Generalized Advantage Estimation.
 * rl-triton API reference, compute_gae; rl-triton paper Table 1 row "GAE",
 * Sec. 3.2 and Sec. 3.3.1; "Technical Deep Dive into the GAE Triton Kernel"
 * Sec. 5.
 *   delta_t = r_t + gamma (1 - term_t) Vn_t - V_t
 *   A_t     = delta_t + gamma lambda (1 - done_t) A_{t+1},   A_T = 0
 * Vn_t, the successor value: with truncateds,
 *   Vn_t = (t < T-1 ? (1 - trunc_t) V_{t+1} : 0) + bs_t;
 * without truncateds, Vn_t = V_{t+1} for t < T-1 and Vn_{T-1} = bs_{T-1}
 * (interior bootstrap entries are not read).  bs = bootstrap_values (zero
 * when NULL); last_value supplies bs_{T-1} alone.
 * Inputs : rewards, values, terminateds [N,T]; truncateds [N,T] nullable;
 *          bootstrap_values [N,T] nullable; last_value [N] nullable.
 * Output : advantages [N,T].
 * Errors : RLSCAN_ERR_ARG_CONFLICT when both bootstrap_values and
 *          last_value are given, or last_value together with truncateds.
 */
rlscan_status rlscan_gae(const float *rewards, const float *values, const float *terminateds,
                         const float *truncateds, const float *bootstrap_values,
                         const float *last_value, int64_t N, int64_t T, int64_t row_stride,
                         float gamma, float lambda, float *advantages,
                         void *ws, size_t ws_bytes, rlscan_stream_t stream);

/*
 * GAE with observation-skip masking.  rl-triton paper Sec. 9.3 plans
 * "observation-skip masking that carries the recurrence across masked
 * tokens (beta_t = 1)"; read here as: at a masked step (mask_t = 0) the
 * advantage is handed through unchanged, A_t = A_{t+1} (alpha_t = 0,
 * beta_t = 1); an unmasked step is the GAE step of rlscan_gae unchanged,
 * including its successor value Vn_t (the stored V_{t+1}, or the bootstrap
 * rule there).  Past the last unmasked step of a row the value is 0.
 *   A_t = m_t delta_t + (m_t gamma lambda (1 - done_t) + 1 - m_t) A_{t+1}
 * For token-level LLM rollouts, mask = 1 on the policy's (response) tokens
 * and 0 on prompt, observation or padding tokens.
 * Inputs : as rlscan_gae, plus mask [N,T] float32 0/1 (required).
 * Outputs: advantages [N,T] (masked steps hold the next unmasked value).
 */
rlscan_status rlscan_gae_masked(const float *rewards, const float *values, const float *terminateds,
                                const float *truncateds, const float *bootstrap_values,
                                const float *last_value, const float *mask, int64_t N, int64_t T,
                                int64_t row_stride, float gamma, float lambda, float *advantages,
                                void *ws, size_t ws_bytes, rlscan_stream_t stream);

/*
 * GAE, lambda-returns and discounted returns from one read of the buffer.
 * The rl-triton paper's planned fused post-scan extensions (Sec. 9.3); the
 * returns tutorial's identity that lambda-returns are the GAE targets
 * (Sec. 6); API reference compute_gae / compute_lambda_returns /
 * compute_discounted_returns for each output.
 *   advantages         = rlscan_gae on the same arguments
 *   lambda_returns     = advantages + values: TD(lambda) returns whose
 *                        V(s_{t+1}) is the successor value rlscan_gae uses
 *                        (values[t+1]; the bootstrap at truncated steps and
 *                        at the window end), i.e. rlscan_lambda_returns with
 *                        next_values built that way
 *   discounted_returns = rlscan_discounted_returns on the same rewards,
 *                        flags and bootstrap (carry bs_{T-1})
 * One kernel runs both recurrences (beta = gamma lambda (1 - done) and
 * gamma (1 - done)) over a single pass of the inputs.
 * Inputs : as rlscan_gae.
 * Outputs: advantages, lambda_returns, discounted_returns [N,T], each
 *          nullable, at least one non-NULL.
 * Errors : as rlscan_gae; RLSCAN_ERR_NULL when every output is NULL.
 */
rlscan_status rlscan_gae_returns(const float *rewards, const float *values,
                                 const float *terminateds, const float *truncateds,
                                 const float *bootstrap_values, const float *last_value,
                                 int64_t N, int64_t T, int64_t row_stride, float gamma,
                                 float lambda, float *advantages, float *lambda_returns,
                                 float *discounted_returns, void *ws, size_t ws_bytes,
                                 rlscan_stream_t stream);

/*
 * GAE without any device allocation, for callers that cannot allocate.
 * The rl-triton pages have no counterpart: this is a deployment variant of
 * rlscan_gae.  Some callers may not allocate device memory when they call
 * in: a plugin inside a framework that owns all device memory through its
 * own pool, a latency-critical loop that bans cudaMalloc/cudaFree after
 * start-up (both can synchronise the device), or an embedded runtime with a
 * fixed memory budget.  Rows longer than one tile need scratch for the
 * cross-block carries; this entry point takes it from a 4 MiB buffer built
 * into the library (each GPU that loads the library keeps it until the
 * process exits) instead of a caller workspace.  That covers shapes with
 * rlscan_workspace_bytes(N, T) <= 4 MiB, i.e. N * ceil(T / 1024) <= 131070
 * (e.g. 32 rows of 4M steps); larger shapes return RLSCAN_ERR_SCRATCH_LIMIT
 * before any device work.  Same arguments and results as rlscan_gae, minus
 * the workspace.  The first call on a device looks up the buffer's address
 * and zeroes it on `stream`; make that first call before any stream
 * capture.  The address is kept for the life of the process: tearing the
 * device's primary context down between calls (cudaDeviceReset) is not
 * supported.  Argument conflicts (as rlscan_gae) are refused before the
 * buffer is touched; a call refused later (a content check with
 * RLSCAN_CHECKS=1, a failed launch) may already have enqueued the header
 * clear, which is harmless.  Every call clears the buffer's header on
 * `stream` before its kernel; calls that share the buffer and overlap on
 * the GPU (unordered streams) race and must not be issued.  A timed-out
 * cross-block wait shows up as NaN outputs (this variant has no status
 * query); later calls are unaffected.
 */
rlscan_status rlscan_gae_noalloc(const float *rewards, const float *values,
                                 const float *terminateds, const float *truncateds,
                                 const float *bootstrap_values, const float *last_value,
                                 int64_t N, int64_t T, int64_t row_stride, float gamma,
                                 float lambda, float *advantages, rlscan_stream_t stream);

/*
 * GAE with its advantages normalised over the whole batch, fused with the
 * returns.  rl-triton paper Sec. 9.3 plans "fused advantage normalization";
 * it is read here as the usual per-batch whitening
 *   adv_t <- (A_t - mean) / (std + eps)
 * with mean and the unbiased (n - 1) standard deviation of all N*T raw GAE
 * advantages A_t of the call (rlscan_gae's values).  The scan kernel also
 * accumulates the batch moments (sum and sum of squares): each thread sums
 * its advantages of a tile in float and carries the totals across tiles as
 * float pairs (unevaluated sums hi + lo, combined with Knuth's TwoSum), the
 * CTA combines its threads' pairs the same way and writes one pair per
 * moment; a second kernel, ordered after it on `stream`, combines the
 * per-CTA pairs in CTA order (every block the same way, so the result is
 * the same bits on every call), derives the mean and standard deviation in
 * float-pair arithmetic and normalises the advantages in place.
 * lambda_returns (A_t + V_t) and discounted_returns are computed from the
 * RAW advantages, as in rlscan_gae_returns; the scan solves one recurrence
 * per step when discounted_returns is NULL and two otherwise.
 * Inputs : as rlscan_gae_returns; eps >= 0 (else RLSCAN_ERR_ARG_VALUE).
 * Outputs: advantages [N,T] (normalised; required); lambda_returns,
 *          discounted_returns [N,T] nullable; moments: nullable device
 *          float[2] receiving (mean, std) of the raw advantages.
 * Workspace: always needed, rlscan_gae_normalized_workspace_bytes(N, T)
 *          bytes, 16-byte aligned, zeroed once by rlscan_workspace_init
 *          (the usual look-back workspace followed by the moments region);
 *          otherwise RLSCAN_ERR_WORKSPACE.
 * With N*T == 1 the standard deviation is undefined and the output is NaN.
 */
size_t rlscan_gae_normalized_workspace_bytes(int64_t N, int64_t T);

rlscan_status rlscan_gae_normalized(const float *rewards, const float *values,
                                    const float *terminateds, const float *truncateds,
                                    const float *bootstrap_values, const float *last_value,
                                    int64_t N, int64_t T, int64_t row_stride, float gamma,
                                    float lambda, float eps, float *advantages,
                                    float *lambda_returns, float *discounted_returns,
                                    float *moments, void *ws, size_t ws_bytes,
                                    rlscan_stream_t stream);

/*
 * Bounds-check diagnostics (no counterpart on the pages).  A library built
 * with RLSCAN_CHECK_BOUNDS=1 tests every global access of its scan kernels,
 * and every bulk copy's source and shared-memory destination, against the
 * extent of the argument it belongs to; a failed test skips the access and
 * counts one violation.  rlscan_bounds_check synchronises the device, then
 * stores the count and the site code of the first violation (1 copy source,
 * 2 copy target, 3 element-wise load, 4 output store, 5 per-row scalar,
 * 6 look-back state, 7 wide input, 8 moments slot, 9 ring stage); reset != 0
 * zeroes them.  Returns 1 in a checked build, 0 in a normal build (nothing
 * is checked; both values 0), -1 on a CUDA error.
 * Positive control (checked build only): with the environment variable
 * RLSCAN_TEST_CHECK_SHORT=1 every [N,T] argument is checked as if it held
 * N-1 rows, so the accesses to the last row (all inside the real arrays)
 * must be reported; their outputs are then not written.
 */
int rlscan_bounds_check(unsigned long long *violations, unsigned long long *first_site, int reset);

/*
 * GAE and fused GAE + returns on compact storage: rewards, values and
 * bootstrap_values in bfloat16, terminateds and truncateds in uint8 (0/1),
 * outputs in float32 or bfloat16 (out_dtype).  rl-triton paper Sec. 9.3
 * plans bfloat16 I/O and Sec. 9.2 defers it "pending a precision-tradeoff
 * analysis"; here the arithmetic stays float32: a bfloat16 value is the
 * float32 with the same upper 16 bits, so every stored input is read
 * exactly and the recurrence is the float32 one of rlscan_gae /
 * rlscan_gae_returns on those values.  The only additional error is the
 * rounding of bfloat16 outputs (to nearest even, at most 2^-9 relative).
 * Bytes per step fall from 16 to 9 (GAE, float32 out) or 7 (bf16 out).
 * Inputs : rewards, values [N,T] bf16; terminateds [N,T] u8; truncateds
 *          [N,T] u8 nullable; bootstrap_values [N,T] bf16 nullable, only
 *          with truncateds (without truncateds the window bootstrap is
 *          last_value, float32 [N], nullable); otherwise
 *          RLSCAN_ERR_ARG_CONFLICT.
 * Outputs: rlscan_gae_compact: advantages; rlscan_gae_returns_compact:
 *          advantages, lambda_returns, discounted_returns (nullable, at
 *          least one), each [N,T] of out_dtype (RLSCAN_F32 or RLSCAN_BF16,
 *          else RLSCAN_ERR_ARG_VALUE).
 * Bulk copies need rows in whole 16-byte units (T and row_stride multiples
 * of 16 for the uint8 flags); other shapes use element-wise loads.  The
 * content checks of RLSCAN_CHECKS do not cover these entry points.
 */
rlscan_status rlscan_gae_compact(const void *rewards, const void *values, const void *terminateds,
                                 const void *truncateds, const void *bootstrap_values,
                                 const float *last_value, int64_t N, int64_t T, int64_t row_stride,
                                 float gamma, float lambda, rlscan_dtype out_dtype, void *advantages,
                                 void *ws, size_t ws_bytes, rlscan_stream_t stream);

rlscan_status rlscan_gae_returns_compact(const void *rewards, const void *values,
                                         const void *terminateds, const void *truncateds,
                                         const void *bootstrap_values, const float *last_value,
                                         int64_t N, int64_t T, int64_t row_stride, float gamma,
                                         float lambda, rlscan_dtype out_dtype, void *advantages,
                                         void *lambda_returns, void *discounted_returns, void *ws,
                                         size_t ws_bytes, rlscan_stream_t stream);

/*
 * V-trace and Retrace(lambda) (per-step inputs) on compact storage, the
 * same bfloat16 I/O plan (rl-triton paper Sec. 9.2-9.3) carried to the
 * off-policy estimators: every value input in bfloat16 (V-trace
 * log_pi_target, log_pi_behavior, values, rewards, bootstrap_values;
 * Retrace pi_taken, mu_taken, q_values, expected_next_q, rewards), the
 * flags in uint8 (0/1), both outputs in out_dtype.  The arithmetic is that
 * of rlscan_vtrace / rlscan_retrace in float32 on the stored values (the
 * ratio exp(lpt - lpb) or pi / mu is formed from the bfloat16 inputs read
 * exactly).  Bytes per step: V-trace 36 -> 20 with float32 outputs, 16 with
 * bf16 outputs (with truncation flags and a 2-D bootstrap); Retrace
 * 32 -> 19 / 15.
 * Inputs : as rlscan_vtrace / rlscan_retrace in the storage types above;
 *          for V-trace the window bootstrap without truncateds is
 *          last_value (float32 [N], nullable), and bootstrap_values
 *          without truncateds is RLSCAN_ERR_ARG_CONFLICT.
 * Outputs: V-trace targets and advantages, or Retrace targets and
 *          advantages, each [N,T] of out_dtype (RLSCAN_F32 or RLSCAN_BF16,
 *          else RLSCAN_ERR_ARG_VALUE).
 * Alignment and content checks as for rlscan_gae_compact.
 */
rlscan_status rlscan_vtrace_compact(const void *log_pi_target, const void *log_pi_behavior,
                                    const void *values, const void *rewards, const void *terminateds,
                                    const void *truncateds, const void *bootstrap_values,
                                    const float *last_value, int64_t N, int64_t T, int64_t row_stride,
                                    float gamma, float rho_bar, float c_bar, rlscan_dtype out_dtype,
                                    void *vtrace_targets, void *vtrace_advantages, void *ws,
                                    size_t ws_bytes, rlscan_stream_t stream);

rlscan_status rlscan_retrace_compact(const void *pi_taken, const void *mu_taken, const void *q_values,
                                     const void *expected_next_q, const void *rewards,
                                     const void *terminateds, const void *truncateds, int64_t N,
                                     int64_t T, int64_t row_stride, float gamma, float lambda,
                                     float c_bar, float rho_bar, rlscan_dtype out_dtype,
                                     void *retrace_targets, void *advantages, void *ws, size_t ws_bytes,
                                     rlscan_stream_t stream);

/*
 * V-trace targets and advantages.
 * rl-triton API reference, compute_vtrace; rl-triton paper Table 1 row
 * "V-Trace" and Sec. 3.3.2.
 *   ratio_t = exp(log_pi_target_t - log_pi_behavior_t)
 *   rho_t = min(rho_bar, ratio_t),  c_t = min(c_bar, ratio_t)
 *   D_t   = rho_t (r_t + gamma (1 - term_t) Vn_t - V_t) + gamma c_t (1 - done_t) D_{t+1},  D_T = 0
 *   vs_t  = D_t + V_t
 *   adv_t = rho_t (r_t + gamma (1 - term_t) vsn_t - V_t)
 * Vn and vsn follow the successor rule of rlscan_gae (vsn with vs in place
 * of V).  last_value may be combined with truncateds (it then supplies
 * bs_{T-1}, interior bootstrap zero).
 * Inputs : log_pi_target, log_pi_behavior, values, rewards, terminateds [N,T];
 *          truncateds, bootstrap_values [N,T] nullable; last_value [N] nullable.
 * Outputs: vtrace_targets, vtrace_advantages [N,T].
 * Errors : RLSCAN_ERR_ARG_CONFLICT when both bootstrap_values and last_value.
 */
rlscan_status rlscan_vtrace(const float *log_pi_target, const float *log_pi_behavior,
                            const float *values, const float *rewards, const float *terminateds,
                            const float *truncateds, const float *bootstrap_values,
                            const float *last_value, int64_t N, int64_t T, int64_t row_stride,
                            float gamma, float rho_bar, float c_bar,
                            float *vtrace_targets, float *vtrace_advantages,
                            void *ws, size_t ws_bytes, rlscan_stream_t stream);

/*
 * Retrace(lambda) targets and advantages from per-step inputs.
 * rl-triton API reference, compute_retrace (recurrence, targets and
 * advantages); rl-triton paper Table 1 row "Retrace" and Sec. 3.3.3;
 * "Retrace(lambda) with Triton Associative Scans" Sec. 3, 4 and 6.
 *   ratio_t = pi_t / mu_t,  c_t = lambda min(c_bar, ratio_t),  rho_t = min(rho_bar, ratio_t)
 *   D_t    = r_t + gamma (1 - term_t) EQ_t - Q_t + gamma c_{t+1} (1 - done_t) D_{t+1}
 *            with c_T = 0 and D_T = 0
 *   Qret_t = Q_t + D_t
 *   adv_t  = rho_t (r_t + gamma (1 - term_t) Qret_{t+1} - Q_t),   Qret_T = 0
 * pi_taken = pi(a_t|s_t), mu_taken = mu(a_t|s_t), expected_next_q =
 * E_pi[Q(s_{t+1}, .)] (the caller supplies Q(s_T, .) at t = T-1).
 * Inputs : pi_taken, mu_taken, q_values, expected_next_q, rewards,
 *          terminateds [N,T]; truncateds [N,T] nullable (zero).
 * Outputs: retrace_targets, advantages [N,T].
 */
rlscan_status rlscan_retrace(const float *pi_taken, const float *mu_taken, const float *q_values,
                             const float *expected_next_q, const float *rewards,
                             const float *terminateds, const float *truncateds,
                             int64_t N, int64_t T, int64_t row_stride,
                             float gamma, float lambda, float c_bar, float rho_bar,
                             float *retrace_targets, float *advantages,
                             void *ws, size_t ws_bytes, rlscan_stream_t stream);

/*
 * Retrace(lambda) targets and advantages from the full action-space inputs,
 * the argument set of the rl-triton API reference's compute_retrace
 * (action_probs_target and next_q_values_all [N,T,A], actions int64 [N,T]).
 * The action dimension is reduced inside the kernel, per step:
 *   EQ_t = sum_a pi_target[t,a] * next_q_values_all[t,a]      (a = 0 .. A-1)
 *   pi_t = pi_target[t, actions[t]]
 * then the recurrence of rlscan_retrace with mu_t = action_probs_behavior[t].
 * The target weights are those stored at the same step t: the API's
 * reduction multiplies the two [N,T,A] tensors element-wise (its
 * mathematical text weights Q(s_{t+1},.) with pi(.|s_{t+1}); a caller who
 * wants that stores pi(.|s_{t+1}) at step t).
 * Layout : action_probs_target and next_q_values_all are float32 [N,T,A]
 *          with element (n,t,a) at n * action_row_stride + t * A + a
 *          (action_row_stride >= T * A, the same for both); actions is int64
 *          [N,T] and every float32 [N,T] argument has row stride row_stride.
 * Inputs : action_probs_target, action_probs_behavior, q_values,
 *          next_q_values_all, actions, rewards, terminateds; truncateds
 *          nullable (zero).
 * Outputs: retrace_targets, advantages [N,T].
 * An action outside [0, A) makes pi_t NaN (its row's outputs are then NaN
 * up to the row start); with RLSCAN_CHECKS=1 such a call returns
 * RLSCAN_ERR_INVALID_INPUT instead.
 * Errors : RLSCAN_ERR_ARG_VALUE when A < 1 or A > 65536; RLSCAN_ERR_SHAPE
 *          when action_row_stride < T * A.
 * The [N,T,A] rows are staged into shared memory with bulk copies when they
 * are 16-byte aligned (action_row_stride a multiple of 4) and a 1024-step
 * tile of them fits the ring (A <= 9); otherwise the kernel reads them from
 * global memory.  Both give the same results.
 */
rlscan_status rlscan_retrace_actions(const float *action_probs_target,
                                     const float *action_probs_behavior, const float *q_values,
                                     const float *next_q_values_all, const int64_t *actions,
                                     const float *rewards, const float *terminateds,
                                     const float *truncateds, int64_t N, int64_t T, int64_t A,
                                     int64_t row_stride, int64_t action_row_stride,
                                     float gamma, float lambda, float c_bar, float rho_bar,
                                     float *retrace_targets, float *advantages,
                                     void *ws, size_t ws_bytes, rlscan_stream_t stream);

/*
 * TD(lambda) returns.
 * rl-triton API reference, compute_lambda_returns; rl-triton paper Table 1
 * row "TD(lambda)" and Sec. 3.3.4; "Returns and Eligibility Traces with
 * Triton Associative Scans" Sec. 2.
 *   G_t = r_t + gamma (1-lambda)(1 - done_t) nv_t + gamma trunc_t bs_t
 *         + gamma lambda (1 - done_t) G_{t+1},        G_T = bs_{T-1}
 * nv = next_values (V(s_{t+1}), zeroed by the caller at truncated steps).
 * bs = bootstrap_values (zero when NULL); last_value supplies bs_{T-1}
 * alone (an addition to the pages' signature: their 1-D window bootstrap).
 * Without truncateds only bs_{T-1} is read.
 * Inputs : rewards, next_values, terminateds [N,T]; truncateds,
 *          bootstrap_values [N,T] nullable; last_value [N] nullable.
 * Output : returns [N,T].
 * Errors : RLSCAN_ERR_ARG_CONFLICT when both bootstrap_values and last_value.
 */
rlscan_status rlscan_lambda_returns(const float *rewards, const float *next_values,
                                    const float *terminateds, const float *truncateds,
                                    const float *bootstrap_values, const float *last_value,
                                    int64_t N, int64_t T, int64_t row_stride,
                                    float gamma, float lambda, float *returns,
                                    void *ws, size_t ws_bytes, rlscan_stream_t stream);

/*
 * Discounted returns (reward-to-go).
 * rl-triton API reference, compute_discounted_returns; rl-triton paper
 * Table 1 row "Disc. Returns" and Sec. 3.3.4; "Returns and Eligibility
 * Traces with Triton Associative Scans" Sec. 1.
 *   G_t = r_t + gamma trunc_t bs_t + gamma (1 - done_t) G_{t+1},   G_T = bs_{T-1}
 * bs and last_value as for rlscan_lambda_returns.
 * Inputs : rewards, terminateds [N,T]; truncateds, bootstrap_values [N,T]
 *          nullable; last_value [N] nullable.
 * Output : returns [N,T].
 * Errors : RLSCAN_ERR_ARG_CONFLICT when both bootstrap_values and last_value.
 */
rlscan_status rlscan_discounted_returns(const float *rewards, const float *terminateds,
                                        const float *truncateds, const float *bootstrap_values,
                                        const float *last_value, int64_t N, int64_t T,
                                        int64_t row_stride, float gamma, float *returns,
                                        void *ws, size_t ws_bytes, rlscan_stream_t stream);

/*
 * Accumulating eligibility traces, forward in time.
 * rl-triton API reference, compute_eligibility_traces; rl-triton paper
 * Table 1 row "Elig. Traces" and Sec. 3.3.5.
 *   z_t = g_t + gamma lambda (1 - d_{t-1}) z_{t-1},   d_{-1} = 0,  z_{-1} = seed
 * dones[t] = 1 means the episode ends at t (pass terminated OR truncated,
 * unshifted).  seed_values [N] nullable (zero).
 * Inputs : gradients, dones [N,T]; seed_values [N] nullable.
 * Output : traces [N,T].
 */
rlscan_status rlscan_eligibility_traces(const float *gradients, const float *dones,
                                        const float *seed_values, int64_t N, int64_t T,
                                        int64_t row_stride, float gamma, float lambda,
                                        float *traces, void *ws, size_t ws_bytes,
                                        rlscan_stream_t stream);

/*
 * Episodic prefix sum, forward in time.
 * rl-triton API reference, compute_episodic_prefix_sum; rl-triton paper
 * Table 1 row "Prefix Sum" and Sec. 3.3.6.
 *   RLSCAN_ENDS_AT:   C_t = x_t + (1 - d_{t-1}) C_{t-1},   d_{-1} = 0
 *   RLSCAN_STARTS_AT: C_t = x_t + (1 - d_t) C_{t-1}
 *   C_{-1} = seed (zero when seed_values is NULL)
 * Inputs : inputs, dones [N,T]; seed_values [N] nullable.
 * Output : prefix_sums [N,T].
 * Errors : RLSCAN_ERR_ARG_VALUE for an unknown boundary.
 */
rlscan_status rlscan_episodic_prefix_sum(const float *inputs, const float *dones,
                                         const float *seed_values, rlscan_boundary boundary,
                                         int64_t N, int64_t T, int64_t row_stride,
                                         float *prefix_sums, void *ws, size_t ws_bytes,
                                         rlscan_stream_t stream);

/*
 * Generic affine recurrence on caller-supplied coefficients.
 * rl-triton paper Eq. 1 (backward) and its forward mirror (Sec. 1); the
 * carry is applied as in Sec. 4.1 step 4.
 *   RLSCAN_BACKWARD: A_t = alpha_t + beta_t A_{t+1},  A_T    = carry
 *   RLSCAN_FORWARD:  A_t = alpha_t + beta_t A_{t-1},  A_{-1} = carry
 * Inputs : alpha, beta [N,T]; carry [N] nullable (zero).
 * Output : out [N,T].
 * Errors : RLSCAN_ERR_ARG_VALUE for an unknown direction.
 */
rlscan_status rlscan_linear_scan(const float *alpha, const float *beta, const float *carry,
                                 rlscan_direction direction, int64_t N, int64_t T,
                                 int64_t row_stride, float *out, void *ws, size_t ws_bytes,
                                 rlscan_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* RLSCAN_H */
