// rlscan_abi.cu -- the extern "C" entry points of librlscan: argument
// validation (the pages' always-on structural checks, rl-triton API
// reference, compute_* functions), choice of the kernel specialisation from
// which optional arguments are present (the pages' HAS_TRUNCATIONS /
// HAS_BOOTSTRAP / HAS_SEED / BOUNDARY_ENDS_AT specialisations, paper
// Sec. 4.2), and the workspace helpers.
#include <cstdlib>
#include <cstring>
#include <initializer_list>

#include <cuda_runtime.h>

#include "params.cuh"
#include "residency.cuh"

namespace rlscan {

#ifndef RLSCAN_CHECK_BOUNDS
#define RLSCAN_CHECK_BOUNDS 0
#endif

// Checked builds: one device counter per process (violations, first site),
// allocated and zeroed at first use; normal builds have none.
unsigned long long *bounds_counter()
{
#if RLSCAN_CHECK_BOUNDS
    static unsigned long long *counter = [] {
        unsigned long long *c = nullptr;
        if (cudaMalloc(&c, 2 * sizeof(unsigned long long)) != cudaSuccess ||
            cudaMemset(c, 0, 2 * sizeof(unsigned long long)) != cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess) {
            cudaGetLastError();
            return static_cast<unsigned long long *>(nullptr);
        }
        return c;
    }();
    return counter;
#else
    return nullptr;
#endif
}

bool check_short()
{
#if RLSCAN_CHECK_BOUNDS
    static const bool on = [] {
        const char *s = std::getenv("RLSCAN_TEST_CHECK_SHORT");
        return s != nullptr && s[0] == '1';
    }();
    return on;
#else
    return false;
#endif
}

uint64_t spin_limit_ns()
{
    static const uint64_t limit = [] {
        const char *s = std::getenv("RLSCAN_SPIN_LIMIT_NS");
        if (s != nullptr) {
            const unsigned long long v = std::strtoull(s, nullptr, 10);
            if (v > 0) return static_cast<uint64_t>(v);
        }
        return static_cast<uint64_t>(1000000000ull);  // one second
    }();
    return limit;
}

int64_t withhold_tile()
{
    static const int64_t tile = [] {
        const char *s = std::getenv("RLSCAN_TEST_WITHHOLD_TILE");
        return s != nullptr ? static_cast<int64_t>(std::strtoll(s, nullptr, 10)) : int64_t(-1);
    }();
    return tile;
}

bool pdl_enabled()
{
    static const bool on = [] {
        const char *s = std::getenv("RLSCAN_PDL");
        return !(s != nullptr && s[0] == '0');
    }();
    return on;
}

namespace {

__global__ void zero_words(uint32_t *p, size_t n)
{
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        p[i] = 0u;
}

inline cudaStream_t cs(rlscan_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// ---- opt-in content checks (RLSCAN_CHECKS=1) --------------------------------
// The rl-triton API reference's correctness-warning checks: terminated and
// truncated are mutually exclusive, and bootstrap_values is zero at interior
// non-truncated steps (compute_gae / compute_vtrace).  Debug only: the call
// synchronises the stream to return the verdict.

__device__ uint32_t g_check_flags;

__global__ void check_inputs(const float *term, const float *trunc, const float *bs, int64_t N,
                             int64_t T, int64_t rs)
{
    uint32_t bad = 0;
    const int64_t total = N * T;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = i / T, t = i - row * T;
        const int64_t e = row * rs + t;
        const float tr = trunc[e];
        if (term != nullptr && term[e] != 0.f && tr != 0.f) bad |= 1u;
        if (bs != nullptr && t < T - 1 && tr == 0.f && bs[e] != 0.f) bad |= 2u;
    }
    if (bad) atomicOr(&g_check_flags, bad);
}

bool checks_enabled()
{
    static const bool on = [] {
        const char *s = std::getenv("RLSCAN_CHECKS");
        return s != nullptr && s[0] == '1';
    }();
    return on;
}

// RLSCAN_OK when the inputs pass (or checks are off), RLSCAN_ERR_INVALID_INPUT otherwise.
rlscan_status run_checks(const float *term, const float *trunc, const float *bs, int64_t N,
                         int64_t T, int64_t rs, cudaStream_t stream)
{
    if (!checks_enabled() || trunc == nullptr) return RLSCAN_OK;
    for (const void *ptr : {static_cast<const void *>(term), static_cast<const void *>(trunc),
                            static_cast<const void *>(bs)})
        if (ptr != nullptr && residency(ptr) == Residency::Unreachable) return RLSCAN_ERR_MEMORY;
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbolAsync(g_check_flags, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                stream) != cudaSuccess)
        return RLSCAN_ERR_CUDA;
    int64_t blocks = (N * T + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    check_inputs<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(term, trunc, bs, N, T, rs);
    uint32_t flags = 0;
    if (cudaGetLastError() != cudaSuccess ||
        cudaMemcpyFromSymbolAsync(&flags, g_check_flags, sizeof(flags), 0, cudaMemcpyDeviceToHost,
                                  stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return RLSCAN_ERR_CUDA;
    return flags ? RLSCAN_ERR_INVALID_INPUT : RLSCAN_OK;
}

// Every action index in [0, A) (compute_retrace gathers pi_target at it).
__global__ void check_actions(const long long *actions, int64_t N, int64_t T, int64_t rs, int64_t A)
{
    uint32_t bad = 0;
    const int64_t total = N * T;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = i / T, t = i - row * T;
        const long long a = actions[row * rs + t];
        if (a < 0 || a >= A) bad = 4u;
    }
    if (bad) atomicOr(&g_check_flags, bad);
}

rlscan_status run_action_checks(const int64_t *actions, int64_t N, int64_t T, int64_t rs, int64_t A,
                                cudaStream_t stream)
{
    if (!checks_enabled()) return RLSCAN_OK;
    if (residency(actions) == Residency::Unreachable) return RLSCAN_ERR_MEMORY;
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbolAsync(g_check_flags, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                stream) != cudaSuccess)
        return RLSCAN_ERR_CUDA;
    int64_t blocks = (N * T + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    check_actions<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        reinterpret_cast<const long long *>(actions), N, T, rs, A);
    uint32_t flags = 0;
    if (cudaGetLastError() != cudaSuccess ||
        cudaMemcpyFromSymbolAsync(&flags, g_check_flags, sizeof(flags), 0, cudaMemcpyDeviceToHost,
                                  stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return RLSCAN_ERR_CUDA;
    return flags ? RLSCAN_ERR_INVALID_INPUT : RLSCAN_OK;
}

inline rlscan_status check_shape(int64_t N, int64_t T, int64_t rs)
{
    if (N < 0 || T < 0 || rs < T) return RLSCAN_ERR_SHAPE;
    return RLSCAN_OK;
}

// An output equal to any input (or to the other output) is a conflict.
inline bool same_as_any(const void *out, std::initializer_list<const void *> others)
{
    for (const void *o : others)
        if (o != nullptr && o == out) return true;
    return false;
}

inline Params base_params(int64_t N, int64_t T, int64_t rs)
{
    Params p;
    std::memset(&p, 0, sizeof(p));
    p.N = N;
    p.T = T;
    p.rs = rs;
    p.rowscalar_stride = 1;
    return p;
}

}  // namespace
}  // namespace rlscan

using namespace rlscan;

#define RLSCAN_TRY(expr)                           \
    do {                                           \
        const rlscan_status st_ = (expr);          \
        if (st_ != RLSCAN_OK) return st_;          \
    } while (0)

#define RLSCAN_API __attribute__((visibility("default")))

extern "C" {

RLSCAN_API int rlscan_version(void) { return (0 << 16) | (1 << 8) | 0; }

RLSCAN_API const char *rlscan_status_string(rlscan_status status)
{
    switch (status) {
    case RLSCAN_OK: return "ok";
    case RLSCAN_ERR_NULL: return "a required pointer is NULL";
    case RLSCAN_ERR_SHAPE: return "invalid shape (N < 0, T < 0 or row_stride < T)";
    case RLSCAN_ERR_ARG_CONFLICT: return "conflicting arguments (exclusive options, or an output equal to an input)";
    case RLSCAN_ERR_ARG_VALUE: return "argument value out of range";
    case RLSCAN_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case RLSCAN_ERR_CUDA: return "CUDA runtime error";
    case RLSCAN_ERR_INVALID_INPUT: return "input content check failed";
    case RLSCAN_ERR_TIMEOUT: return "a cross-block wait timed out";
    case RLSCAN_ERR_SCRATCH_LIMIT: return "shape needs more scratch than the built-in no-allocation buffer holds";
    case RLSCAN_ERR_MEMORY: return "a pointer is in memory the GPU cannot reach (pageable host memory)";
    }
    return "unknown status";
}

RLSCAN_API int rlscan_bounds_check(unsigned long long *violations, unsigned long long *first_site, int reset)
{
    if (violations != nullptr) *violations = 0;
    if (first_site != nullptr) *first_site = 0;
    unsigned long long *c = bounds_counter();
    if (c == nullptr) return 0;
    unsigned long long h[2] = {0, 0};
    if (cudaDeviceSynchronize() != cudaSuccess || cudaMemcpy(h, c, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (violations != nullptr) *violations = h[0];
    if (first_site != nullptr) *first_site = h[1];
    if (reset && (cudaMemset(c, 0, sizeof(h)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)) {
        cudaGetLastError();
        return -1;
    }
    return 1;
}

RLSCAN_API size_t rlscan_workspace_bytes(int64_t N, int64_t T)
{
    if (N <= 0 || T <= 0 || T <= kSmallestTile) return 0;
    const int64_t tiles = N * ((T + kMinTile - 1) / kMinTile);
    return kHeaderBytes + kStateBytes * kMaxScans * static_cast<size_t>(tiles);
}

RLSCAN_API size_t rlscan_gae_normalized_workspace_bytes(int64_t N, int64_t T)
{
    if (N <= 0 || T <= 0) return 0;
    size_t scan = rlscan_workspace_bytes(N, T);
    if (scan < kHeaderBytes) scan = kHeaderBytes;
    return (scan + 255) / 256 * 256 + kMomentBytes;
}

RLSCAN_API rlscan_status rlscan_workspace_init(void *ws, size_t ws_bytes, rlscan_stream_t stream)
{
    if (ws == nullptr) return RLSCAN_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(ws) & 15u) != 0 || ws_bytes % 4 != 0 || residency(ws) != Residency::Device)
        return RLSCAN_ERR_WORKSPACE;
    const size_t words = ws_bytes / 4;
    if (words == 0) return RLSCAN_OK;
    size_t blocks = (words + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    zero_words<<<static_cast<unsigned>(blocks), 256, 0, cs(stream)>>>(static_cast<uint32_t *>(ws), words);
    return cudaGetLastError() == cudaSuccess ? RLSCAN_OK : RLSCAN_ERR_CUDA;
}

RLSCAN_API rlscan_status rlscan_workspace_status(void *ws, size_t ws_bytes, rlscan_stream_t stream)
{
    if (cudaStreamSynchronize(cs(stream)) != cudaSuccess) return RLSCAN_ERR_CUDA;
    if (ws == nullptr || ws_bytes < kHeaderBytes) return RLSCAN_OK;
    uint32_t *hdr = static_cast<uint32_t *>(ws);
    uint32_t code = 0;
    if (cudaMemcpy(&code, hdr + kHdrError, sizeof(code), cudaMemcpyDeviceToHost) != cudaSuccess)
        return RLSCAN_ERR_CUDA;
    if (code != 0) {
        const uint32_t zero[2] = {0u, 0u};
        if (cudaMemcpy(hdr + kHdrError, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return RLSCAN_ERR_CUDA;
    }
    return static_cast<rlscan_status>(code);
}

RLSCAN_API rlscan_status rlscan_gae(const float *rewards, const float *values, const float *terminateds,
                         const float *truncateds, const float *bootstrap_values,
                         const float *last_value, int64_t N, int64_t T, int64_t row_stride,
                         float gamma, float lambda, float *advantages,
                         void *ws, size_t ws_bytes, rlscan_stream_t stream)
{
    RLSCAN_TRY(check_shape(N, T, row_stride));
    if (N == 0 || T == 0) return RLSCAN_OK;
    if (!rewards || !values || !terminateds || !advantages) return RLSCAN_ERR_NULL;
    if (bootstrap_values && last_value) return RLSCAN_ERR_ARG_CONFLICT;
    if (last_value && truncateds) return RLSCAN_ERR_ARG_CONFLICT;
    if (same_as_any(advantages, {rewards, values, terminateds, truncateds, bootstrap_values, last_value}))
        return RLSCAN_ERR_ARG_CONFLICT;
    RLSCAN_TRY(run_checks(terminateds, truncateds, bootstrap_values, N, T, row_stride, cs(stream)));
    Params p = base_params(N, T, row_stride);
    p.c0 = gamma;
    p.c1 = lambda;
    p.out[0] = advantages;
    p.in[0] = rewards;
    p.in[1] = values;
    p.in[2] = terminateds;
    if (truncateds) {
        p.in[3] = truncateds;
        p.in[4] = bootstrap_values;
        return launch_gae(true, bootstrap_values != nullptr, p, ws, ws_bytes, cs(stream));
    }
    if (last_value) {
        p.rowscalar = last_value;
    } else if (bootstrap_values) {  // window bootstrap column only
        p.rowscalar = bootstrap_values + (T - 1);
        p.rowscalar_stride = row_stride;
    }
    return launch_gae(false, false, p, ws, ws_bytes, cs(stream));
}

RLSCAN_API rlscan_status rlscan_gae_masked(const float *rewards, const float *values,
                                           const float *terminateds, const float *truncateds,
                                           const float *bootstrap_values, const float *last_value,
                                           const float *mask, int64_t N, int64_t T, int64_t row_stride,
                                           float gamma, float lambda, float *advantages, void *ws,
                                           size_t ws_bytes, rlscan_stream_t stream)
{
    RLSCAN_TRY(check_shape(N, T, row_stride));
    if (N == 0 || T == 0) return RLSCAN_OK;
    if (!rewards || !values || !terminateds || !mask || !advantages) return RLSCAN_ERR_NULL;
    if (bootstrap_values && last_value) return RLSCAN_ERR_ARG_CONFLICT;
    if (last_value && truncateds) return RLSCAN_ERR_ARG_CONFLICT;
    if (same_as_any(advantages, {rewards, values, terminateds, truncateds, bootstrap_values, last_value, mask}))
        return RLSCAN_ERR_ARG_CONFLICT;
    RLSCAN_TRY(run_checks(terminateds, truncateds, bootstrap_values, N, T, row_stride, cs(stream)));
    Params p = base_params(N, T, row_stride);
    p.c0 = gamma;
    p.c1 = lambda;
    p.out[0] = advantages;
    p.in[0] = rewards;
    p.in[1] = values;
    p.in[2] = terminateds;
    if (truncateds) {
        p.in[3] = truncateds;
        if (bootstrap_values) {
            p.in[4] = bootstrap_values;
            p.in[5] = mask;
        } else {
            p.in[4] = mask;
        }
        return launch_gae_masked(true, bootstrap_values != nullptr, p, ws, ws_bytes, cs(stream));
    }
    p.in[3] = mask;
    if (last_value) {
        p.rowscalar = last_value;
    } else if (bootstrap_values) {
        p.rowscalar = bootstrap_values + (T - 1);
        p.rowscalar_stride = row_stride;
    }
    return launch_gae_masked(false, false, p, ws, ws_bytes, cs(stream));
}

RLSCAN_API rlscan_status rlscan_gae_returns(const float *rewards, const float *values,
                                            const float *terminateds, const float *truncateds,
                                            const float *bootstrap_values, const float *last_value,
                                            int64_t N, int64_t T, int64_t row_stride, float gamma,
                                            float lambda, float *advantages, float *lambda_returns,
                                            float *discounted_returns, void *ws, size_t ws_bytes,
                                            rlscan_stream_t stream)
{
    RLSCAN_TRY(check_shape(N, T, row_stride));
    if (N == 0 || T == 0) return RLSCAN_OK;
    if (!rewards || !values || !terminateds) return RLSCAN_ERR_NULL;
    if (!advantages && !lambda_returns && !discounted_returns) return RLSCAN_ERR_NULL;
    if (bootstrap_values && last_value) return RLSCAN_ERR_ARG_CONFLICT;
    if (last_value && truncateds) return RLSCAN_ERR_ARG_CONFLICT;
    for (const float *o : {static_cast<const float *>(advantages), static_cast<const float *>(lambda_returns),
                           static_cast<const float *>(discounted_returns)}) {
        if (o == nullptr) continue;
        if (same_as_any(o, {rewards, values, terminateds, truncateds, bootstrap_values, last_value}))
            return RLSCAN_ERR_ARG_CONFLICT;
    }
    if ((advantages && (advantages == lambda_returns || advantages == discounted_returns)) ||
        (lambda_returns && lambda_returns == discounted_returns))
        return RLSCAN_ERR_ARG_CONFLICT;
    RLSCAN_TRY(run_checks(terminateds, truncateds, bootstrap_values, N, T, row_stride, cs(stream)));
    Params p = base_params(N, T, row_stride);
    p.c0 = gamma;
    p.c1 = lambda;
    p.out[0] = advantages;
    p.out[1] = lambda_returns;
    p.out[2] = discounted_returns;
    p.in[0] = rewards;
    p.in[1] = values;
    p.in[2] = terminateds;
    if (truncateds) {
        p.in[3] = truncateds;
        p.in[4] = bootstrap_values;
        return launch_gae_returns(true, bootstrap_values != nullptr, p, ws, ws_bytes, cs(stream));
    }
    if (last_value) {
        p.rowscalar = last_value;
    } else if (bootstrap_values) {
        p.rowscalar = bootstrap_values + (T - 1);
        p.rowscalar_stride = row_stride;
    }
    return launch_gae_returns(false, false, p, ws, ws_bytes, cs(stream));
}

RLSCAN_API rlscan_status rlscan_gae_normalized(const float *rewards, const float *values,
                                               const float *terminateds, const float *truncateds,
                                               const float *bootstrap_values, const float *last_value,
                                               int64_t N, int64_t T, int64_t row_stride, float gamma,
                                               float lambda, float eps, float *advantages,
                                               float *lambda_returns, float *discounted_returns,
                                               float *moments, void *ws, size_t ws_bytes,
                                               rlscan_stream_t stream)
{
    RLSCAN_TRY(check_shape(N, T, row_stride));
    if (N == 0 || T == 0) return RLSCAN_OK;
    if (!rewards || !values || !terminateds || !advantages) return RLSCAN_ERR_NULL;
    if (!(eps >= 0.f)) return RLSCAN_ERR_ARG_VALUE;
    if (bootstrap_values && last_value) return RLSCAN_ERR_ARG_CONFLICT;
    if (last_value && truncateds) return RLSCAN_ERR_ARG_CONFLICT;
    for (const float *o : {static_cast<const float *>(advantages), static_cast<const float *>(lambda_returns),
                           static_cast<const float *>(discounted_returns), static_cast<const float *>(moments)}) {
        if (o == nullptr) continue;
        if (same_as_any(o, {rewards, values, terminateds, truncateds, bootstrap_values, last_value}))
            return RLSCAN_ERR_ARG_CONFLICT;
    }
    if (advantages == lambda_returns || advantages == discounted_returns || advantages == moments ||
        (lambda_returns && (lambda_returns == discounted_returns || lambda_returns == moments)) ||
        (discounted_returns && discounted_returns == moments))
        return RLSCAN_ERR_ARG_CONFLICT;
    const size_t need = rlscan_gae_normalized_workspace_bytes(N, T);
    if (ws == nullptr || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 15u) != 0 ||
        residency(ws) != Residency::Device)
        return RLSCAN_ERR_WORKSPACE;
    if (moments != nullptr && residency(moments) == Residency::Unreachable) return RLSCAN_ERR_MEMORY;
    RLSCAN_TRY(run_checks(terminateds, truncateds, bootstrap_values, N, T, row_stride, cs(stream)));
    Params p = base_params(N, T, row_stride);
    p.c0 = gamma;
    p.c1 = lambda;
    p.out[0] = advantages;
    p.out[1] = lambda_returns;
    p.out[2] = discounted_returns;
    p.in[0] = rewards;
    p.in[1] = values;
    p.in[2] = terminateds;
    p.c2 = eps;
    p.mom_part = reinterpret_cast<float *>(static_cast<char *>(ws) + (need - kMomentBytes));
    {
        // 1 / n and 1 / (n - 1) as float pairs (NaN for n = 1)
        const double n = static_cast<double>(N) * static_cast<double>(T);
        const double inv[2] = {1.0 / n, n > 1.0 ? 1.0 / (n - 1.0) : __builtin_nan("")};
        for (int i = 0; i < 2; ++i) {
            p.mom_inv[2 * i] = static_cast<float>(inv[i]);
            p.mom_inv[2 * i + 1] = static_cast<float>(inv[i] - static_cast<double>(p.mom_inv[2 * i]));
        }
    }
    const bool disc = discounted_returns != nullptr;
    if (truncateds) {
        p.in[3] = truncateds;
        p.in[4] = bootstrap_values;
        return launch_gae_normalized(true, bootstrap_values != nullptr, disc, p, moments, ws, ws_bytes, cs(stream));
    } else {
        if (last_value) {
            p.rowscalar = last_value;
        } else if (bootstrap_values) {
            p.rowscalar = bootstrap_values + (T - 1);
            p.rowscalar_stride = row_stride;
        }
        return launch_gae_normalized(false, false, disc, p, moments, ws, ws_bytes, cs(stream));
    }
}

namespace {
// Shared checks and parameter block of the compact-storage GAE entry points.
rlscan_status compact_params(const void *rewards, const void *values, const void *terminateds,
                             const void *truncateds, const void *bootstrap_values, const float *last_value,
                             int64_t N, int64_t T, int64_t row_stride, float gamma, float lambda,
                             rlscan_dtype out_dtype, std::initializer_list<const void *> outs, Params &p)
{
    RLSCAN_TRY(check_shape(N, T, row_stride));
    if (out_dtype != RLSCAN_F32 && out_dtype != RLSCAN_BF16) return RLSCAN_ERR_ARG_VALUE;
    if (N == 0 || T == 0) return RLSCAN_OK;
    if (!rewards || !values || !terminateds) return RLSCAN_ERR_NULL;
    if (bootstrap_values && last_value) return RLSCAN_ERR_ARG_CONFLICT;
    if (last_value && truncateds) return RLSCAN_ERR_ARG_CONFLICT;
    if (bootstrap_values && !truncateds) return RLSCAN_ERR_ARG_CONFLICT;  // window bootstrap: last_value
    const void *o_prev = nullptr;
    for (const void *o : outs) {
        if (o == nullptr) continue;
        if (same_as_any(o, {rewards, values, terminateds, truncateds, bootstrap_values, last_value}) || o == o_prev)
            return RLSCAN_ERR_ARG_CONFLICT;
        o_prev = o;
    }
    p = base_params(N, T, row_stride);
    p.c0 = gamma;
    p.c1 = lambda;
    p.in[0] = static_cast<const float *>(rewards);
    p.in[1] = static_cast<const float *>(values);
    p.in[2] = static_cast<const float *>(terminateds);
    if (truncateds) {
        p.in[3] = static_cast<const float *>(truncateds);
        p.in[4] = static_cast<const float *>(bootstrap_values);
    } else {
        p.rowscalar = last_value;
    }
    return RLSCAN_OK;
}
}  // namespace

RLSCAN_API rlscan_status rlscan_gae_compact(const void *rewards, const void *values, const void *terminateds,
                                            const void *truncateds, const void *bootstrap_values,
                                            const float *last_value, int64_t N, int64_t T, int64_t row_stride,
                                            float gamma, float lambda, rlscan_dtype out_dtype, void *advantages,
                                            void *ws, size_t ws_bytes, rlscan_stream_t stream)
{
    if (N > 0 && T > 0 && advantages == nullptr) return RLSCAN_ERR_NULL;
    Params p;
    RLSCAN_TRY(compact_params(rewards, values, terminateds, truncateds, bootstrap_values, last_value, N, T,
                              row_stride, gamma, lambda, out_dtype, {advantages}, p));
    if (N == 0 || T == 0) return RLSCAN_OK;
    p.out[0] = static_cast<float *>(advantages);
    return launch_gae_compact(truncateds != nullptr, bootstrap_values != nullptr, out_dtype == RLSCAN_BF16, p,
                              ws, ws_bytes, cs(stream));
}

RLSCAN_API rlscan_status rlscan_gae_returns_compact(const void *rewards, const void *values,
                                                    const void *terminateds, const void *truncateds,
                                                    const void *bootstrap_values, const float *last_value,
                                                    int64_t N, int64_t T, int64_t row_stride, float gamma,
                                                    float lambda, rlscan_dtype out_dtype, void *advantages,
                                                    void *lambda_returns, void *discounted_returns, void *ws,
                                                    size_t ws_bytes, rlscan_stream_t stream)
{
    if (N > 0 && T > 0 && !advantages && !lambda_returns && !discounted_returns) return RLSCAN_ERR_NULL;
    if ((advantages && (advantages == lambda_returns || advantages == discounted_returns)) ||
        (lambda_returns && lambda_returns == discounted_returns))
        return RLSCAN_ERR_ARG_CONFLICT;
    Params p;
    RLSCAN_TRY(compact_params(rewards, values, terminateds, truncateds, bootstrap_values, last_value, N, T,
                              row_stride, gamma, lambda, out_dtype, {advantages, lambda_returns, discounted_returns},
                              p));
    if (N == 0 || T == 0) return RLSCAN_OK;
    p.out[0] = static_cast<float *>(advantages);
    p.out[1] = static_cast<float *>(lambda_returns);
    p.out[2] = static_cast<float *>(discounted_returns);
    return launch_gae_returns_compact(truncateds != nullptr, bootstrap_values != nullptr, out_dtype == RLSCAN_BF16,
                                      p, ws, ws_bytes, cs(stream));
}

RLSCAN_API rlscan_status rlscan_vtrace_compact(const void *log_pi_target, const void *log_pi_behavior,
                                               const void *values, const void *rewards, const void *terminateds,
                                               const void *truncateds, const void *bootstrap_values,
                                               const float *last_value, int64_t N, int64_t T, int64_t row_stride,
                                               float gamma, float rho_bar, float c_bar, rlscan_dtype out_dtype,
                                               void *vtrace_targets, void *vtrace_advantages, void *ws,
                                               size_t ws_bytes, rlscan_stream_t stream)
{
    RLSCAN_TRY(check_shape(N, T, row_stride));
    if (out_dtype != RLSCAN_F32 && out_dtype != RLSCAN_BF16) return RLSCAN_ERR_ARG_VALUE;
    if (N == 0 || T == 0) return RLSCAN_OK;
    if (!log_pi_target || !log_pi_behavior || !values || !rewards || !terminateds || !vtrace_targets ||
        !vtrace_advantages)
        return RLSCAN_ERR_NULL;
    if (bootstrap_values && last_value) return RLSCAN_ERR_ARG_CONFLICT;
    if (bootstrap_values && !truncateds) return RLSCAN_ERR_ARG_CONFLICT;  // window bootstrap: last_value
    for (const void *o : {vtrace_targets, vtrace_advantages})
        if (same_as_any(o, {log_pi_target, log_pi_behavior, values, rewards, terminateds, truncateds,
                            bootstrap_values, last_value}))
            return RLSCAN_ERR_ARG_CONFLICT;
    if (vtrace_targets == vtrace_advantages) return RLSCAN_ERR_ARG_CONFLICT;
    Params p = base_params(N, T, row_stride);
    p.c0 = gamma;
    p.c1 = rho_bar;
    p.c2 = c_bar;
    p.out[0] = static_cast<float *>(vtrace_targets);
    p.out[1] = static_cast<float *>(vtrace_advantages);
    p.in[0] = static_cast<const float *>(log_pi_target);
    p.in[1] = static_cast<const float *>(log_pi_behavior);
    p.in[2] = static_cast<const float *>(values);
    p.in[3] = static_cast<const float *>(rewards);
    p.in[4] = static_cast<const float *>(terminateds);
    p.rowscalar = last_value;
    if (truncateds) {
        p.in[5] = static_cast<const float *>(truncateds);
        p.in[6] = static_cast<const float *>(bootstrap_values);
    }
    return launch_vtrace_compact(truncateds != nullptr, bootstrap_values != nullptr, out_dtype == RLSCAN_BF16, p, ws,
                                 ws_bytes, cs(stream));
}

RLSCAN_API rlscan_status rlscan_retrace_compact(const void *pi_taken, const void *mu_taken, const void *q_values,
                                                const void *expected_next_q, const void *rewards,
                                                const void *terminateds, const void *truncateds, int64_t N,
                                                int64_t T, int64_t row_stride, float gamma, float lambda,
                                                float c_bar, float rho_bar, rlscan_dtype out_dtype,
                                                void *retrace_targets, void *advantages, void *ws, size_t ws_bytes,
                                                rlscan_stream_t stream)
{
    RLSCAN_TRY(check_shape(N, T, row_stride));
    if (out_dtype != RLSCAN_F32 && out_dtype != RLSCAN_BF16) return RLSCAN_ERR_ARG_VALUE;
    if (N == 0 || T == 0) return RLSCAN_OK;
    if (!pi_taken || !mu_taken || !q_values || !expected_next_q || !rewards || !terminateds || !retrace_targets ||
        !advantages)
        return RLSCAN_ERR_NULL;
    for (const void *o : {retrace_targets, advantages})
        if (same_as_any(o, {pi_taken, mu_taken, q_values, expected_next_q, rewards, terminateds, truncateds}))
            return RLSCAN_ERR_ARG_CONFLICT;
    if (retrace_targets == advantages) return RLSCAN_ERR_ARG_CONFLICT;
    Params p = base_params(N, T, row_stride);
    p.c0 = gamma;
    p.c1 = lambda;
    p.c2 = c_bar;
    p.c3 = rho_bar;
    p.out[0] = static_cast<float *>(retrace_targets);
    p.out[1] = static_cast<float *>(advantages);
    p.in[0] = static_cast<const float *>(pi_taken);
    p.in[1] = static_cast<const float *>(mu_taken);
    p.in[2] = static_cast<const float *>(q_values);
    p.in[3] = static_cast<const float *>(expected_next_q);
    p.in[4] = static_cast<const float *>(rewards);
    p.in[5] = static_cast<const float *>(terminateds);
    p.in[6] = static_cast<const float *>(truncateds);
    return launch_retrace_compact(truncateds != nullptr, out_dtype == RLSCAN_BF16, p, ws, ws_bytes, cs(stream));
}

RLSCAN_API rlscan_status rlscan_vtrace(const float *log_pi_target, const float *log_pi_behavior,
                            const float *values, const float *rewards, const float *terminateds,
                            const float *truncateds, const float *bootstrap_values,
                            const float *last_value, int64_t N, int64_t T, int64_t row_stride,
                            float gamma, float rho_bar, float c_bar,
                            float *vtrace_targets, float *vtrace_advantages,
                            void *ws, size_t ws_bytes, rlscan_stream_t stream)
{
    RLSCAN_TRY(check_shape(N, T, row_stride));
    if (N == 0 || T == 0) return RLSCAN_OK;
    if (!log_pi_target || !log_pi_behavior || !values || !rewards || !terminateds || !vtrace_targets ||
        !vtrace_advantages)
        return RLSCAN_ERR_NULL;
    if (bootstrap_values && last_value) return RLSCAN_ERR_ARG_CONFLICT;
    for (const float *o : {static_cast<const float *>(vtrace_targets), static_cast<const float *>(vtrace_advantages)})
        if (same_as_any(o, {log_pi_target, log_pi_behavior, values, rewards, terminateds, truncateds,
                            bootstrap_values, last_value}))
            return RLSCAN_ERR_ARG_CONFLICT;
    if (vtrace_targets == vtrace_advantages) return RLSCAN_ERR_ARG_CONFLICT;
    RLSCAN_TRY(run_checks(terminateds, truncateds, bootstrap_values, N, T, row_stride, cs(stream)));
    Params p = base_params(N, T, row_stride);
    p.c0 = gamma;
    p.c1 = rho_bar;
    p.c2 = c_bar;
    p.out[0] = vtrace_targets;
    p.out[1] = vtrace_advantages;
    p.in[0] = log_pi_target;
    p.in[1] = log_pi_behavior;
    p.in[2] = values;
    p.in[3] = rewards;
    p.in[4] = terminateds;
    if (truncateds) {
        p.in[5] = truncateds;
        p.in[6] = bootstrap_values;
        p.rowscalar = last_value;  // last_value with truncations: bs_{T-1} only
        return launch_vtrace(true, bootstrap_values != nullptr, p, ws, ws_bytes, cs(stream));
    }
    if (last_value) {
        p.rowscalar = last_value;
    } else if (bootstrap_values) {
        p.rowscalar = bootstrap_values + (T - 1);
        p.rowscalar_stride = row_stride;
    }
    return launch_vtrace(false, false, p, ws, ws_bytes, cs(stream));
}

RLSCAN_API rlscan_status rlscan_retrace(const float *pi_taken, const float *mu_taken, const float *q_values,
                             const float *expected_next_q, const float *rewards,
                             const float *terminateds, const float *truncateds,
                             int64_t N, int64_t T, int64_t row_stride,
                             float gamma, float lambda, float c_bar, float rho_bar,
                             float *retrace_targets, float *advantages,
                             void *ws, size_t ws_bytes, rlscan_stream_t stream)
{
    RLSCAN_TRY(check_shape(N, T, row_stride));
    if (N == 0 || T == 0) return RLSCAN_OK;
    if (!pi_taken || !mu_taken || !q_values || !expected_next_q || !rewards || !terminateds ||
        !retrace_targets || !advantages)
        return RLSCAN_ERR_NULL;
    for (const float *o : {static_cast<const float *>(retrace_targets), static_cast<const float *>(advantages)})
        if (same_as_any(o, {pi_taken, mu_taken, q_values, expected_next_q, rewards, terminateds, truncateds}))
            return RLSCAN_ERR_ARG_CONFLICT;
    if (retrace_targets == advantages) return RLSCAN_ERR_ARG_CONFLICT;
    RLSCAN_TRY(run_checks(terminateds, truncateds, nullptr, N, T, row_stride, cs(stream)));
    Params p = base_params(N, T, row_stride);
    p.c0 = gamma;
    p.c1 = lambda;
    p.c2 = c_bar;
    p.c3 = rho_bar;
    p.out[0] = retrace_targets;
    p.out[1] = advantages;
    p.in[0] = pi_taken;
    p.in[1] = mu_taken;
    p.in[2] = q_values;
    p.in[3] = expected_next_q;
    p.in[4] = rewards;
    p.in[5] = terminateds;
    p.in[6] = truncateds;
    return launch_retrace(truncateds != nullptr, p, ws, ws_bytes, cs(stream));
}

RLSCAN_API rlscan_status rlscan_retrace_actions(const float *action_probs_target,
                                                const float *action_probs_behavior,
                                                const float *q_values, const float *next_q_values_all,
                                                const int64_t *actions, const float *rewards,
                                                const float *terminateds, const float *truncateds,
                                                int64_t N, int64_t T, int64_t A, int64_t row_stride,
                                                int64_t action_row_stride, float gamma, float lambda,
                                                float c_bar, float rho_bar, float *retrace_targets,
                                                float *advantages, void *ws, size_t ws_bytes,
                                                rlscan_stream_t stream)
{
    if (A < 1 || A > 65536) return RLSCAN_ERR_ARG_VALUE;
    RLSCAN_TRY(check_shape(N, T, row_stride));
    if (action_row_stride < T * A) return RLSCAN_ERR_SHAPE;
    if (N == 0 || T == 0) return RLSCAN_OK;
    if (!action_probs_target || !action_probs_behavior || !q_values || !next_q_values_all || !actions ||
        !rewards || !terminateds || !retrace_targets || !advantages)
        return RLSCAN_ERR_NULL;
    for (const float *o : {static_cast<const float *>(retrace_targets), static_cast<const float *>(advantages)})
        if (same_as_any(o, {action_probs_target, action_probs_behavior, q_values, next_q_values_all,
                            actions, rewards, terminateds, truncateds}))
            return RLSCAN_ERR_ARG_CONFLICT;
    if (retrace_targets == advantages) return RLSCAN_ERR_ARG_CONFLICT;
    RLSCAN_TRY(run_checks(terminateds, truncateds, nullptr, N, T, row_stride, cs(stream)));
    RLSCAN_TRY(run_action_checks(actions, N, T, row_stride, A, cs(stream)));
    Params p = base_params(N, T, row_stride);
    p.c0 = gamma;
    p.c1 = lambda;
    p.c2 = c_bar;
    p.c3 = rho_bar;
    p.out[0] = retrace_targets;
    p.out[1] = advantages;
    p.in[1] = action_probs_behavior;
    p.in[2] = q_values;
    p.in[4] = rewards;
    p.in[5] = terminateds;
    p.in[6] = truncateds;
    p.A = static_cast<int32_t>(A);
    p.wide[0] = action_probs_target;
    p.wide[1] = next_q_values_all;
    p.wide[2] = actions;
    p.wide_rs[0] = action_row_stride;
    p.wide_rs[1] = action_row_stride;
    p.wide_rs[2] = 2 * row_stride;
    return launch_retrace_actions(truncateds != nullptr, p, ws, ws_bytes, cs(stream));
}

RLSCAN_API rlscan_status rlscan_lambda_returns(const float *rewards, const float *next_values,
                                    const float *terminateds, const float *truncateds,
                                    const float *bootstrap_values, const float *last_value,
                                    int64_t N, int64_t T, int64_t row_stride,
                                    float gamma, float lambda, float *returns,
                                    void *ws, size_t ws_bytes, rlscan_stream_t stream)
{
    RLSCAN_TRY(check_shape(N, T, row_stride));
    if (N == 0 || T == 0) return RLSCAN_OK;
    if (!rewards || !next_values || !terminateds || !returns) return RLSCAN_ERR_NULL;
    if (bootstrap_values && last_value) return RLSCAN_ERR_ARG_CONFLICT;
    if (same_as_any(returns, {rewards, next_values, terminateds, truncateds, bootstrap_values, last_value}))
        return RLSCAN_ERR_ARG_CONFLICT;
    RLSCAN_TRY(run_checks(terminateds, truncateds, nullptr, N, T, row_stride, cs(stream)));
    Params p = base_params(N, T, row_stride);
    p.c0 = gamma;
    p.c1 = lambda;
    p.out[0] = returns;
    p.in[0] = rewards;
    p.in[1] = next_values;
    p.in[2] = terminateds;
    if (truncateds) {
        p.in[3] = truncateds;
        p.in[4] = bootstrap_values;
        p.rowscalar = last_value;
        return launch_lambda_returns(true, bootstrap_values != nullptr, p, ws, ws_bytes, cs(stream));
    }
    if (last_value) {
        p.rowscalar = last_value;
    } else if (bootstrap_values) {
        p.rowscalar = bootstrap_values + (T - 1);
        p.rowscalar_stride = row_stride;
    }
    return launch_lambda_returns(false, false, p, ws, ws_bytes, cs(stream));
}

RLSCAN_API rlscan_status rlscan_discounted_returns(const float *rewards, const float *terminateds,
                                        const float *truncateds, const float *bootstrap_values,
                                        const float *last_value, int64_t N, int64_t T,
                                        int64_t row_stride, float gamma, float *returns,
                                        void *ws, size_t ws_bytes, rlscan_stream_t stream)
{
    RLSCAN_TRY(check_shape(N, T, row_stride));
    if (N == 0 || T == 0) return RLSCAN_OK;
    if (!rewards || !terminateds || !returns) return RLSCAN_ERR_NULL;
    if (bootstrap_values && last_value) return RLSCAN_ERR_ARG_CONFLICT;
    if (same_as_any(returns, {rewards, terminateds, truncateds, bootstrap_values, last_value}))
        return RLSCAN_ERR_ARG_CONFLICT;
    RLSCAN_TRY(run_checks(terminateds, truncateds, nullptr, N, T, row_stride, cs(stream)));
    Params p = base_params(N, T, row_stride);
    p.c0 = gamma;
    p.out[0] = returns;
    p.in[0] = rewards;
    p.in[1] = terminateds;
    if (truncateds) {
        p.in[2] = truncateds;
        p.in[3] = bootstrap_values;
        p.rowscalar = last_value;
        return launch_discounted(true, bootstrap_values != nullptr, p, ws, ws_bytes, cs(stream));
    }
    if (last_value) {
        p.rowscalar = last_value;
    } else if (bootstrap_values) {
        p.rowscalar = bootstrap_values + (T - 1);
        p.rowscalar_stride = row_stride;
    }
    return launch_discounted(false, false, p, ws, ws_bytes, cs(stream));
}

RLSCAN_API rlscan_status rlscan_eligibility_traces(const float *gradients, const float *dones,
                                        const float *seed_values, int64_t N, int64_t T,
                                        int64_t row_stride, float gamma, float lambda,
                                        float *traces, void *ws, size_t ws_bytes,
                                        rlscan_stream_t stream)
{
    RLSCAN_TRY(check_shape(N, T, row_stride));
    if (N == 0 || T == 0) return RLSCAN_OK;
    if (!gradients || !dones || !traces) return RLSCAN_ERR_NULL;
    if (same_as_any(traces, {gradients, dones, seed_values})) return RLSCAN_ERR_ARG_CONFLICT;
    Params p = base_params(N, T, row_stride);
    p.c0 = gamma;
    p.c1 = lambda;
    p.out[0] = traces;
    p.in[0] = gradients;
    p.in[1] = dones;
    p.rowscalar = seed_values;
    return launch_eligibility(p, ws, ws_bytes, cs(stream));
}

RLSCAN_API rlscan_status rlscan_episodic_prefix_sum(const float *inputs, const float *dones,
                                         const float *seed_values, rlscan_boundary boundary,
                                         int64_t N, int64_t T, int64_t row_stride,
                                         float *prefix_sums, void *ws, size_t ws_bytes,
                                         rlscan_stream_t stream)
{
    if (boundary != RLSCAN_ENDS_AT && boundary != RLSCAN_STARTS_AT) return RLSCAN_ERR_ARG_VALUE;
    RLSCAN_TRY(check_shape(N, T, row_stride));
    if (N == 0 || T == 0) return RLSCAN_OK;
    if (!inputs || !dones || !prefix_sums) return RLSCAN_ERR_NULL;
    if (same_as_any(prefix_sums, {inputs, dones, seed_values})) return RLSCAN_ERR_ARG_CONFLICT;
    Params p = base_params(N, T, row_stride);
    p.out[0] = prefix_sums;
    p.in[0] = inputs;
    p.in[1] = dones;
    p.rowscalar = seed_values;
    return launch_prefix(boundary == RLSCAN_STARTS_AT, p, ws, ws_bytes, cs(stream));
}

RLSCAN_API rlscan_status rlscan_linear_scan(const float *alpha, const float *beta, const float *carry,
                                 rlscan_direction direction, int64_t N, int64_t T,
                                 int64_t row_stride, float *out, void *ws, size_t ws_bytes,
                                 rlscan_stream_t stream)
{
    if (direction != RLSCAN_BACKWARD && direction != RLSCAN_FORWARD) return RLSCAN_ERR_ARG_VALUE;
    RLSCAN_TRY(check_shape(N, T, row_stride));
    if (N == 0 || T == 0) return RLSCAN_OK;
    if (!alpha || !beta || !out) return RLSCAN_ERR_NULL;
    if (same_as_any(out, {alpha, beta, carry})) return RLSCAN_ERR_ARG_CONFLICT;
    Params p = base_params(N, T, row_stride);
    p.out[0] = out;
    p.in[0] = alpha;
    p.in[1] = beta;
    p.rowscalar = carry;
    return launch_linear(direction == RLSCAN_FORWARD, p, ws, ws_bytes, cs(stream));
}

}  // extern "C"
