// k_normalize.cu -- fused GAE + returns with the batch moments of the
// advantages, and the pass that normalises the advantages with them
// (advantage normalisation, the planned extension of the rl-triton paper,
// Sec. 9.3, read as the usual per-batch whitening
// (A - mean) / (std + eps) with the unbiased standard deviation).
#include "dfloat.cuh"
#include "launch.cuh"

namespace rlscan {

rlscan_status launch_gae_moments(bool trunc, bool bs2d, Params p, void *ws, size_t ws_bytes, cudaStream_t s,
                                 int64_t *grid)
{
    if (!trunc) return launch_scan<est::GAEReturnsMoments<false, false>>(p, ws, ws_bytes, s, grid);
    if (!bs2d) return launch_scan<est::GAEReturnsMoments<true, false>>(p, ws, ws_bytes, s, grid);
    return launch_scan<est::GAEReturnsMoments<true, true>>(p, ws, ws_bytes, s, grid);
}

namespace {

constexpr int kNormThreads = 256;
constexpr int kVecPerThread = 8;

// x <- (x - mean) / (std + eps) over an [N, T] buffer with row stride rs.
// Every block first combines the scan kernel's per-CTA slots
// (sum and sum of squares as float pairs) in the same fixed order -- so all
// blocks agree bit for bit -- into mean = S / n and the unbiased variance
// (Q - S mean) / (n - 1) (inv_n = 1 / n and inv_nm1 = 1 / (n - 1) from the
// host; NaN for n = 1).  Contiguous buffers are walked as one flat array
// (float4 when aligned, four vectors in flight per thread), strided ones row
// by row.
__global__ void __launch_bounds__(kNormThreads) normalize_kernel(float *x, int64_t N, int64_t T, int64_t rs,
                                                                 const float *parts, int nparts, double inv_n,
                                                                 double inv_nm1, float eps, float *moments_out,
                                                                 int vec)
{
    ptx::pdl_trigger_dependents();
    ptx::pdl_wait_prerequisites();  // the scan kernel's outputs and moments are complete
    // flat buffers: this block's first vectors are requested before the
    // moments are combined, so their latency overlaps the combination
    const bool flat = rs == T && vec;
    float4 *x4 = reinterpret_cast<float4 *>(x);
    const int64_t n4 = N * T / 4;
    int64_t base = blockIdx.x * static_cast<int64_t>(kVecPerThread * kNormThreads);
    float4 v[kVecPerThread];
    auto load_chunk = [&] {
#pragma unroll
        for (int u = 0; u < kVecPerThread; ++u) {
            const int64_t i = base + u * kNormThreads + threadIdx.x;
            if (i < n4) v[u] = x4[i];
        }
    };
    if (flat) load_chunk();
    __shared__ DF s_red[kNormThreads / 32][2];
    __shared__ float s_mi[2];
    {
        DF sum, sumsq;
        combine_moment_slots<kNormThreads>(parts, nparts, threadIdx.x, s_red, [] { __syncthreads(); }, sum, sumsq);
        if (threadIdx.x == 0) {
            const Whitening w = whitening(sum, sumsq, inv_n, inv_nm1, eps);
            s_mi[0] = w.mean;
            s_mi[1] = w.inv;
            if (moments_out != nullptr && blockIdx.x == 0) {
                moments_out[0] = w.mean;
                moments_out[1] = w.sd;
            }
        }
    }
    __syncthreads();
    const float m = s_mi[0], inv = s_mi[1];
    if (flat) {
        // block b owns kVecPerThread * kNormThreads consecutive vectors per
        // step of the grid; all of a thread's loads are issued before its stores
        const int64_t step = static_cast<int64_t>(gridDim.x) * kVecPerThread * kNormThreads;
        for (bool first = true; base < n4; base += step, first = false) {
            if (!first) load_chunk();
#pragma unroll
            for (int u = 0; u < kVecPerThread; ++u) {
                const int64_t i = base + u * kNormThreads + threadIdx.x;
                if (i < n4) {
                    v[u].x = (v[u].x - m) * inv;
                    v[u].y = (v[u].y - m) * inv;
                    v[u].z = (v[u].z - m) * inv;
                    v[u].w = (v[u].w - m) * inv;
                    x4[i] = v[u];
                }
            }
        }
        return;
    }
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kNormThreads;
    const int64_t first = blockIdx.x * static_cast<int64_t>(kNormThreads) + threadIdx.x;
    if (rs == T) {
        const int64_t n = N * T;
        for (int64_t i = first; i < n; i += stride) x[i] = (x[i] - m) * inv;
        return;
    }
    for (int64_t row = blockIdx.x; row < N; row += gridDim.x) {
        float *r = x + row * rs;
        if (vec) {
            float4 *r4 = reinterpret_cast<float4 *>(r);
            for (int64_t c = threadIdx.x; c < T / 4; c += kNormThreads) {
                float4 v = r4[c];
                v.x = (v.x - m) * inv;
                v.y = (v.y - m) * inv;
                v.z = (v.z - m) * inv;
                v.w = (v.w - m) * inv;
                r4[c] = v;
            }
        } else {
            for (int64_t c = threadIdx.x; c < T; c += kNormThreads) r[c] = (r[c] - m) * inv;
        }
    }
}

}  // namespace

rlscan_status launch_normalize(float *x, int64_t N, int64_t T, int64_t rs, const float *parts, int64_t nparts,
                               float eps, float *moments_out, cudaStream_t stream)
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return RLSCAN_ERR_CUDA;
    const bool vec = (T % 4 == 0) && (rs % 4 == 0) && aligned16(x);
    int64_t blocks;
    if (rs == T && vec) {
        blocks = (N * T / 4 + kVecPerThread * kNormThreads - 1) / (kVecPerThread * kNormThreads);
    } else {
        const int64_t work = rs == T ? N * T : N * kNormThreads;
        blocks = (work + kNormThreads - 1) / kNormThreads;
    }
    const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * 8;  // one wave; each block re-reads the slots
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const double n = static_cast<double>(N) * static_cast<double>(T);
    const double inv_n = 1.0 / n;
    const double inv_nm1 = n > 1.0 ? 1.0 / (n - 1.0) : __builtin_nan("");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kNormThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, normalize_kernel, x, N, T, rs, parts, static_cast<int>(nparts), inv_n, inv_nm1, eps,
                           moments_out, vec ? 1 : 0) != cudaSuccess) {
        cudaGetLastError();
        return RLSCAN_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? RLSCAN_OK : RLSCAN_ERR_CUDA;
}

}  // namespace rlscan
