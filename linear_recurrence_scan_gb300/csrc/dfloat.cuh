// dfloat.cuh -- sums carried as unevaluated pairs of floats (hi + lo), for
// reductions whose partial sums need more than float precision.  GB300's
// double-precision rate is a small fraction of its float rate, so the
// batch-moment reductions add in float pairs instead: Knuth's TwoSum gives
// the exact rounding error of a float addition, and the pair sum keeps it
// (Dekker's double-length addition, about 48 significant bits).  Products
// take the leading product with __fmul_rn (never contracted into a
// multiply-add) and its exact rounding error from one fmaf (Dekker's
// TwoProduct), so no contraction can change the error terms either.  The
// whitening constants are derived in these pairs too: on GB300 a chain of
// double-precision operations costs microseconds.
#pragma once

namespace rlscan {

struct DF {
    float hi, lo;
};

// a + b = s + e exactly, s = fl(a + b)
__device__ __forceinline__ DF two_sum(float a, float b)
{
    const float s = a + b;
    const float bb = s - a;
    const float e = (a - (s - bb)) + (b - bb);
    return DF{s, e};
}

__device__ __forceinline__ DF df_add(DF a, DF b)
{
    const DF s = two_sum(a.hi, b.hi);
    const float e = s.lo + (a.lo + b.lo);
    const float h = s.hi + e;  // renormalise: |e| is small next to s.hi
    return DF{h, e - (h - s.hi)};
}

__device__ __forceinline__ DF df_shfl_down(DF v, int off)
{
    return DF{__shfl_down_sync(0xffffffffu, v.hi, off), __shfl_down_sync(0xffffffffu, v.lo, off)};
}

__device__ __forceinline__ DF df_neg(DF a) { return DF{-a.hi, -a.lo}; }

// a * b: the leading product, its rounding error (exact, from one fmaf) and
// the cross terms, renormalised
__device__ __forceinline__ DF df_mul(DF a, DF b)
{
    const float p = __fmul_rn(a.hi, b.hi);
    const float e = fmaf(a.hi, b.hi, -p);
    const float t = fmaf(a.hi, b.lo, fmaf(a.lo, b.hi, e));
    const float h = p + t;
    return DF{h, t - (h - p)};
}

// Whitening constants from the combined sum S and sum of squares Q of n
// values (inv_n = 1 / n and inv_nm1 = 1 / (n - 1) as float pairs, the
// latter NaN for n = 1): the mean S / n, the unbiased standard deviation
// sqrt((Q - S mean) / (n - 1)) (a negative rounding residue reads as 0) and
// 1 / (sd + eps).
struct Whitening {
    float mean, sd, inv;
};
__device__ __forceinline__ Whitening whitening(DF sum, DF sumsq, DF inv_n, DF inv_nm1, float eps)
{
    const DF mean = df_mul(sum, inv_n);
    const DF var = df_mul(df_add(sumsq, df_neg(df_mul(sum, mean))), inv_nm1);
    const float v = var.hi;
    const float sd = sqrtf(v > 0.f ? v : (v == v ? 0.f : v));
    return Whitening{mean.hi, sd, 1.f / (sd + eps)};
}

// Combine the per-CTA moment slots parts[c] = (sum hi, sum lo, sumsq hi,
// sumsq lo), c < nparts, over threads 0..NT-1 in a fixed order (thread t
// takes slots t, t + NT, ..., loading eight before adding them; then a warp
// tree; then thread 0 adds the warps in order), so every caller gets the
// same bits.  red holds NT / 32 pairs of DF; sync() is a barrier over the NT
// threads.  The result is valid in thread 0.
template <int NT, class Sync>
__device__ __forceinline__ void combine_moment_slots(const float *parts, int nparts, int tid, DF (*red)[2], Sync sync,
                                                     DF &sum, DF &sumsq)
{
    DF a{0.f, 0.f}, b{0.f, 0.f};
    constexpr int kBatch = 8;  // slot loads in flight per thread before their adds
    for (int c0 = tid; c0 < nparts; c0 += kBatch * NT) {
        float4 v[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int c = c0 + u * NT;
            v[u] = c < nparts ? __ldcg(reinterpret_cast<const float4 *>(parts + 4 * c)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            a = df_add(a, DF{v[u].x, v[u].y});
            b = df_add(b, DF{v[u].z, v[u].w});
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a = df_add(a, df_shfl_down(a, o));
        b = df_add(b, df_shfl_down(b, o));
    }
    if ((tid & 31) == 0) {
        red[tid >> 5][0] = a;
        red[tid >> 5][1] = b;
    }
    sync();
    if (tid == 0) {
        a = DF{0.f, 0.f};
        b = DF{0.f, 0.f};
        for (int w = 0; w < NT / 32; ++w) {
            a = df_add(a, red[w][0]);
            b = df_add(b, red[w][1]);
        }
        sum = a;
        sumsq = b;
    }
}

}  // namespace rlscan
