// dfloat.cuh -- sums carried as unevaluated pairs of floats (hi + lo), for
// reductions whose partial sums need more than float precision.  GB300's
// double-precision rate is a small fraction of its float rate, so the
// batch-moment reductions add in float pairs instead: Knuth's TwoSum gives
// the exact rounding error of a float addition, and the pair sum keeps it
// (Dekker's double-length addition, about 48 significant bits).  Only
// additions and subtractions appear, so no multiply-add contraction can
// change the error terms.
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

__device__ __forceinline__ double df_value(DF v) { return static_cast<double>(v.hi) + static_cast<double>(v.lo); }

}  // namespace rlscan
