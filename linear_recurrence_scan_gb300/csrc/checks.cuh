// checks.cuh -- bounds checks of a checked build (RLSCAN_CHECK_BOUNDS=1).
//
// Every global access of the scan kernels, and every bulk copy's source and
// destination range, can be tested against the extent of the argument it
// belongs to: an [N,T] array with row stride rs spans ((N-1) rs + T)
// elements from its base.  In a checked build a failed test counts one
// violation (and keeps the first site code) in the launch's counter and the
// access is skipped; in a normal build the tests compile to nothing.
#pragma once

#include <cstdint>

#include "params.cuh"

#ifndef RLSCAN_CHECK_BOUNDS
#define RLSCAN_CHECK_BOUNDS 0
#endif

namespace rlscan {

// Site codes (the first failing one is kept).
enum BoundsSite : uint32_t {
    kSiteCopySource = 1,   // bulk copy: global source range
    kSiteCopyTarget = 2,   // bulk copy: shared destination range
    kSiteElementLoad = 3,  // element-wise staging load
    kSiteStore = 4,        // output store
    kSiteRowScalar = 5,    // per-row scalar load
    kSiteState = 6,        // look-back tile state
    kSiteWide = 7,         // wide input read from global memory
    kSiteMoments = 8,      // moments slot
    kSiteRing = 9,         // ring stage inside the dynamic shared memory
};

#if RLSCAN_CHECK_BOUNDS
__device__ __noinline__ inline void bounds_violation(const Params &p, uint32_t site)
{
    if (p.bounds == nullptr) return;
    atomicAdd(&p.bounds[0], 1ull);
    atomicCAS(&p.bounds[1], 0ull, static_cast<unsigned long long>(site));
}
#endif

// [addr, addr + len) inside [base, base + extent) (bytes)
__device__ __forceinline__ bool span_ok(const Params &p, const void *base, uint64_t extent, const void *addr,
                                        uint64_t len, uint32_t site)
{
#if RLSCAN_CHECK_BOUNDS
    const uint64_t b = reinterpret_cast<uintptr_t>(base), a = reinterpret_cast<uintptr_t>(addr);
    const bool ok = base != nullptr && a >= b && a + len <= b + extent;
    if (!ok) bounds_violation(p, site);
    return ok;
#else
    (void)p, (void)base, (void)extent, (void)addr, (void)len, (void)site;
    return true;
#endif
}

// bytes spanned by an [N,T] array of `eb`-byte elements
__device__ __forceinline__ uint64_t array_extent(const Params &p, int eb)
{
    return p.check_rows > 0 ? static_cast<uint64_t>((p.check_rows - 1) * p.rs + p.T) * static_cast<uint64_t>(eb) : 0;
}

// bytes spanned by wide array w: (N-1) wide_rs + T wide_words 4-byte words
__device__ __forceinline__ uint64_t wide_extent(const Params &p, int w)
{
    return p.check_rows > 0 ? static_cast<uint64_t>((p.check_rows - 1) * p.wide_rs[w] + p.T * p.wide_words[w]) * 4u
                            : 0;
}

// [addr, addr + len) inside this CTA's dynamic shared memory
__device__ __forceinline__ bool smem_ok(const Params &p, const void *smem_base, const void *addr, uint64_t len,
                                        uint32_t site)
{
#if RLSCAN_CHECK_BOUNDS
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    return span_ok(p, smem_base, dyn, addr, len, site);
#else
    (void)p, (void)smem_base, (void)addr, (void)len, (void)site;
    return true;
#endif
}

// state word index w (two words per tile and scan) inside the workspace
__device__ __forceinline__ bool state_ok(const Params &p, int64_t w, int K)
{
#if RLSCAN_CHECK_BOUNDS
    const bool ok = p.states != nullptr && w >= 0 && w < 2 * K * p.num_tiles;
    if (!ok) bounds_violation(p, kSiteState);
    return ok;
#else
    (void)p, (void)w, (void)K;
    return true;
#endif
}

}  // namespace rlscan
