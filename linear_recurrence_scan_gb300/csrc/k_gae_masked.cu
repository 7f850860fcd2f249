// k_gae_masked.cu -- GAE with observation-skip masking.
#include "launch.cuh"

namespace rlscan {

rlscan_status launch_gae_masked(bool trunc, bool bs2d, Params p, void *ws, size_t ws_bytes, cudaStream_t s)
{
    if (!trunc) return launch_scan<est::GAEMasked<false, false>>(p, ws, ws_bytes, s);
    if (!bs2d) return launch_scan<est::GAEMasked<true, false>>(p, ws, ws_bytes, s);
    return launch_scan<est::GAEMasked<true, true>>(p, ws, ws_bytes, s);
}

}  // namespace rlscan
