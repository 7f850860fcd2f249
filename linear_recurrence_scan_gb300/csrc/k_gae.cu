// k_gae.cu -- GAE, fused GAE + returns, and V-trace instantiations of the scan kernel.
#include "launch.cuh"

namespace rlscan {

rlscan_status launch_gae(bool trunc, bool bs2d, Params p, void *ws, size_t ws_bytes, cudaStream_t s)
{
    if (!trunc) return launch_scan<est::GAE<false, false>>(p, ws, ws_bytes, s);
    if (!bs2d) return launch_scan<est::GAE<true, false>>(p, ws, ws_bytes, s);
    return launch_scan<est::GAE<true, true>>(p, ws, ws_bytes, s);
}

rlscan_status launch_gae_returns(bool trunc, bool bs2d, Params p, void *ws, size_t ws_bytes,
                                 cudaStream_t s)
{
    if (!trunc) return launch_scan<est::GAEReturns<false, false>>(p, ws, ws_bytes, s);
    if (!bs2d) return launch_scan<est::GAEReturns<true, false>>(p, ws, ws_bytes, s);
    return launch_scan<est::GAEReturns<true, true>>(p, ws, ws_bytes, s);
}

rlscan_status launch_vtrace(bool trunc, bool bs2d, Params p, void *ws, size_t ws_bytes, cudaStream_t s)
{
    if (!trunc) return launch_scan<est::VTrace<false, false>>(p, ws, ws_bytes, s);
    if (!bs2d) return launch_scan<est::VTrace<true, false>>(p, ws, ws_bytes, s);
    return launch_scan<est::VTrace<true, true>>(p, ws, ws_bytes, s);
}

}  // namespace rlscan
