// k_retrace.cu -- Retrace(lambda) instantiations of the scan kernel.
#include "launch.cuh"

namespace rlscan {

rlscan_status launch_retrace(bool trunc, Params p, void *ws, size_t ws_bytes, cudaStream_t s)
{
    if (!trunc) return launch_scan<est::Retrace<false>>(p, ws, ws_bytes, s);
    return launch_scan<est::Retrace<true>>(p, ws, ws_bytes, s);
}

}  // namespace rlscan
