// k_forward.cu -- eligibility traces, episodic prefix sums and the generic
// affine scan.
#include "launch.cuh"

namespace rlscan {

rlscan_status launch_eligibility(Params p, void *ws, size_t ws_bytes, cudaStream_t s)
{
    return launch_scan<est::Eligibility>(p, ws, ws_bytes, s);
}

rlscan_status launch_prefix(bool starts_at, Params p, void *ws, size_t ws_bytes, cudaStream_t s)
{
    if (starts_at) return launch_scan<est::Prefix<true>>(p, ws, ws_bytes, s);
    return launch_scan<est::Prefix<false>>(p, ws, ws_bytes, s);
}

rlscan_status launch_linear(bool forward, Params p, void *ws, size_t ws_bytes, cudaStream_t s)
{
    if (forward) return launch_scan<est::Linear<true>>(p, ws, ws_bytes, s);
    return launch_scan<est::Linear<false>>(p, ws, ws_bytes, s);
}

}  // namespace rlscan
