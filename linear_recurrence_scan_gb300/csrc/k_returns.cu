// k_returns.cu -- TD(lambda) and discounted-return instantiations of the scan kernel.
#include "launch.cuh"

namespace rlscan {

rlscan_status launch_lambda_returns(bool trunc, bool bs2d, Params p, void *ws, size_t ws_bytes,
                                    cudaStream_t s)
{
    if (!trunc) return launch_scan<est::LambdaReturns<false, false>>(p, ws, ws_bytes, s);
    if (!bs2d) return launch_scan<est::LambdaReturns<true, false>>(p, ws, ws_bytes, s);
    return launch_scan<est::LambdaReturns<true, true>>(p, ws, ws_bytes, s);
}

rlscan_status launch_discounted(bool trunc, bool bs2d, Params p, void *ws, size_t ws_bytes,
                                cudaStream_t s)
{
    if (!trunc) return launch_scan<est::Discounted<false, false>>(p, ws, ws_bytes, s);
    if (!bs2d) return launch_scan<est::Discounted<true, false>>(p, ws, ws_bytes, s);
    return launch_scan<est::Discounted<true, true>>(p, ws, ws_bytes, s);
}

}  // namespace rlscan
