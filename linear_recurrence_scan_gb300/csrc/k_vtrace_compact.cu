// k_vtrace_compact.cu -- V-trace on compact storage: bfloat16 log-probabilities,
// values, rewards and bootstrap values, uint8 flags, float or bfloat16
// outputs (float arithmetic).
#include "launch.cuh"

namespace rlscan {

namespace {
template <int OB>
rlscan_status launch_out(bool trunc, bool bs2d, Params p, void *ws, size_t ws_bytes, cudaStream_t s)
{
    if (!trunc) return launch_scan<est::Compact<est::VTrace<false, false>, 2, 1, OB>>(p, ws, ws_bytes, s);
    if (!bs2d) return launch_scan<est::Compact<est::VTrace<true, false>, 2, 1, OB>>(p, ws, ws_bytes, s);
    return launch_scan<est::Compact<est::VTrace<true, true>, 2, 1, OB>>(p, ws, ws_bytes, s);
}
}  // namespace

rlscan_status launch_vtrace_compact(bool trunc, bool bs2d, bool bf16_out, Params p, void *ws, size_t ws_bytes,
                                    cudaStream_t s)
{
    if (bf16_out) return launch_out<2>(trunc, bs2d, p, ws, ws_bytes, s);
    return launch_out<4>(trunc, bs2d, p, ws, ws_bytes, s);
}

}  // namespace rlscan
