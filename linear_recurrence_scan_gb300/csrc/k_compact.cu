// k_compact.cu -- GAE and fused GAE + returns on compact storage: bfloat16
// values, uint8 flags, float or bfloat16 outputs (float arithmetic).
#include "launch.cuh"

namespace rlscan {

namespace {
template <template <bool, bool> class Est, int OB>
rlscan_status launch_compact_out(bool trunc, bool bs2d, Params p, void *ws, size_t ws_bytes, cudaStream_t s)
{
    if (!trunc) return launch_scan<est::Compact<Est<false, false>, 2, 1, OB>>(p, ws, ws_bytes, s);
    if (!bs2d) return launch_scan<est::Compact<Est<true, false>, 2, 1, OB>>(p, ws, ws_bytes, s);
    return launch_scan<est::Compact<Est<true, true>, 2, 1, OB>>(p, ws, ws_bytes, s);
}
}  // namespace

rlscan_status launch_gae_compact(bool trunc, bool bs2d, bool bf16_out, Params p, void *ws, size_t ws_bytes,
                                 cudaStream_t s)
{
    if (bf16_out) return launch_compact_out<est::GAE, 2>(trunc, bs2d, p, ws, ws_bytes, s);
    return launch_compact_out<est::GAE, 4>(trunc, bs2d, p, ws, ws_bytes, s);
}

rlscan_status launch_gae_returns_compact(bool trunc, bool bs2d, bool bf16_out, Params p, void *ws, size_t ws_bytes,
                                         cudaStream_t s)
{
    if (bf16_out) return launch_compact_out<est::GAEReturns, 2>(trunc, bs2d, p, ws, ws_bytes, s);
    return launch_compact_out<est::GAEReturns, 4>(trunc, bs2d, p, ws, ws_bytes, s);
}

}  // namespace rlscan
