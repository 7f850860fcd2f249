// k_retrace_compact.cu -- Retrace(lambda) from per-step inputs on compact
// storage: bfloat16 probabilities, Q-values and rewards, uint8 flags, float or
// bfloat16 outputs (float arithmetic).
#include "launch.cuh"

namespace rlscan {

rlscan_status launch_retrace_compact(bool trunc, bool bf16_out, Params p, void *ws, size_t ws_bytes,
                                     cudaStream_t s)
{
    if (bf16_out) {
        if (!trunc) return launch_scan<est::Compact<est::Retrace<false>, 2, 1, 2>>(p, ws, ws_bytes, s);
        return launch_scan<est::Compact<est::Retrace<true>, 2, 1, 2>>(p, ws, ws_bytes, s);
    }
    if (!trunc) return launch_scan<est::Compact<est::Retrace<false>, 2, 1, 4>>(p, ws, ws_bytes, s);
    return launch_scan<est::Compact<est::Retrace<true>, 2, 1, 4>>(p, ws, ws_bytes, s);
}

}  // namespace rlscan
