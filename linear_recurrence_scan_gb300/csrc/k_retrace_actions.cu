// k_retrace_actions.cu -- Retrace(lambda) from the full action-space inputs
// ([N,T,A] target probabilities and successor Q-values, int64 actions).
#include "launch.cuh"

namespace rlscan {

rlscan_status launch_retrace_actions(bool trunc, Params p, void *ws, size_t ws_bytes, cudaStream_t s)
{
    for (int w = 0; w < est::RetraceActions<false>::NWIDE; ++w)
        p.wide_words[w] = est::RetraceActions<false>::wide_words(w, p.A);
    if (!trunc) return launch_scan<est::RetraceActions<false>>(p, ws, ws_bytes, s);
    return launch_scan<est::RetraceActions<true>>(p, ws, ws_bytes, s);
}

}  // namespace rlscan
