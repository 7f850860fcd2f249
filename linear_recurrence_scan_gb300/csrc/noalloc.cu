// noalloc.cu -- rlscan_gae_noalloc: GAE for callers that may not allocate
// device memory.
//
// Long rows are scanned by several thread blocks that hand carries to each
// other through scratch memory (the look-back tile states).  rlscan_gae
// takes that scratch from the caller.  Some callers cannot provide it: code
// running inside a host framework that owns every device allocation through
// its own pool, a latency-critical loop whose policy forbids cudaMalloc and
// cudaFree after start-up (both can synchronise the whole device), or an
// embedded runtime with a memory budget fixed before the first call.  This
// entry point serves them from a fixed buffer that is part of the library
// image: it allocates nothing, ever.
//
// The buffer is a file-scope __device__ array, so every GPU that loads the
// library holds kScratchBytes of it until the process exits.  In host code
// the array's name is only a host-side stand-in; its device address is
// looked up with cudaGetSymbolAddress once per device, with that device
// current, the first time this entry point runs there, and kept for the
// life of the process (a cudaDeviceReset, or any other teardown of the
// device's primary context, between calls is not supported: the module is
// reloaded and the kept address may no longer be the buffer's).  That
// first call also zeroes the buffer, so it should happen before any stream
// capture.
// All calls share the buffer: each call clears the buffer header (tile
// ticket and counters) on its stream before launching, and the tile states
// themselves are tagged per call, so stale contents are never consumed.
// Calls whose executions overlap on the GPU (different streams, no
// ordering) race on the buffer and must not be issued.
#include <initializer_list>
#include <mutex>

#include <cuda_runtime.h>

#include "params.cuh"

#define RLSCAN_API __attribute__((visibility("default")))

namespace {

// Header + 16 bytes per (tile of at least 1024 steps, scan), sized by
// rlscan_workspace_bytes: N * ceil(T / 1024) <= 131,070, e.g. 32 rows of 4M
// steps or 2048 rows of 64K steps.
constexpr size_t kScratchBytes = size_t(4) << 20;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDev];

// Device address of g_scratch on the current device; on the first call per
// device also zero the whole buffer on `stream`.
rlscan_status scratch_for_current_device(cudaStream_t stream, void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return RLSCAN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || ptr == nullptr)
            return RLSCAN_ERR_CUDA;
        if (cudaMemsetAsync(ptr, 0, kScratchBytes, stream) != cudaSuccess) return RLSCAN_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return RLSCAN_OK;
}

}  // namespace

extern "C" RLSCAN_API rlscan_status rlscan_gae_noalloc(
    const float *rewards, const float *values, const float *terminateds, const float *truncateds,
    const float *bootstrap_values, const float *last_value, int64_t N, int64_t T,
    int64_t row_stride, float gamma, float lambda, float *advantages, rlscan_stream_t stream)
{
    if (N < 0 || T < 0 || row_stride < T) return RLSCAN_ERR_SHAPE;
    if (N == 0 || T == 0) return RLSCAN_OK;
    if (!rewards || !values || !terminateds || !advantages) return RLSCAN_ERR_NULL;
    // rlscan_gae's own argument conflicts, checked before the shared buffer
    // is touched, so a rejected call enqueues nothing
    if (bootstrap_values && last_value) return RLSCAN_ERR_ARG_CONFLICT;
    if (last_value && truncateds) return RLSCAN_ERR_ARG_CONFLICT;
    for (const void *in : {static_cast<const void *>(rewards), static_cast<const void *>(values),
                           static_cast<const void *>(terminateds), static_cast<const void *>(truncateds),
                           static_cast<const void *>(bootstrap_values), static_cast<const void *>(last_value)})
        if (in != nullptr && in == static_cast<const void *>(advantages)) return RLSCAN_ERR_ARG_CONFLICT;
    const size_t need = rlscan_workspace_bytes(N, T);
    if (need > kScratchBytes) return RLSCAN_ERR_SCRATCH_LIMIT;
    void *ws = nullptr;
    size_t ws_bytes = 0;
    if (need > 0) {
        cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        const rlscan_status st = scratch_for_current_device(s, &ws);
        if (st != RLSCAN_OK) return st;
        // ticket, exit count and error words start at zero for every call;
        // the epoch word (kHdrEpoch) is kept, so earlier calls' tile states
        // stay stale
        if (cudaMemsetAsync(ws, 0, rlscan::kHdrEpoch * sizeof(uint32_t), s) != cudaSuccess) return RLSCAN_ERR_CUDA;
        ws_bytes = kScratchBytes;
    }
    return rlscan_gae(rewards, values, terminateds, truncateds, bootstrap_values, last_value, N, T,
                      row_stride, gamma, lambda, advantages, ws, ws_bytes, stream);
}
