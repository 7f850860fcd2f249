// launch.cuh -- host side of the scan kernel: tile geometry, staging path,
// workspace binding and grid sizing for one estimator instantiation.
#pragma once

#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "params.cuh"
#include "scan_kernel.cuh"

namespace rlscan {

// Launch shape per estimator: 256 threads; 8 steps per thread (2048-step
// tiles) for the light estimators, 4 (1024-step tiles) for those with five
// or more input streams, so that STAGES stages of every input fit twice per
// SM.  The ring holds up to ~96 KB per CTA.
template <class E>
struct Shape {
    static constexpr int THREADS = 256;
    static constexpr int ITEMS = (E::NIN >= 5) ? 4 : 8;
    static constexpr int TILE = THREADS * ITEMS;
    static constexpr int STAGE_BYTES = E::NIN * (TILE + 8) * 4;
    static constexpr int RAW = (96 * 1024) / STAGE_BYTES;
    static constexpr int STAGES = RAW < 2 ? 2 : (RAW > 4 ? 4 : RAW);
};

constexpr int kMaxDevices = 64;

inline bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

template <class E>
rlscan_status launch_scan(Params p, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    using S = Shape<E>;
    constexpr int TILE = S::TILE;
    auto kernel = scan_kernel<E, S::THREADS, S::ITEMS, S::STAGES>;
    const size_t smem = static_cast<size_t>(S::STAGES) * S::STAGE_BYTES;

    if (p.T <= TILE) {
        p.packed = 1;
        p.C = static_cast<int32_t>((p.T + S::ITEMS - 1) / S::ITEMS * S::ITEMS);
        p.R = TILE / p.C;
        p.tiles_per_row = 1;
        p.num_tiles = (p.N + p.R - 1) / p.R;
        p.dynamic = 0;
        p.hdr = nullptr;
        p.states = nullptr;
        p.epoch = 0;
    } else {
        p.packed = 0;
        p.C = TILE;
        p.R = 1;
        p.tiles_per_row = (p.T + TILE - 1) / TILE;
        p.num_tiles = p.N * p.tiles_per_row;
        const size_t need = kHeaderBytes + kStateBytes * static_cast<size_t>(p.num_tiles);
        if (ws == nullptr || ws_bytes < need || !aligned16(ws)) return RLSCAN_ERR_WORKSPACE;
        p.dynamic = 1;
        p.hdr = static_cast<uint32_t *>(ws);
        p.states = reinterpret_cast<unsigned long long *>(static_cast<char *>(ws) + kHeaderBytes);
        p.epoch = next_epoch();
    }

    bool tma = (p.T % 4 == 0) && (p.rs % 4 == 0);
    for (int j = 0; j < E::NIN; ++j) tma = tma && aligned16(p.in[j]);
    for (int q = 0; q < E::NOUT; ++q) tma = tma && aligned16(p.out[q]);
    p.tma = tma ? 1 : 0;
    p.spin_limit_ns = spin_limit_ns();

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RLSCAN_ERR_CUDA;
    static std::mutex mu;
    static int blocks_per_sm[kMaxDevices];
    static int sm_count[kMaxDevices];
    {
        std::lock_guard<std::mutex> lock(mu);
        if (sm_count[dev] == 0) {
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem)) != cudaSuccess)
                return RLSCAN_ERR_CUDA;
            int occ = 0, sms = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, S::THREADS, smem) != cudaSuccess ||
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                return RLSCAN_ERR_CUDA;
            blocks_per_sm[dev] = occ > 0 ? occ : 1;
            sm_count[dev] = sms > 0 ? sms : 1;
        }
    }
    const int64_t slots = static_cast<int64_t>(sm_count[dev]) * blocks_per_sm[dev];
    const int64_t grid = p.num_tiles < slots ? p.num_tiles : slots;
    kernel<<<static_cast<unsigned>(grid), S::THREADS, smem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? RLSCAN_OK : RLSCAN_ERR_CUDA;
}

}  // namespace rlscan
