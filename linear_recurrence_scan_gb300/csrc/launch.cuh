// launch.cuh -- host side of the scan kernel: tile geometry, staging path,
// workspace binding and grid sizing for one estimator instantiation.
#pragma once

#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "params.cuh"
#include "residency.cuh"
#include "scan_kernel.cuh"

namespace rlscan {

// Launch shape per estimator, from the bytes one time step moves
// (4 * (inputs + outputs)): tiles of 1024, 2048 or 4096 steps, whichever is
// closest to TILE_BYTES_TARGET bytes of traffic, so the per-tile fixed cost
// (barrier, warp scans, look-back) is amortised over enough data; 256
// compute threads (4, 8 or 16 steps each); as many ring stages
// (2..MAX_STAGES) as fit in SMEM_BUDGET_KB per CTA, of which packed tiles
// use PACKED_STAGES.  Sweeps on GB300 chose the defaults: short kernels are
// bound by each CTA's serial path through its tiles, so they prefer short
// per-thread chains (more warps per tile) and a shallow ring (every CTA's
// first tile arrives sooner); split rows that finish at once keep a deeper
// ring, and the deferred kernels of long rows a ring of DEFER_STAGES.  The
// macros exist for such sweeps.
#ifndef RLSCAN_TILE_BYTES_TARGET
#define RLSCAN_TILE_BYTES_TARGET 30000
#endif
#ifndef RLSCAN_SMEM_BUDGET_KB
#define RLSCAN_SMEM_BUDGET_KB 64
#endif
#ifndef RLSCAN_MAX_STAGES
#define RLSCAN_MAX_STAGES 3
#endif
// Compact storage (bf16 / uint8) moves about half the bytes per step and
// is bound by its issue rate: a deeper ring of split-row tiles keeps more
// copies in flight while its two CTAs per SM compute (3 stages: V-trace
// 2048 x 4096 26.9 -> 26.6 us, Retrace 1024 x 16384 46.3 -> 45.7 us).
#ifndef RLSCAN_LOWP_SMEM_BUDGET_KB
#define RLSCAN_LOWP_SMEM_BUDGET_KB 80
#endif
#ifndef RLSCAN_LOWP_MAX_STAGES
#define RLSCAN_LOWP_MAX_STAGES 3
#endif
// Packed tiles (whole rows, no look-back) use at most this many of the
// ring's stages: a shallower ring gets every CTA's first tile sooner, while
// split rows keep the deeper ring to hide their look-back waits.
#ifndef RLSCAN_PACKED_STAGES
#define RLSCAN_PACKED_STAGES 2
#endif
#ifndef RLSCAN_THREADS_2048
#define RLSCAN_THREADS_2048 256
#endif
#ifndef RLSCAN_LOWP_TILE_CAP
#define RLSCAN_LOWP_TILE_CAP 2048
#endif
#ifndef RLSCAN_THREADS_1024
#define RLSCAN_THREADS_1024 256
#endif
#ifndef RLSCAN_LOWP_THREADS_1024
#define RLSCAN_LOWP_THREADS_1024 256
#endif
// Packed launches with a workspace at hand: the last RLSCAN_PACKED_DYN_TAIL
// tiles per CTA are drawn from the workspace ticket instead of assigned
// statically (0: all static).  Measured on 4096 x 1024: GAE 13.88 -> 13.35
// us, TD(lambda) 13.53 -> 12.83, discounted returns 11.00 -> 10.69, V-trace
// 25.4 -> 23.9 (two or three dynamic tiles per CTA did no better).
#ifndef RLSCAN_PACKED_DYN_TAIL
#define RLSCAN_PACKED_DYN_TAIL 1
#endif
// Estimators with wide inputs (several words per step, e.g. [N,T,A]) move
// far more bytes per step: 1024-step tiles, and a ring of WIDE_STAGES stages
// whose size depends on the runtime width (one CTA per SM at A = 4).
#ifndef RLSCAN_WIDE_THREADS
#define RLSCAN_WIDE_THREADS 256
#endif
#ifndef RLSCAN_WIDE_STAGES
#define RLSCAN_WIDE_STAGES 2
#endif
// Long rows with several tiles of each row in flight finish every tile
// after the next tile's first half (deferred look-back); the pending tile
// keeps its stage, so the ring needs at least three.  RLSCAN_DEFER_MODE:
// -1 decide from the shape (several tiles of each row in flight, and the
// deeper ring keeps three CTAs per SM or as many as before), 0 never,
// 1 whenever rows span several tiles.
#ifndef RLSCAN_DEFER_STAGES
#define RLSCAN_DEFER_STAGES 3
#endif
#ifndef RLSCAN_DEFER_MODE
#define RLSCAN_DEFER_MODE -1
#endif

// Ring of the deferred kernel: RLSCAN_DEFER_STAGES unless the estimator
// declares DEFER_RING (eligibility traces: 4, 141 -> 138 us on 64 rows of
// 2^20 steps; the other long-row kernels lost with a fourth stage).
template <class E, class = void>
struct DeferRingOf {
    static constexpr int value = RLSCAN_DEFER_STAGES;
};
template <class E>
struct DeferRingOf<E, std::void_t<decltype(E::DEFER_RING)>> {
    static constexpr int value = E::DEFER_RING;
};

// Tile of a wide-input estimator: 1024 steps unless it declares WIDE_TILE
// (a smaller tile keeps two or three CTAs per SM when its stage is large).
template <class E, class = void>
struct WideTileOf {
    static constexpr int value = 1024;
};
template <class E>
struct WideTileOf<E, std::void_t<decltype(E::WIDE_TILE)>> {
    static constexpr int value = E::WIDE_TILE;
};

template <class E>
struct Shape {
    static constexpr bool WIDE = WideOf<E>::NWIDE > 0;
    static constexpr int in_sum()
    {
        int n = 0;
        for (int j = 0; j < E::NIN; ++j) n += IoOf<E>::in(j);
        return n;
    }
    static constexpr int BYTES_PER_STEP = in_sum() + IoOf<E>::OUT * E::NOUT;
    // compact storage sizes its tile as if its outputs were bfloat16 either
    // way, so float32 and bfloat16 outputs come from the same arithmetic (the
    // bfloat16 ones are the float32 ones rounded)
    static constexpr int SHAPE_BYTES = IoOf<E>::LOWP ? in_sum() + 2 * E::NOUT : BYTES_PER_STEP;
    static constexpr int TILE_RAW = RLSCAN_TILE_BYTES_TARGET / SHAPE_BYTES;
    // compact storage moves few bytes per step: cap at 2048 (8 steps per
    // thread; estimators with four or more inputs then run two CTAs per SM,
    // whose register budget holds their 8 steps)
    static constexpr int TILE_BY_BYTES = TILE_RAW >= 3072 ? 4096 : (TILE_RAW >= 1536 ? 2048 : 1024);
    static constexpr int TILE = WIDE ? WideTileOf<E>::value
                                     : ((IoOf<E>::LOWP && TILE_BY_BYTES > RLSCAN_LOWP_TILE_CAP)
                                            ? RLSCAN_LOWP_TILE_CAP : TILE_BY_BYTES);
    static constexpr int THREADS = WIDE ? (TILE < 1024 ? 128 : RLSCAN_WIDE_THREADS)
                                        : (TILE >= 4096 ? 256 : (TILE >= 2048 ? RLSCAN_THREADS_2048
                                                                              : (IoOf<E>::LOWP ? RLSCAN_LOWP_THREADS_1024
                                                                                               : RLSCAN_THREADS_1024)));
    static constexpr int ITEMS = TILE / THREADS;
    static constexpr int STAGE_BYTES = narrow_bytes<E, TILE>();  // narrow arrays
    static constexpr int RAW = ((IoOf<E>::LOWP ? RLSCAN_LOWP_SMEM_BUDGET_KB : RLSCAN_SMEM_BUDGET_KB) * 1024) /
                               STAGE_BYTES;
    static constexpr int MAXST = IoOf<E>::LOWP ? RLSCAN_LOWP_MAX_STAGES : RLSCAN_MAX_STAGES;
    // ring of an immediate-finish launch, and of a deferred one
    static constexpr int SHORT_STAGES = WIDE ? RLSCAN_WIDE_STAGES : (RAW < 2 ? 2 : (RAW > MAXST ? MAXST : RAW));
    static constexpr int PACKED_STAGES = SHORT_STAGES < RLSCAN_PACKED_STAGES ? SHORT_STAGES : RLSCAN_PACKED_STAGES;
    static constexpr int DEFER_RING = DeferRingOf<E>::value;
    static constexpr int DEFER_STAGES = (WIDE || DEFER_RING < 3) ? 0
                                        : (DEFER_RING > SHORT_STAGES ? DEFER_RING : SHORT_STAGES);
    static_assert(TILE == THREADS * ITEMS, "tile shape");
};

#ifndef RLSCAN_SHORT_THREADS
#define RLSCAN_SHORT_THREADS 128
#endif
#ifndef RLSCAN_SHORT_STAGES
#define RLSCAN_SHORT_STAGES 2
#endif
#ifndef RLSCAN_MOM_SHORT
#define RLSCAN_MOM_SHORT 1
#endif
// Compact storage on split rows: 1024-step tiles on 128 threads x 8 with a
// three-stage ring from this many rows on (fewer rows keep the regular
// shape, whose deferred kernel they need).  Measured: compact V-trace
// 2048 x 4096 26.5 -> 25.7 us, compact Retrace 1024 x 16384 45.8 -> 45.2.
#ifndef RLSCAN_LOWP_SPLIT_MIN_ROWS
#define RLSCAN_LOWP_SPLIT_MIN_ROWS 512
#endif
#ifndef RLSCAN_LOWP_SPLIT_STAGES
#define RLSCAN_LOWP_SPLIT_STAGES 3
#endif
// Packed launches (whole rows, T <= 1024) of single-scan or compact-storage
// estimators whose own shape is 2048 steps or more: 1024-step tiles on 128
// threads x 8 steps.  Rows this short gain from the smaller CTAs (five per
// SM instead of three, a shorter serial path through each tile, a 4-warp
// composition); measured on 4096 x 1024: GAE 14.65 -> 14.28 us, discounted
// returns 11.83 -> 11.17, TD(lambda) 14.31 -> 13.64, compact GAE 11.56 ->
// 11.06, compact fused GAE + returns 14.88 -> 13.84 (the float32 two-scan
// step and the 1024-step estimators lost with this shape and keep their
// own).
template <class E>
struct ShortShape {
    static constexpr bool ENABLED = !Shape<E>::WIDE && (E::K == 1 || IoOf<E>::LOWP) &&
                                    (Shape<E>::TILE >= 2048 || (RLSCAN_MOM_SHORT && MomentsOf<E>::value));
    static constexpr bool WIDE = false;
    static constexpr int TILE = 1024;
    static constexpr int THREADS = RLSCAN_SHORT_THREADS;
    static constexpr int ITEMS = TILE / THREADS;
    static constexpr int STAGE_BYTES = narrow_bytes<E, TILE>();
    static constexpr int DEFER_STAGES = 0;
};

constexpr int kMaxDevices = 64;

#define RLSCAN_LAUNCH_TRY(expr)                 \
    do {                                        \
        const rlscan_status st_ = (expr);       \
        if (st_ != RLSCAN_OK) return st_;       \
    } while (0)

inline bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }


// Per-device launch facts of one kernel: SM count, the dynamic shared
// memory a CTA may opt into (the device limit less the kernel's static
// shared memory), and resident CTAs for the last dynamic size used.
struct KernelFacts {
    std::mutex mu;
    int sm_count[kMaxDevices] = {};
    size_t max_dyn[kMaxDevices] = {};
    int blocks_per_sm[kMaxDevices] = {};
    size_t occ_smem[kMaxDevices] = {};
};

template <class Kernel>
rlscan_status kernel_facts(KernelFacts &f, Kernel kernel, int dev, int threads, size_t largest, bool opt_in_max,
                           size_t smem, size_t *dyn_limit, int64_t *slots)
{
    std::lock_guard<std::mutex> lock(f.mu);
    if (f.sm_count[dev] == 0) {
        int sms = 0, optin = 0;
        cudaFuncAttributes fa;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaFuncGetAttributes(&fa, kernel) != cudaSuccess)
            return RLSCAN_ERR_CUDA;
        const size_t dyn = static_cast<size_t>(optin) > fa.sharedSizeBytes ? optin - fa.sharedSizeBytes : 0;
        if (dyn < largest) return RLSCAN_ERR_CUDA;
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(opt_in_max ? dyn : largest)) != cudaSuccess)
            return RLSCAN_ERR_CUDA;
        f.max_dyn[dev] = dyn;
        f.sm_count[dev] = sms > 0 ? sms : 1;
    }
    if (dyn_limit != nullptr) *dyn_limit = f.max_dyn[dev];
    if (slots != nullptr) {
        if (f.occ_smem[dev] != smem) {
            int occ = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, smem) != cudaSuccess)
                return RLSCAN_ERR_CUDA;
            f.blocks_per_sm[dev] = occ > 0 ? occ : 1;
            f.occ_smem[dev] = smem;
        }
        *slots = static_cast<int64_t>(f.sm_count[dev]) * f.blocks_per_sm[dev];
    }
    return RLSCAN_OK;
}

template <class Kernel>
rlscan_status launch_kernel(Kernel kernel, const Params &p, int64_t grid, int threads, size_t smem,
                            cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, p) != cudaSuccess) {
        cudaGetLastError();
        return RLSCAN_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? RLSCAN_OK : RLSCAN_ERR_CUDA;
}

// Staging path and limits of a launch: bulk copies and vector stores when
// every row is whole 16-byte units and the arrays are aligned (bulk copies
// only from device memory).  Returns whether the tiles are bulk-copied.
template <class E>
rlscan_status bind_io(Params &p, bool *tma_out)
{
    bool tma = true;
    for (int j = 0; j < E::NIN; ++j) {
        const int units = 16 / IoOf<E>::in(j);
        tma = tma && (p.T % units == 0) && (p.rs % units == 0) && aligned16(p.in[j]);
    }
    for (int q = 0; q < E::NOUT; ++q) {
        const int units = 16 / IoOf<E>::OUT;
        tma = tma && (p.T % units == 0) && (p.rs % units == 0) && (p.out[q] == nullptr || aligned16(p.out[q]));
    }
    p.vec = tma ? 1 : 0;
    bool on_host = false, unreachable = false;
    auto note = [&](const void *ptr, bool input) {
        if (ptr == nullptr) return;
        const Residency r = residency(ptr);
        unreachable = unreachable || r == Residency::Unreachable;
        on_host = on_host || (input && r == Residency::Host);
    };
    for (int j = 0; j < E::NIN; ++j) note(p.in[j], true);
    for (int w = 0; w < WideOf<E>::NWIDE; ++w) note(p.wide[w], true);
    for (int q = 0; q < E::NOUT; ++q) note(p.out[q], false);
    note(p.rowscalar, false);
    if (unreachable) return RLSCAN_ERR_MEMORY;
    tma = tma && !on_host;
    p.tma = tma ? 1 : 0;
    p.spin_limit_ns = spin_limit_ns();
    p.copy_limit_ns = 2000000000ull;  // bulk copies land in microseconds; never cut short
    p.withhold_tile = withhold_tile();
    p.bounds = bounds_counter();
    p.check_rows = p.N - (check_short() ? 1 : 0);
    *tma_out = tma;
    return RLSCAN_OK;
}

// Packed tiling (whole rows per tile) of an estimator's shape.
template <class E, class S>
void bind_packed(Params &p)
{
    p.packed = 1;
    p.C = static_cast<int32_t>((p.T + S::ITEMS - 1) / S::ITEMS * S::ITEMS);
    p.R = S::TILE / p.C;
    p.tiles_per_row = 1;
    p.num_tiles = (p.N + p.R - 1) / p.R;
    p.dynamic = 0;
    p.hdr = nullptr;
    p.states = nullptr;
}

// One launch of shape S with an immediate-finish ring of ST stages (or, for
// split rows with several tiles of each row in flight, the deferred kernel).
template <class E, class S, int ST>
rlscan_status launch_scan_ring(Params p, void *ws, size_t ws_bytes, cudaStream_t stream, int64_t *grid_out)
{
    constexpr int TILE = S::TILE;
    constexpr int BT = block_threads<S::THREADS>();
    auto kernel = scan_kernel<E, S::THREADS, S::ITEMS, ST, false>;
    size_t smem = static_cast<size_t>(ST) * S::STAGE_BYTES;

    if (p.T <= TILE) {
        bind_packed<E, S>(p);
    } else {
        p.packed = 0;
        p.C = TILE;
        p.R = 1;
        p.tiles_per_row = (p.T + TILE - 1) / TILE;
        p.num_tiles = p.N * p.tiles_per_row;
        const size_t need = kHeaderBytes + kStateBytes * E::K * static_cast<size_t>(p.num_tiles);
        if (ws == nullptr || ws_bytes < need || !aligned16(ws) || residency(ws) != Residency::Device)
            return RLSCAN_ERR_WORKSPACE;
        p.dynamic = 1;
        p.hdr = static_cast<uint32_t *>(ws);
        p.states = reinterpret_cast<unsigned long long *>(static_cast<char *>(ws) + kHeaderBytes);
    }

    bool tma = false;
    RLSCAN_LAUNCH_TRY(bind_io<E>(p, &tma));

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RLSCAN_ERR_CUDA;
    static KernelFacts facts;
    size_t dyn_limit = 0;
    RLSCAN_LAUNCH_TRY(kernel_facts(facts, kernel, dev, BT, smem, S::WIDE, smem, &dyn_limit, nullptr));
    if constexpr (S::WIDE) {
        // stage the wide arrays when they are aligned and the ring fits
        int64_t wide_floats = 0;
        bool wide_ok = tma;
        for (int w = 0; w < WideOf<E>::NWIDE; ++w) {
            wide_floats += static_cast<int64_t>(TILE + 4) * p.wide_words[w];
            wide_ok = wide_ok && aligned16(p.wide[w]) && (p.wide_rs[w] % 4 == 0);
        }
        // copied narrow arrays, then the wide region, which the derived
        // arrays overlay (they need a region of their own when not staged)
        const int64_t copied = static_cast<int64_t>(narrow_copied<E>()) * (TILE + 8);
        const int64_t derived = static_cast<int64_t>(E::NIN - narrow_copied<E>()) * (TILE + 8);
        const int64_t staged_floats = copied + (wide_floats > derived ? wide_floats : derived);
        wide_ok = wide_ok && static_cast<size_t>(ST) * staged_floats * 4 <= dyn_limit;
        p.wide_staged = wide_ok ? 1 : 0;
        p.stage_floats = static_cast<int32_t>(wide_ok ? staged_floats : copied + derived);
        smem = static_cast<size_t>(ST) * p.stage_floats * 4;
    }
    int64_t slots = 0;
    RLSCAN_LAUNCH_TRY(kernel_facts(facts, kernel, dev, BT, smem, S::WIDE, smem, nullptr, &slots));

    // Deferred finishing when several tiles of each row are in flight at
    // once (their look-backs would otherwise wait on one another).
    if constexpr (S::DEFER_STAGES >= 3) {
        const bool want = !p.packed && (RLSCAN_DEFER_MODE == 1 ||
                                        (RLSCAN_DEFER_MODE < 0 && slots * ST >= 2 * p.N));
        if (want) {
            auto dkernel = scan_kernel<E, S::THREADS, S::ITEMS, S::DEFER_STAGES, true>;
            static KernelFacts dfacts;
            const size_t dsmem = static_cast<size_t>(S::DEFER_STAGES) * S::STAGE_BYTES;
            int64_t dslots = 0;
            RLSCAN_LAUNCH_TRY(kernel_facts(dfacts, dkernel, dev, BT, dsmem, false, dsmem, nullptr, &dslots));
            // only while the deeper ring keeps three CTAs per SM resident (or
            // as many as the immediate kernel); forced: always
            if (MomentsOf<E>::value && dslots > kMaxMomentCtas) dslots = kMaxMomentCtas;
            if (RLSCAN_DEFER_MODE == 1 || dslots >= slots || dslots >= 3 * static_cast<int64_t>(facts.sm_count[dev])) {
                const int64_t grid = p.num_tiles < dslots ? p.num_tiles : dslots;
                if (grid_out != nullptr) *grid_out = grid;
                return launch_kernel(dkernel, p, grid, BT, dsmem, stream);
            }
        }
    }
    if (MomentsOf<E>::value && slots > kMaxMomentCtas) slots = kMaxMomentCtas;  // one moments slot per CTA
    const int64_t grid = p.num_tiles < slots ? p.num_tiles : slots;
    // Packed tiles: all but the last RLSCAN_PACKED_DYN_TAIL per CTA go out
    // statically (no atomic on the producer's path); the rest come from the
    // workspace ticket, so CTAs on faster SMs take more of them and all end
    // together.  Kernels that accumulate moments keep the static order (their
    // per-CTA sums, and so the normalised outputs, are the same bits on
    // every call); without a usable workspace all tiles are static.
    if (p.packed && RLSCAN_PACKED_DYN_TAIL > 0 && !MomentsOf<E>::value && ws != nullptr &&
        ws_bytes >= kHeaderBytes && aligned16(ws) && residency(ws) == Residency::Device) {
        const int64_t per_cta = p.num_tiles / grid;
        if (per_cta > RLSCAN_PACKED_DYN_TAIL) {
            p.dynamic = 1;
            p.hdr = static_cast<uint32_t *>(ws);
            p.static_tiles = (per_cta - RLSCAN_PACKED_DYN_TAIL) * grid;
        }
    }
    if (grid_out != nullptr) *grid_out = grid;
    return launch_kernel(kernel, p, grid, BT, smem, stream);
}

template <class E>
rlscan_status launch_scan(Params p, void *ws, size_t ws_bytes, cudaStream_t stream, int64_t *grid_out = nullptr)
{
    using S = Shape<E>;
    if constexpr (ShortShape<E>::ENABLED) {
        using Q = ShortShape<E>;
        if (p.T <= Q::TILE) return launch_scan_ring<E, Q, RLSCAN_SHORT_STAGES>(p, ws, ws_bytes, stream, grid_out);
    }
    if constexpr (ShortShape<E>::ENABLED && IoOf<E>::LOWP) {
        // compact storage: the short-row shape for split rows too (a
        // three-stage ring), unless the rows are few enough for the
        // deferred kernel of the regular shape
        using Q = ShortShape<E>;
        if (p.T > S::TILE && p.N >= RLSCAN_LOWP_SPLIT_MIN_ROWS)
            return launch_scan_ring<E, Q, RLSCAN_LOWP_SPLIT_STAGES>(p, ws, ws_bytes, stream, grid_out);
    }
    if (p.T <= S::TILE) return launch_scan_ring<E, S, S::PACKED_STAGES>(p, ws, ws_bytes, stream, grid_out);
    return launch_scan_ring<E, S, S::SHORT_STAGES>(p, ws, ws_bytes, stream, grid_out);
}

}  // namespace rlscan
