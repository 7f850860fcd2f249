// params.cuh -- the argument block every scan kernel receives, and the
// internal launcher entry points the C ABI dispatches to.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "rlscan.h"

namespace rlscan {

constexpr int kMaxIn = 8;
constexpr int kMaxWide = 3;  // staged arrays with several 4-byte words per step

// Workspace layout: a 64-byte header followed by one 16-byte state per tile
// and scan (an estimator solves up to kMaxScans recurrences per step).
//   bytes  0.. 7  u64 tile ticket (dynamic tile ids, reset by the last CTA)
//   bytes  8..11  u32 count of CTAs that finished (reset by the last CTA)
//   bytes 12..15  u32 first error code recorded on the device (0 = none)
//   bytes 16..19  u32 detail of that error (tile index / stage)
constexpr size_t kHeaderBytes = 64;
constexpr size_t kStateBytes = 16;
constexpr int kMaxScans = 2;
//   bytes 20..23  u32 epoch: tag of the current call's tile states (advanced by the last CTA)
enum HeaderWord : int { kHdrExit = 2, kHdrError = 3, kHdrDetail = 4, kHdrEpoch = 5 };

// Batch moments of the advantages (normalising entry point): after the
// header and tile states, at a 256-byte boundary, one 16-byte slot per CTA
// of the scan kernel: its sum and sum of squares, each a float pair (hi, lo).
constexpr int kMaxMomentCtas = 4096;
constexpr size_t kMomentBytes = 16 * static_cast<size_t>(kMaxMomentCtas);

// The workspace size query counts 1024-step tiles and kMaxScans scans per
// tile: kernels with 1024-step or longer tiles fit it with up to kMaxScans
// scans, 512-step tiles with one scan.  Rows of up to 512 steps never need
// a workspace.
constexpr int kMinTile = 1024;
constexpr int kSmallestTile = 512;

struct Params {
    const float *in[kMaxIn];   // [N, rs] inputs, order defined by the estimator
    float *out[3];             // [N, rs] outputs (optional ones may be null)
    const float *rowscalar;    // per-row scalar (bootstrap / carry / seed), nullable
    int64_t rowscalar_stride;  // elements between consecutive rows' scalars
    int64_t N, T, rs;
    float c0, c1, c2, c3;      // estimator constants (gamma, lambda, clips)

    // tiling, filled by the launcher
    int64_t num_tiles;         // tiles in the whole problem
    int64_t tiles_per_row;     // 1 when whole rows are packed into a tile
    int32_t C;                 // smem row pitch of a tile (elements)
    int32_t R;                 // rows per tile (packed) or 1
    int32_t packed;            // 1: tiles hold whole rows; 0: rows split into tiles
    int32_t tma;               // 1: bulk asynchronous copies; 0: element-wise loads
    int32_t vec;               // 1: rows in whole 16-byte units: vector stores
    int32_t dynamic;           // 1: tile ids from the workspace ticket (look-back, or a packed tail)
    int64_t static_tiles;      // tiles [0, static_tiles) go to CTAs statically (b, b + grid, ...)
    unsigned long long *states;
    uint32_t *hdr;
    uint64_t spin_limit_ns;    // bound on every look-back wait
    uint64_t copy_limit_ns;    // bound on every wait for a bulk copy
    int64_t withhold_tile;     // test hook: this tile never publishes (-1: none)

    // wide inputs (several 4-byte words per step, e.g. [N, T, A] arrays),
    // used only by estimators that declare them
    const void *wide[kMaxWide];
    int64_t wide_rs[kMaxWide];    // row stride in 4-byte words
    int32_t wide_words[kMaxWide]; // 4-byte words per step
    int32_t wide_staged;          // 1: copied into the stage; 0: read from global memory
    int32_t stage_floats;         // floats per ring stage (narrow and wide regions)
    int32_t A;                    // number of actions

    // batch moments of output 0 (estimators that declare MOMENTS); c2 holds
    // eps, mom_inv the normalising pass's 1 / n and 1 / (n - 1) (n = N T)
    // as float pairs (hi, lo)
    float *mom_part;              // [gridDim.x][4] per-CTA sum and sum of squares, each a float pair
    float mom_inv[4];

    // checked builds only: violations counted and the first site (else NULL),
    // and the rows the checks take each [N,T] array to span (N; fewer under
    // the RLSCAN_TEST_CHECK_SHORT test hook, which must then be reported)
    unsigned long long *bounds;
    int64_t check_rows;
};

// Launchers (one translation unit per estimator family).
rlscan_status launch_gae(bool trunc, bool bs2d, Params p, void *ws, size_t ws_bytes, cudaStream_t s);
rlscan_status launch_gae_returns(bool trunc, bool bs2d, Params p, void *ws, size_t ws_bytes, cudaStream_t s);
rlscan_status launch_gae_normalized(bool trunc, bool bs2d, bool discounted, Params p, float *moments_out,
                                    void *ws, size_t ws_bytes, cudaStream_t s);
rlscan_status launch_gae_masked(bool trunc, bool bs2d, Params p, void *ws, size_t ws_bytes, cudaStream_t s);
rlscan_status launch_gae_compact(bool trunc, bool bs2d, bool bf16_out, Params p, void *ws, size_t ws_bytes,
                                 cudaStream_t s);
rlscan_status launch_gae_returns_compact(bool trunc, bool bs2d, bool bf16_out, Params p, void *ws, size_t ws_bytes,
                                         cudaStream_t s);
rlscan_status launch_vtrace(bool trunc, bool bs2d, Params p, void *ws, size_t ws_bytes, cudaStream_t s);
rlscan_status launch_vtrace_compact(bool trunc, bool bs2d, bool bf16_out, Params p, void *ws, size_t ws_bytes,
                                    cudaStream_t s);
rlscan_status launch_retrace_compact(bool trunc, bool bf16_out, Params p, void *ws, size_t ws_bytes,
                                     cudaStream_t s);
rlscan_status launch_retrace(bool trunc, Params p, void *ws, size_t ws_bytes, cudaStream_t s);
rlscan_status launch_retrace_actions(bool trunc, Params p, void *ws, size_t ws_bytes, cudaStream_t s);
rlscan_status launch_lambda_returns(bool trunc, bool bs2d, Params p, void *ws, size_t ws_bytes, cudaStream_t s);
rlscan_status launch_discounted(bool trunc, bool bs2d, Params p, void *ws, size_t ws_bytes, cudaStream_t s);
rlscan_status launch_eligibility(Params p, void *ws, size_t ws_bytes, cudaStream_t s);
rlscan_status launch_prefix(bool starts_at, Params p, void *ws, size_t ws_bytes, cudaStream_t s);
rlscan_status launch_linear(bool forward, Params p, void *ws, size_t ws_bytes, cudaStream_t s);

// Host helpers shared by the launchers (rlscan_abi.cu).
uint64_t spin_limit_ns();
int64_t withhold_tile();  // RLSCAN_TEST_WITHHOLD_TILE, -1 when unset
bool pdl_enabled();  // programmatic dependent launch (RLSCAN_PDL=0 disables)
// checked builds: the device counter of bounds violations (NULL otherwise)
unsigned long long *bounds_counter();
bool check_short();  // RLSCAN_TEST_CHECK_SHORT=1 in a checked build

}  // namespace rlscan
