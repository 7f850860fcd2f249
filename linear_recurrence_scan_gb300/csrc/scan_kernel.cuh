// scan_kernel.cuh -- the one kernel template behind every entry point.
//
// Problem: for each row of an [N, T] buffer, A_t = alpha_t + beta_t A_{t-+1}
// with (alpha_t, beta_t) built in registers by an estimator functor
// (estimators.cuh).  The recurrence is an associative scan of affine maps
// f_t(x) = alpha_t + beta_t x under composition (rl-triton paper Eq. 2 and
// Prop. 1); the backward recurrences scan in decreasing time (Sec. 2.2).
//
// GB300 design:
//  * Persistent CTAs (grid = SMs x resident CTAs) walk a sequence of tiles.
//    A tile is THREADS*ITEMS elements: either several whole rows ("packed",
//    T <= tile) or one segment of a long row.
//  * Staging: one thread issues bulk asynchronous copies (cp.async.bulk, the
//    TMA engine's non-tensor form) of every input array of a tile into a
//    shared-memory stage, completing on an mbarrier.  STAGES stages form a
//    ring, so the copies of the next STAGES-1 tiles are in flight while one
//    tile is computed.  Unaligned shapes fall back to element-wise loads.
//  * Scan inside a tile: each thread owns ITEMS consecutive steps and folds
//    them serially; a warp shuffle scan combines the 32 threads; warp 0
//    combines the warps.  Then each thread re-runs its serial recurrence
//    from its exact incoming value, so every output is one fused multiply-add
//    chain from a known value (no separate "apply carry" pass).
//  * Row boundaries are folded into the coefficients: at the row's first
//    element in scan order (t = T-1 backward, t = 0 forward) the kernel sets
//    alpha += beta * boundary and beta = 0.  A packed tile is then one flat
//    scan (beta = 0 severs rows), and the first tile of a long row never
//    depends on anything before it.
//  * Long rows: decoupled look-back.  Each tile publishes its aggregate
//    (a, b) and later its inclusive value in a 16-byte state in the caller's
//    workspace; a tile waits only for its predecessors' aggregates.  Each
//    64-bit state word carries a 32-bit tag (call epoch << 2 | kind) next to
//    its payload, so a reader validates it without fences and stale words of
//    earlier calls are never mistaken for fresh ones (no memset per call).
//    Tiles are handed out by an atomic ticket in the order (position in row,
//    row): a tile's predecessor in its row was handed out N tickets earlier,
//    so it is usually finished before it is needed, and every predecessor is
//    held by a CTA that is already running (no deadlock).  The predecessor's
//    state is fetched when the tile starts, off the critical path.
//  * Launched with programmatic stream serialization: the next kernel may be
//    scheduled while this one drains, and this one touches global memory
//    only after griddepcontrol.wait (previous kernel complete and visible).
//  * Roles (warp specialisation): lane 0 of an extra producer warp draws
//    tickets and issues the copies, gated per stage by an "empty" mbarrier
//    that the compute warps arrive on; the compute warps wait on the stage's
//    "full" mbarrier.  The compute warps share one named barrier per tile:
//    after it each warp composes the aggregates of the warps before it
//    (double-buffered in shared memory) and, for a chained tile, its lane 0
//    reads the predecessor states itself; the warp holding the tile's last
//    element in scan order publishes.
//  * Every wait (mbarrier phase, predecessor state) is bounded in time; on
//    expiry the kernel records RLSCAN_ERR_TIMEOUT in the workspace, uses NaN
//    for the missing value and carries on, so it always terminates.
#pragma once

#include <cstdint>
#include <type_traits>

#include <cuda_bf16.h>

#include "dfloat.cuh"
#include "estimators.cuh"
#include "params.cuh"
#include "checks.cuh"
#include "ptx.cuh"

namespace rlscan {

struct Pair {
    float a, b;
};

// Wide inputs of an estimator (none unless it declares NWIDE / DERIVED):
// NWIDE arrays of several words per step staged after the narrow arrays,
// and the narrow arrays (bit mask) that prepass() derives from them instead
// of reading global memory.
template <class E, class = void>
struct WideOf {
    static constexpr int NWIDE = 0;
    static constexpr unsigned DERIVED = 0u;
};
template <class E>
struct WideOf<E, std::void_t<decltype(E::NWIDE)>> {
    static constexpr int NWIDE = E::NWIDE;
    static constexpr unsigned DERIVED = E::DERIVED;
};

// Element sizes of an estimator's narrow inputs and outputs: 4-byte floats
// unless it declares in_bytes(j) / OUT_BYTES (bf16 values, uint8 flags).
template <class E, class = void>
struct IoOf {
    static constexpr bool LOWP = false;
    __host__ __device__ static constexpr int in(int) { return 4; }
    static constexpr int OUT = 4;
};
template <class E>
struct IoOf<E, std::void_t<decltype(E::OUT_BYTES)>> {
    static constexpr bool LOWP = true;
    __host__ __device__ static constexpr int in(int j) { return E::in_bytes(j); }
    static constexpr int OUT = E::OUT_BYTES;
};

// Estimators whose kernel accumulates the batch moments of output 0.
template <class E, class = void>
struct MomentsOf {
    static constexpr bool value = false;
};
template <class E>
struct MomentsOf<E, std::void_t<decltype(E::MOMENTS)>> {
    static constexpr bool value = E::MOMENTS;
};

// Estimators whose tile aggregates usually keep a nonzero decay (beta = 1
// within episodes: prefix sums, the generic scan): a chained tile cannot
// resolve its carry from its nearest predecessor's aggregate alone, so the
// deferred kernel prefetches a window of predecessor states (see
// RLSCAN_LB_WINDOW) instead of one.
template <class E, class = void>
struct ChainOf {
    static constexpr bool value = false;
};
template <class E>
struct ChainOf<E, std::void_t<decltype(E::LB_CHAIN)>> {
    static constexpr bool value = E::LB_CHAIN;
};

// Estimators whose look-back states are laid out row-major (see state_pos):
// the chain estimators and those that declare LB_ROW_MAJOR.
template <class E, class = void>
struct RowMajorDecl {
    static constexpr bool value = false;
};
template <class E>
struct RowMajorDecl<E, std::void_t<decltype(E::LB_ROW_MAJOR)>> {
    static constexpr bool value = E::LB_ROW_MAJOR;
};
template <class E>
struct RowMajorOf {
    static constexpr bool value = ChainOf<E>::value || RowMajorDecl<E>::value;
};

// Shared-memory slot of narrow input j within a stage: the copied arrays
// first, in input order, then the derived ones.  The wide region starts
// after the copied arrays and overlays the derived slots: prepass() reads
// the wide rows, then writes the derived values over them.
template <class E>
__host__ __device__ constexpr int narrow_copied()
{
    int n = 0;
    for (int j = 0; j < E::NIN; ++j) n += ((WideOf<E>::DERIVED >> j) & 1u) ? 0 : 1;
    return n;
}
template <class E>
__host__ __device__ constexpr int slot_of(int j)
{
    constexpr unsigned D = WideOf<E>::DERIVED;
    const bool derived = (D >> j) & 1u;
    int below = 0;
    for (int i = 0; i < j; ++i) below += (((D >> i) & 1u) != 0) == derived ? 1 : 0;
    return derived ? narrow_copied<E>() + below : below;
}

// Shared-memory region of narrow input j in a stage: 16 bytes for the step
// before the tile, the tile's steps, 16 bytes for the step after it.
// Regions follow one another in slot order; 4-byte inputs give the float
// layout (TILE + 8) floats per array, data from float 4.
template <class E, int TILE>
__host__ __device__ constexpr int region_bytes(int j) { return TILE * IoOf<E>::in(j) + 32; }
template <class E, int TILE>
__host__ __device__ constexpr int region_off(int j)
{
    int off = 0;
    for (int i = 0; i < E::NIN; ++i)
        if (slot_of<E>(i) < slot_of<E>(j)) off += region_bytes<E, TILE>(i);
    return off;
}
template <class E, int TILE>
__host__ __device__ constexpr int narrow_bytes()
{
    int n = 0;
    for (int i = 0; i < E::NIN; ++i) n += region_bytes<E, TILE>(i);
    return n;
}
// step 0 of the tile in array j's region
template <class E, int TILE>
__device__ __forceinline__ char *elem0(float *stage, int j)
{
    return reinterpret_cast<char *>(stage) + region_off<E, TILE>(j) + 16;
}
template <class E, int TILE>
__device__ __forceinline__ const char *elem0(const float *stage, int j)
{
    return reinterpret_cast<const char *>(stage) + region_off<E, TILE>(j) + 16;
}

// Byte r of w (an integer 0..255) as a float.  RLSCAN_U8_PRMT=1: one byte
// permute builds the float 2^23 + byte (bits 0x4B0000bb) and one subtraction
// removes 2^23, exact for every byte; 0: integer extract and conversion.
#ifndef RLSCAN_U8_PRMT
#define RLSCAN_U8_PRMT 1
#endif
__device__ __forceinline__ float u8_to_float(uint32_t w, int r)
{
    if (RLSCAN_U8_PRMT)
        return __uint_as_float(__byte_perm(w, 0x4B000000u, static_cast<uint32_t>(r) | 0x7540u)) - 8388608.f;
    return static_cast<float>((w >> (8 * r)) & 0xffu);
}

// one stored element of `bytes` bytes as a float: bf16 (the upper half of a
// float), uint8 (an integer 0..255) or float
template <int BYTES>
__device__ __forceinline__ float to_float(const char *ptr)
{
    if constexpr (BYTES == 4) return *reinterpret_cast<const float *>(ptr);
    else if constexpr (BYTES == 2) return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const unsigned short *>(ptr)) << 16);
    else return static_cast<float>(*reinterpret_cast<const unsigned char *>(ptr));
}
template <int BYTES>
__device__ __forceinline__ void copy_elem(char *dst, const char *src)
{
    if constexpr (BYTES == 4) *reinterpret_cast<float *>(dst) = __ldg(reinterpret_cast<const float *>(src));
    else if constexpr (BYTES == 2) *reinterpret_cast<unsigned short *>(dst) = __ldg(reinterpret_cast<const unsigned short *>(src));
    else *reinterpret_cast<unsigned char *>(dst) = __ldg(reinterpret_cast<const unsigned char *>(src));
}

// outer o inner: x -> outer.a + outer.b * (inner.a + inner.b * x)
__device__ __forceinline__ Pair compose(Pair outer, Pair inner)
{
    return Pair{fmaf(outer.b, inner.a, outer.a), outer.b * inner.b};
}

constexpr uint32_t kTagAgg = 1u, kTagPrefix = 2u;



// Longest pause between two polls of a predecessor's state (ns); the pause
// starts at 32 ns and doubles.  0: poll without pausing.  An estimator may
// declare its own (LB_NAP_MAX): V-trace polls without pausing (64 rows of
// 2^20 steps 367 -> 363 us; 512 ns cost it 21 %).
#ifndef RLSCAN_LB_NAP_MAX
#define RLSCAN_LB_NAP_MAX 128
#endif
template <class E, class = void>
struct NapOf {
    static constexpr int value = RLSCAN_LB_NAP_MAX;
};
template <class E>
struct NapOf<E, std::void_t<decltype(E::LB_NAP_MAX)>> {
    static constexpr int value = E::LB_NAP_MAX;
};

__device__ __forceinline__ unsigned long long pack_word(uint32_t tag, float v)
{
    return (static_cast<unsigned long long>(tag) << 32) | __float_as_uint(v);
}

__device__ __forceinline__ void record_error(const Params &p, uint32_t code, uint32_t detail)
{
    if (p.hdr == nullptr) return;
    if (atomicCAS(&p.hdr[kHdrError], 0u, code) == 0u) atomicExch(&p.hdr[kHdrDetail], detail);
}

// Where tile (row, j)'s states sit in the workspace (in units of K states):
// ticket order (j N + row: the tiles in flight together side by side) or
// row-major (row tiles_per_row + j: a row's tiles side by side, so the tiles
// that run together write different cache lines and a tile's predecessors
// share its line).  The predecessor of position q is q - state_step<RM>(p).
// The layout is private to one launch; each estimator takes the one that
// measured faster for it (RowMajorOf), RLSCAN_STATE_ROW_MAJOR = 0 or 1
// forces one for all.
#ifndef RLSCAN_STATE_ROW_MAJOR
#define RLSCAN_STATE_ROW_MAJOR -1
#endif
template <bool RM>
__device__ __forceinline__ int64_t state_pos(const Params &p, int64_t g, int64_t row, int64_t j)
{
    return RM ? row * p.tiles_per_row + j : g;  // ticket g = j N + row
}
template <bool RM>
__device__ __forceinline__ int64_t state_step(const Params &p) { return RM ? 1 : p.N; }

struct TileGeo {
    int64_t row0;  // first row of the tile
    int64_t t0;    // first time step held by the tile
    int64_t j;     // position of the tile within its row, in scan order
    int64_t pos;   // position of the tile's look-back states (state_pos)
    int32_t nrows; // rows present (packed) or 1
    int32_t len;   // time steps present per row
};

// Tile g -> rows and time range.  Packed: rows [g R, g R + R).  Long rows:
// ticket g = j * N + row (all rows' j-th tiles before any (j+1)-th tile);
// j counts tiles in scan order (from t = T-1 backward, from t = 0 forward).
template <bool FWD, int TILE, bool RM>
__device__ __forceinline__ TileGeo decode_tile(const Params &p, int64_t g)
{
    TileGeo tg;
    if (p.packed) {
        tg.row0 = g * p.R;
        const int64_t rem = p.N - tg.row0;
        tg.nrows = rem < p.R ? static_cast<int32_t>(rem) : p.R;
        tg.t0 = 0;
        tg.len = static_cast<int32_t>(p.T);
        tg.j = 0;
        tg.pos = 0;
    } else {
        tg.j = g / p.N;
        tg.row0 = g - tg.j * p.N;
        const int64_t chrono = FWD ? tg.j : (p.tiles_per_row - 1 - tg.j);
        tg.t0 = chrono * TILE;
        const int64_t rem = p.T - tg.t0;
        tg.len = rem < TILE ? static_cast<int32_t>(rem) : TILE;
        tg.nrows = 1;
        tg.pos = state_pos<RM>(p, g, tg.row0, tg.j);
    }
    return tg;
}

// Issue the bulk copies of one tile into `stage` (called by one thread).
// Narrow array j occupies region_bytes(j): its data start 16 bytes in, with
// the 16 bytes before the tile in front and the 16 bytes after it behind
// (the neighbour step of a HALO input: copies are whole 16-byte units).
// Wide array w (when staged) follows the narrow arrays and occupies
// (TILE + 4) * words floats: step e of the tile at e * words, the step after
// the tile right behind the last one.
template <class E, int TILE, int AST>
__device__ void issue_tile_copies(const Params &p, const TileGeo &tg, float *stage, uint64_t *bar,
                                  const float *smem_base)
{
    constexpr int NW = WideOf<E>::NWIDE;
    constexpr unsigned DER = WideOf<E>::DERIVED;
    const bool wide = NW > 0 && p.wide_staged;
    float *wsm = stage + narrow_copied<E>() * AST;
    // every copy of the tile as (shared destination, global source, bytes,
    // the source array's base and extent), in issue order
    uint32_t bytes = 0;
    auto each = [&](auto &&f) {
        if (p.packed) {
            bool contig = p.rs == p.T && p.C == p.T;  // rows contiguous in global and in shared memory
#pragma unroll
            for (int w = 0; w < NW; ++w) contig = contig && (!wide || p.wide_rs[w] == p.T * p.wide_words[w]);
            const int copies = contig ? 1 : tg.nrows;
            const int64_t steps = contig ? static_cast<int64_t>(tg.nrows) * p.T : p.T;
            const uint32_t nb = static_cast<uint32_t>(steps * 4);
            for (int i = 0; i < copies; ++i) {
#pragma unroll
                for (int j = 0; j < E::NIN; ++j) {
                    if (!((DER >> j) & 1u)) {
                        const int eb = IoOf<E>::in(j);
                        f(elem0<E, TILE>(stage, j) + static_cast<int64_t>(i) * p.C * eb,
                          reinterpret_cast<const char *>(p.in[j]) + (tg.row0 + i) * p.rs * eb,
                          static_cast<uint32_t>(steps * eb), p.in[j], array_extent(p, eb));
                    }
                }
                if (wide) {
                    float *dst = wsm;
#pragma unroll
                    for (int w = 0; w < NW; ++w) {
                        const int W = p.wide_words[w];
                        f(reinterpret_cast<char *>(dst + static_cast<int64_t>(i) * p.C * W),
                          reinterpret_cast<const char *>(static_cast<const float *>(p.wide[w]) +
                                                         (tg.row0 + i) * p.wide_rs[w]),
                          nb * static_cast<uint32_t>(W), p.wide[w], wide_extent(p, w));
                        dst += (TILE + 4) * W;
                    }
                }
            }
            return;
        }
        const int64_t base = tg.row0 * p.rs;
#pragma unroll
        for (int j = 0; j < E::NIN; ++j) {
            const int halo = 16 / IoOf<E>::in(j);  // steps in 16 bytes
            int64_t lo = tg.t0, hi = tg.t0 + tg.len;
            if ((E::HALO >> j) & 1u) {
                if (!E::FWD && hi < p.T) hi += halo;   // next step (T a multiple of halo keeps it in the row)
                if (E::FWD && lo > 0) lo -= halo;      // previous step
            }
            if (!((DER >> j) & 1u)) {
                const int eb = IoOf<E>::in(j);
                f(elem0<E, TILE>(stage, j) + (lo - tg.t0) * eb,
                  reinterpret_cast<const char *>(p.in[j]) + (base + lo) * eb, static_cast<uint32_t>((hi - lo) * eb),
                  p.in[j], array_extent(p, eb));
            }
        }
        if (wide) {
            // wide arrays: the tile and, backward, the four steps after it
            const int64_t whi = (!E::FWD && tg.t0 + tg.len < p.T) ? tg.t0 + tg.len + 4 : tg.t0 + tg.len;
            float *dst = wsm;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const int W = p.wide_words[w];
                f(reinterpret_cast<char *>(dst),
                  reinterpret_cast<const char *>(static_cast<const float *>(p.wide[w]) + tg.row0 * p.wide_rs[w] +
                                                 tg.t0 * W),
                  static_cast<uint32_t>((whi - tg.t0) * 4 * W), p.wide[w], wide_extent(p, w));
                dst += (TILE + 4) * W;
            }
        }
    };
    bool ok = true;
    each([&](char *dst, const char *src, uint32_t n, const void *base, uint64_t extent) {
        bytes += n;
        if constexpr (RLSCAN_CHECK_BOUNDS) {
            const bool src_ok = span_ok(p, base, extent, src, n, kSiteCopySource);
            ok = smem_ok(p, smem_base, dst, n, kSiteCopyTarget) && src_ok && ok;
        }
    });
    if (!ok) {  // checked build: no copy of this tile is issued; the phase completes without data
        ptx::mbar_arrive(bar);
        return;
    }
    ptx::mbar_arrive_expect_tx(bar, bytes);
    each([&](char *dst, const char *src, uint32_t n, const void *, uint64_t) { ptx::bulk_g2s(dst, src, n, bar); });
}

// Element e of array j's tile region (e = -1: the step before the tile,
// e = TILE: the step after it) from global element `src`.
template <class E, int TILE>
__device__ __forceinline__ void load_elem(const Params &p, float *stage, int j, int e, int64_t src)
{
    const int eb = IoOf<E>::in(j);
    char *dst = elem0<E, TILE>(stage, j) + static_cast<int64_t>(e) * eb;
    const char *from = reinterpret_cast<const char *>(p.in[j]) + src * eb;
    if (!span_ok(p, p.in[j], array_extent(p, eb), from, eb, kSiteElementLoad)) return;
    if (eb == 4) copy_elem<4>(dst, from);
    else if (eb == 2) copy_elem<2>(dst, from);
    else copy_elem<1>(dst, from);
}

// Element-wise cooperative load of one tile (any alignment), same layout.
template <class E, int TILE, int AST>
__device__ void load_tile_elementwise(const Params &p, const TileGeo &tg, float *stage, int nthreads)
{
    constexpr unsigned DER = WideOf<E>::DERIVED;
    const int total = tg.nrows * p.C;
    for (int e = threadIdx.x; e < total; e += nthreads) {
        const int i = e / p.C;
        const int c = e - i * p.C;
        if (c < tg.len) {
            const int64_t src = (tg.row0 + i) * p.rs + tg.t0 + c;
#pragma unroll
            for (int j = 0; j < E::NIN; ++j)
                if (!((DER >> j) & 1u)) load_elem<E, TILE>(p, stage, j, e, src);
        }
    }
    if (!p.packed) {
        const int64_t base = tg.row0 * p.rs;
#pragma unroll
        for (int j = 0; j < E::NIN; ++j) {
            if (threadIdx.x == j && (((E::HALO & ~DER) >> j) & 1u)) {
                if (!E::FWD && tg.t0 + tg.len < p.T) load_elem<E, TILE>(p, stage, j, TILE, base + tg.t0 + tg.len);
                if (E::FWD && tg.t0 > 0) load_elem<E, TILE>(p, stage, j, -1, base + tg.t0 - 1);
            }
        }
    }
}

__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t start = ptx::globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((n & 31u) == 0 && ptx::globaltimer_ns() - start > limit_ns) return false;
    }
}

// Decoupled look-back.  Tile g holds one 16-byte state per scan it solves
// (K of them, slot g * K + scan): two 64-bit words, each a 32-bit tag
// (call epoch << 2 | kind) beside a float payload.  The epoch is a counter
// in the workspace header: every CTA reads it at start, the last CTA out
// advances it, so the next call on the workspace (a stream-ordered launch,
// or a replay of a captured graph) sees the states of this one as stale.
//
// Publishing side (one thread per tile and scan): the tile's aggregate map
// `total`, or directly its inclusive value when that does not depend on
// anything before the tile (first tile of the row, or b == 0).
template <int K>
__device__ __forceinline__ void publish_first(const Params &p, uint32_t epoch, int64_t slot, int64_t g,
                                              int64_t j, Pair total)
{
    if (g == p.withhold_tile) return;  // test hook: successors must time out
    unsigned long long *st = p.states;
    if (!state_ok(p, 2 * slot + 1, K)) return;
    if (j == 0 || total.b == 0.f) {
        ptx::st_relaxed(&st[2 * slot], pack_word((epoch << 2) | kTagPrefix, total.a));
    } else {
        ptx::st_relaxed(&st[2 * slot + 1], pack_word((epoch << 2) | kTagAgg, total.b));
        ptx::st_relaxed(&st[2 * slot], pack_word((epoch << 2) | kTagAgg, total.a));
    }
}

template <int K>
__device__ __forceinline__ void publish_inclusive(const Params &p, uint32_t epoch, int64_t slot, int64_t g,
                                                  float v)
{
    if (g == p.withhold_tile) return;
    if (!state_ok(p, 2 * slot, K)) return;
    ptx::st_relaxed(&p.states[2 * slot], pack_word((epoch << 2) | kTagPrefix, v));
}

// Reading side (one thread per warp and scan): the value entering tile g
// (state position pos, position j > 0 of its row) from its scan-order
// predecessor, i.e. A at the step just outside the tile, for scan `sc` of K.
// (w0, w1) are the predecessor's state words as fetched earlier.  Walks back
// through aggregates until an inclusive value, a zero decay, or the row's
// first tile; every wait is bounded.
template <int K, bool RM, int NAP>
__device__ inline float lookback_read(const Params &p, uint32_t epoch, int64_t g, int64_t pos, int64_t j, int sc,
                                      unsigned long long w0, unsigned long long w1)
{
    const unsigned long long *st = p.states;
    const uint32_t tagA = (epoch << 2) | kTagAgg;
    const uint32_t tagP = (epoch << 2) | kTagPrefix;
    Pair acc{0.f, 1.f};
    const int64_t step = state_step<RM>(p);
    int64_t k = pos - step;  // state position of the tile being read
    int64_t left = j;  // predecessors not yet folded in
    uint64_t waited_since = 0;
    uint32_t nap = 32;
    bool fresh = true;  // (w0, w1) hold a probe of tile k
    for (;;) {
        if (!fresh) {
            if (!state_ok(p, 2 * (k * K + sc) + 1, K)) return __int_as_float(0x7fc00000);
            w0 = ptx::ld_relaxed(&st[2 * (k * K + sc)]);
            w1 = ptx::ld_relaxed(&st[2 * (k * K + sc) + 1]);
        }
        fresh = false;
        const uint32_t tag = static_cast<uint32_t>(w0 >> 32);
        if (tag == tagP) return fmaf(acc.b, __uint_as_float(static_cast<uint32_t>(w0)), acc.a);
        if (tag == tagA && static_cast<uint32_t>(w1 >> 32) == tagA) {
            acc = compose(acc, Pair{__uint_as_float(static_cast<uint32_t>(w0)),
                                    __uint_as_float(static_cast<uint32_t>(w1))});
            if (acc.b == 0.f || --left == 0) return acc.a;
            k -= step;
            waited_since = 0;
            nap = 32;
            continue;
        }
        const uint64_t now = ptx::globaltimer_ns();
        if (waited_since == 0) {
            waited_since = now;
        } else if (now - waited_since > p.spin_limit_ns) {
            record_error(p, RLSCAN_ERR_TIMEOUT, static_cast<uint32_t>(g));
            return __int_as_float(0x7fc00000);
        }
        if (NAP > 0) {
            __nanosleep(nap);
            if (nap < NAP) nap <<= 1;
        }
    }
}

template <bool FWD>
__device__ __forceinline__ Pair shfl_pred(Pair v, int off)
{
    Pair o;
    if (FWD) {
        o.a = __shfl_up_sync(0xffffffffu, v.a, off);
        o.b = __shfl_up_sync(0xffffffffu, v.b, off);
    } else {
        o.a = __shfl_down_sync(0xffffffffu, v.a, off);
        o.b = __shfl_down_sync(0xffffffffu, v.b, off);
    }
    return o;
}

// Inclusive warp scan in scan order: lane l ends with f_l o f_{pred} o ...
template <bool FWD>
__device__ __forceinline__ Pair warp_inclusive(Pair v, int lane)
{
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const Pair o = shfl_pred<FWD>(v, off);
        const bool has = FWD ? (lane >= off) : (lane + off < 32);
        if (has) v = compose(v, o);
    }
    return v;
}

template <bool FWD>
__device__ __forceinline__ Pair warp_exclusive_from(Pair inc, int lane)
{
    Pair ex = shfl_pred<FWD>(inc, 1);
    if (FWD ? (lane == 0) : (lane == 31)) ex = Pair{0.f, 1.f};
    return ex;
}

// Where this thread's ITEMS steps sit in a tile: number of valid steps (kv)
// and the index of the row's boundary step within the range (kb; -1 if
// none).  `col` is the thread's first column within the tile's row segment.
struct ThreadSpan {
    int kv, kb;
};

template <bool FWD, int ITEMS>
__device__ __forceinline__ ThreadSpan thread_span(const Params &p, const TileGeo &tg, int rit, int col)
{
    ThreadSpan sp;
    const bool row_ok = rit < tg.nrows;
    const int rem = tg.len - col;
    sp.kv = row_ok ? (rem < 0 ? 0 : (rem > ITEMS ? ITEMS : rem)) : 0;
    sp.kb = -1;
    // only a packed tile or a row's first tile in scan order holds the boundary
    if (row_ok && (p.packed || tg.j == 0)) {
        const int d = FWD ? -col : (tg.len - 1 - col);
        if (d >= 0 && d < ITEMS) sp.kb = d;
    }
    return sp;
}

// Block = THREADS compute threads + one producer warp.
template <int THREADS>
constexpr int block_threads() { return THREADS + 32; }
#ifndef RLSCAN_MIN_BLOCKS
#define RLSCAN_MIN_BLOCKS 3
#endif
// Two scans need more registers: three CTAs per SM at four steps per
// thread, two at eight (four for a small 128-thread CTA); two CTAs per SM is
// the most the wide stages leave room for, and what compact-storage
// estimators with four or more inputs get at eight steps per thread
// (their staged inputs unpack into many registers).
#ifndef RLSCAN_LOWP_BLOCKS
#define RLSCAN_LOWP_BLOCKS 2
#endif
#ifndef RLSCAN_K2_SHORT_BLOCKS
#define RLSCAN_K2_SHORT_BLOCKS 3
#endif
// 1: in immediate-finish kernels each warp releases its share of a ring
// slot as soon as its inputs are in registers (0: after the tile's warp scans)
#ifndef RLSCAN_EARLY_RELEASE
#define RLSCAN_EARLY_RELEASE 1
#endif
// Look-back window of the deferred kernels of chain estimators: lanes
// 0..W-1 of every warp fetch the states of the W nearest predecessors when
// the pending tile's finishing iteration starts, and the walk composes them
// with a shuffle reduction (one round trip, already in flight, instead of a
// chain of dependent loads); it falls back to the serial walk when the
// window holds no resolved value.  0: off.  RLSCAN_LB_WINDOW_ALL=1 applies
// it to every single-scan estimator.
#ifndef RLSCAN_LB_WINDOW
#define RLSCAN_LB_WINDOW 8
#endif
#ifndef RLSCAN_LB_WINDOW_ALL
#define RLSCAN_LB_WINDOW_ALL 0
#endif
// Start-up: the barriers are initialised (and made visible) before the
// wait for the previous kernel, so the producer issues its first copies as
// soon as that wait ends (1; 0: one block-wide barrier after the wait).
// Measured: 0.3-1.3 % on every kernel, the short ones most.
#ifndef RLSCAN_EARLY_START
#define RLSCAN_EARLY_START 1
#endif
// Where a CTA counts itself out of a dynamic launch: right after its
// producer's last ticket draw (1), or at the end of the kernel after a block
// barrier and a fence (0).
#ifndef RLSCAN_EARLY_EXIT_COUNT
#define RLSCAN_EARLY_EXIT_COUNT 1
#endif
// 1: bf16 inputs at 8 steps per thread take their neighbour step by a
// shuffle too (0: a 2-byte shared-memory read with its bank conflicts)
#ifndef RLSCAN_HALO_SHFL_NARROW
#define RLSCAN_HALO_SHFL_NARROW 0
#endif
// 1: the swapped float32 reads at 8 steps per thread (0: plain reads with
// their two-way conflicts; measured 4-5 % slower on 2^20-step rows)
#ifndef RLSCAN_F32_SWAP
#define RLSCAN_F32_SWAP 1
#endif
// Deferred kernels fetch the pending tile's predecessor states when the
// next tile's data has landed, or, for estimators that declare LB_LATE,
// after the next tile's warp scans (fresher: eligibility traces, whose
// predecessors publish their inclusive values at once, 137.9 -> 134.9 us on
// 64 rows of 2^20 steps; later or earlier cost the others 1-10 %).
template <class E, class = void>
struct LateOf {
    static constexpr bool value = false;
};
template <class E>
struct LateOf<E, std::void_t<decltype(E::LB_LATE)>> {
    static constexpr bool value = E::LB_LATE;
};
#ifndef RLSCAN_DEFER_MIN_BLOCKS
#define RLSCAN_DEFER_MIN_BLOCKS 0  // 0: as the immediate-finish kernel
#endif
// Resident CTAs the 128-thread short-row kernels are compiled for (their
// register budget): 4 measured best (GAE 4096 x 1024 13.35 -> 13.06 us; 5
// and 6 lost on discounted returns and TD(lambda)).
#ifndef RLSCAN_SHORT_MIN_BLOCKS
#define RLSCAN_SHORT_MIN_BLOCKS 4
#endif
template <class E, bool DEFER, int THREADS, int ITEMS>
constexpr int min_blocks()
{
    return (DEFER && RLSCAN_DEFER_MIN_BLOCKS > 0) ? RLSCAN_DEFER_MIN_BLOCKS
           : (THREADS <= 128 && E::K == 1 && WideOf<E>::NWIDE == 0) ? RLSCAN_SHORT_MIN_BLOCKS
           : WideOf<E>::NWIDE > 0 ? 2
           : (IoOf<E>::LOWP && E::NIN >= 4 && ITEMS >= 8) ? RLSCAN_LOWP_BLOCKS
           : (E::K > 1) ? (ITEMS <= 4 ? RLSCAN_K2_SHORT_BLOCKS : (THREADS <= 128 && !DEFER ? 4 : 2))
           : RLSCAN_MIN_BLOCKS;
}

template <class E, int THREADS, int ITEMS, int STAGES, bool DEFER>
__global__ void __launch_bounds__(block_threads<THREADS>(), min_blocks<E, DEFER, THREADS, ITEMS>())
scan_kernel(const __grid_constant__ Params p)
{
    constexpr int NIN = E::NIN, NOUT = E::NOUT, K = E::K;
    constexpr int TILE = THREADS * ITEMS, AST = TILE + 8, WARPS = THREADS / 32;
    constexpr bool FWD = E::FWD;
    static_assert(K >= 1 && K <= kMaxScans, "scans per step");
    constexpr int PUB_WARP = FWD ? WARPS - 1 : 0;   // warp holding the tile's last element in scan order
    constexpr int COMPUTE_BAR = 1;                  // named barrier of the compute warps
    static_assert(STAGES >= 2, "the ring needs two stages");
    static_assert(ITEMS % 4 == 0, "items per thread are moved as float4");
    static_assert(TILE >= kSmallestTile && K * (TILE >= kMinTile ? 1 : kMinTile / TILE) <= kMaxScans,
                  "the workspace holds kMaxScans states per 1024 steps");
    constexpr int NWIDE = WideOf<E>::NWIDE;
    constexpr int LBW = (DEFER && K == 1 && (ChainOf<E>::value || RLSCAN_LB_WINDOW_ALL)) ? RLSCAN_LB_WINDOW : 0;
    constexpr bool RM = RLSCAN_STATE_ROW_MAJOR < 0 ? RowMajorOf<E>::value : RLSCAN_STATE_ROW_MAJOR != 0;
    constexpr int LBNAP = NapOf<E>::value;
    constexpr bool LBLATE = LateOf<E>::value;
    static_assert(LBW >= 0 && LBW <= 32, "look-back window: at most one warp of states");
    static_assert(NWIDE == 0 || !FWD, "wide inputs are staged for backward recurrences only");

    extern __shared__ __align__(128) float smem[];
    __shared__ __align__(8) uint64_t full_bar[STAGES];   // stage data (and tile id) ready
    __shared__ __align__(8) uint64_t meta_bar[STAGES];   // tile id and geometry recorded
    __shared__ __align__(8) uint64_t empty_bar[STAGES];  // every compute warp is done reading it
    __shared__ int64_t tile_ids[STAGES];
    __shared__ TileGeo s_geo[STAGES];
    __shared__ Pair wagg[2][WARPS][K];  // warp aggregates per scan, double-buffered by tile parity

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const bool tma = p.tma != 0;
    const bool vec = p.vec != 0;
    static_assert(!(IoOf<E>::LOWP && NWIDE > 0), "wide inputs are float only");
    const int SST = NWIDE > 0 ? p.stage_floats : narrow_bytes<E, TILE>() / 4;  // floats per ring stage
    constexpr int NST = STAGES;                                // ring stages
    static_assert(!DEFER || STAGES >= 3, "a deferred tile holds its stage: the ring needs three");

    ptx::pdl_trigger_dependents();
    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full_bar[s], 1);
            ptx::mbar_init(&meta_bar[s], 1);
            ptx::mbar_init(&empty_bar[s], WARPS);
        }
        ptx::fence_mbar_init();
    }
    __shared__ uint32_t s_epoch;
    if (RLSCAN_EARLY_START) {
        // the barriers are initialised while the previous kernel drains; after
        // the wait the producer issues its first copies at once, and only the
        // compute warps meet to share the epoch
        __syncthreads();
        ptx::pdl_wait_prerequisites();
        if (warp < WARPS) {
            if (tid == 0) s_epoch = p.dynamic ? (ptx::ld_relaxed_u32(&p.hdr[kHdrEpoch]) & 0x3FFFFFFFu) : 0u;
            ptx::named_barrier(1, THREADS);
        }
    } else {
        // nothing global is touched before the previous kernel has completed
        ptx::pdl_wait_prerequisites();
        if (tid == 0) s_epoch = p.dynamic ? (ptx::ld_relaxed_u32(&p.hdr[kHdrEpoch]) & 0x3FFFFFFFu) : 0u;
        __syncthreads();
    }
    const uint32_t epoch = warp < WARPS ? s_epoch : 0u;  // tag of this call's tile states (compute warps)

    if (warp == WARPS) {
        // Producer (lane 0 of the extra warp): for ring slot s of iteration
        // it, wait until every compute warp has released the slot (iteration
        // it - STAGES), draw the next ticket, record the tile and start its copies.  An
        // exhausted ticket completes the slot's phase without data, which
        // tells the compute warps to stop.  Tickets are drawn just before
        // their copies can start, so tiles are processed in close to ticket
        // order.
        if (lane == 0) {
            int64_t static_next = blockIdx.x;
            for (int it = 0;; ++it) {
                const int s = it % NST;
                if (it >= NST &&
                    !wait_phase(&empty_bar[s], static_cast<uint32_t>((it / NST - 1) & 1),
                                p.spin_limit_ns + p.copy_limit_ns))
                    record_error(p, RLSCAN_ERR_TIMEOUT, 0x40000000u | static_cast<uint32_t>(s));
                int64_t g;
                if (static_next < p.static_tiles || !p.dynamic) {
                    g = static_next;
                    static_next += gridDim.x;
                } else {
                    g = p.static_tiles +
                        static_cast<int64_t>(atomicAdd(reinterpret_cast<unsigned long long *>(p.hdr), 1ull));
                }
                tile_ids[s] = g;
                if (g >= p.num_tiles) {
                    ptx::mbar_arrive(&meta_bar[s]);
                    ptx::mbar_arrive(&full_bar[s]);
                    // Every ticket this CTA draws has been drawn (the draw that
                    // just returned g is performed): count this CTA out.  The
                    // last one re-arms the ticket and advances the epoch for
                    // the next call on the workspace (whose CTAs read them only
                    // after this kernel has completed); this call's CTAs keep
                    // the epoch they read at start.  Done here, a tile or two
                    // before the CTA's compute ends, the round trips stay off
                    // the kernel's end.
                    if (RLSCAN_EARLY_EXIT_COUNT && p.dynamic) {
                        const uint32_t done = atomicAdd(&p.hdr[kHdrExit], 1u);
                        if (done == gridDim.x - 1) {
                            atomicExch(reinterpret_cast<unsigned long long *>(p.hdr), 0ull);
                            atomicExch(&p.hdr[kHdrExit], 0u);
                            atomicAdd(&p.hdr[kHdrEpoch], 1u);
                        }
                    }
                    break;
                }
                const TileGeo tg = decode_tile<FWD, TILE, RM>(p, g);
                s_geo[s] = tg;
                ptx::mbar_arrive(&meta_bar[s]);  // the tile is known before its data lands
                if (tma) issue_tile_copies<E, TILE, AST>(p, tg, smem + s * SST, &full_bar[s], smem);
                else ptx::mbar_arrive(&full_bar[s]);
            }
        }
    } else {

    const int li = tid * ITEMS;
    const int rit = p.packed ? li / p.C : 0;
    const int col = p.packed ? li - rit * p.C : li;

    // Row scalar of this thread's row when the row's boundary step falls in
    // its range.  Fetched as soon as its tile is known (the slot's meta phase
    // has completed; its data may still be in flight): for the next tile when
    // a tile starts, else for this tile before waiting for its data, so the
    // load's latency never holds the tile (one thread's wait would hold the
    // whole CTA at the tile's barrier).
    auto load_row_scalar = [&](int s) -> float {
        if (tile_ids[s] >= p.num_tiles) return 0.f;
        const TileGeo tg = s_geo[s];
        if (thread_span<FWD, ITEMS>(p, tg, rit, col).kb < 0) return 0.f;
        const float *rs_ptr = p.rowscalar + (tg.row0 + rit) * p.rowscalar_stride;
        const uint64_t rs_ext = static_cast<uint64_t>((p.check_rows - 1) * p.rowscalar_stride + 1) * 4u;
        if (!span_ok(p, p.rowscalar, rs_ext, rs_ptr, 4, kSiteRowScalar)) return 0.f;
        return __ldg(rs_ptr);
    };
    constexpr bool kRowScalar = E::ROWSCALAR;
    const bool use_rsc = kRowScalar && p.rowscalar != nullptr;
    float rsc_next = 0.f;
    bool rsc_ready = false;
    uint32_t lost_stages = 0, lost_parity = 0;  // waits that timed out (thread 0)

    using Keep = typename E::template Keep<ITEMS>;
    constexpr bool MOM = MomentsOf<E>::value;
    // this thread's share of the batch moments: a float sum per tile, carried
    // across tiles (and combined across the CTA and the grid) as float pairs
    DF mom_s{0.f, 0.f}, mom_q{0.f, 0.f};

    // inputs of this thread's ITEMS steps, plus the neighbour step
    auto load_inputs = [&](const float *stage, float (&x)[NIN][ITEMS], float (&xn)[NIN]) {
#pragma unroll
        for (int j = 0; j < NIN; ++j) {
            const int eb = IoOf<E>::in(j);
            const char *aj = elem0<E, TILE>(stage, j) + li * eb;
            // four consecutive steps of array j from `q` (one 16-, 8- or
            // 4-byte shared-memory load): float32, bf16 (a float's upper 16
            // bits each) or uint8
            auto load4 = [&](const char *q, float (&v)[4]) {
                if (eb == 4) {
                    const float4 w = *reinterpret_cast<const float4 *>(q);
                    v[0] = w.x;
                    v[1] = w.y;
                    v[2] = w.z;
                    v[3] = w.w;
                } else if (eb == 2) {
                    const uint2 w = *reinterpret_cast<const uint2 *>(q);
                    v[0] = __uint_as_float(w.x << 16);
                    v[1] = __uint_as_float(w.x & 0xffff0000u);
                    v[2] = __uint_as_float(w.y << 16);
                    v[3] = __uint_as_float(w.y & 0xffff0000u);
                } else {
                    const uint32_t w = *reinterpret_cast<const uint32_t *>(q);
#pragma unroll
                    for (int r = 0; r < 4; ++r) v[r] = u8_to_float(w, r);
                }
            };
            if constexpr (ITEMS == 8) {
                if (eb == 2) {  // eight bf16 in one 16-byte load (lanes 16 bytes apart: conflict-free)
                    const uint4 w = *reinterpret_cast<const uint4 *>(aj);
                    const uint32_t h[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        x[j][2 * q] = __uint_as_float(h[q] << 16);
                        x[j][2 * q + 1] = __uint_as_float(h[q] & 0xffff0000u);
                    }
                } else if (eb == 1) {  // eight uint8 in one 8-byte load (conflict-free)
                    const uint2 w = *reinterpret_cast<const uint2 *>(aj);
                    const uint32_t h[2] = {w.x, w.y};
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
#pragma unroll
                        for (int r = 0; r < 4; ++r) x[j][4 * q + r] = u8_to_float(h[q], r);
                    }
                } else {
                    // Two 16-byte chunks per thread: consecutive lanes' first
                    // chunks lie 2 chunks apart, so in one shared-memory
                    // wavefront (8 lanes of 16-byte loads) lanes l and l + 4
                    // would hit the same banks.  Lanes 4..7 of each group of 8
                    // read their second chunk first (two-way conflicts gone),
                    // then the chunks are put back in order.
                    const bool sw = RLSCAN_F32_SWAP && ((lane >> 2) & 1) != 0;
                    float c0[4], c1[4];
                    load4(aj + (sw ? 16 : 0), c0);
                    load4(aj + (sw ? 0 : 16), c1);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        x[j][q] = sw ? c1[q] : c0[q];
                        x[j][q + 4] = sw ? c0[q] : c1[q];
                    }
                }
            } else {
#pragma unroll
                for (int k = 0; k < ITEMS; k += 4) {
                    float v[4];
                    load4(aj + k * eb, v);
#pragma unroll
                    for (int q = 0; q < 4; ++q) x[j][k + q] = v[q];
                }
            }
            float nb = 0.f;
            if ((E::HALO >> j) & 1u) {
                const char *q = FWD ? aj - eb : aj + ITEMS * eb;
                if (ITEMS == 8 && (eb == 4 || (RLSCAN_HALO_SHFL_NARROW && eb == 2))) {
                    // the neighbour step is the adjacent lane's last (forward)
                    // or first (backward) step: a shuffle, and a shared-memory
                    // read only at the warp's edge (lanes 32 bytes apart
                    // reading one float each would be an 8-way bank conflict);
                    // at 4 steps per thread or narrower types the read's
                    // smaller conflict measured cheaper than the shuffle
                    nb = FWD ? __shfl_up_sync(0xffffffffu, x[j][ITEMS - 1], 1)
                             : __shfl_down_sync(0xffffffffu, x[j][0], 1);
                    if (lane == (FWD ? 0 : 31)) nb = eb == 4 ? to_float<4>(q) : to_float<2>(q);
                } else {
                    nb = eb == 4 ? to_float<4>(q) : (eb == 2 ? to_float<2>(q) : to_float<1>(q));
                }
            }
            xn[j] = nb;
        }
    };

    // coefficients of the thread's steps: the row's boundary values folded
    // in (and the recurrence severed) there, the identity map outside the data
    auto make_coeffs = [&](const float (&x)[NIN][ITEMS], const float (&xn)[NIN], const ThreadSpan &sp, float rsc,
                           float (&a)[K][ITEMS], float (&b)[K][ITEMS], Keep &keep) {
        const bool edge = sp.kb >= 0 || sp.kv < ITEMS;
        if (!edge) {
            E::template coeffs<ITEMS, false>(x, xn, -1, p, rsc, a, b, keep);
            return;
        }
        E::template coeffs<ITEMS, true>(x, xn, sp.kb, p, rsc, a, b, keep);
#pragma unroll
        for (int k = 0; k < ITEMS; ++k) {
            if (k == sp.kb) {
                float bv[K];
                E::template boundary<ITEMS>(x, k, rsc, p, bv);
#pragma unroll
                for (int sc = 0; sc < K; ++sc) {
                    a[sc][k] = fmaf(b[sc][k], bv[sc], a[sc][k]);
                    b[sc][k] = 0.f;
                }
            }
            if (k >= sp.kv) {
#pragma unroll
                for (int sc = 0; sc < K; ++sc) {
                    a[sc][k] = 0.f;
                    b[sc][k] = 1.f;
                }
            }
        }
    };

    // serial recurrence of each scan from its exact incoming value, the
    // estimator's outputs, and the stores
    auto finish = [&](const float (&x)[NIN][ITEMS], const float (&xn)[NIN], const float (&a)[K][ITEMS],
                      const float (&b)[K][ITEMS], const Keep &keep, const ThreadSpan &sp, const TileGeo &tg,
                      float rsc, const float (&x_in)[K]) {
        float A[K][ITEMS];
#pragma unroll
        for (int sc = 0; sc < K; ++sc) {
            float v = x_in[sc];
            if (FWD) {
#pragma unroll
                for (int k = 0; k < ITEMS; ++k) {
                    v = fmaf(b[sc][k], v, a[sc][k]);
                    A[sc][k] = v;
                }
            } else {
#pragma unroll
                for (int k = ITEMS - 1; k >= 0; --k) {
                    v = fmaf(b[sc][k], v, a[sc][k]);
                    A[sc][k] = v;
                }
            }
        }
        float o[NOUT][ITEMS];
        const bool edge = sp.kb >= 0 || sp.kv < ITEMS;
        if (!edge) E::template post<ITEMS, false>(x, xn, -1, p, rsc, A, x_in, keep, o);
        else E::template post<ITEMS, true>(x, xn, sp.kb, p, rsc, A, x_in, keep, o);
        if constexpr (MOM) {  // this tile's share of the batch moments of output 0
            float s1 = 0.f, s2 = 0.f;
#pragma unroll
            for (int k = 0; k < ITEMS; ++k) {
                if (k < sp.kv) {
                    s1 += o[0][k];
                    s2 = fmaf(o[0][k], o[0][k], s2);
                }
            }
            mom_s = df_add(mom_s, DF{s1, 0.f});
            mom_q = df_add(mom_q, DF{s2, 0.f});
        }
        if (sp.kv > 0) {
            const int64_t off = (tg.row0 + rit) * p.rs + tg.t0 + col;
#pragma unroll
            for (int q = 0; q < NOUT; ++q) {
                if (NOUT > 1 && p.out[q] == nullptr) continue;  // optional output
                if constexpr (IoOf<E>::OUT == 2) {  // bf16, rounded to nearest even
                    __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.out[q]) + off;
                    if (vec) {
#pragma unroll
                        for (int k = 0; k < ITEMS; k += 4) {
                            if (k < sp.kv) {
                                const __nv_bfloat162 lo2 = __floats2bfloat162_rn(o[q][k], o[q][k + 1]);
                                const __nv_bfloat162 hi2 = __floats2bfloat162_rn(o[q][k + 2], o[q][k + 3]);
                                uint2 w;
                                w.x = *reinterpret_cast<const uint32_t *>(&lo2);
                                w.y = *reinterpret_cast<const uint32_t *>(&hi2);
                                if (span_ok(p, p.out[q], array_extent(p, 2), dst + k, 8, kSiteStore))
                                    *reinterpret_cast<uint2 *>(dst + k) = w;
                            }
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < ITEMS; ++k)
                            if (k < sp.kv && span_ok(p, p.out[q], array_extent(p, 2), dst + k, 2, kSiteStore))
                                dst[k] = __float2bfloat16_rn(o[q][k]);
                    }
                } else if (vec) {
#pragma unroll
                    for (int k = 0; k < ITEMS; k += 4) {
                        if (k < sp.kv && span_ok(p, p.out[q], array_extent(p, 4), p.out[q] + off + k, 16, kSiteStore))
                            *reinterpret_cast<float4 *>(p.out[q] + off + k) =
                                make_float4(o[q][k], o[q][k + 1], o[q][k + 2], o[q][k + 3]);
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < ITEMS; ++k)
                        if (k < sp.kv && span_ok(p, p.out[q], array_extent(p, 4), p.out[q] + off + k, 4, kSiteStore))
                            p.out[q][off + k] = o[q][k];
                }
            }
        }
    };

    // Value entering a chained tile per scan (lane sc < K walks scan sc from
    // the prefetched predecessor words), broadcast to the warp; the
    // publishing warp then publishes the tile's inclusive values.
    auto carry_in = [&](int64_t g, int64_t pos, int64_t j, const Pair (&total)[K], unsigned long long w0,
                        unsigned long long w1, float (&carry)[K]) {
        float mine = 0.f;
        if (lane < K) mine = lookback_read<K, RM, LBNAP>(p, epoch, g, pos, j, lane, w0, w1);
#pragma unroll
        for (int sc = 0; sc < K; ++sc) carry[sc] = __shfl_sync(0xffffffffu, mine, sc);
        if (warp == PUB_WARP && lane == 0) {
#pragma unroll
            for (int sc = 0; sc < K; ++sc)
                if (total[sc].b != 0.f)
                    publish_inclusive<K>(p, epoch, pos * K + sc, g, fmaf(total[sc].b, carry[sc], total[sc].a));
        }
    };

    // Windowed variant (chain estimators, deferred tiles, one scan): lane l
    // holds the state words of the tile l + 1 positions back in the row.  The
    // nearest lane with a resolved value (an inclusive value, or an
    // aggregate with b = 0), all lanes before it holding aggregates, gives
    // the carry as the composition of lanes 0..f in order (lane 0 outermost),
    // reduced across the warp; otherwise lane 0 walks serially from its own
    // words (waits, timeouts and NaN as in lookback_read).
    auto carry_in_window = [&](int64_t g, int64_t pos, int64_t j, const Pair (&total)[K], unsigned long long w0,
                               unsigned long long w1, float (&carry)[K]) {
        const uint32_t tagA = (epoch << 2) | kTagAgg;
        const uint32_t tagP = (epoch << 2) | kTagPrefix;
        const int n = j < LBW ? static_cast<int>(j) : LBW;
        const bool in = lane < n;
        const bool isP = in && static_cast<uint32_t>(w0 >> 32) == tagP;
        const bool isA = in && !isP && static_cast<uint32_t>(w0 >> 32) == tagA &&
                         static_cast<uint32_t>(w1 >> 32) == tagA;
        Pair v{0.f, 1.f};
        if (isP) v = Pair{__uint_as_float(static_cast<uint32_t>(w0)), 0.f};
        else if (isA) v = Pair{__uint_as_float(static_cast<uint32_t>(w0)), __uint_as_float(static_cast<uint32_t>(w1))};
        const unsigned resolved = __ballot_sync(0xffffffffu, isP || (isA && v.b == 0.f));
        const unsigned missing = __ballot_sync(0xffffffffu, in && !isP && !isA);
        const int f = __ffs(resolved) - 1;  // nearest resolved lane, -1 if none
        float c;
        if (resolved != 0u && (missing & ((2u << f) - 1u)) == 0u) {
            if (lane > f) v = Pair{0.f, 1.f};
#pragma unroll
            for (int off = 1; off < LBW; off <<= 1) {
                Pair o;
                o.a = __shfl_down_sync(0xffffffffu, v.a, off);
                o.b = __shfl_down_sync(0xffffffffu, v.b, off);
                if (lane + off < 32) v = compose(v, o);
            }
            c = __shfl_sync(0xffffffffu, v.a, 0);
        } else {
            float mine = 0.f;
            if (lane == 0) mine = lookback_read<K, RM, LBNAP>(p, epoch, g, pos, j, 0, w0, w1);
            c = __shfl_sync(0xffffffffu, mine, 0);
        }
        carry[0] = c;
        if (warp == PUB_WARP && lane == 0 && total[0].b != 0.f)
            publish_inclusive<K>(p, epoch, pos * K, g, fmaf(total[0].b, c, total[0].a));
    };

    // Deferred finishing (long rows with several tiles of a row in flight):
    // a tile's look-back, rescan and stores run after the next tile's first
    // half, so the predecessors have had that long to publish.  The pending
    // tile keeps its stage (inputs are re-read from it) until it is done.
    constexpr bool defer = DEFER;
    bool pend = false;
    int ps = 0;
    int64_t pg = 0;
    // state position of the pending tile (its geometry stays in s_geo[ps])
    auto pending_pos = [&]() { return RM ? s_geo[ps].pos : pg; };
    float prsc = 0.f;
    Pair pex[K], pwe[K], ptot[K];
    unsigned long long pw0 = 0, pw1 = 0;
    // the pending tile's geometry stays in s_geo[ps] (and its id in
    // tile_ids[ps]) until its stage is released, as the producer rewrites
    // them only for the slot's next use
    auto finish_pending = [&]() {
        const TileGeo tg = s_geo[ps];
        float carry[K];
#pragma unroll
        for (int sc = 0; sc < K; ++sc) carry[sc] = 0.f;
        if (tg.j > 0) {
            if constexpr (LBW > 0) carry_in_window(pg, pending_pos(), tg.j, ptot, pw0, pw1, carry);
            else carry_in(pg, pending_pos(), tg.j, ptot, pw0, pw1, carry);
        }
        const ThreadSpan sp = thread_span<FWD, ITEMS>(p, tg, rit, col);
        float x[NIN][ITEMS], xn[NIN];
        load_inputs(smem + ps * SST, x, xn);
        float a[K][ITEMS], b[K][ITEMS];
        Keep keep;
        make_coeffs(x, xn, sp, prsc, a, b, keep);
        float x_in[K];
#pragma unroll
        for (int sc = 0; sc < K; ++sc) x_in[sc] = fmaf(pex[sc].b, fmaf(pwe[sc].b, carry[sc], pwe[sc].a), pex[sc].a);
        finish(x, xn, a, b, keep, sp, tg, prsc, x_in);
        if (lane == 0) ptx::mbar_arrive(&empty_bar[ps]);  // the pending tile's stage is free
        pend = false;
    };
    auto prefetch_pending = [&]() {  // nearest predecessor states of the pending tile
        if constexpr (LBW > 0) {  // lane l: the tile l + 1 positions back (one scan)
            pw0 = pw1 = 0ull;
            if (lane < LBW && lane < s_geo[ps].j) {
                const int64_t slot = pending_pos() - static_cast<int64_t>(lane + 1) * state_step<RM>(p);
                if (state_ok(p, 2 * slot + 1, K)) {
                    pw0 = ptx::ld_relaxed(&p.states[2 * slot]);
                    pw1 = ptx::ld_relaxed(&p.states[2 * slot + 1]);
                }
            }
            return;
        }
        if (s_geo[ps].j > 0 && lane < K) {
            const int64_t slot = (pending_pos() - state_step<RM>(p)) * K + lane;
            if (state_ok(p, 2 * slot + 1, K)) {
                pw0 = ptx::ld_relaxed(&p.states[2 * slot]);
                pw1 = ptx::ld_relaxed(&p.states[2 * slot + 1]);
            }
        }
    };

    for (int it = 0;; ++it) {
        const int s = it % NST;
        const uint32_t parity = static_cast<uint32_t>((it / NST) & 1);
        if (!wait_phase(&full_bar[s], parity, p.copy_limit_ns) && tid == 0) {
            lost_stages |= 1u << s;
            lost_parity = (lost_parity & ~(1u << s)) | (parity << s);
            record_error(p, RLSCAN_ERR_TIMEOUT, 0x80000000u | static_cast<uint32_t>(s));
        }
        if (!LBLATE && pend) prefetch_pending();
        const int64_t g = tile_ids[s];
        if (g >= p.num_tiles) break;
        const TileGeo tg = s_geo[s];
        const float rsc = !use_rsc ? 0.f : (rsc_ready ? rsc_next : load_row_scalar(s));
        float *stage = smem + s * SST;
        if constexpr (RLSCAN_CHECK_BOUNDS) smem_ok(p, smem, stage, static_cast<uint64_t>(SST) * 4u, kSiteRing);
        const bool chained = !p.packed && tg.j > 0;  // needs its predecessor's value


        // predecessor states for an immediate look-back (lane sc < K reads
        // scan sc), fetched early so their latency overlaps the tile's work
        unsigned long long cw0 = 0, cw1 = 0;
        if (!defer && chained && lane < K) {
            const int64_t slot = ((RM ? tg.pos : g) - state_step<RM>(p)) * K + lane;
            if (state_ok(p, 2 * slot + 1, K)) {
                cw0 = ptx::ld_relaxed(&p.states[2 * slot]);
                cw1 = ptx::ld_relaxed(&p.states[2 * slot + 1]);
            }
        }

        if (!tma) {
            load_tile_elementwise<E, TILE, AST>(p, tg, stage, THREADS);
            ptx::named_barrier(COMPUTE_BAR, THREADS);
        }
        if constexpr (NWIDE > 0) {  // derive the per-step inputs from the wide arrays
            E::template prepass<TILE, AST, THREADS, COMPUTE_BAR>(p, tg, stage + slot_of<E>(E::PI) * AST,
                                                                 stage + slot_of<E>(E::EQ) * AST,
                                                                 stage + narrow_copied<E>() * AST,
                                                                 tma && p.wide_staged, tid);
            ptx::named_barrier(COMPUTE_BAR, THREADS);
        }

        const ThreadSpan sp = thread_span<FWD, ITEMS>(p, tg, rit, col);
        float x[NIN][ITEMS], xn[NIN];
        load_inputs(stage, x, xn);
        if constexpr (RLSCAN_EARLY_RELEASE && !DEFER) {
            // this warp's inputs are in registers: its share of the slot is free
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&empty_bar[s]);
        }
        float a[K][ITEMS], b[K][ITEMS];
        Keep keep;
        make_coeffs(x, xn, sp, rsc, a, b, keep);

        // per scan: thread aggregate in scan order, warp scan
        Pair ex[K];
        Pair(*wa)[K] = wagg[it & 1];
#pragma unroll
        for (int sc = 0; sc < K; ++sc) {
            Pair agg;
            if (FWD) {
                agg = Pair{a[sc][0], b[sc][0]};
#pragma unroll
                for (int k = 1; k < ITEMS; ++k) agg = compose(Pair{a[sc][k], b[sc][k]}, agg);
            } else {
                agg = Pair{a[sc][ITEMS - 1], b[sc][ITEMS - 1]};
#pragma unroll
                for (int k = ITEMS - 2; k >= 0; --k) agg = compose(Pair{a[sc][k], b[sc][k]}, agg);
            }
            const Pair inc = warp_inclusive<FWD>(agg, lane);
            ex[sc] = warp_exclusive_from<FWD>(inc, lane);
            if (lane == (FWD ? 31 : 0)) wa[warp][sc] = inc;
        }
        if (LBLATE && pend) prefetch_pending();
        ptx::named_barrier(COMPUTE_BAR, THREADS);  // warp aggregates visible
        // every input is in registers: unless the tile is finished later, the slot is free
        if (!RLSCAN_EARLY_RELEASE && !defer && lane == 0) ptx::mbar_arrive(&empty_bar[s]);

        if (use_rsc) {
            const int s1 = (it + 1) % NST;
            rsc_ready = ptx::mbar_test_wait(&meta_bar[s1], static_cast<uint32_t>(((it + 1) / NST) & 1));
            if (rsc_ready) rsc_next = load_row_scalar(s1);
        }

        // map entering this warp's range from the warps before it in scan order
        Pair we[K];
#pragma unroll
        for (int sc = 0; sc < K; ++sc) {
            we[sc] = Pair{0.f, 1.f};
            if (FWD) {
#pragma unroll
                for (int w2 = 0; w2 < WARPS - 1; ++w2)
                    if (w2 < warp) we[sc] = compose(wa[w2][sc], we[sc]);
            } else {
#pragma unroll
                for (int w2 = WARPS - 1; w2 > 0; --w2)
                    if (w2 > warp) we[sc] = compose(wa[w2][sc], we[sc]);
            }
        }
        if (!p.packed && warp == PUB_WARP && lane == 0) {
#pragma unroll
            for (int sc = 0; sc < K; ++sc)
                publish_first<K>(p, epoch, (RM ? tg.pos : g) * K + sc, g, tg.j,
                                 compose(wa[PUB_WARP][sc], we[sc]));
        }

        if (!defer) {
            float carry[K];
#pragma unroll
            for (int sc = 0; sc < K; ++sc) carry[sc] = 0.f;
            if (chained) {
                Pair total[K];
#pragma unroll
                for (int sc = 0; sc < K; ++sc) total[sc] = compose(wa[PUB_WARP][sc], we[sc]);
                carry_in(g, (RM ? tg.pos : g), tg.j, total, cw0, cw1, carry);
            }
            float x_in[K];
#pragma unroll
            for (int sc = 0; sc < K; ++sc) x_in[sc] = fmaf(ex[sc].b, fmaf(we[sc].b, carry[sc], we[sc].a), ex[sc].a);
            finish(x, xn, a, b, keep, sp, tg, rsc, x_in);
        } else {
            if (pend) finish_pending();
            pend = true;
            ps = s;
            pg = g;
            prsc = rsc;
#pragma unroll
            for (int sc = 0; sc < K; ++sc) {
                pex[sc] = ex[sc];
                pwe[sc] = we[sc];
                // the aggregate map, kept for the publishing warp (wagg is
                // reused two tiles later, possibly before this tile is done)
                ptot[sc] = compose(wa[PUB_WARP][sc], we[sc]);
            }
        }
    }
    if (pend) {
        if (LBLATE) prefetch_pending();  // the loop ended before its late fetch
        finish_pending();
    }

    if constexpr (MOM) {
        // CTA total of the moments (float pairs), delivered to this CTA's
        // slot; every block of the normalising pass combines the slots in
        // CTA order after this kernel (the same bits on every call)
        __shared__ DF s_mom[WARPS][2];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            mom_s = df_add(mom_s, df_shfl_down(mom_s, o));
            mom_q = df_add(mom_q, df_shfl_down(mom_q, o));
        }
        if (lane == 0) {
            s_mom[warp][0] = mom_s;
            s_mom[warp][1] = mom_q;
        }
        ptx::named_barrier(COMPUTE_BAR, THREADS);
        if (tid == 0) {
            DF cs{0.f, 0.f}, cq{0.f, 0.f};
            for (int w2 = 0; w2 < WARPS; ++w2) {
                cs = df_add(cs, s_mom[w2][0]);
                cq = df_add(cq, s_mom[w2][1]);
            }
            if (span_ok(p, p.mom_part, kMomentBytes, p.mom_part + 4 * static_cast<int64_t>(blockIdx.x), 16,
                        kSiteMoments))
                *reinterpret_cast<float4 *>(p.mom_part + 4 * static_cast<int64_t>(blockIdx.x)) =
                    make_float4(cs.hi, cs.lo, cq.hi, cq.lo);
        }
    }

    // A copy whose wait timed out may still be landing: give it one more
    // bounded wait before the shared memory is released.
    if (lost_stages != 0 && tid == 0) {
        for (int s2 = 0; s2 < NST; ++s2)
            if ((lost_stages >> s2) & 1u) wait_phase(&full_bar[s2], (lost_parity >> s2) & 1u, p.copy_limit_ns);
    }
    }  // compute warps
    if (!RLSCAN_EARLY_EXIT_COUNT && p.dynamic) {
        __syncthreads();  // every ticket this CTA will draw has been drawn
        if (tid == THREADS) {
            __threadfence();
            const uint32_t done = atomicAdd(&p.hdr[kHdrExit], 1u);
            if (done == gridDim.x - 1) {  // last CTA out: re-arm the ticket, advance the epoch
                atomicExch(reinterpret_cast<unsigned long long *>(p.hdr), 0ull);
                atomicExch(&p.hdr[kHdrExit], 0u);
                atomicAdd(&p.hdr[kHdrEpoch], 1u);
                __threadfence();
            }
        }
    }
}

}  // namespace rlscan
