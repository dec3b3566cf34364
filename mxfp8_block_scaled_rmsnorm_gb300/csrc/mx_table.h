// mx_table.h -- launch descriptor table shared by the C-ABI layer and the
// kernels. One table describes one launch over a list of matrices; it is
// passed by value as a __grid_constant__ kernel parameter (no device-side
// allocation), so it must stay under the 32 KB kernel-parameter limit.
#pragma once

#include <stdint.h>

namespace mx {

// Thread tile: kRows rows x 8 columns (one 16-byte bf16 vector per row). The
// 32 lanes of a warp split into kGroups row groups of kGroupLanes lanes; group
// q takes rows [q * kRows, (q + 1) * kRows) of a 32-row stripe and its lanes
// take consecutive 8-column vectors, so a warp covers 32 rows x kWarpCols
// columns and a CTA covers 32 rows x kChunk columns (one "pass").
template <int ROWS, int CHUNK>
struct TileGeo {
    static constexpr int kRows = ROWS;               // 16 or 8
    static constexpr int kGroups = 32 / ROWS;        // 2 or 4
    static constexpr int kGroupLanes = 32 / kGroups; // 16 or 8 (== kRows)
    static constexpr int kWarpCols = 8 * kGroupLanes;
    static constexpr int kChunk = CHUNK;             // columns of one CTA pass
    static constexpr int kWarps = CHUNK / kWarpCols;
    static constexpr int kThreads = 32 * kWarps;
    static_assert(ROWS == 16 || ROWS == 8, "supported thread tiles");
    static_assert(kGroupLanes == kRows, "row-sum reduce-scatter maps one row per lane");
    static_assert(CHUNK % kWarpCols == 0 && kWarps >= 1 && kWarps <= 32, "whole warps");
};

// The fused kernel holds 8-row tiles (64 registers a thread) in 256-thread
// CTAs over 512-column passes, four CTAs per SM, so that some CTAs load while
// others store and a launch has many small work units (measured against
// 512-thread CTAs over 1024 columns, two per SM: +1.2 % at 32768 x 8192,
// +10 % at 8192 x 4096), with or without a residual input: the residual form
// is held to the same 64 registers (a few bytes spill) because occupancy,
// not register room, bounds it (128-thread CTAs over 256 columns measured 6 %
// slower). The quantize kernel holds 16-row tiles (fewer shuffles, more bytes
// in flight per thread) in 128-thread CTAs, four per SM (+1 % on lists of
// tensors against two 256-thread CTAs).
using FusedGeo = TileGeo<8, 512>;
using QuantGeo = TileGeo<16, 512>;

constexpr int kBlock = 32;                            // MXFP8 block size
// Largest cluster. Sizes above 8 are non-portable and opted into per kernel;
// they keep a CTA's slice (and so the L2 footprint of the pass-2 re-reads) at
// most 2048 columns up to C = 32768.
constexpr int kMaxCluster = 16;
constexpr int kPortableCluster = 8;
// Fused kernel: a CTA takes up to kTargetChunks passes of its row stripe
// (the re-read of the earlier passes is served by L2; four passes per CTA
// with fewer, larger slices measured 6-13 % slower).
constexpr int kTargetChunks = 2;

// One non-empty list entry, with its place in the launch's flattened work.
struct DevDesc {
    const uint16_t* x;
    const uint16_t* gamma;
    uint16_t* normed;
    uint8_t* q_row;
    uint8_t* s_row;
    uint8_t* q_col;
    uint8_t* s_col;
    const uint16_t* res_in;   // fused with residual: added to x (NULL: none)
    uint16_t* res_out;        // fused with residual: x + residual as normalized (NULL: none)
    int64_t rows;
    int64_t cols;
    int64_t unit_begin;  // first flattened work unit of this entry
    float eps;
    float offset;
    int32_t cta_cols;    // fused: columns owned by each CTA of a cluster
    int32_t col_tiles;   // quant: QuantGeo::kWarpCols-column tiles across a row
};

template <int MAXN>
struct Table {
    DevDesc d[MAXN];
    int32_t n;           // live entries (ascending unit_begin)
    int32_t rowwise;
    int32_t columnwise;
    int32_t cluster;     // fused: CTAs per 32-row stripe (cluster size)
    int32_t scale_layout;  // 0: compact; 1: tiled GEMM-operand layout; 2: padded row-major
    int32_t residual;      // fused: entries may carry a residual input / output
    int32_t stage;         // fused, residual: stage residual tiles in shared memory
    int64_t total_units; // fused: stripes; quant: warp tiles
};

// Small lists use a small table so that a launch copies few parameter bytes.
constexpr int kSmallTable = 8;
constexpr int kLargeTable = 256;
static_assert(sizeof(Table<kLargeTable>) < 32000, "kernel parameter limit");

// Launchers (mxfp8_kernels.cu). They return the cudaError_t of the launch.
int launch_fused(const Table<kSmallTable>& t, int64_t grid, void* stream);
int launch_fused(const Table<kLargeTable>& t, int64_t grid, void* stream);
int launch_quant(const Table<kSmallTable>& t, int64_t grid, void* stream);
int launch_quant(const Table<kLargeTable>& t, int64_t grid, void* stream);

// Columns of one CTA pass of the fused kernel (with or without a residual).
int fused_chunk_cols();

// Largest cluster size <= kMaxCluster (above kPortableCluster only where the
// device allows non-portable sizes) that the current device can co-schedule
// for the fused kernel; queried once per device.
int fused_max_cluster();

// CTAs of the fused kernel the current device holds at once (SMs x CTAs per
// SM, from the occupancy calculator); queried once per device, 0 if the query
// fails.
int fused_resident_ctas();

// Status word of the bounds-checking build (always 0 in the normal build),
// read with a synchronizing copy; cleared when asked.
int bounds_status(bool clear, unsigned long long* out);

// Test hooks (mxfp8_set_test_hook, mxfp8_api.cu). hook_launch_error():
// cudaErrorInvalidValue while a launch failure is being injected (every
// launcher returns it before touching the device), else cudaSuccess.
// hook_max_cluster(): a cap on the fused kernel's cluster size, 0 for none.
int hook_launch_error();
int hook_max_cluster();

}  // namespace mx
