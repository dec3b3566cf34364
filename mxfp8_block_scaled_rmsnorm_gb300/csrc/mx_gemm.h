// mx_gemm.h -- launch parameters of the block-scaled MXFP8 GEMM
// (mxfp8_gemm.cu), shared with the C-ABI layer (mxfp8_mm.cu). Passed by value
// as a __grid_constant__ kernel parameter (CUtensorMap carries its own
// 128-byte alignment, which the TMA instructions need).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace mx {

// The general form: 256 x 256 output tiles per CTA pair.
struct GemmParams {
    CUtensorMap tma_a;     // A codes [M, K] (K-major), boxes 128 B x 128 rows, 128-byte swizzle
    CUtensorMap tma_b;     // B codes [N, K] (K-major), boxes 128 B x 128 rows
    CUtensorMap tma_sfa;   // A scales (tiled layout) as 32-bit words [M/128][K/128][128]
    CUtensorMap tma_sfb;   // B scales, same view; boxes of two 128-row tiles
    CUtensorMap tma_out;   // bf16 output [M, N] (row-major), boxes 32 x 32, 64-byte swizzle
    int32_t M, N, K;
    int32_t m_tiles, n_tiles, k_tiles;  // 256-row, 256-column and 128-byte tiles
    int32_t num_tiles;                  // m_tiles * n_tiles output tiles (one per CTA pair)
};

// The form for few activation rows (M <= 64, and up to kSkinnyMaxM where it
// is estimated faster than the general form's few 256 x 256 tiles): the operands swap
// roles, so that the weight's rows fill the MMA's 256 rows and the activation
// rows are its N (32, 64 or 128); the K steps of a 256-column output block are
// split over the CTA pairs of one cluster, whose float32 partial sums meet in
// distributed shared memory.
constexpr int64_t kSkinnyMaxM = 2048;
struct SkinnyParams {
    CUtensorMap tma_w;     // B codes [N, K] (the weight), boxes 128 B x 128 rows
    CUtensorMap tma_x;     // A codes [M, K] (the activation), boxes 128 B x mt/2 rows
    CUtensorMap tma_sfw;   // B scales as 32-bit words [N/128][K/128][128], boxes of one tile
    CUtensorMap tma_sfx;   // A scales, same view
    CUtensorMap tma_out;   // bf16 output [M, N] (row-major), boxes 32 columns x mt rows
    int32_t M, N, K;
    int32_t mt;               // activation rows per MMA (32, 64 or 128)
    int32_t m_blocks;         // blocks of mt activation rows (1 unless mt = 128)
    int32_t n_tiles, k_tiles; // 256-column output blocks; 128-byte K steps
    int32_t num_tiles;        // n_tiles * m_blocks work tiles, block n of tile t:
                              // t / m_blocks, activation block t % m_blocks
    int32_t splits;           // CTA pairs per cluster, each taking one K range
    int32_t steps_per_split;  // K steps per range (the last range may be shorter)
    int32_t resident;         // (planning) clusters of the chosen split held at once
    int32_t weight_early;     // the weight and its scales may be read before the
                              // dependency wait (see below)
    int64_t cost;             // (planning) waves x (K steps per pair + hand-overs)
};

// weight_early (0 unless the caller sets it after gemm_plan): the GEMMs are
// launched as programmatic dependents of the kernel before them on the stream
// and read nothing before that kernel has completed. When that kernel is
// known to leave the weight and its scales alone, and itself started only
// after everything before it had completed, the weight is already final when
// the GEMM starts, so the swapped form's first ring stages of weight copies go
// out before the wait and overlap the previous kernel. mm_mxfp8 sets it: its
// GEMM follows its own activation quantize, an ordinary launch that writes
// only the activation's scratch. (The 256 x 256-tile form measured no gain
// from the same and does not take it.)

struct GemmPlan {
    bool skinny;
    GemmParams general;
    SkinnyParams thin;
};

// Fills plan for out[M, N] = A [M, K] x B [N, K]^T (E4M3 codes with tiled
// UE8M0 scales), choosing the form by M. Returns 0, or -1 / -2 / -3 when a
// tensor map of A / B (codes or scales) / the output cannot be made (a driver
// without cuTensorMapEncodeTiled, or an address or stride TMA rejects).
int gemm_plan(GemmPlan* plan, const uint8_t* a, const uint8_t* sfa, const uint8_t* b,
              const uint8_t* sfb, uint16_t* out, int64_t M, int64_t N, int64_t K);

// One persistent launch of the planned form on `stream` (general: CTA pairs
// in clusters of two, at most one pair per output tile; skinny: clusters of
// `splits` pairs, at most one cluster per output block); returns the
// cudaError_t of the launch.
int gemm_launch(const GemmPlan& plan, void* stream);

// The GEMM's device status word (0: no wait has given up since it was last
// cleared), read with a synchronizing copy; cleared when asked.
int gemm_status(bool clear, unsigned long long* out);

// Test hooks (mxfp8_set_test_hook, mxfp8_api.cu): the form the planner is
// held to (0 its own choice, 1 the 256 x 256-tile form, 2 the swapped form
// where M <= kSkinnyMaxM) and the K split of the swapped form (0 its own
// choice, else that many pairs, at most the K steps).
int hook_gemm_form();
int hook_gemm_splits();

}  // namespace mx
