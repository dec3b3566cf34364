// mx_update.h -- launch table of the plane update (mxfp8_update.cu), shared
// by the C-ABI layer and the kernel; passed by value as a __grid_constant__
// kernel parameter, so it must stay under the 32 KB kernel-parameter limit.
#pragma once

#include <stdint.h>

namespace mx {

// Plane update (mxfp8_update.cu): one launch over a list of tensors. Each
// entry's selected planes are cut into chunks, one CTA per chunk, in the
// order [row scales][column scales][row codes][column codes]: scales (byte
// by byte re-lay, slower per byte) in 8 KB chunks and first, so they do not
// trail the launch; codes in 64 KB chunks. A plane whose source pointers are
// NULL is cleared instead of copied.
struct UpdEntry {
    const uint8_t* src[4];  // q_row, s_row, q_col, s_col (compact scales); NULL: plane absent
    uint8_t* dst[4];        // same planes; scales in the table's layout
    int64_t rows, cols;
    int64_t chunk_begin;    // first CTA chunk of this entry
};
constexpr int64_t kUpdChunkBytes = 65536;      // code bytes per CTA chunk
constexpr int64_t kUpdScaleChunkBytes = 8192;  // scale bytes per CTA chunk
constexpr int kUpdThreads = 256;
struct UpdTable {
    UpdEntry e[256];
    int32_t n;
    int32_t rowwise, columnwise;
    int32_t layout;         // destination scale layout: 0 compact, 1 tiled, 2 padded
    int64_t total_chunks;
};
static_assert(sizeof(UpdTable) < 32000, "kernel parameter limit");
int launch_update(const UpdTable& t, void* stream);
int hook_launch_error();  // mxfp8_api.cu: an injected launch error, else cudaSuccess

}  // namespace mx
