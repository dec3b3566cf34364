// mxfp8_update.cu -- in-place update of MXFP8 planes from a compact source
// (Megatron-FSDP page
// "core.distributed.fsdp.src.megatron_fsdp.experimental.quantized_dbuffer",
// `update_mxfp8_tensor`: the selected planes are taken from the compact
// source with padded scales, unselected planes stay as they are, and selected
// planes that the source lacks are cleared).
//
// One launch covers the whole list. Every selected plane of every entry is
// cut into chunks (scales first, 8 KB; then codes, 64 KB), one CTA per chunk;
// a CTA finds its entry by binary search over the entries' first chunks,
// then its plane and part (codes or scales) from the per-entry chunk counts.
// Codes move as 16-byte vectors, eight in flight per thread; a scale chunk
// reads 16 source bytes per thread step and writes them as one vector when
// they stay in one row of a row-major destination at a 16-byte boundary,
// else one by one at their place in the destination layout.
#include <cuda_runtime.h>
#include <stdint.h>

#include "mx_update.h"

namespace mx {
namespace {

__device__ __forceinline__ int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }
__device__ __forceinline__ int64_t chunks_of(int64_t bytes, int64_t chunk) {
    return (bytes + chunk - 1) / chunk;
}

// Byte offset of scale (m, k) in the tiled GEMM-operand layout (tiles of 128
// rows x 4 scale columns, 512 bytes each, row tiles outer; inside a tile
// (m % 32) * 16 + ((m / 32) % 4) * 4 + k % 4), for kb scale columns.
__device__ __forceinline__ int64_t tiled_off(int64_t m, int64_t k, int64_t kb) {
    const int64_t col_tiles = (kb + 3) >> 2;
    return (((m >> 7) * col_tiles + (k >> 2)) << 9) + ((m & 31) << 4) + (((m >> 5) & 3) << 2) +
           (k & 3);
}

// Bytes of a destination scale plane in `layout` (cleared whole when absent).
__device__ __forceinline__ int64_t dst_scale_bytes(int layout, bool colw, int64_t R, int64_t C) {
    if (layout == 0) return R * C / 32;
    if (!colw) return round_up(R, 128) * round_up(C / 32, 4);
    return layout == 2 ? round_up(R / 32, 4) * round_up(C, 128)
                       : round_up(C, 128) * round_up(R / 32, 4);
}

// Copy (src != NULL) or clear a byte range [b0, b1) of a code plane; the
// planes are whole 16-byte vectors.
__device__ __forceinline__ void move_codes(uint8_t* dst, const uint8_t* src, int64_t b0,
                                           int64_t b1) {
    constexpr int kDepth = 8;
    uint4* d = reinterpret_cast<uint4*>(dst);
    const int64_t v0 = b0 >> 4, v1 = b1 >> 4;
    if (src == nullptr) {
        for (int64_t v = v0 + threadIdx.x; v < v1; v += kUpdThreads) d[v] = make_uint4(0, 0, 0, 0);
        return;
    }
    const uint4* s = reinterpret_cast<const uint4*>(src);
    for (int64_t base = v0; base < v1; base += (int64_t)kDepth * kUpdThreads) {
        uint4 buf[kDepth];
#pragma unroll
        for (int u = 0; u < kDepth; ++u) {
            const int64_t v = base + u * kUpdThreads + threadIdx.x;
            if (v < v1) buf[u] = __ldcs(s + v);
        }
#pragma unroll
        for (int u = 0; u < kDepth; ++u) {
            const int64_t v = base + u * kUpdThreads + threadIdx.x;
            if (v < v1) __stcs(d + v, buf[u]);
        }
    }
}

// Clear bytes [b0, b1) of a scale plane (any byte count; b0 is 16-aligned).
__device__ __forceinline__ void clear_bytes(uint8_t* dst, int64_t b0, int64_t b1) {
    const int64_t v0 = b0 >> 4, v1 = b1 >> 4;
    uint4* d = reinterpret_cast<uint4*>(dst);
    for (int64_t v = v0 + threadIdx.x; v < v1; v += kUpdThreads) d[v] = make_uint4(0, 0, 0, 0);
    for (int64_t b = v1 * 16 + threadIdx.x; b < b1; b += kUpdThreads) dst[b] = 0;
}

// Re-lay compact source scale bytes [b0, b1) into the destination layout.
// Rowwise source [R, C/32]: byte i is (r, k) = divmod(i, C/32). Columnwise
// source [R/32, C]: byte i is (b, c) = divmod(i, C); as a GEMM operand its row
// is the column c and its scale column the row block b.
__device__ __forceinline__ void move_scales(uint8_t* dst, const uint8_t* src, int layout,
                                            bool colw, int64_t R, int64_t C, int64_t b0,
                                            int64_t b1) {
    const int64_t width = colw ? C : C / 32;  // source row length (a multiple of 1, not 16)
    // destination row pitch of the row-major layouts (compact: width)
    const int64_t pitch = layout == 2 ? (colw ? round_up(C, 128) : round_up(C / 32, 4)) : width;
    for (int64_t i0 = b0 + 16 * threadIdx.x; i0 < b1; i0 += 16 * kUpdThreads) {
        const int64_t n = b1 - i0 < 16 ? b1 - i0 : 16;
        uint8_t v[16];
        if (n == 16 && (reinterpret_cast<uintptr_t>(src + i0) & 15) == 0) {
            *reinterpret_cast<uint4*>(v) = *reinterpret_cast<const uint4*>(src + i0);
        } else {
            for (int j = 0; j < n; ++j) v[j] = src[i0 + j];
        }
        int64_t row = i0 / width, col = i0 - row * width;
        if (layout != 1 && n == 16 && col + 16 <= width) {
            uint8_t* d = dst + row * pitch + col;
            if ((reinterpret_cast<uintptr_t>(d) & 15) == 0) {
                *reinterpret_cast<uint4*>(d) = *reinterpret_cast<const uint4*>(v);
                continue;
            }
        }
        for (int j = 0; j < n; ++j) {
            int64_t off;
            if (layout != 1) off = row * pitch + col;
            else off = colw ? tiled_off(col, row, R / 32) : tiled_off(row, col, C / 32);
            dst[off] = v[j];
            if (++col == width) {
                col = 0;
                ++row;
            }
        }
    }
}

__global__ void __launch_bounds__(kUpdThreads)
update_planes_kernel(const __grid_constant__ UpdTable T) {
    const int64_t chunk = blockIdx.x;
    int lo = 0, hi = T.n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (T.e[mid].chunk_begin <= chunk) lo = mid;
        else hi = mid - 1;
    }
    const UpdEntry& E = T.e[lo];
    const int64_t R = E.rows, C = E.cols;
    int64_t local = chunk - E.chunk_begin;
    // parts: 0 row codes, 1 row scales, 2 col codes, 3 col scales; scales first
    for (int step = 0; step < 4; ++step) {
        const int part = step < 2 ? 2 * step + 1 : 2 * (step - 2);
        const bool colw = part >= 2;
        if (!(colw ? T.columnwise : T.rowwise)) continue;
        const bool scales = part & 1;
        const uint8_t* src = E.src[part];
        const int64_t bytes = !scales ? R * C
                            : (src ? R * C / 32 : dst_scale_bytes(T.layout, colw, R, C));
        const int64_t chunk_bytes = scales ? kUpdScaleChunkBytes : kUpdChunkBytes;
        const int64_t n = chunks_of(bytes, chunk_bytes);
        if (local >= n) {
            local -= n;
            continue;
        }
        const int64_t b0 = local * chunk_bytes;
        const int64_t b1 = b0 + chunk_bytes < bytes ? b0 + chunk_bytes : bytes;
        if (!scales) move_codes(E.dst[part], src, b0, b1);
        else if (src == nullptr) clear_bytes(E.dst[part], b0, b1);
        else move_scales(E.dst[part], src, T.layout, colw, R, C, b0, b1);
        return;
    }
}

}  // namespace

int launch_update(const UpdTable& t, void* stream) {
    if (const int e = hook_launch_error()) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)t.total_chunks, 1, 1);
    cfg.blockDim = dim3(kUpdThreads, 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cfg.numAttrs = 0;
    return (int)cudaLaunchKernelEx(&cfg, update_planes_kernel, t);
}

}  // namespace mx
