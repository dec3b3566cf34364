// mxfp8_kernels.cu -- sm_103a kernels for fused RMSNorm + MXFP8 quantization.
//
// What is computed (per list entry, bf16 matrix [R, C], row-major):
//   fused:  normed = bf16((x * 1/sqrt(sum(x^2)/C + eps)) * (gamma + offset)),
//           per row in float32 (MAX Mojo page
//           "DistributedAllGatherRMSNormQuantMXFP8", Args gammas, epsilons,
//           weight_offsets, outputs_normed), then both MXFP8 planes of that
//           same bf16 (the page's description: the quantize reads the bf16 that
//           lands in outputs_normed).
//   quant:  both MXFP8 planes of x itself (Megatron inference page
//           "core.inference.quantization.utils", quantize_params_to_mxfp8).
// MXFP8 planes: 32-element blocks (Megatron-FSDP page
// "core.distributed.fsdp.src.megatron_fsdp.experimental.quantized_dbuffer",
// _MXFP8_BLOCK_SIZE), E4M3 codes with one E8M0 scale per block; rowwise
// blocks run along a row (scales [R, C/32]), columnwise blocks down 32 rows of
// a column (scales [R/32, C], the page's _columnwise_scale_layout and
// _block_atomic_to_flat), and both code planes are [R, C] row-major.
// Scale rule: amax == 0 -> byte 0, else byte = clamp(floor(log2 amax) - 8,
// -127, 127) + 127; codes are RNE(v * 2^-e) saturated to +-448.
//
// Design (HBM-bound: ~6 B per element moved, no contraction, so no tensor
// cores; the instruction budget per element is the second limit):
//  - Thread tile: kRows rows x 8 columns, one 16-byte bf16 vector per row
//    (TileGeo in mx_table.h: 8 rows in the fused kernel, 16 in the quantize).
//    Each row group of a warp reads kGroupLanes * 16
//    contiguous bytes per row, so every load and store is fully coalesced.
//  - The tile stays in registers from load to store, so x is read from HBM
//    once. A rowwise block (32 columns) spans 4 lanes: amax by two xor
//    shuffles. A columnwise block (32 rows) spans the kGroups row groups of
//    a warp: per-thread column maxima plus log2(kGroups) xor shuffles.
//  - Fused kernel: a 32-row stripe of C columns is split over a thread-block
//    cluster of K CTAs (ceil(C / 1024) up to 8, up to 16 for wider rows
//    where the device allows; launches too small to fill the device once
//    take one 512-column pass per CTA instead). Row partial sums of squares
//    meet in each CTA's shared memory and are summed across the cluster
//    through distributed shared memory, in rank order, so every CTA derives
//    the same 1/rms for a row. A CTA's slice is kTargetChunks 512-column
//    passes wide when the row allows: after the row sums, the last pass is
//    still in registers and the earlier ones are read again from L2.
//  - L2 policy: outputs are written with streaming (evict-first) stores, so
//    the pass-2 re-reads hit L2 and x crosses DRAM once; a residual input is
//    staged per pass in shared memory by cp.async (evict-first) while x loads
//    to registers, keeping both input streams in flight at 64 registers.
//  - Quant kernel: every warp owns one 32 x kWarpCols tile of the flattened list.
//  - Arithmetic: x^2 is summed with mixed-precision fma.rn.f32.bf16 (the bf16
//    product is exact in float32); the normalization runs on packed
//    mul.rn.f32x2; amax is max.xorsign.abs.bf16x2 on the bf16 values; the scale
//    byte is the bf16 exponent field of amax minus 8 (clamped at 0), which is
//    the rule above for every finite bf16 amax; cvt.rn.satfinite.e4m3x2.f32
//    rounds to nearest even and saturates.
//  - v * 2^-e is one correctly rounded float32 product (exact whenever it can
//    matter; products below 2^-126 quantize to a signed zero either way). The
//    fused kernel forms it with fma.rn.f32.bf16 and the scale kept as bf16
//    (quantize_tile: fewer live registers, which keeps it at 64 registers and
//    four 256-thread CTAs per SM); the quantize kernel unpacks each bf16 pair once and
//    multiplies it by float32 scale pairs with mul.rn.f32x2 for both planes
//    (emit_planes: fewer instructions). Both give the same float32 value and
//    the same E4M3 code for every input, so the fused planes are
//    byte-identical to a standalone quantize of the fused normed output.
#include <cuda_runtime.h>
#include <stdint.h>

#include "mx_table.h"

namespace mx {

// Bounds-checking build (-DMXFP8_DEBUG_BOUNDS): every global access of the two
// kernels is checked against the extent of its buffer that the C ABI states
// for the entry's shape and scale layout; an access outside it is skipped and
// the first one is recorded in g_bounds_status (bits 48-55: 0x80 | the access
// site; bits 0-47: the element offset), which mxfp8_device_status reports.
// In the normal build the checks compile to nothing.
#ifdef MXFP8_DEBUG_BOUNDS
__device__ unsigned long long g_bounds_status = 0;
#endif

namespace {

enum BoundsSite : uint32_t {
    kSiteX = 1, kSiteResIn, kSiteResOut, kSiteGamma, kSiteNormed,
    kSiteQRow, kSiteSRow, kSiteQCol, kSiteSCol
};

#ifdef MXFP8_DEBUG_BOUNDS
__device__ __noinline__ bool in_bounds(int64_t off, int64_t len, int64_t extent, uint32_t site) {
    if (off >= 0 && off + len <= extent) return true;
    atomicCAS(&g_bounds_status, 0ull,
              ((unsigned long long)(0x80u | site) << 48) |
                  ((unsigned long long)off & 0xFFFFFFFFFFFFull));
    return false;
}
#define MX_IN(off, len, extent, site) in_bounds((off), (len), (extent), (site))
#else
#define MX_IN(off, len, extent, site) true
#endif

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// acc + lo^2 + hi^2 for the two bf16 of w (each product exact in float32).
__device__ __forceinline__ float sumsq2(uint32_t w, float acc) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\t"
        "fma.rn.f32.bf16 %0, l, l, %0;\n\tfma.rn.f32.bf16 %0, h, h, %0;\n\t}"
        : "+f"(acc) : "r"(w));
    return acc;
}

__device__ __forceinline__ uint64_t pair(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

// bf16x2( (x * r) * w ) for the two bf16 of x; r and w are float32 pairs.
__device__ __forceinline__ uint32_t norm2(uint32_t x, uint64_t rr, uint64_t ww) {
    const uint64_t xf = pair(bf16lo(x), bf16hi(x));
    uint64_t t, y;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(t) : "l"(xf), "l"(rr));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(y) : "l"(t), "l"(ww));
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(y));
    uint32_t out;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(hi), "f"(lo));
    return out;
}

// Two E4M3 codes (lo in bits 0-7) of the bf16 pair w, each multiplied by the
// bf16 power of two in the matching half of s2 (one rounding, like a float32
// multiply), then RNE with saturation to +-448. Adding -0 keeps the sign of
// zero products.
__device__ __forceinline__ uint32_t quant2(uint32_t w, uint32_t s2) {
    unsigned short q;
    asm("{\n\t.reg .b16 xl, xh, sl, sh;\n\t.reg .f32 fa, fb;\n\t"
        "mov.b32 {xl, xh}, %1;\n\tmov.b32 {sl, sh}, %2;\n\t"
        "fma.rn.f32.bf16 fa, xl, sl, 0f80000000;\n\t"
        "fma.rn.f32.bf16 fb, xh, sh, 0f80000000;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 %0, fb, fa;\n\t}"
        : "=h"(q) : "r"(w), "r"(s2));
    return q;
}

__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// The two bf16 of w as an exact float32 pair.
__device__ __forceinline__ uint64_t unpack2(uint32_t w) { return pair(bf16lo(w), bf16hi(w)); }

// Four E4M3 codes (element 0 in bits 0-7) of the float32 pairs a and b:
// round to nearest even, magnitudes past 448 saturate to 448, signs kept.
__device__ __forceinline__ uint32_t e4m3x4(uint64_t a, uint64_t b) {
    uint32_t r;
    asm("{\n\t.reg .b16 u, v;\n\t.reg .f32 a0, a1, b0, b1;\n\t"
        "mov.b64 {a0, a1}, %1;\n\tmov.b64 {b0, b1}, %2;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 u, a1, a0;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 v, b1, b0;\n\t"
        "mov.b32 %0, {u, v};\n\t}"
        : "=r"(r) : "l"(a), "l"(b));
    return r;
}

// 2^-(byte - 127) as float32 (a normal number for every byte <= 246).
__device__ __forceinline__ float inv_scale(uint32_t byte) {
    return __uint_as_float((254u - byte) << 23);
}

// Per 16-bit half: the larger magnitude of a and b (the sign bit of the
// result is not used).
__device__ __forceinline__ uint32_t maxabs2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Per 16-bit half: E8M0 scale byte of a block whose amax has the bf16
// magnitude bits in that half (the sign bit is ignored).
__device__ __forceinline__ uint32_t scale_bytes2(uint32_t m2) {
    const uint32_t b = (m2 >> 7) & 0x00FF00FFu;
    return __vsub2(__vmaxu2(b, 0x00080008u), 0x00080008u);
}

// Per 16-bit half: the bf16 bits of 2^-(byte - 127) (a normal number for
// every byte <= 246).
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t bytes2) {
    return (0x00FE00FEu - bytes2) << 7;
}

__device__ __forceinline__ uint2 quant8(const uint4& y, uint32_t s01, uint32_t s23,
                                        uint32_t s45, uint32_t s67) {
    return make_uint2(quant2(y.x, s01) | (quant2(y.y, s23) << 16),
                      quant2(y.z, s45) | (quant2(y.w, s67) << 16));
}

// Running maxima of a thread tile. colmax[k]: magnitudes of columns 2k, 2k+1
// over the rows folded so far. rowpk[j]: 8-column maxima of rows 2j (bits
// 0-15) and 2j+1 (bits 16-31).
template <class G>
struct TileMax {
    uint32_t colmax[4];
    uint32_t rowpk[G::kRows / 2];
};

__device__ __forceinline__ uint32_t row_max8(const uint4& y) {
    return maxabs2(maxabs2(y.x, y.y), maxabs2(y.z, y.w));
}

template <class M>
__device__ __forceinline__ void fold_col(M& m, const uint4& y) {
    m.colmax[0] = maxabs2(m.colmax[0], y.x);
    m.colmax[1] = maxabs2(m.colmax[1], y.y);
    m.colmax[2] = maxabs2(m.colmax[2], y.z);
    m.colmax[3] = maxabs2(m.colmax[3], y.w);
}

// Row maxima of rows 2j and 2j+1 packed into rowpk[j].
template <class M>
__device__ __forceinline__ void fold_rows(M& m, int j, const uint4& y0, const uint4& y1) {
    const uint32_t a = row_max8(y0), b = row_max8(y1);
    m.rowpk[j] = maxabs2(__byte_perm(a, b, 0x5410), __byte_perm(a, b, 0x7632));
}

// Where one thread tile lands in the outputs.
struct TileAt {
    int64_t row0;      // first row of the thread's rows
    int64_t col;       // first of the thread's 8 columns
    int64_t cols;      // C
    int64_t stripe;    // 32-row block index (columnwise scale row)
    int64_t rows;      // R
    int nrows;         // of the thread's rows, those inside the matrix (ragged R)
    bool col_ok;       // the 8 columns lie inside the matrix (or this CTA's slice)
    bool mma;          // scales in the tiled GEMM-operand layout
    bool padded;       // row-major scales with padded pitches (TE's allocation shape)
};

__device__ __forceinline__ int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// Extents (in bytes) of the scale buffers of the entry `at` belongs to, as the
// C ABI states them for each layout.
__device__ __forceinline__ int64_t srow_extent(const TileAt& at) {
    const int64_t nb = at.cols / kBlock;
    return (at.mma || at.padded) ? round_up(at.rows, 128) * round_up(nb, 4) : at.rows * nb;
}
__device__ __forceinline__ int64_t scol_extent(const TileAt& at) {
    const int64_t sb = at.rows / kBlock;
    return (at.mma || at.padded) ? round_up(sb, 4) * round_up(at.cols, 128) : sb * at.cols;
}

// Byte offset of scale (m, k) in the tiled GEMM-operand layout: tiles of 128
// rows x 4 scale columns, 512 bytes each, row tiles outer; inside a tile, row
// m and column k sit at (m % 32) * 16 + ((m / 32) % 4) * 4 + k % 4.
// col_tiles = ceil(scale columns / 4).
__device__ __forceinline__ int64_t mma_off(int64_t m, int64_t k, int64_t col_tiles) {
    return (((m >> 7) * col_tiles + (k >> 2)) << 9) + ((m & 31) << 4) + (((m >> 5) & 3) << 2) +
           (k & 3);
}

// Where the rowwise scales of a thread's rows start, and how far apart they
// are, for its column block kb. Row-major layouts: rows are nb = C / 32
// (compact) or roundup(nb, 4) (padded) bytes apart. Tiled: the thread's rows
// lie inside one 32-row group (row0 % 32 + i < 32), so they share the tile and
// the (m / 32) % 4 slot and sit 16 bytes apart.
__device__ __forceinline__ uint8_t* row_scale_base(uint8_t* s_row, const TileAt& at, int64_t kb,
                                                   int64_t nb, int64_t& pitch) {
    if (at.mma) {
        pitch = 16;
        return s_row + mma_off(at.row0, kb, (nb + 3) >> 2);
    }
    pitch = at.padded ? round_up(nb, 4) : nb;
    return s_row + at.row0 * pitch + kb;
}

// Columnwise scales of the thread's 8 columns for its 32-row block: bytes of
// columns col..col+3 in lo4, col+4..col+7 in hi4. In the tiled layout the
// columnwise scales are those of an operand whose rows are the C columns and
// whose scale columns are the R / 32 row blocks; col % 8 == 0, so the 8
// columns lie inside one 32-column group and sit 16 bytes apart.
__device__ __forceinline__ void store_col_scales(uint8_t* s_col, const TileAt& at, uint32_t lo4,
                                                 uint32_t hi4) {
    if (!at.mma) {
        const int64_t cp = at.padded ? round_up(at.cols, 128) : at.cols;
        if (MX_IN(at.stripe * cp + at.col, 8, scol_extent(at), kSiteSCol))
            *reinterpret_cast<uint2*>(s_col + at.stripe * cp + at.col) = make_uint2(lo4, hi4);
        return;
    }
    const int64_t o = mma_off(at.col, at.stripe, ((at.rows >> 5) + 3) >> 2);
    uint8_t* sc = s_col + o;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (MX_IN(o + 16 * j, 1, scol_extent(at), kSiteSCol))
            sc[16 * j] = (uint8_t)(((j < 4 ? lo4 : hi4) >> (8 * (j & 3))) & 0xFFu);
}

// Both planes of a thread tile y[] whose maxima were folded into m, with bf16
// scales and mixed-precision products (the fused kernel's register-lean
// path). Codes are written with streaming (evict-first) stores: the kernel
// never reads them, and in L2 they would displace the x tiles that pass 2
// reads again. Every code and scale depends only on the block's values.
// Executed by all 32 lanes (the shuffles need them); stores are guarded per
// row/column.
template <class G>
__device__ __forceinline__ void quantize_tile(const uint4 (&y)[G::kRows], TileMax<G>& m,
                                              const TileAt& at,
                                              uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                                              uint8_t* s_col, bool do_row, bool do_col, int g,
                                              int q) {
    const int64_t base = at.row0 * at.cols + at.col;
    if (do_row) {
        // a rowwise block is 4 lanes wide (lanes 4j..4j+3 of a row group)
#pragma unroll
        for (int j = 0; j < G::kRows / 2; ++j) {
            m.rowpk[j] = maxabs2(m.rowpk[j], __shfl_xor_sync(0xFFFFFFFFu, m.rowpk[j], 1));
            m.rowpk[j] = maxabs2(m.rowpk[j], __shfl_xor_sync(0xFFFFFFFFu, m.rowpk[j], 2));
        }
        const int64_t nb = at.cols / kBlock;
        uint8_t* qr = q_row + base;
        int64_t rp;
        uint8_t* sr = row_scale_base(s_row, at, at.col / kBlock, nb, rp);
        if (at.mma) {
            // Tiled scales. After the reduction all 4 lanes of a block hold
            // its maxima of all the thread's rows, so lane i of the 4 stores
            // the scale bytes of rows 2i and 2i + 1: two stores per pass with
            // every lane active, where one lane in four storing all 8 rows
            // takes eight (measured 3 % faster in this layout, whose 16-byte
            // tile rows hold the bytes of four stripes; 0.5 % slower in the
            // row-major ones, which keep the form below).
            const int i4 = g & 3;
            uint32_t mine = 0;  // the scale bytes of rows 2 i4 (bits 0-7) and 2 i4 + 1 (16-23)
#pragma unroll
            for (int j = 0; j < G::kRows / 2; ++j) {
                const uint32_t bytes2 = scale_bytes2(m.rowpk[j]);
                if (j == i4) mine = bytes2;
                const uint32_t sc2 = scale_bf16x2(bytes2);
                const uint32_t s_even = __byte_perm(sc2, 0, 0x1010);  // row 2j scale, both halves
                const uint32_t s_odd = __byte_perm(sc2, 0, 0x3232);   // row 2j+1
                if (at.col_ok) {
                    if (2 * j < at.nrows &&
                        MX_IN(base + (2 * j) * at.cols, 8, at.rows * at.cols, kSiteQRow))
                        __stcs(reinterpret_cast<uint2*>(qr + (2 * j) * at.cols),
                               quant8(y[2 * j], s_even, s_even, s_even, s_even));
                    if (2 * j + 1 < at.nrows &&
                        MX_IN(base + (2 * j + 1) * at.cols, 8, at.rows * at.cols, kSiteQRow))
                        __stcs(reinterpret_cast<uint2*>(qr + (2 * j + 1) * at.cols),
                               quant8(y[2 * j + 1], s_odd, s_odd, s_odd, s_odd));
                }
            }
            if (at.col_ok) {
                uint8_t* sl = sr + (2 * i4) * rp;
                const int64_t so = (sl - s_row);
                if (2 * i4 < at.nrows && MX_IN(so, 1, srow_extent(at), kSiteSRow))
                    sl[0] = (uint8_t)(mine & 0xFFu);
                if (2 * i4 + 1 < at.nrows && MX_IN(so + rp, 1, srow_extent(at), kSiteSRow))
                    sl[rp] = (uint8_t)(mine >> 16);
            }
        } else {
            const bool writes_scale = (g & 3) == 0;
#pragma unroll
            for (int j = 0; j < G::kRows / 2; ++j) {
                const uint32_t bytes2 = scale_bytes2(m.rowpk[j]);
                const uint32_t sc2 = scale_bf16x2(bytes2);
                const uint32_t s_even = __byte_perm(sc2, 0, 0x1010);  // row 2j scale, both halves
                const uint32_t s_odd = __byte_perm(sc2, 0, 0x3232);   // row 2j+1
                if (at.col_ok) {
                    if (2 * j < at.nrows) {
                        if (MX_IN(base + (2 * j) * at.cols, 8, at.rows * at.cols, kSiteQRow))
                            __stcs(reinterpret_cast<uint2*>(qr + (2 * j) * at.cols),
                                   quant8(y[2 * j], s_even, s_even, s_even, s_even));
                        if (writes_scale &&
                            MX_IN((sr - s_row) + (2 * j) * rp, 1, srow_extent(at), kSiteSRow))
                            sr[(2 * j) * rp] = (uint8_t)(bytes2 & 0xFFu);
                    }
                    if (2 * j + 1 < at.nrows) {
                        if (MX_IN(base + (2 * j + 1) * at.cols, 8, at.rows * at.cols, kSiteQRow))
                            __stcs(reinterpret_cast<uint2*>(qr + (2 * j + 1) * at.cols),
                                   quant8(y[2 * j + 1], s_odd, s_odd, s_odd, s_odd));
                        if (writes_scale &&
                            MX_IN((sr - s_row) + (2 * j + 1) * rp, 1, srow_extent(at), kSiteSRow))
                            sr[(2 * j + 1) * rp] = (uint8_t)(bytes2 >> 16);
                    }
                }
            }
        }
    }
    if (do_col) {
        // a columnwise block is the kGroups row groups of the warp
        uint32_t sc[4], bytes[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int o = G::kGroupLanes; o < 32; o <<= 1)
                m.colmax[k] = maxabs2(m.colmax[k], __shfl_xor_sync(0xFFFFFFFFu, m.colmax[k], o));
            bytes[k] = scale_bytes2(m.colmax[k]);
            sc[k] = scale_bf16x2(bytes[k]);
        }
        if (at.col_ok) {
            if (q == 0) {
                store_col_scales(s_col, at, __byte_perm(bytes[0], bytes[1], 0x6420),
                                 __byte_perm(bytes[2], bytes[3], 0x6420));
            }
            uint8_t* qc = q_col + base;
#pragma unroll
            for (int i = 0; i < G::kRows; ++i)
                if (i < at.nrows && MX_IN(base + i * at.cols, 8, at.rows * at.cols, kSiteQCol))
                    __stcs(reinterpret_cast<uint2*>(qc + i * at.cols),
                           quant8(y[i], sc[0], sc[1], sc[2], sc[3]));
        }
    }
}

// Both planes of a thread tile y[] whose maxima were folded into m, with one
// unpack per bf16 pair and float32 scale pairs (the quantize kernel's
// instruction-lean path; same codes as quantize_tile). Codes go out with
// streaming (evict-first) stores when code rows start on 128-byte lines
// (C % 128 == 0): measured +4 % on large tensors, while on lists of narrow
// tensors whose rows split lines the early evictions cost 3 %. Executed by all 32
// lanes (the shuffles need them). FULL: the caller has checked,
// warp-uniformly, that every row and column of the tile lies inside the
// matrix, so no store is guarded.
// 8 code bytes, with a streaming (evict-first) store when asked.
__device__ __forceinline__ void st_code8(uint2* p, uint2 v, bool streaming) {
    if (streaming) __stcs(p, v);
    else *p = v;
}

template <class G, bool FULL>
__device__ __forceinline__ void emit_planes(const uint4 (&y)[G::kRows], TileMax<G>& m,
                                            const TileAt& at, uint8_t* q_row, uint8_t* s_row,
                                            uint8_t* q_col, uint8_t* s_col, bool do_row,
                                            bool do_col, int g, int q) {
    constexpr int kR = G::kRows;
    uint32_t rbytes[kR / 2];  // rowwise scale bytes of rows 2j (bits 0-7) and 2j+1 (16-23)
    if (do_row) {
        // a rowwise block is 4 lanes wide (lanes 4j..4j+3 of a row group)
#pragma unroll
        for (int j = 0; j < kR / 2; ++j) {
            m.rowpk[j] = maxabs2(m.rowpk[j], __shfl_xor_sync(0xFFFFFFFFu, m.rowpk[j], 1));
            m.rowpk[j] = maxabs2(m.rowpk[j], __shfl_xor_sync(0xFFFFFFFFu, m.rowpk[j], 2));
            rbytes[j] = scale_bytes2(m.rowpk[j]);
        }
    }
    uint32_t cbytes[4];  // columnwise scale bytes of columns 2k (bits 0-7), 2k+1 (16-23)
    uint64_t cscale[4];
    if (do_col) {
        // a columnwise block is the kGroups row groups of the warp
#pragma unroll
        for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int o = G::kGroupLanes; o < 32; o <<= 1)
                m.colmax[k] = maxabs2(m.colmax[k], __shfl_xor_sync(0xFFFFFFFFu, m.colmax[k], o));
            cbytes[k] = scale_bytes2(m.colmax[k]);
            cscale[k] = pair(inv_scale(cbytes[k] & 0xFFu), inv_scale(cbytes[k] >> 16));
        }
    }
    if (!FULL && !at.col_ok) return;
    const int64_t C = at.cols;
    const int64_t base = at.row0 * C + at.col;
    if (do_col && q == 0) {
        store_col_scales(s_col, at, __byte_perm(cbytes[0], cbytes[1], 0x6420),
                         __byte_perm(cbytes[2], cbytes[3], 0x6420));
    }
    int64_t rp;
    uint8_t* sr = row_scale_base(s_row, at, at.col / kBlock, C / kBlock, rp);
    if (do_row) {
        // After the reduction all 4 lanes of a block hold its maxima of all
        // the thread's rows, so lane i of the 4 stores the scale bytes of rows
        // 4i .. 4i + 3: four stores per tile with every lane active, where one
        // lane in four storing all 16 rows took sixteen (128 ragged tensors:
        // 674 -> 668 us with compact scales, 680 -> 660 us tiled).
        const int i4 = g & 3;
        uint32_t lo = 0, hi = 0;  // scale bytes of rows 4 i4, +1 (bits 0-7, 16-23); +2, +3
#pragma unroll
        for (int j = 0; j < kR / 2; ++j) {
            if (j == 2 * i4) lo = rbytes[j];
            if (j == 2 * i4 + 1) hi = rbytes[j];
        }
        uint8_t* sl = sr + (4 * i4) * rp;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const uint32_t w = t < 2 ? lo : hi;
            if ((FULL || 4 * i4 + t < at.nrows) &&
                MX_IN((sl - s_row) + t * rp, 1, srow_extent(at), kSiteSRow))
                sl[t * rp] = (uint8_t)((t & 1) ? (w >> 16) : w);
        }
    }
    const bool lines = (C & 127) == 0;  // code rows start on 128-byte lines
#pragma unroll
    for (int i = 0; i < kR; ++i) {
        if (!FULL && i >= at.nrows) continue;
        const uint64_t p0 = unpack2(y[i].x), p1 = unpack2(y[i].y);
        const uint64_t p2 = unpack2(y[i].z), p3 = unpack2(y[i].w);
        if (do_row) {
            const uint32_t byte = (i & 1) ? (rbytes[i >> 1] >> 16) : (rbytes[i >> 1] & 0xFFu);
            const float s = inv_scale(byte);
            const uint64_t ss = pair(s, s);
            if (MX_IN(base + i * C, 8, at.rows * C, kSiteQRow))
                st_code8(reinterpret_cast<uint2*>(q_row + base + i * C),
                       make_uint2(e4m3x4(mul2(p0, ss), mul2(p1, ss)),
                                  e4m3x4(mul2(p2, ss), mul2(p3, ss))), lines);
        }
        if (do_col && MX_IN(base + i * C, 8, at.rows * C, kSiteQCol))
            st_code8(reinterpret_cast<uint2*>(q_col + base + i * C),
                   make_uint2(e4m3x4(mul2(p0, cscale[0]), mul2(p1, cscale[1])),
                              e4m3x4(mul2(p2, cscale[2]), mul2(p3, cscale[3]))), lines);
    }
}

template <int MAXN>
__device__ __forceinline__ int find_entry(const Table<MAXN>& T, int64_t u) {
    int lo = 0, hi = T.n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (T.d[mid].unit_begin <= u) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Reduce-scatter over the N lanes of a row group (N == rows per thread): each
// lane starts with N per-row partial sums and ends with the group total of
// row g (its lane index within the group), using N/2 + N/4 + ... + 1 shuffles.
template <int O, int N>
__device__ __forceinline__ void rs_step(float (&v)[N], int g) {
    const bool up = (g & O) != 0;
#pragma unroll
    for (int j = 0; j < O; ++j) {
        const float send = up ? v[j] : v[j + O];
        const float keep = up ? v[j + O] : v[j];
        v[j] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, O);
    }
}

template <int N>
__device__ __forceinline__ float reduce_scatter_rows(float (&v)[N], int g) {
    if constexpr (N >= 16) rs_step<8>(v, g);
    rs_step<4>(v, g);
    rs_step<2>(v, g);
    rs_step<1>(v, g);
    return v[0];
}

__device__ __forceinline__ float sumsq8(const uint4& v, float acc) {
    acc = sumsq2(v.x, acc);
    acc = sumsq2(v.y, acc);
    acc = sumsq2(v.z, acc);
    return sumsq2(v.w, acc);
}

// Rows of an n-row thread tile starting at row0 that lie inside R rows.
__device__ __forceinline__ int rows_inside(int64_t R, int64_t row0, int n) {
    const int64_t k = R - row0;
    return k <= 0 ? 0 : (k >= n ? n : (int)k);
}

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

// ---- thread-block cluster primitives (distributed shared memory) ----

__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// Read a float at the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ float ld_cluster_f32(const float* local, uint32_t rank) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(remote) : "r"(a), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];\n" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

__device__ __forceinline__ uint4 ld_x(const uint16_t* p, bool keep_in_l2) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
    return keep_in_l2 ? __ldcg(q) : __ldcs(q);
}

// Load the kR rows of a thread tile starting at p (row stride C elements).
// FULL: every row and column is inside the matrix, so no load is guarded;
// otherwise rows past nrows and columns outside the slice read as zero.
// KEEP: the data will be read again soon, so keep it in L2 (ld.global.cg);
// otherwise stream it (ld.global.cs, evict first).
template <int kR, bool FULL, bool KEEP>
__device__ __forceinline__ void load_tile(uint4 (&xv)[kR], const uint16_t* p, int64_t C,
                                          bool col_ok, int nrows, int64_t off, int64_t extent) {
#pragma unroll
    for (int i = 0; i < kR; ++i) {
        if ((FULL || (col_ok && i < nrows)) && MX_IN(off + i * C, 8, extent, kSiteX)) {
            const uint4* a = reinterpret_cast<const uint4*>(p + i * C);
            xv[i] = KEEP ? __ldcg(a) : __ldcs(a);
        } else {
            xv[i] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

// h = bf16(x + residual) per element: add.rn.bf16x2 rounds the exact sum once.
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Asynchronous 16-byte global -> shared copy, cached in L2 only and marked
// evict-first there (read once: it must not push out the tiles that pass 2
// reads again); the copies a thread issues complete for that thread at
// cp_async_wait_all.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;\n"
                 ::"r"(s), "l"(gmem), "l"(pol) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;\n" ::: "memory");
}

// Residual stream of one thread tile: xv += residual (when the entry has one)
// and, when asked, write the sum to res_out. Rows past nrows and columns
// outside the slice are skipped (they hold zeros and are never stored).
// keep: the residual will be read again in pass 2, so keep it in L2.
template <int kR>
__device__ __forceinline__ void add_residual_tile(uint4 (&xv)[kR], const DevDesc& D,
                                                  int64_t base, int64_t C, bool ok, int nrows,
                                                  bool write_out, bool keep) {
    if (D.res_in != nullptr) {
#pragma unroll
        for (int i = 0; i < kR; ++i) {
            if (ok && i < nrows && MX_IN(base + i * C, 8, D.rows * C, kSiteResIn)) {
                const uint4* a = reinterpret_cast<const uint4*>(D.res_in + base + i * C);
                const uint4 r = keep ? __ldcg(a) : __ldcs(a);
                xv[i].x = add_bf16x2(xv[i].x, r.x);
                xv[i].y = add_bf16x2(xv[i].y, r.y);
                xv[i].z = add_bf16x2(xv[i].z, r.z);
                xv[i].w = add_bf16x2(xv[i].w, r.w);
            }
        }
    }
    if (write_out && D.res_out != nullptr) {
#pragma unroll
        for (int i = 0; i < kR; ++i)
            if (ok && i < nrows && MX_IN(base + i * C, 8, D.rows * C, kSiteResOut))
                *reinterpret_cast<uint4*>(D.res_out + base + i * C) = xv[i];
    }
}

// Whether every lane of the warp holds a whole tile (warp-uniform result).
__device__ __forceinline__ bool warp_full(bool lane_full) {
    return __all_sync(0xFFFFFFFFu, lane_full);
}

// ---------------------------------------------------------------------------
// Fused RMSNorm + MXFP8. Grid: K CTAs (one cluster) per 32-row stripe of each
// entry, stripes of all entries laid end to end. CTA `rank` owns columns
// [rank * cta_cols, (rank + 1) * cta_cols) of its stripe.
// ---------------------------------------------------------------------------
template <int MAXN, bool MMA, bool RES>
__global__ void __launch_bounds__(FusedGeo::kThreads, 4)
fused_rmsnorm_quant_kernel(const __grid_constant__ Table<MAXN> T) {
    // let a dependent launch that opted in (the GEMM after a quantize) start
    // its set-up now: it reads nothing before this grid has completed
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    using G = FusedGeo;
    constexpr int kChunkCols = G::kChunk;
    constexpr int kR = G::kRows;
    __shared__ float red[G::kWarps][kBlock];
    __shared__ float part[kBlock];
    __shared__ float inv_rms[kBlock];
    // T.stage (residual inputs): each thread's residual rows of the current
    // pass, copied in asynchronously while x is loaded to registers, so both
    // input streams are in flight at once within the 64-register budget
    // ([kR][kThreads]).
    extern __shared__ uint4 rstage[];

    const int K = T.cluster;
    const int64_t unit = blockIdx.x / K;
    const int rank = (int)(blockIdx.x - unit * K);  // cluster rank for 1-D clusters
    const DevDesc& D = T.d[find_entry(T, unit)];
    const int64_t R = D.rows, C = D.cols;
    const int64_t stripe = unit - D.unit_begin;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane % G::kGroupLanes, q = lane / G::kGroupLanes;

    TileAt at;
    at.row0 = stripe * kBlock + q * kR;
    at.cols = C;
    at.rows = R;
    at.stripe = stripe;
    at.nrows = rows_inside(R, at.row0, kR);
    at.mma = MMA;  // compile-time: the row-major paths carry no tiled state
    at.padded = T.scale_layout == 2;
    const int64_t c_lo = (int64_t)rank * D.cta_cols;
    const int64_t c_hi = min64(C, c_lo + D.cta_cols);
    const int nch = c_hi > c_lo ? (int)((c_hi - c_lo + kChunkCols - 1) / kChunkCols) : 0;
    const int64_t col_in_chunk = (int64_t)warp * G::kWarpCols + g * 8;

    // pass 1: load the tile (kept in registers when the slice is one pass wide)
    uint4 xv[kR];
    float ss[kR];
#pragma unroll
    for (int i = 0; i < kR; ++i) ss[i] = 0.f;
    for (int ch = 0; ch < nch; ++ch) {
        const int64_t c = c_lo + (int64_t)ch * kChunkCols + col_in_chunk;
        const bool ok = c < c_hi;
        const uint16_t* p = D.x + at.row0 * C + c;
        const bool reread = ch + 1 < nch;  // every chunk but the last is read again in pass 2
        // x itself is read again unless pass 2 reads the written-out x + residual
        const bool keep_x = reread && !(RES && D.res_out != nullptr);
        const bool staged = RES && T.stage != 0 && D.res_in != nullptr;
        if (staged) {
#pragma unroll
            for (int i = 0; i < kR; ++i)
                if (ok && i < at.nrows &&
                    MX_IN(at.row0 * C + c + i * C, 8, R * C, kSiteResIn))
                    cp_async16(&rstage[i * G::kThreads + tid], D.res_in + at.row0 * C + c + i * C);
        }
        if (warp_full(ok && at.nrows == kR)) {
#pragma unroll
            for (int i = 0; i < kR; ++i)
                xv[i] = MX_IN(at.row0 * C + c + i * C, 8, R * C, kSiteX) ? ld_x(p + i * C, keep_x)
                                                                          : make_uint4(0, 0, 0, 0);
        } else {
#pragma unroll
            for (int i = 0; i < kR; ++i)
                xv[i] = (ok && i < at.nrows && MX_IN(at.row0 * C + c + i * C, 8, R * C, kSiteX))
                            ? ld_x(p + i * C, keep_x)
                            : make_uint4(0, 0, 0, 0);
        }
        // h = x + residual, written out here; the residual is kept in L2 for
        // the pass-2 re-read only when h is not written (else h is re-read)
        if (staged) {
            cp_async_wait_all();
#pragma unroll
            for (int i = 0; i < kR; ++i) {
                if (ok && i < at.nrows) {
                    // (the staged copy was skipped, and this slot is stale, only
                    // where the bounds-checking build reports an access)
                    const uint4 r = rstage[i * G::kThreads + tid];
                    xv[i].x = add_bf16x2(xv[i].x, r.x);
                    xv[i].y = add_bf16x2(xv[i].y, r.y);
                    xv[i].z = add_bf16x2(xv[i].z, r.z);
                    xv[i].w = add_bf16x2(xv[i].w, r.w);
                    if (D.res_out != nullptr &&
                        MX_IN(at.row0 * C + c + i * C, 8, R * C, kSiteResOut))
                        *reinterpret_cast<uint4*>(D.res_out + at.row0 * C + c + i * C) = xv[i];
                }
            }
        } else if (RES) {
            add_residual_tile<kR>(xv, D, at.row0 * C + c, C, ok, at.nrows, true,
                                  reread && D.res_out == nullptr);
        }
#pragma unroll
        for (int i = 0; i < kR; ++i) ss[i] = sumsq8(xv[i], ss[i]);
    }

    // row sums: row-group reduce-scatter, then across warps, then the cluster
    red[warp][q * kR + g] = reduce_scatter_rows(ss, g);
    __syncthreads();
    if (tid < kBlock) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < G::kWarps; ++w) s += red[w][tid];
        part[tid] = s;
    }
    if (K > 1) {
        // only warp 0 wrote `part`: its arrival releases those writes to the
        // peers; the other warps arrive without a release, which would wait
        // for their own memory operations to complete (measured 1.8 % of a
        // launch at 32768 x 8192)
        if (warp == 0)
            cluster_arrive_release();
        else
            asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
        cluster_wait_acquire();
        if (tid < kBlock) {
            // every peer's partial in flight at once, then added in rank order
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (j < K) v[j] = ld_cluster_f32(&part[tid], (uint32_t)j);
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (j < K) s += v[j];
            inv_rms[tid] = 1.0f / sqrtf(s / (float)C + D.eps);
        }
        // done reading the peers' shared memory (the loads have completed:
        // their values are already used, so no release ordering is needed)
        asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
    } else if (tid < kBlock) {
        inv_rms[tid] = 1.0f / sqrtf(part[tid] / (float)C + D.eps);
    }
    __syncthreads();

    // pass 2: normalize, write normed, quantize both planes. Chunks run in
    // reverse so that the last chunk of pass 1 is still in registers.
    const bool do_row = T.rowwise != 0, do_col = T.columnwise != 0;
    for (int k = 0; k < nch; ++k) {
        const int ch = nch - 1 - k;
        at.col = c_lo + (int64_t)ch * kChunkCols + col_in_chunk;
        at.col_ok = at.col < c_hi;
        const int64_t base = at.row0 * C + at.col;
        if (k > 0) {
            // pass 2 of an earlier chunk: with a residual whose sum was written
            // in pass 1, read that sum back (one stream, fresh in L2)
            const uint16_t* src = (RES && D.res_out != nullptr) ? D.res_out : D.x;
#pragma unroll
            for (int i = 0; i < kR; ++i)
                xv[i] = (at.col_ok && i < at.nrows &&
                         MX_IN(base + i * C, 8, R * C, src == D.x ? kSiteX : kSiteResOut))
                            ? ld_x(src + base + i * C, false)
                            : make_uint4(0, 0, 0, 0);
            if (RES && D.res_out == nullptr)
                add_residual_tile<kR>(xv, D, base, C, at.col_ok, at.nrows, false, false);
        }
        uint64_t ww[4];
        if (at.col_ok && MX_IN(at.col, 8, C, kSiteGamma)) {
            const uint4 gv = __ldg(reinterpret_cast<const uint4*>(D.gamma + at.col));
            const float o = D.offset;
            ww[0] = pair(bf16lo(gv.x) + o, bf16hi(gv.x) + o);
            ww[1] = pair(bf16lo(gv.y) + o, bf16hi(gv.y) + o);
            ww[2] = pair(bf16lo(gv.z) + o, bf16hi(gv.z) + o);
            ww[3] = pair(bf16lo(gv.w) + o, bf16hi(gv.w) + o);
        } else {
            ww[0] = ww[1] = ww[2] = ww[3] = 0ull;
        }
        TileMax<G> m;
        m.colmax[0] = m.colmax[1] = m.colmax[2] = m.colmax[3] = 0u;
        uint16_t* nrm = D.normed + base;
#pragma unroll
        for (int i = 0; i < kR; ++i) {
            const float r = inv_rms[q * kR + i];
            const uint64_t rr = pair(r, r);
            const uint4 xi = xv[i];
            uint4 y;
            y.x = norm2(xi.x, rr, ww[0]);
            y.y = norm2(xi.y, rr, ww[1]);
            y.z = norm2(xi.z, rr, ww[2]);
            y.w = norm2(xi.w, rr, ww[3]);
            xv[i] = y;
            // streaming store, as for the codes (never read by this kernel)
            if (at.col_ok && i < at.nrows && MX_IN(base + i * C, 8, R * C, kSiteNormed))
                __stcs(reinterpret_cast<uint4*>(nrm + i * C), y);
            fold_col(m, y);
            if (i & 1) fold_rows(m, i >> 1, xv[i - 1], y);
        }
        quantize_tile<G>(xv, m, at, D.q_row, D.s_row, D.q_col, D.s_col, do_row, do_col, g, q);
    }

    if (K > 1) cluster_wait_acquire();  // peers may still read this CTA's `part`
}

// ---------------------------------------------------------------------------
// MXFP8 quantize (no norm). Every warp owns one 32-row x kWarpCols-column tile
// of the flattened list; tiles of an entry run row-stripe major.
// ---------------------------------------------------------------------------
template <int MAXN, bool MMA>
__global__ void __launch_bounds__(QuantGeo::kThreads, 4)
quant_kernel(const __grid_constant__ Table<MAXN> T) {
    // let a dependent launch that opted in (the GEMM after a quantize) start
    // its set-up now: it reads nothing before this grid has completed
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    using G = QuantGeo;
    constexpr int kR = G::kRows;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane % G::kGroupLanes, q = lane / G::kGroupLanes;
    const int64_t u = (int64_t)blockIdx.x * G::kWarps + warp;
    if (u >= T.total_units) return;  // whole warp leaves; no block barrier follows
    const DevDesc& D = T.d[find_entry(T, u)];
    const int64_t local = u - D.unit_begin;
    const int64_t stripe = local / D.col_tiles;
    const int64_t tile = local - stripe * D.col_tiles;

    TileAt at;
    at.row0 = stripe * kBlock + q * kR;
    at.col = tile * G::kWarpCols + g * 8;
    at.cols = D.cols;
    at.rows = D.rows;
    at.stripe = stripe;
    at.nrows = rows_inside(D.rows, at.row0, kR);
    at.mma = MMA;  // compile-time: the row-major paths carry no tiled state
    at.padded = T.scale_layout == 2;
    at.col_ok = at.col < D.cols;

    const uint16_t* p = D.x + at.row0 * at.cols + at.col;
    const bool do_row = T.rowwise != 0, do_col = T.columnwise != 0;
    uint4 xv[kR];
    TileMax<G> m;
    m.colmax[0] = m.colmax[1] = m.colmax[2] = m.colmax[3] = 0u;
    if (warp_full(at.col_ok && at.nrows == kR)) {
        load_tile<kR, true, false>(xv, p, at.cols, at.col_ok, at.nrows,
                                   at.row0 * at.cols + at.col, at.rows * at.cols);
#pragma unroll
        for (int i = 0; i < kR; ++i) {
            fold_col(m, xv[i]);
            if (i & 1) fold_rows(m, i >> 1, xv[i - 1], xv[i]);
        }
        emit_planes<G, true>(xv, m, at, D.q_row, D.s_row, D.q_col, D.s_col, do_row, do_col, g, q);
    } else {
        load_tile<kR, false, false>(xv, p, at.cols, at.col_ok, at.nrows,
                                    at.row0 * at.cols + at.col, at.rows * at.cols);
#pragma unroll
        for (int i = 0; i < kR; ++i) {
            fold_col(m, xv[i]);
            if (i & 1) fold_rows(m, i >> 1, xv[i - 1], xv[i]);
        }
        emit_planes<G, false>(xv, m, at, D.q_row, D.s_row, D.q_col, D.s_col, do_row, do_col, g, q);
    }
}

// An ordinary launch (no programmatic dependency on the kernel before it):
// the kernel starts after all earlier work on the stream has completed.
// mm_mxfp8 relies on this for its activation quantize: the GEMM after it
// fetches the weight before its own dependency wait.
template <typename Kern, int MAXN>
int launch(Kern kern, const Table<MAXN>& t, int64_t grid, int threads, int cluster,
           void* stream, int smem = 0) {
    if (const int e = hook_launch_error()) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    cfg.numAttrs = 0;
    if (cluster > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)cluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.numAttrs = 1;
    }
    cfg.attrs = attr;
    return (int)cudaLaunchKernelEx(&cfg, kern, t);
}

// Dynamic shared memory of the residual staging buffer (one pass of a CTA).
constexpr int kStageBytes = FusedGeo::kRows * FusedGeo::kThreads * 16;

// Fused launches, with the residual staging buffer when T.stage. Dynamic
// shared memory above the default limit is allowed once per instantiation
// and device (the cache lives in each instantiation: the kernels all have
// the same pointer type).
template <int MAXN, bool MMA, bool RES>
int launch_staged(const Table<MAXN>& t, int64_t grid, void* stream) {
    auto kern = fused_rmsnorm_quant_kernel<MAXN, MMA, RES>;
    if (const int e = hook_launch_error()) return e;
    const bool big = t.cluster > kPortableCluster;
    if (t.stage || big) {
        constexpr int kMaxDevices = 64;
        static bool staged[kMaxDevices] = {false}, wide[kMaxDevices] = {false};
        int dev = 0;
        int err = (int)cudaGetDevice(&dev);
        if (err != cudaSuccess) return err;
        const bool known = dev >= 0 && dev < kMaxDevices;
        if (t.stage && !(known && staged[dev])) {
            err = (int)cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            kStageBytes);
            if (err != cudaSuccess) return err;
            if (known) staged[dev] = true;
        }
        if (big && !(known && wide[dev])) {
            err = (int)cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                            1);
            if (err != cudaSuccess) return err;
            if (known) wide[dev] = true;
        }
    }
    return launch(kern, t, grid, FusedGeo::kThreads, t.cluster, stream,
                  t.stage ? kStageBytes : 0);
}

template <int MAXN>
int launch_fused_t(const Table<MAXN>& t, int64_t grid, void* stream) {
    if (t.residual)
        return t.scale_layout == 1 ? launch_staged<MAXN, true, true>(t, grid, stream)
                                   : launch_staged<MAXN, false, true>(t, grid, stream);
    return t.scale_layout == 1 ? launch_staged<MAXN, true, false>(t, grid, stream)
                               : launch_staged<MAXN, false, false>(t, grid, stream);
}

}  // namespace

int launch_fused(const Table<kSmallTable>& t, int64_t grid, void* stream) {
    return launch_fused_t(t, grid, stream);
}
int launch_fused(const Table<kLargeTable>& t, int64_t grid, void* stream) {
    return launch_fused_t(t, grid, stream);
}
int launch_quant(const Table<kSmallTable>& t, int64_t grid, void* stream) {
    return t.scale_layout == 1
        ? launch(quant_kernel<kSmallTable, true>, t, grid, QuantGeo::kThreads, 1, stream)
        : launch(quant_kernel<kSmallTable, false>, t, grid, QuantGeo::kThreads, 1, stream);
}
int launch_quant(const Table<kLargeTable>& t, int64_t grid, void* stream) {
    return t.scale_layout == 1
        ? launch(quant_kernel<kLargeTable, true>, t, grid, QuantGeo::kThreads, 1, stream)
        : launch(quant_kernel<kLargeTable, false>, t, grid, QuantGeo::kThreads, 1, stream);
}

int fused_chunk_cols() { return FusedGeo::kChunk; }

int bounds_status(bool clear, unsigned long long* out) {
    *out = 0;
#ifdef MXFP8_DEBUG_BOUNDS
    int err = (int)cudaDeviceSynchronize();
    if (err != cudaSuccess) return err;
    err = (int)cudaMemcpyFromSymbol(out, g_bounds_status, sizeof *out);
    if (err != cudaSuccess) return err;
    if (clear && *out != 0) {
        const unsigned long long zero = 0;
        err = (int)cudaMemcpyToSymbol(g_bounds_status, &zero, sizeof zero);
    }
    return err;
#else
    (void)clear;
    return cudaSuccess;
#endif
}

int fused_resident_ctas() {
    constexpr int kMaxDevices = 64;
    static int cache[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (dev >= 0 && dev < kMaxDevices && cache[dev] > 0) return cache[dev];
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm, fused_rmsnorm_quant_kernel<kLargeTable, false, false>, FusedGeo::kThreads,
            0) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    const int n = sms * per_sm;
    if (dev >= 0 && dev < kMaxDevices) cache[dev] = n;
    return n;
}

int fused_max_cluster() {
    constexpr int kMaxDevices = 64;
    static int cache[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    if (dev >= 0 && dev < kMaxDevices && cache[dev] > 0) return cache[dev];
    // sizes above the portable limit only where the device allows them
    int top = kPortableCluster;
    if (cudaFuncSetAttribute(fused_rmsnorm_quant_kernel<kLargeTable, false, false>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess)
        top = kMaxCluster;
    else
        cudaGetLastError();
    int best = 1;
    for (int k = top; k >= 2; --k) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(k * 64), 1, 1);
        cfg.blockDim = dim3(FusedGeo::kThreads, 1, 1);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)k;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, fused_rmsnorm_quant_kernel<kLargeTable, false, false>,
                                           &cfg) ==
                cudaSuccess && n > 0) {
            best = k;
            break;
        }
        cudaGetLastError();
    }
    if (dev >= 0 && dev < kMaxDevices) cache[dev] = best;
    return best;
}

}  // namespace mx
