// mx_umma.h -- bit layouts of the tcgen05 (5th-generation tensor core)
// descriptors used by the block-scaled MXFP8 GEMM (mxfp8_gemm.cu). Plain
// integer encoders, compiled for host and device, so that the CPU tests can
// check every field against hand-worked values.
//
// Field positions follow the PTX ISA's tcgen05 chapter ("Shared memory
// descriptor" and "Instruction descriptor" for .kind::mxf8f6f4):
//
// Shared-memory matrix descriptor (64 bits):
//   [ 0,14) matrix start address >> 4        [16,30) leading byte offset >> 4
//   [32,46) stride byte offset >> 4          [46,49) fixed 0b001
//   [49,52) matrix base offset (0 here)      [52]    leading-offset mode (0)
//   [61,64) swizzle: 0 none, 2 128-byte, 4 64-byte, 6 32-byte
// Instruction descriptor, block-scaled kinds (32 bits):
//   [ 4, 6) scale-factor id of B (which byte of the 32-bit scale word)
//   [ 7,10) A format (E4M3 = 0)     [10,13) B format (E4M3 = 0)
//   [13] negate A  [14] negate B    [15] A MN-major  [16] B MN-major (0: K-major)
//   [17,23) N >> 3                  [23] scale format (1: UE8M0)
//   [24,29) M >> 4                  [29,31) scale-factor id of A
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define MX_HD __host__ __device__ __forceinline__
#else
#define MX_HD inline
#endif

namespace mx {
namespace umma {

constexpr uint32_t kSwizzleNone = 0;
constexpr uint32_t kSwizzle128B = 2;

// Descriptor of an operand tile in shared memory.
MX_HD uint64_t smem_desc(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                         uint32_t swizzle) {
    return (uint64_t)((smem_addr & 0x3FFFFu) >> 4) |
           ((uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) |
           ((uint64_t)(swizzle & 7u) << 61);
}

// K-major operand, rows of 128 bytes written by a 128-byte-swizzled TMA load:
// 8-row groups of 1024 bytes (the stride offset); the leading offset is not
// used by swizzled K-major layouts (set to 16 bytes).
MX_HD uint64_t kmajor_sw128_desc(uint32_t smem_addr) {
    return smem_desc(smem_addr, 16, 1024, kSwizzle128B);
}

// A 32-row x 16-byte block of scale factors (one 128 x 4 scale tile of the
// tiled layout, 512 contiguous bytes), no swizzle: 8-row core matrices of
// 128 bytes, 128 bytes apart.
MX_HD uint64_t scale_tile_desc(uint32_t smem_addr) {
    return smem_desc(smem_addr, 0, 128, kSwizzleNone);
}

// kind::mxf8f6f4 with block scaling: E4M3 x E4M3, UE8M0 scales, both operands
// K-major, float32 accumulation; sf_a / sf_b pick the byte of each 32-bit
// scale word that this K = 32 step uses.
MX_HD uint32_t idesc_mxf8(uint32_t M, uint32_t N, uint32_t sf_a, uint32_t sf_b) {
    return ((sf_b & 3u) << 4) | ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24) |
           ((sf_a & 3u) << 29);
}

// Tensor-memory address: lane in bits 16-31, column in bits 0-15.
MX_HD uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col) {
    return base + (lane << 16) + col;
}

}  // namespace umma
}  // namespace mx
