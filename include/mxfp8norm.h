/*
 * mxfp8norm.h -- C ABI of the fused RMSNorm + MXFP8 block-quantization library
 * (libmxfp8norm.so, sm_103a).
 *
 * What the calls compute
 * ----------------------
 * MXFP8 here is 32-element blocks (Megatron-FSDP page
 * "core.distributed.fsdp.src.megatron_fsdp.experimental.quantized_dbuffer",
 * Data `_MXFP8_BLOCK_SIZE`) of float8_e4m3fn codes sharing one float8_e8m0fnu
 * scale byte (MAX Mojo page "DistributedAllGatherRMSNormQuantMXFP8",
 * Parameters `quant_dtype`, `scales_dtype`). Each call writes up to two planes
 * of every input matrix v [rows, cols]:
 *
 *   rowwise    q_row [rows, cols] row-major and s_row [rows, cols/32]: one scale
 *              per 32 consecutive columns of a row (the Mojo page, Args
 *              `outputs_quant`, `outputs_scale` [rows, cols / 32]).
 *   columnwise q_col [rows, cols] in the SAME row-major layout as q_row (not
 *              transposed) and s_col [rows/32, cols]: one scale per 32
 *              consecutive rows (starting at a multiple of 32) of a column
 *              (the FSDP page, `_columnwise_scale_layout`, `_block_atomic_to_flat`).
 *
 * Scales are compact and unswizzled by default (the FSDP page, class
 * `QuantizedDBuffer` and `get_tensor_view`); the *_ex calls can write them in
 * the tiled layout of a block-scaled GEMM operand instead. For a block with
 * largest magnitude amax:
 * amax == 0 gives scale byte 0; otherwise e = clamp(floor(log2(amax)) - 8,
 * -127, 127), the byte is e + 127, and every element v is coded as the E4M3
 * value nearest to v * 2^-e (ties to even, magnitudes past 448 clamped to 448,
 * sign kept). The pages do not state this rule; it is this library's choice.
 *
 * rmsnorm_quant_mxfp8 first computes, per row in float32,
 *   normed = bf16( (x * 1/sqrt(mean(x^2) + eps)) * (gamma + weight_offset) )
 * (the Mojo page, Args `gammas`, `epsilons` (float32), `weight_offsets`,
 * `outputs_normed`) and quantizes that same bf16 (the Mojo page's description:
 * the quantize reads the bf16 that lands in outputs_normed, so it is
 * byte-identical to quant_mxfp8 applied to `normed`). quant_mxfp8 quantizes its
 * bf16 input directly (weight storage: the Megatron inference page
 * "core.inference.quantization.utils", `quantize_params_to_mxfp8`, `_to_bf16`).
 *
 * Conventions for every call
 * --------------------------
 *  - All buffers are DEVICE memory of the current device, owned by the caller;
 *    the library allocates no memory and never synchronizes (except
 *    mxfp8_device_status). Outputs are overwritten in place, so a capture of
 *    the quantize calls in a CUDA graph stays valid across replays on the same
 *    buffers (the inference page, `quantize_params_to_mxfp8`, persistent
 *    buffers).
 *  - Matrices are dense row-major: element (r, c) at index r * cols + c.
 *  - Every pointer that a call uses must be non-NULL and 16-byte aligned.
 *    Pointers of disabled planes are ignored and may be NULL.
 *  - cols must be a multiple of 32; with columnwise, rows too. rows == 0 or
 *    cols == 0 makes an entry a no-op.
 *  - The whole list is processed by ONE kernel launch enqueued on `stream`
 *    (a cudaStream_t; NULL is the legacy default stream). The call returns as
 *    soon as the launch is enqueued.
 *  - Inputs must not overlap outputs. NaN and infinite inputs are outside the
 *    contract: the kernels do not fault or hang on them, but the codes written
 *    for their blocks are unspecified.
 *  - Return value: MXFP8_OK (0) or a negative MXFP8_ERR_* code, in which case
 *    nothing was launched and mxfp8_last_error() describes the problem.
 */
#ifndef MXFP8NORM_H
#define MXFP8NORM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MXFP8_ABI_VERSION 7
#define MXFP8_BLOCK_SIZE 32
#define MXFP8_MAX_TENSORS 256
#define MXFP8_MAX_UPDATE 256

/* Scale layouts (the scale_layout argument of the *_ex calls). */
#define MXFP8_SCALES_COMPACT 0   /* s_row [rows, cols/32], s_col [rows/32, cols], row-major */
#define MXFP8_SCALES_MMA_TILED 1 /* tiled layout of a block-scaled GEMM operand, below   */
#define MXFP8_SCALES_PADDED 2    /* row-major, pitches padded to TE's allocation shape   */

#define MXFP8_OK 0
#define MXFP8_ERR_POINTER (-1) /* a used pointer is NULL or not 16-byte aligned */
#define MXFP8_ERR_SHAPE (-2)   /* negative size, cols % 32 != 0, or rows % 32 != 0 with columnwise */
#define MXFP8_ERR_FLAGS (-3)   /* neither plane requested, or unknown scale layout */
#define MXFP8_ERR_COUNT (-4)   /* desc == NULL, n < 1 or n > MXFP8_MAX_TENSORS */
#define MXFP8_ERR_CUDA (-5)    /* the CUDA runtime rejected the launch */

/* One list entry. The fused call reads x, gamma, eps and weight_offset and
 * writes normed; both calls write the planes their flags select. */
typedef struct mxfp8_desc {
    const void* x;       /* in:  bf16 [rows, cols]                          */
    const void* gamma;   /* in:  bf16 [cols]           (fused call only)    */
    void* normed;        /* out: bf16 [rows, cols]     (fused call only)    */
    void* q_row;         /* out: e4m3 codes [rows, cols]      (rowwise)     */
    void* s_row;         /* out: e8m0 bytes [rows, cols/32]   (rowwise)     */
    void* q_col;         /* out: e4m3 codes [rows, cols]      (columnwise)  */
    void* s_col;         /* out: e8m0 bytes [rows/32, cols]   (columnwise)  */
    int64_t rows;
    int64_t cols;
    float eps;           /* float32 epsilon inside the square root (fused)  */
    float weight_offset; /* float32 added to every gamma element (fused)    */
} mxfp8_desc;

/* Fused RMSNorm + MXFP8 quantization of n matrices in one launch.
 * rowwise / columnwise (0 or 1) select the planes; at least one must be set.
 * Errors: MXFP8_ERR_COUNT, MXFP8_ERR_FLAGS, MXFP8_ERR_SHAPE, MXFP8_ERR_POINTER,
 * MXFP8_ERR_CUDA. */
int rmsnorm_quant_mxfp8(const mxfp8_desc* desc, int n, int rowwise, int columnwise,
                        void* stream);

/* MXFP8 quantization (no norm) of the bf16 matrices desc[i].x in one launch;
 * gamma, normed, eps and weight_offset are ignored. Same flags and errors. */
int quant_mxfp8(const mxfp8_desc* desc, int n, int rowwise, int columnwise,
                void* stream);

/* The same two calls under the names of the library's first interface
 * sketch (mxfp8_rmsnorm_quant == rmsnorm_quant_mxfp8, mxfp8_quant ==
 * quant_mxfp8): identical arguments, behaviour and errors. */
int mxfp8_rmsnorm_quant(const mxfp8_desc* desc, int n, int rowwise, int columnwise,
                        void* stream);
int mxfp8_quant(const mxfp8_desc* desc, int n, int rowwise, int columnwise, void* stream);

/* The same calls with a choice of scale layout (NEXT item of the FSDP page:
 * TE pads its scale planes for compute, `_pad_rowwise_scale`,
 * `_pad_columnwise_scale`, without stating the shapes; the tiled layout here
 * is the one Blackwell block-scaled matrix multiplies document for 1-D
 * 32-element UE8M0 scale vectors, so the planes can feed such a GEMM as is).
 *
 * MXFP8_SCALES_MMA_TILED: take an operand with M rows (its non-reduced
 * dimension) and Kb scale columns (K / 32). Its scales occupy
 * roundup(M, 128) * roundup(Kb, 4) bytes cut into tiles of 128 rows x 4 scale
 * columns, 512 contiguous bytes each, row tiles outer; inside a tile, row m
 * and scale column k sit at byte (m % 32) * 16 + ((m / 32) % 4) * 4 + k % 4.
 *   s_row: the rowwise plane is an operand with M = rows, Kb = cols / 32,
 *          so s_row needs roundup(rows, 128) * roundup(cols / 32, 4) bytes.
 *   s_col: the columnwise plane is an operand with M = cols, Kb = rows / 32
 *          (its blocks run down the rows), so s_col needs
 *          roundup(cols, 128) * roundup(rows / 32, 4) bytes.
 * MXFP8_SCALES_PADDED: the compact row-major arrays with padded pitches, i.e.
 * TE's physical allocation shape (the FSDP page's `_pad_rowwise_scale`,
 * `_pad_columnwise_scale`; the shapes are this library's reading):
 *   s_row [roundup(rows, 128), roundup(cols / 32, 4)], scale (r, k) at
 *         r * roundup(cols / 32, 4) + k;
 *   s_col [roundup(rows / 32, 4), roundup(cols, 128)], scale (b, c) at
 *         b * roundup(cols, 128) + c.
 * In both non-compact layouts the calls write only the unpadded positions; the
 * padding keeps whatever the buffer held (zero it once when it is allocated).
 * Errors: as above, and MXFP8_ERR_FLAGS for an unknown scale_layout. */
int rmsnorm_quant_mxfp8_ex(const mxfp8_desc* desc, int n, int rowwise, int columnwise,
                           int scale_layout, void* stream);
int quant_mxfp8_ex(const mxfp8_desc* desc, int n, int rowwise, int columnwise,
                   int scale_layout, void* stream);

/* Residual stream of one list entry (add_rmsnorm_quant_mxfp8). */
typedef struct mxfp8_residual {
    const void* residual; /* in:  bf16 [rows, cols] added to x, or NULL (nothing added) */
    void* residual_out;   /* out: bf16 [rows, cols] h = x + residual, or NULL (not written) */
} mxfp8_residual;

/* Fused residual add + RMSNorm + MXFP8 (the single-GPU counterpart of the Mojo
 * page's outputs_residual: the pre-norm activations that the normalization
 * reads, written out for the next residual connection). Per element,
 * h = bf16(x + residual) with one round-to-nearest-even of the exact sum;
 * residual_out = h; then normed = RMSNorm(h) and both planes of normed, as in
 * rmsnorm_quant_mxfp8_ex. res[i] belongs to desc[i]; both of its pointers may
 * be NULL; non-NULL ones must be 16-byte aligned and must not overlap x
 * (residual_out may not alias x or residual). Errors as for
 * rmsnorm_quant_mxfp8_ex; MXFP8_ERR_POINTER if res is NULL. */
int add_rmsnorm_quant_mxfp8(const mxfp8_desc* desc, const mxfp8_residual* res, int n,
                            int rowwise, int columnwise, int scale_layout, void* stream);

/* The four planes of one MXFP8 tensor [rows, cols] (mxfp8_update_planes). */
typedef struct mxfp8_planes {
    void* q_row; /* e4m3 codes [rows, cols]                       */
    void* s_row; /* e8m0 rowwise scales (layout set by the call)   */
    void* q_col; /* e4m3 codes [rows, cols], same layout as q_row  */
    void* s_col; /* e8m0 columnwise scales (layout set by the call) */
    int64_t rows;
    int64_t cols;
} mxfp8_planes;

/* In-place plane update (the FSDP page, `update_mxfp8_tensor`): dst[i] takes
 * the planes that rowwise / columnwise select from src[i], whose scales are
 * compact ([rows, cols/32] and [rows/32, cols]); dst's scales are written in
 * dst_scale_layout (MXFP8_SCALES_*), padding untouched. A selected plane that
 * src lacks (both of its pointers NULL) is cleared in dst: its codes and its
 * whole scale buffer (padding included) are set to zero. Unselected planes of
 * dst are not touched; src is only read. One launch for the whole list.
 * Shapes of src[i] and dst[i] must match (cols % 32 == 0; rows % 32 == 0 when
 * columnwise is selected); dst buffers of selected planes must be non-NULL and
 * 16-byte aligned; src may not overlap dst. n in [1, MXFP8_MAX_UPDATE].
 * Errors: MXFP8_ERR_COUNT, MXFP8_ERR_FLAGS, MXFP8_ERR_SHAPE, MXFP8_ERR_POINTER,
 * MXFP8_ERR_CUDA. */
int mxfp8_update_planes(const mxfp8_planes* src, const mxfp8_planes* dst, int n, int rowwise,
                        int columnwise, int dst_scale_layout, void* stream);

/* MXFP8 matrix multiply consuming the planes (the Megatron inference page,
 * `mm_mxfp8`: the bf16 activation is quantized on the fly, the weight is
 * already quantized): out[M, N] = x[M, K] w^T, where
 *   x    bf16 [M, K] row-major;
 *   w_q  e4m3 codes [N, K] row-major: the rowwise plane of the weight [N, K];
 *   w_s  its scales in MXFP8_SCALES_MMA_TILED layout (an operand with N rows
 *        and K / 32 scale columns), as quant_mxfp8_ex writes them;
 *   out  bf16 [M, N] row-major.
 * x is quantized rowwise (the encoder of quant_mxfp8) into `workspace` (codes,
 * then tiled scales), then this library's block-scaled GEMM on the tensor
 * cores (tcgen05, E4M3 x E4M3 with UE8M0 block scales, float32 accumulation,
 * one rounding to bf16) writes out: two launches on `stream`.
 * Requirements: M, N, K in [1, 2^31), K % 32 == 0, N % 16 == 0; every pointer
 * 256-byte aligned; workspace_bytes >= mm_mxfp8_workspace_size(M, K). The
 * caller owns the workspace; calls that share it must not overlap on the GPU.
 * Errors: MXFP8_ERR_SHAPE, MXFP8_ERR_POINTER, MXFP8_ERR_CUDA (a launch the
 * runtime rejects, or a TMA tensor map the driver cannot make). */
size_t mm_mxfp8_workspace_size(int64_t M, int64_t K);

/* The GEMM of mm_mxfp8 alone, for an activation that is already quantized
 * (for instance the rowwise plane that rmsnorm_quant_mxfp8_ex writes with
 * MXFP8_SCALES_MMA_TILED, so that a norm + quantize feeds the matrix multiply
 * without the bf16 being read again): out[M, N] = deq(x_q, x_s) deq(w_q, w_s)^T
 * with deq(q, s)[r, k] = e4m3(q[r, k]) * 2^(s(r, k / 32) - 127), where
 *   x_q  e4m3 codes [M, K] row-major;
 *   x_s  their scales in MXFP8_SCALES_MMA_TILED layout (an operand with M rows
 *        and K / 32 scale columns);
 *   w_q, w_s, out  as for mm_mxfp8.
 * One launch on `stream`, no scratch. The tiled buffers' padding (rows past M
 * or N, scale columns past K / 32) is never read. The same kernel as the
 * second launch of mm_mxfp8: on the same quantized operands the two give the
 * same bytes.
 * Requirements and errors as for mm_mxfp8 (every pointer 256-byte aligned);
 * there is no workspace. */
int mm_mxfp8_quantized(const void* x_q, const void* x_s, int64_t M, int64_t K, const void* w_q,
                       const void* w_s, int64_t N, void* out, void* stream);
int mm_mxfp8(const void* x, int64_t M, int64_t K, const void* w_q, const void* w_s, int64_t N,
             void* out, void* workspace, size_t workspace_bytes, void* stream);

/* mm_mxfp8 for callers that cannot allocate device memory: the same product,
 * with its scratch (the quantized activation) taken from a fixed device array
 * inside this library instead of a caller-provided workspace. It is meant for
 * code that may not call cudaMalloc: a plugin or callback running inside
 * another framework whose caching allocator owns all device memory and cannot
 * be reached from here, or a latency-critical loop where cudaMalloc's implicit
 * device synchronization is not allowed. The pages have no counterpart of this
 * entry point.
 *
 *  - The array holds MXFP8_MM_STATIC_SCRATCH_BYTES bytes on every GPU that
 *    loads the library, until the process exits. Problems whose quantized
 *    activation, M * K code bytes plus roundup(M, 128) * roundup(K / 32, 4)
 *    scale bytes (each rounded up to 256), does not fit are rejected with
 *    MXFP8_ERR_SHAPE; everything that fits runs.
 *  - The first call on a device does the set-up: it looks up the array's
 *    device address (cudaGetSymbolAddress). Make that first call before any
 *    stream capture. No call allocates device memory (no cudaMalloc, cudaFree
 *    or allocating library routine).
 *  - Every call shares the one array and leaves its contents behind (nothing in
 *    it needs to start at zero); calls that overlap on the GPU (e.g. on two
 *    streams) race and must not be used.
 *  - Arguments, layouts and errors as for mm_mxfp8. */
#define MXFP8_MM_STATIC_SCRATCH_BYTES (32ull << 20)
int mm_mxfp8_static(const void* x, int64_t M, int64_t K, const void* w_q, const void* w_s,
                    int64_t N, void* out, void* stream);

/* Device-side status of this library's kernels on the current device: 0 if
 * nothing was recorded since the last clear, else a positive code:
 *  - bits 48-55 in 1..4: a wait of the GEMM on its own pipeline gave up after
 *    2 s instead of hanging (bits 0-47: the CTA); that launch left its output
 *    incomplete;
 *  - bits 48-55 in 0x81..0x89 (bounds-checking build libmxfp8norm_bounds.so
 *    only): a quantize kernel computed an access outside the extent this
 *    header states for a buffer, and skipped it (bits 0-47: the element
 *    offset; 0x81 x, 0x82 residual, 0x83 residual_out, 0x84 gamma,
 *    0x85 normed, 0x86 q_row, 0x87 s_row, 0x88 q_col, 0x89 s_col).
 * Synchronizes the device; clear != 0 resets the status. Returns
 * MXFP8_ERR_CUDA if the status cannot be read. The pages have no
 * counterpart. */
int64_t mxfp8_device_status(int clear);

/* Testing hooks, process-wide, for exercising error paths (the pages have no
 * counterpart):
 *   MXFP8_HOOK_FAIL_LAUNCH  value != 0: every later call that passes its
 *       argument checks returns MXFP8_ERR_CUDA ("invalid argument") as if the
 *       CUDA runtime had rejected its launch; nothing is launched. 0 restores.
 *   MXFP8_HOOK_MAX_CLUSTER  value > 0: the fused calls use thread-block
 *       clusters of at most `value` CTAs (1: one CTA per 32-row stripe, the
 *       path taken where the device co-schedules no cluster); 0 lifts the cap.
 *   MXFP8_HOOK_GEMM_FORM  the form of the matrix multiplies: 1 the 256 x 256
 *       output-tile form, 2 the swapped-operand form (where M <= 2048; the
 *       tile form above), 0 the planner's choice.
 *   MXFP8_HOOK_GEMM_SPLITS  value 1-3: the swapped-operand form splits K over
 *       that many CTA pairs (fewer where K has fewer 128-element steps);
 *       0 the planner's choice. Larger values are rejected.
 * Returns the hook's previous value, or MXFP8_ERR_FLAGS for an unknown hook
 * or a value out of range. Not meant to be set while other threads call. */
#define MXFP8_HOOK_FAIL_LAUNCH 1
#define MXFP8_HOOK_MAX_CLUSTER 2
#define MXFP8_HOOK_GEMM_FORM 3
#define MXFP8_HOOK_GEMM_SPLITS 4
int mxfp8_set_test_hook(int hook, int value);

/* Text of the last error raised by a call on this host thread ("" if none).
 * The pointer stays valid until the next call on the same thread. */
const char* mxfp8_last_error(void);

/* MXFP8_ABI_VERSION of the loaded library. */
int mxfp8_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MXFP8NORM_H */
