// mxfp8_mm.cu -- MXFP8 matrix multiply consumer of the planes (Megatron
// inference page "core.inference.quantization.utils", `mm_mxfp8`: quantize the
// bf16 activation on the fly, the weight already quantized, then a
// block-scaled GEMM).
//
// Here: the activation x [M, K] is quantized rowwise by this library's
// quantize kernel, with its scales in the tiled GEMM-operand layout, into a
// scratch area; this library's tcgen05 block-scaled GEMM (mxfp8_gemm.cu) then
// computes out = x_q w_q^T with float32 accumulation and a bf16 result. Two
// launches on the caller's stream (mm_mxfp8_quantized: the GEMM alone, on an
// activation the caller quantized).
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "mx_gemm.h"
#include "mx_table.h"
#include "mx_trace.h"
#include "mxfp8norm.h"

namespace mx {
int set_error(int code, const char* fmt, ...);  // mxfp8_api.cu
}

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t align256(int64_t v) { return (v + 255) / 256 * 256; }

// Bytes of the quantized activation in the scratch: codes, then tiled scales.
int64_t act_bytes(int64_t M, int64_t K) {
    return align256(M * K) + align256(ceil_div(M, 128) * 128 * ceil_div(K / 32, 4) * 4);
}

int gemm_error(int err) {
    cudaGetLastError();
    return mx::set_error(MXFP8_ERR_CUDA, "GEMM launch failed: %s",
                         cudaGetErrorString(static_cast<cudaError_t>(err)));
}

// The product with a given scratch area (quantized activation: codes, then
// scales). Pointers and sizes are already checked.
int mm_run(const void* x, int64_t M, int64_t K, const void* w_q, const void* w_s, int64_t N,
           void* out, uint8_t* scratch, void* stream) {
    // 1. quantize x rowwise into the scratch, scales tiled for the GEMM. The
    // tiled buffer's padding (rows past M, scale columns past K / 32) is never
    // read: the GEMM's rows past M are not stored and its last K step issues
    // only the 32-column blocks that exist.
    uint8_t* xq = scratch;
    uint8_t* xs = xq + align256(M * K);
    mx::GemmPlan plan;
    std::memset(&plan, 0, sizeof plan);
    const int mr = mx::gemm_plan(&plan, xq, xs, static_cast<const uint8_t*>(w_q),
                                 static_cast<const uint8_t*>(w_s), static_cast<uint16_t*>(out),
                                 M, N, K);
    if (mr != 0)
        return mx::set_error(MXFP8_ERR_CUDA, "cannot make the TMA tensor map of %s",
                             mr == -1 ? "x" : mr == -2 ? "w_q" : "out");
    // the quantize below writes only the scratch and is an ordinary launch
    // (it starts after all earlier work): the GEMM after it may fetch the
    // weight before its dependency wait
    plan.thin.weight_early = 1;
    mx::Table<mx::kSmallTable> t;
    std::memset(&t, 0, sizeof t);
    t.n = 1;
    t.rowwise = 1;
    t.columnwise = 0;
    t.scale_layout = MXFP8_SCALES_MMA_TILED;
    t.d[0].x = static_cast<const uint16_t*>(x);
    t.d[0].q_row = xq;
    t.d[0].s_row = xs;
    t.d[0].rows = M;
    t.d[0].cols = K;
    t.d[0].col_tiles = (int32_t)ceil_div(K, mx::QuantGeo::kWarpCols);
    t.total_units = ceil_div(M, mx::kBlock) * t.d[0].col_tiles;
    int err = mx::launch_quant(t, ceil_div(t.total_units, mx::QuantGeo::kWarps), stream);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return mx::set_error(MXFP8_ERR_CUDA, "quantize launch failed: %s",
                             cudaGetErrorString(static_cast<cudaError_t>(err)));
    }
    // 2. out = x_q w_q^T on the tensor cores
    err = mx::gemm_launch(plan, stream);
    return err != cudaSuccess ? gemm_error(err) : MXFP8_OK;
}

int check_mm_args(const void* x, int64_t M, int64_t K, const void* w_q, const void* w_s,
                  int64_t N, void* out) {
    constexpr int64_t kMax = (int64_t(1) << 31) - 1;
    if (M <= 0 || N <= 0 || K <= 0 || K % 32 != 0 || N % 16 != 0 || M > kMax || N > kMax ||
        K > kMax || ceil_div(M, 128) * ceil_div(N, 256) > kMax)
        return mx::set_error(MXFP8_ERR_SHAPE,
                             "mm_mxfp8 needs M, N, K in [1, 2^31), K %% 32 == 0 and "
                             "N %% 16 == 0 (got M=%lld N=%lld K=%lld)", (long long)M,
                             (long long)N, (long long)K);
    const void* ptrs[] = {x, w_q, w_s, out};
    const char* names[] = {"x", "w_q", "w_s", "out"};
    for (int i = 0; i < 4; ++i)
        if (ptrs[i] == nullptr || (reinterpret_cast<uintptr_t>(ptrs[i]) & 255u) != 0)
            return mx::set_error(MXFP8_ERR_POINTER, "%s must be non-NULL and 256-byte aligned",
                                 names[i]);
    return MXFP8_OK;
}

// ---------------------------------------------------------------------------
// Scratch for callers that cannot allocate device memory (mm_mxfp8_static).
// A file-scope device array: every GPU that loads this library holds it until
// the process exits. Its device address is looked up once per device.
// ---------------------------------------------------------------------------
static __device__ __align__(256) uint8_t g_mm_static_scratch[MXFP8_MM_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
uint8_t* g_static_ptr[kMaxDevices] = {nullptr};

// Device address of the static scratch on the current device (set-up on the
// first use per device: the host-side name of the array is only a stand-in).
int static_scratch(uint8_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return mx::set_error(MXFP8_ERR_CUDA, "no usable current device");
    }
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (g_static_ptr[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_mm_static_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return mx::set_error(MXFP8_ERR_CUDA, "cudaGetSymbolAddress of the scratch failed: %s",
                                 cudaGetErrorString(e));
        }
        g_static_ptr[dev] = static_cast<uint8_t*>(p);
    }
    *out = g_static_ptr[dev];
    return MXFP8_OK;
}

}  // namespace

extern "C" {

size_t mm_mxfp8_workspace_size(int64_t M, int64_t K) {
    if (M <= 0 || K <= 0 || K % 32 != 0) return 0;
    return (size_t)act_bytes(M, K);
}

int mm_mxfp8(const void* x, int64_t M, int64_t K, const void* w_q, const void* w_s, int64_t N,
             void* out, void* workspace, size_t workspace_bytes, void* stream) {
    const mx::TraceRange trace("mm_mxfp8");
    mx::set_error(MXFP8_OK, "");
    int rc = check_mm_args(x, M, K, w_q, w_s, N, out);
    if (rc != MXFP8_OK) return rc;
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return mx::set_error(MXFP8_ERR_POINTER, "workspace must be non-NULL and 256-byte aligned");
    const int64_t need_act = act_bytes(M, K);
    if ((int64_t)workspace_bytes < need_act)
        return mx::set_error(MXFP8_ERR_SHAPE, "workspace of %zu bytes < %lld needed",
                             workspace_bytes, (long long)need_act);
    return mm_run(x, M, K, w_q, w_s, N, out, static_cast<uint8_t*>(workspace), stream);
}

int mm_mxfp8_quantized(const void* x_q, const void* x_s, int64_t M, int64_t K, const void* w_q,
                       const void* w_s, int64_t N, void* out, void* stream) {
    const mx::TraceRange trace("mm_mxfp8_quantized");
    mx::set_error(MXFP8_OK, "");
    int rc = check_mm_args(x_q, M, K, w_q, w_s, N, out);
    if (rc != MXFP8_OK) return rc;
    if (x_s == nullptr || (reinterpret_cast<uintptr_t>(x_s) & 255u) != 0)
        return mx::set_error(MXFP8_ERR_POINTER, "x_s must be non-NULL and 256-byte aligned");
    mx::GemmPlan plan;
    std::memset(&plan, 0, sizeof plan);
    const int mr = mx::gemm_plan(&plan, static_cast<const uint8_t*>(x_q),
                                 static_cast<const uint8_t*>(x_s), static_cast<const uint8_t*>(w_q),
                                 static_cast<const uint8_t*>(w_s), static_cast<uint16_t*>(out), M,
                                 N, K);
    if (mr != 0)
        return mx::set_error(MXFP8_ERR_CUDA, "cannot make the TMA tensor map of %s",
                             mr == -1 ? "x_q" : mr == -2 ? "w_q" : "out");
    const int err = mx::gemm_launch(plan, stream);
    return err != cudaSuccess ? gemm_error(err) : MXFP8_OK;
}

int mm_mxfp8_static(const void* x, int64_t M, int64_t K, const void* w_q, const void* w_s,
                    int64_t N, void* out, void* stream) {
    const mx::TraceRange trace("mm_mxfp8_static");
    mx::set_error(MXFP8_OK, "");
    int rc = check_mm_args(x, M, K, w_q, w_s, N, out);
    if (rc != MXFP8_OK) return rc;
    const int64_t need_act = act_bytes(M, K);
    if (need_act > (int64_t)MXFP8_MM_STATIC_SCRATCH_BYTES)
        return mx::set_error(MXFP8_ERR_SHAPE,
                             "mm_mxfp8_static: the quantized activation of M=%lld K=%lld needs "
                             "%lld bytes, more than the %lld-byte static scratch",
                             (long long)M, (long long)K, (long long)need_act,
                             (long long)MXFP8_MM_STATIC_SCRATCH_BYTES);
    uint8_t* scratch = nullptr;
    rc = static_scratch(&scratch);
    if (rc != MXFP8_OK) return rc;
    return mm_run(x, M, K, w_q, w_s, N, out, scratch, stream);
}

int64_t mxfp8_device_status(int clear) {
    mx::set_error(MXFP8_OK, "");
    unsigned long long gemm = 0, bounds = 0;
    int err = mx::gemm_status(clear != 0, &gemm);
    if (err == cudaSuccess) err = mx::bounds_status(clear != 0, &bounds);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return mx::set_error(MXFP8_ERR_CUDA, "cannot read the device status: %s",
                             cudaGetErrorString(static_cast<cudaError_t>(err)));
    }
    return (int64_t)(gemm != 0 ? gemm : bounds);
}

}  // extern "C"
