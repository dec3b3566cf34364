// mxfp8_api.cu -- the C ABI (include/mxfp8norm.h): argument checks, the
// per-launch descriptor table, and one kernel launch per call.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "mx_table.h"
#include "mx_update.h"
#include "mx_trace.h"
#include "mxfp8norm.h"

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

bool aligned16(const void* p) {
    return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Checks one entry; returns MXFP8_OK or an error code with the message set.
int check_entry(const mxfp8_desc& e, int i, bool fused, bool rowwise, bool columnwise) {
    if (e.rows < 0 || e.cols < 0)
        return fail(MXFP8_ERR_SHAPE, "entry %d: negative shape [%lld, %lld]", i,
                    (long long)e.rows, (long long)e.cols);
    if (e.cols % mx::kBlock != 0)
        return fail(MXFP8_ERR_SHAPE, "entry %d: cols = %lld is not a multiple of 32", i,
                    (long long)e.cols);
    if (columnwise && e.rows % mx::kBlock != 0)
        return fail(MXFP8_ERR_SHAPE,
                    "entry %d: rows = %lld is not a multiple of 32 (columnwise plane)", i,
                    (long long)e.rows);
    if (e.rows > (int64_t(1) << 31) || e.cols > (int64_t(1) << 31) ||
        (e.rows > 0 && e.cols > (int64_t(1) << 46) / e.rows))
        return fail(MXFP8_ERR_SHAPE, "entry %d: shape [%lld, %lld] is too large", i,
                    (long long)e.rows, (long long)e.cols);
    if (e.rows == 0 || e.cols == 0) return MXFP8_OK;
    struct {
        const void* p;
        const char* name;
        bool used;
    } ptrs[] = {
        {e.x, "x", true},
        {e.gamma, "gamma", fused},
        {e.normed, "normed", fused},
        {e.q_row, "q_row", rowwise},
        {e.s_row, "s_row", rowwise},
        {e.q_col, "q_col", columnwise},
        {e.s_col, "s_col", columnwise},
    };
    for (const auto& p : ptrs)
        if (p.used && !aligned16(p.p))
            return fail(MXFP8_ERR_POINTER, "entry %d: %s is %s", i, p.name,
                        p.p ? "not 16-byte aligned" : "NULL");
    return MXFP8_OK;
}

template <int MAXN>
int fill_and_launch(bool fused, const mxfp8_desc* d, const mxfp8_residual* res, int n,
                    bool rowwise, bool columnwise, int scale_layout, int64_t max_cols,
                    void* stream) {
    mx::Table<MAXN> tab;
    std::memset(&tab, 0, sizeof tab);
    tab.rowwise = rowwise;
    tab.columnwise = columnwise;
    tab.scale_layout = scale_layout;
    tab.residual = res != nullptr;
    tab.stage = res != nullptr;
    int cluster = 1;
    if (fused) {
        // kTargetChunks passes per CTA. Past the portable cluster size, the
        // plain call keeps 8-CTA clusters while a CTA's slice stays within
        // kWideSlicePasses passes (its stripes' pass-2 re-reads still fit L2;
        // 16 CTAs measured 3 % slower at C = 16384) and grows the cluster only
        // beyond that (C = 32768: 74 % -> 83 % of HBM bandwidth); the residual
        // form, whose re-read is of h, does better with the larger cluster at
        // once (16384: +2.7 %).
        //
        // A launch whose CTAs at that size would not fill the device once
        // (fewer than it holds at a time) is bound by the latency of its
        // passes, not by bandwidth: it takes one pass per CTA instead, in
        // larger clusters (256 x 1024: 11.1 -> 9.3 us, 64 x 8192: 14.8 ->
        // 10.7 us, 16384 x 1024: 25.1 -> 23.2 us with the L2 flushed; raising
        // the threshold to two or more device fills slowed 8192 x 4096 and
        // 8192 x 8192 by 4-10 %).
        constexpr int64_t kWideSlicePasses = 4;
        const int64_t chunk = mx::fused_chunk_cols();
        int64_t want = ceil_div(max_cols, chunk * mx::kTargetChunks);
        if (want > mx::kPortableCluster && res == nullptr) {
            const int64_t wide = ceil_div(max_cols, chunk * kWideSlicePasses);
            want = wide > mx::kPortableCluster ? wide : mx::kPortableCluster;
        }
        int64_t stripes = 0;
        for (int i = 0; i < n; ++i)
            if (d[i].rows > 0 && d[i].cols > 0) stripes += ceil_div(d[i].rows, mx::kBlock);
        if (stripes * want < mx::fused_resident_ctas()) {
            const int64_t one_pass = ceil_div(max_cols, chunk);
            if (one_pass > want) want = one_pass;
        }
        int most = mx::fused_max_cluster();
        const int cap = mx::hook_max_cluster();
        if (cap > 0 && cap < most) most = cap;
        cluster = (int)(want < most ? want : most);
        if (cluster < 1) cluster = 1;
    }
    tab.cluster = cluster;
    int64_t units = 0;
    int m = 0;
    for (int i = 0; i < n; ++i) {
        const mxfp8_desc& e = d[i];
        if (e.rows == 0 || e.cols == 0) continue;
        mx::DevDesc& o = tab.d[m++];
        o.x = static_cast<const uint16_t*>(e.x);
        o.gamma = static_cast<const uint16_t*>(fused ? e.gamma : nullptr);
        o.normed = static_cast<uint16_t*>(fused ? e.normed : nullptr);
        o.q_row = static_cast<uint8_t*>(rowwise ? e.q_row : nullptr);
        o.s_row = static_cast<uint8_t*>(rowwise ? e.s_row : nullptr);
        o.q_col = static_cast<uint8_t*>(columnwise ? e.q_col : nullptr);
        o.s_col = static_cast<uint8_t*>(columnwise ? e.s_col : nullptr);
        o.res_in = static_cast<const uint16_t*>(res ? res[i].residual : nullptr);
        o.res_out = static_cast<uint16_t*>(res ? res[i].residual_out : nullptr);
        o.rows = e.rows;
        o.cols = e.cols;
        o.eps = e.eps;
        o.offset = e.weight_offset;
        o.unit_begin = units;
        const int64_t stripes = ceil_div(e.rows, mx::kBlock);
        if (fused) {
            o.cta_cols = (int32_t)(ceil_div(ceil_div(e.cols, cluster), mx::kBlock) * mx::kBlock);
            o.col_tiles = 0;
            units += stripes;
        } else {
            o.cta_cols = 0;
            o.col_tiles = (int32_t)ceil_div(e.cols, mx::QuantGeo::kWarpCols);
            units += stripes * o.col_tiles;
        }
    }
    tab.n = m;
    tab.total_units = units;
    const int64_t grid = fused ? units * cluster : ceil_div(units, mx::QuantGeo::kWarps);
    if (grid > 0x7FFFFFFFLL)
        return fail(MXFP8_ERR_SHAPE, "list needs %lld CTAs, more than one launch allows",
                    (long long)grid);
    const int err = fused ? mx::launch_fused(tab, grid, stream) : mx::launch_quant(tab, grid, stream);
    if (err != cudaSuccess) {
        cudaGetLastError();  // clear a non-sticky launch error
        return fail(MXFP8_ERR_CUDA, "kernel launch failed: %s",
                    cudaGetErrorString(static_cast<cudaError_t>(err)));
    }
    return MXFP8_OK;
}

int run(bool fused, const mxfp8_desc* d, const mxfp8_residual* res, int n, int rowwise,
        int columnwise, int scale_layout, void* stream) {
    g_err.clear();
    if (d == nullptr) return fail(MXFP8_ERR_COUNT, "desc is NULL");
    if (n < 1 || n > MXFP8_MAX_TENSORS)
        return fail(MXFP8_ERR_COUNT, "n = %d is outside [1, %d]", n, MXFP8_MAX_TENSORS);
    if (!rowwise && !columnwise)
        return fail(MXFP8_ERR_FLAGS, "neither rowwise nor columnwise requested");
    if (scale_layout != MXFP8_SCALES_COMPACT && scale_layout != MXFP8_SCALES_MMA_TILED &&
        scale_layout != MXFP8_SCALES_PADDED)
        return fail(MXFP8_ERR_FLAGS, "unknown scale layout %d", scale_layout);
    int live = 0;
    int64_t max_cols = 0;
    for (int i = 0; i < n; ++i) {
        const int rc = check_entry(d[i], i, fused, rowwise != 0, columnwise != 0);
        if (rc != MXFP8_OK) return rc;
        if (res != nullptr && d[i].rows > 0 && d[i].cols > 0) {
            if (res[i].residual != nullptr && !aligned16(res[i].residual))
                return fail(MXFP8_ERR_POINTER, "entry %d: residual is not 16-byte aligned", i);
            if (res[i].residual_out != nullptr && !aligned16(res[i].residual_out))
                return fail(MXFP8_ERR_POINTER, "entry %d: residual_out is not 16-byte aligned", i);
        }
        if (d[i].rows > 0 && d[i].cols > 0) {
            ++live;
            if (d[i].cols > max_cols) max_cols = d[i].cols;
        }
    }
    if (live == 0) return MXFP8_OK;
    if (live <= mx::kSmallTable)
        return fill_and_launch<mx::kSmallTable>(fused, d, res, n, rowwise != 0, columnwise != 0,
                                                scale_layout, max_cols, stream);
    return fill_and_launch<mx::kLargeTable>(fused, d, res, n, rowwise != 0, columnwise != 0,
                                            scale_layout, max_cols, stream);
}

}  // namespace

namespace mx {
namespace {
std::atomic<int> g_hook_fail_launch{0};
std::atomic<int> g_hook_max_cluster{0};
std::atomic<int> g_hook_gemm_form{0};
std::atomic<int> g_hook_gemm_splits{0};
}  // namespace

int hook_launch_error() {
    return g_hook_fail_launch.load(std::memory_order_relaxed) ? (int)cudaErrorInvalidValue
                                                              : (int)cudaSuccess;
}
int hook_max_cluster() { return g_hook_max_cluster.load(std::memory_order_relaxed); }
int hook_gemm_form() { return g_hook_gemm_form.load(std::memory_order_relaxed); }
int hook_gemm_splits() { return g_hook_gemm_splits.load(std::memory_order_relaxed); }

TraceRange::TraceRange(const char* name) { nvtxRangePushA(name); }
TraceRange::~TraceRange() { nvtxRangePop(); }

// Sets this thread's last-error text (used by the other translation units).
int set_error(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}
}  // namespace mx

extern "C" {

int rmsnorm_quant_mxfp8(const mxfp8_desc* desc, int n, int rowwise, int columnwise,
                        void* stream) {
    const mx::TraceRange trace("rmsnorm_quant_mxfp8");
    return run(true, desc, nullptr, n, rowwise, columnwise, MXFP8_SCALES_COMPACT, stream);
}

int quant_mxfp8(const mxfp8_desc* desc, int n, int rowwise, int columnwise, void* stream) {
    const mx::TraceRange trace("quant_mxfp8");
    return run(false, desc, nullptr, n, rowwise, columnwise, MXFP8_SCALES_COMPACT, stream);
}

int rmsnorm_quant_mxfp8_ex(const mxfp8_desc* desc, int n, int rowwise, int columnwise,
                           int scale_layout, void* stream) {
    const mx::TraceRange trace("rmsnorm_quant_mxfp8_ex");
    return run(true, desc, nullptr, n, rowwise, columnwise, scale_layout, stream);
}

int quant_mxfp8_ex(const mxfp8_desc* desc, int n, int rowwise, int columnwise,
                   int scale_layout, void* stream) {
    const mx::TraceRange trace("quant_mxfp8_ex");
    return run(false, desc, nullptr, n, rowwise, columnwise, scale_layout, stream);
}

int add_rmsnorm_quant_mxfp8(const mxfp8_desc* desc, const mxfp8_residual* res, int n,
                            int rowwise, int columnwise, int scale_layout, void* stream) {
    const mx::TraceRange trace("add_rmsnorm_quant_mxfp8");
    if (res == nullptr) {
        g_err.clear();
        return fail(MXFP8_ERR_POINTER, "residual array is NULL");
    }
    return run(true, desc, res, n, rowwise, columnwise, scale_layout, stream);
}

int mxfp8_update_planes(const mxfp8_planes* src, const mxfp8_planes* dst, int n, int rowwise,
                        int columnwise, int dst_scale_layout, void* stream) {
    const mx::TraceRange trace("mxfp8_update_planes");
    g_err.clear();
    if (src == nullptr || dst == nullptr) return fail(MXFP8_ERR_COUNT, "src or dst is NULL");
    if (n < 1 || n > MXFP8_MAX_UPDATE)
        return fail(MXFP8_ERR_COUNT, "n = %d is outside [1, %d]", n, MXFP8_MAX_UPDATE);
    if (!rowwise && !columnwise)
        return fail(MXFP8_ERR_FLAGS, "neither rowwise nor columnwise selected");
    if (dst_scale_layout < MXFP8_SCALES_COMPACT || dst_scale_layout > MXFP8_SCALES_PADDED)
        return fail(MXFP8_ERR_FLAGS, "unknown scale layout %d", dst_scale_layout);
    mx::UpdTable tab;
    std::memset(&tab, 0, sizeof tab);
    tab.rowwise = rowwise != 0;
    tab.columnwise = columnwise != 0;
    tab.layout = dst_scale_layout;
    auto r128 = [](int64_t v) { return ceil_div(v, 128) * 128; };
    auto r4 = [](int64_t v) { return ceil_div(v, 4) * 4; };
    auto chunks = [](int64_t bytes) { return ceil_div(bytes, mx::kUpdChunkBytes); };
    auto scale_chunks = [](int64_t bytes) { return ceil_div(bytes, mx::kUpdScaleChunkBytes); };
    int64_t total = 0;
    int m = 0;
    for (int i = 0; i < n; ++i) {
        const mxfp8_planes& S = src[i];
        const mxfp8_planes& D = dst[i];
        const int64_t R = D.rows, C = D.cols;
        if (S.rows != R || S.cols != C)
            return fail(MXFP8_ERR_SHAPE, "entry %d: src [%lld, %lld] and dst [%lld, %lld] differ",
                        i, (long long)S.rows, (long long)S.cols, (long long)R, (long long)C);
        if (R < 0 || C < 0 || C % 32 != 0 || (columnwise && R % 32 != 0) ||
            R > (int64_t(1) << 31) || C > (int64_t(1) << 31))
            return fail(MXFP8_ERR_SHAPE, "entry %d: bad shape [%lld, %lld]", i, (long long)R,
                        (long long)C);
        if (R == 0 || C == 0) continue;
        mx::UpdEntry& e = tab.e[m];
        const void* sp[4] = {S.q_row, S.s_row, S.q_col, S.s_col};
        void* dp[4] = {D.q_row, D.s_row, D.q_col, D.s_col};
        int64_t entry_chunks = 0;
        for (int plane = 0; plane < 2; ++plane) {
            if (!(plane == 0 ? rowwise : columnwise)) continue;
            const char* name = plane == 0 ? "rowwise" : "columnwise";
            const void* sq = sp[2 * plane];
            const void* ss = sp[2 * plane + 1];
            if (!aligned16(dp[2 * plane]) || !aligned16(dp[2 * plane + 1]))
                return fail(MXFP8_ERR_POINTER, "entry %d: dst %s plane pointers must be non-NULL "
                            "and 16-byte aligned", i, name);
            if ((sq == nullptr) != (ss == nullptr))
                return fail(MXFP8_ERR_POINTER, "entry %d: src %s plane is half present", i, name);
            if (sq != nullptr && (!aligned16(sq) || !aligned16(ss)))
                return fail(MXFP8_ERR_POINTER, "entry %d: src %s plane is not 16-byte aligned",
                            i, name);
            int64_t scale_bytes = R * C / 32;  // copied: the compact source bytes
            if (sq == nullptr && dst_scale_layout == MXFP8_SCALES_PADDED)
                scale_bytes = plane == 0 ? r128(R) * r4(C / 32) : r4(R / 32) * r128(C);
            else if (sq == nullptr && dst_scale_layout == MXFP8_SCALES_MMA_TILED)
                scale_bytes = plane == 0 ? r128(R) * r4(C / 32) : r128(C) * r4(R / 32);
            entry_chunks += chunks(R * C) + scale_chunks(scale_bytes);
        }
        for (int k = 0; k < 4; ++k) {
            e.src[k] = static_cast<const uint8_t*>(sp[k]);
            e.dst[k] = static_cast<uint8_t*>(dp[k]);
        }
        e.rows = R;
        e.cols = C;
        e.chunk_begin = total;
        total += entry_chunks;
        ++m;
    }
    if (m == 0) return MXFP8_OK;
    if (total > 0x7FFFFFFFLL) return fail(MXFP8_ERR_SHAPE, "update too large for one launch");
    tab.n = m;
    tab.total_chunks = total;
    const int err = mx::launch_update(tab, stream);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return fail(MXFP8_ERR_CUDA, "kernel launch failed: %s",
                    cudaGetErrorString(static_cast<cudaError_t>(err)));
    }
    return MXFP8_OK;
}

int mxfp8_rmsnorm_quant(const mxfp8_desc* desc, int n, int rowwise, int columnwise,
                        void* stream) {
    const mx::TraceRange trace("mxfp8_rmsnorm_quant");
    return run(true, desc, nullptr, n, rowwise, columnwise, MXFP8_SCALES_COMPACT, stream);
}

int mxfp8_quant(const mxfp8_desc* desc, int n, int rowwise, int columnwise, void* stream) {
    const mx::TraceRange trace("mxfp8_quant");
    return run(false, desc, nullptr, n, rowwise, columnwise, MXFP8_SCALES_COMPACT, stream);
}

int mxfp8_set_test_hook(int hook, int value) {
    g_err.clear();
    if (value < 0) return fail(MXFP8_ERR_FLAGS, "test hook %d: negative value %d", hook, value);
    switch (hook) {
        case MXFP8_HOOK_FAIL_LAUNCH:
            return mx::g_hook_fail_launch.exchange(value != 0 ? 1 : 0);
        case MXFP8_HOOK_MAX_CLUSTER:
            return mx::g_hook_max_cluster.exchange(value);
        case MXFP8_HOOK_GEMM_FORM:
            if (value > 2) return fail(MXFP8_ERR_FLAGS, "GEMM form hook: %d is not 0, 1 or 2", value);
            return mx::g_hook_gemm_form.exchange(value);
        case MXFP8_HOOK_GEMM_SPLITS:
            if (value > 3) return fail(MXFP8_ERR_FLAGS, "GEMM split hook: %d is past 3", value);
            return mx::g_hook_gemm_splits.exchange(value);
        default:
            return fail(MXFP8_ERR_FLAGS, "unknown test hook %d", hook);
    }
}

const char* mxfp8_last_error(void) { return g_err.c_str(); }

int mxfp8_abi_version(void) { return MXFP8_ABI_VERSION; }

}  // extern "C"
