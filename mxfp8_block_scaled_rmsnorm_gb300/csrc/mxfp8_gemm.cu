// mxfp8_gemm.cu -- block-scaled MXFP8 GEMM on the 5th-generation tensor cores
// (sm_103a: tcgen05.mma kind::mxf8f6f4 with UE8M0 block scales), the matrix
// multiply behind mm_mxfp8 (Megatron inference page
// "core.inference.quantization.utils", `mm_mxfp8`: quantized activation times
// the quantized weight, float32 accumulation, bf16 output).
//
// out[M, N] = sum_k (a[m, k] * 2^(sa[m, k/32] - 127)) * (b[n, k] * 2^(sb[n, k/32] - 127))
// with a [M, K] and b [N, K] E4M3 codes (K-major: row-major with K contiguous)
// and sa, sb their scale bytes in the tiled GEMM-operand layout that the
// quantize kernels write (tiles of 128 rows x 4 scale columns, 512 bytes).
//
// Design: pairs of CTAs on two SMs (a thread-block cluster of 2) compute
// 256 x 256 output tiles with the two-SM form of the MMA (cta_group::2):
// CTA r of the pair holds rows 128r .. 128r+127 of the A tile and of the B
// tile (B split along N), and its tensor memory receives its 128 rows of the
// float32 accumulator over all 256 columns. Per SM and K step of 128 bytes
// that is 32 KB of operands for 128 x 256 x 128 multiply-adds (the one-SM
// 128 x 256 form moves 48 KB). Persistent: the pairs the device holds at once
// walk the output tiles.
// The issuing roles below are whole warps: every lane runs the role's loop
// (barrier waits, stage counters, descriptor words: the same value in each
// lane) and one elected lane issues the TMA, tcgen05 and commit instructions.
// Kept warp-uniform, those operands need no per-instruction conversion from
// per-thread registers; the same loops run on one thread (lane 0 alone)
// issued 6-8 % slower over the whole GEMM.
//  - warp 0 of each CTA: producer. Per K step it loads its A and B
//    halves (TMA, 128-byte swizzle) and the scale tiles (TMA over a 3-D view
//    of the tiled scales: its own A tile, both 128-row B tiles, since its
//    accumulator rows span all 256 columns) into a 6-stage ring. All copies
//    of both CTAs complete on the leader CTA's "full" barrier.
//  - warp 1 of the leader CTA: MMA issuer. Per K step it copies the stage's
//    scale tiles of both CTAs into their tensor memory (tcgen05.cp
//    32x128b.warpx4, one column slot per stage), issues four 256 x 256 x 32
//    MMAs (scale byte k of each 32-bit scale word for the k-th 32-element
//    block), then commits to the "empty" barrier of both CTAs; after the last
//    K step, to "tmem_full". A scale copy and the MMAs after it, issued by
//    the same thread, run in issue order on the tensor pipe, so the MMAs need
//    no wait for the copy. The loop is kept to these instructions and
//    precomputed descriptor words: each tcgen05 issue costs the issuing lane
//    tens of cycles.
//  - warp 2 of each CTA: allocates (and at the end frees) 512 tensor-memory
//    columns, collectively for the pair: the accumulator (256 columns) and
//    per-stage scale columns. Warp 3 has no role.
//  - warps 4-11: epilogue. Each reads its 32 accumulator lanes (its TMEM lane
//    quarter, warp % 4) over 128 columns with tcgen05.ld, converts to bf16
//    (round to nearest even), releases the accumulator (an arrival on the
//    leader's "tmem_empty"), then stores: per 32-column chunk its 32 rows go
//    to a shared-memory staging buffer (64-byte swizzle, one per warp) and
//    one lane issues a TMA store of the 32 x 32 box, clipped at the matrix
//    edges. Whole lines reach L2, and the stores overlap the next tile's
//    MMAs; stores by each lane of its own row, 16 bytes at a time, had
//    delayed the next tile's first operand loads and the release behind
//    them by thousands of cycles per tile.
//  - Every mbarrier wait gives up after a time limit: it records the site in a
//    device status word (read by mxfp8_device_status), raises a CTA-wide abort
//    flag that ends the CTA's other waits, the leader waits (bounded) for the
//    pair's copies and MMAs in flight, and both CTAs meet at a cluster barrier,
//    free their tensor memory and exit.
//
// Skinny form (decoding steps, M <= 64, and mid-size M where the planner
// estimates it faster): a 256-row output tile would be mostly empty, and few
// tiles would leave most SMs idle, so the operands swap roles. The weight's
// 256-row block fills the MMA's M (128 rows per CTA of the pair) and the
// activation rows are its N (32, 64 or 128, zero rows past M; more rows run
// as several 128-row activation blocks, each a work tile), so out^T is
// accumulated: weight row n in tensor-memory lane n, activation row m in
// column m. The tensor cores have
// little to do and the kernel streams the weight; what bounds it is the MMA
// warp's issue rate, so a stage holds two K steps (one wait and one commit
// per eight MMAs) and the four 32-element blocks of a K step add into four
// separate accumulators (one for N = 128; summed by the epilogue; MMAs into
// one accumulator wait for each other). With few output blocks the K range is
// split over two or three pairs of a cluster; in turn, each CTA of a later
// pair writes its float32 partial straight into the shared memory of the
// first pair's CTA with the same lanes (st.async, counted on that CTA's
// mbarrier), which adds it. That CTA then stages its bf16 output in the same
// shared memory and writes it with TMA stores.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "mx_gemm.h"
#include "mx_table.h"
#include "mx_umma.h"

namespace mx {

__device__ unsigned long long g_gemm_status = 0;

namespace {

constexpr int kBM = 128;   // A rows per CTA (256 per pair)
constexpr int kBN = 256;   // output columns per tile; B rows per CTA: kBN / 2
constexpr int kBK = 128;   // bytes = E4M3 elements per K step
constexpr int kStages = 6;
constexpr int kThreads = 384;
constexpr int kEpilogueWarp0 = 4;
constexpr uint32_t kTileA = kBM * kBK;        // 16 KB
constexpr uint32_t kTileB = (kBN / 2) * kBK;  // 16 KB
constexpr uint32_t kSfTile = 512;             // one 128-row x 4 scale tile
constexpr uint32_t kSfStage = 3 * kSfTile;    // A tile, then the two B tiles
constexpr uint32_t kStageTx = kTileA + kTileB + kSfStage;  // bytes one CTA loads per stage
constexpr uint32_t kOffB = kStages * kTileA;
constexpr uint32_t kOffSf = kOffB + kStages * kTileB;
// epilogue staging: per epilogue warp one buffer of one 32-row x 32-column
// bf16 chunk (64 bytes a row, 64-byte swizzle), the source of its TMA stores
// (one buffer, not two, so that the ring has a sixth stage: the ring refills
// after each tile switch, and five stages left the MMAs waiting there)
constexpr uint32_t kEpiBuf = 32 * 64;
constexpr uint32_t kOffEpi = (kOffSf + kStages * kSfStage + 1023) / 1024 * 1024;
constexpr uint32_t kOffBar = kOffEpi + 8 * kEpiBuf;
constexpr uint32_t kBarBytes = 256;
constexpr uint32_t kSmemBytes = 1024 + kOffBar + kBarBytes;  // + alignment slack
static_assert(8 * (2 * kStages + 3) + 8 <= kBarBytes, "barriers, tensor-memory slot, abort flag");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColSfa = kBN;                // 4 columns per stage
constexpr uint32_t kColSfb = kBN + 4 * kStages;  // 8 columns per stage
static_assert(kColSfb + 8 * kStages <= kTmemCols, "tensor memory budget");
static_assert(kSmemBytes <= 232448, "shared memory budget");

// The skinny form (few activation rows; see SkinnyParams): 256 threads (warp 0
// producer, warp 1 MMA issuer of the pair's leader, warp 2 tensor-memory
// allocator, warps 4-7 epilogue), a ring of stages of two K steps each (the
// weight's 128-row tile, the activation's mt/2 rows and both scale tiles per
// CTA and K step), and a float32 partial-sum area for the split of K over the
// cluster's pairs. Two instances: up to 64 activation rows (mt 32 or 64) and
// up to 128 (mt 128), whose larger activation tiles and partial rows leave
// shared memory for three stages instead of four.
constexpr int kSkThreads = 256;
constexpr int kSkSub = 2;                 // K steps per stage: one wait and one commit per 8 MMAs
constexpr uint32_t kSkTileW = 128 * kBK;  // 16 KB per K step
constexpr uint32_t kSkSf = 2 * 512;       // per K step: weight tile, activation tile
constexpr uint32_t kSkTmemCols = 512;
template <int MT>  // the largest mt of the instance: 64 or 128
struct SkLayout {
    static constexpr int kStages = MT <= 64 ? 4 : 3;
    static constexpr uint32_t kTileX = (MT / 2) * kBK;  // slot per K step (mt/2 rows used)
    static constexpr uint32_t kStageW = kSkSub * kSkTileW;
    static constexpr uint32_t kStageX = kSkSub * kTileX;
    static constexpr uint32_t kSfStage = kSkSub * kSkSf;
    static constexpr uint32_t kOffX = kStages * kStageW;
    static constexpr uint32_t kOffSf = kOffX + kStages * kStageX;
    // the adding CTA's receive area for the other pair's partial sums: for
    // each accumulator lane (128) MT float32, per epilogue warp q a region of
    // float4 groups [MT / 4][32 lanes] (so a warp's 16-byte accesses cover
    // 512 contiguous bytes), which then holds the warp's bf16 output staging
    static constexpr uint32_t kOffP = kOffSf + kStages * kSfStage;
    static constexpr uint32_t kOffBar = kOffP + 128 * MT * 4;
    static constexpr uint32_t kSmemBytes = 1024 + kOffBar + kBarBytes;
    static constexpr int kNumBars = 2 * kStages + 5;
    // One accumulator per 32-element block of a K step (block k adds into
    // accumulator k % kChains, at columns MT * (k % kChains) ..): MMAs into one
    // accumulator wait for each other, and with mt <= 64 columns each is too
    // short to hide that (a K step took as long as a 256-column one); the
    // epilogue adds the accumulators. Four of 64 columns; at 128 columns one
    // (measured 1-2 % faster than two, which had been faster than three).
    static constexpr int kChains = MT <= 64 ? 4 : 1;
    static constexpr uint32_t kColSfw = kChains * MT;                  // 4 columns per K step
    static constexpr uint32_t kColSfx = kColSfw + 4 * kSkSub * kStages;  // 4 columns per K step
    static_assert(8 * kNumBars + 8 <= kBarBytes, "barriers, tensor-memory slot, abort flag");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kOffX % 1024 == 0 && kOffSf % 1024 == 0 && kOffP % 1024 == 0,
                  "128-byte-swizzled tiles start on 1024-byte boundaries");
    static_assert(kColSfx + 4 * kSkSub * kStages <= kSkTmemCols, "tensor memory budget");
};
// K split over at most 3 pairs (clusters of up to 6 CTAs); pair 0 receives
// the other pairs' partial sums in turn. Four pairs in 8-CTA clusters
// measured slower than three on every shape tried (1.3-2x; fewer such
// clusters are resident at once).
constexpr int kSkMaxSplits = 3;

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait

// Status codes of the sites that can give up (bits 48-55 of the status word;
// the low bits hold the CTA index).
enum : uint32_t { kSiteEmpty = 1, kSiteTmemEmpty = 2, kSiteFull = 3, kSiteTmemFull = 4 };

// ------------------------------------------------------------ primitives ---

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The shared::cluster address of the same shared-memory offset in CTA `rank`.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// Arrival on a barrier given by its shared::cluster address (this CTA's or the peer's).
__device__ __forceinline__ void bar_arrive_cluster(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ bool bar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits until the phase of `bar` with parity `parity` has completed. Gives up
// after kWaitLimitNs (recording `site` and raising the abort flag), or as soon
// as another thread of the CTA has given up. Returns whether the phase completed.
// The first poll is inline (the common case in the MMA warp's loop, whose
// issue rate bounds the tensor pipe); the rest is an out-of-line call.
__device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, volatile uint32_t* abort,
                                           uint32_t site) {
    const uint64_t t0 = global_ns();
    while (true) {
        for (int i = 0; i < 32; ++i)
            if (bar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            *abort = 1u;
            atomicCAS(&g_gemm_status, 0ull, ((unsigned long long)site << 48) | blockIdx.x);
            return false;
        }
    }
}
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort,
                                         uint32_t site) {
    return bar_try_wait(bar, parity) || wait_bar_slow(bar, parity, abort, site);
}


// The lowest lane of a converged warp, which issues the warp's tensor-core and
// TMA operations (always the same lane, so its commits cover its own MMAs and
// copies); the rest of the warp keeps the loop's values warp-uniform.
__device__ __forceinline__ bool elect_one() {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r));
    return r != 0;
}
// wait_bar by every lane of a converged warp, with the same result in all lanes.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity,
                                              volatile uint32_t* abort, uint32_t site) {
    return __all_sync(0xFFFFFFFFu, wait_bar(bar, parity, abort, site));
}

// The same wait, used while draining after an abort: bounded, and not cut
// short by the abort flag.
__device__ void drain_bar(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = global_ns();
    while (!bar_try_wait(bar, parity))
        if (global_ns() - t0 > kWaitLimitNs) return;
}

// TMA loads into this CTA's shared memory, completing on the barrier at the
// shared::cluster address `bar` (the leader CTA's, for both CTAs of the pair).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, int32_t z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// TMA store of a 2-D box from this CTA's shared memory, in the thread's
// bulk async-group; the tensor map clips the parts of the box outside the
// tensor.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x,
                                             int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Until all of this thread's bulk groups have completed (writes performed).
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}
// Orders this thread's shared-memory writes before later TMA reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Copy one 512-byte scale tile (32 rows x 16 bytes in shared memory) to four
// tensor-memory columns, replicated into all four 32-lane quarters, in both
// CTAs of the pair (each from its own shared memory).
__device__ __forceinline__ void tc_copy_scales(uint32_t taddr, uint64_t desc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc)
                 : "memory");
}

// A 64-bit descriptor from its two 32-bit words.
__device__ __forceinline__ uint64_t desc64(uint32_t lo, uint32_t hi) {
    return ((uint64_t)hi << 32) | lo;
}

// D (+)= A x B with block scales over the pair; accumulate selects D += (else D =).
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X"
        " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
        : "memory");
}

// Arrive on the barrier at offset `bar` in the CTAs of `mask` once every
// tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar), "h"(mask)
        : "memory");
}

// 32 consecutive float32 columns of this thread's accumulator lane.
__device__ __forceinline__ void tc_load32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
        " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
        " [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
// The same into float registers (the load moves 32-bit words).
__device__ __forceinline__ void tc_load32f(uint32_t taddr, float (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
        " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
        " [%32];"
        : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]),
          "=f"(r[7]), "=f"(r[8]), "=f"(r[9]), "=f"(r[10]), "=f"(r[11]), "=f"(r[12]),
          "=f"(r[13]), "=f"(r[14]), "=f"(r[15]), "=f"(r[16]), "=f"(r[17]), "=f"(r[18]),
          "=f"(r[19]), "=f"(r[20]), "=f"(r[21]), "=f"(r[22]), "=f"(r[23]), "=f"(r[24]),
          "=f"(r[25]), "=f"(r[26]), "=f"(r[27]), "=f"(r[28]), "=f"(r[29]), "=f"(r[30]),
          "=f"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tc_wait_load() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t bf16x2(uint32_t lo_f32, uint32_t hi_f32) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(__uint_as_float(hi_f32)),
        "f"(__uint_as_float(lo_f32)));
    return r;
}

// Output tile t of the launch: tiles are taken in groups of kGroupN column
// blocks, row blocks fastest within a group, so that the tiles in flight at
// once (one per pair) share a few column blocks of B and a band of A rows,
// which stay in L2 instead of the whole of A being re-read per column block.
constexpr int kGroupN = 8;
__device__ __forceinline__ void tile_coords(const GemmParams& p, int t, int& m_pair, int& n_blk) {
    const int per_group = kGroupN * p.m_tiles;
    const int g = t / per_group;
    const int first = g * kGroupN;
    const int width = p.n_tiles - first < kGroupN ? p.n_tiles - first : kGroupN;
    const int in = t - g * per_group;
    n_blk = first + in % width;
    m_pair = in / width;
}

// ----------------------------------------------------------------- kernel ---

__global__ void __launch_bounds__(kThreads, 1) mxfp8_gemm_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    // 128-byte-swizzled tiles must start on 1024-byte boundaries (the same
    // offsets in both CTAs of the pair, as the two-SM MMA requires)
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    // bars[0, S): full; [S, 2S): empty; 2S: tmem_full; 2S+1: tmem_empty;
    // 2S+2: drain (MMA issuer)
    const uint32_t bar0 = smem_u32(bars);
    auto full = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto empty = [&](int s) { return bar0 + 8u * (uint32_t)(kStages + s); };
    const uint32_t tmem_full = bar0 + 8u * (2 * kStages);
    const uint32_t tmem_empty = bar0 + 8u * (2 * kStages + 1);
    const uint32_t drain = bar0 + 8u * (2 * kStages + 2);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * (2 * kStages + 3));
    volatile uint32_t* abort = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1, pairs = gridDim.x >> 1;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            bar_init(full(s), 1);  // the leader's producer; bytes from both CTAs
            bar_init(empty(s), 1);
        }
        bar_init(tmem_full, 1);
        bar_init(tmem_empty, 16);  // one arrival per epilogue warp of the pair
        bar_init(drain, 1);
        *abort = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------- producer
        const uint32_t lead_full0 = peer_addr(full(0), 0);
        int s = 0;
        uint32_t ph = 0;
        uint32_t used = 0, last_par = 0;  // per stage: filled at all; parity of its last fill
        bool ok = true;
        // launched as a programmatic dependent of the previous kernel on the
        // stream (which may have written A, B or their scales): nothing is
        // read before it has completed; the set-up above overlapped its tail
        asm volatile("griddepcontrol.wait;" ::: "memory");
        for (int tile = pair; ok && tile < p.num_tiles; tile += pairs) {
            int m_pair, n_blk;
            tile_coords(p, tile, m_pair, n_blk);
            const int m_tile = 2 * m_pair + (int)rank;  // this CTA's 128-row tile of A
            for (int kt = 0; kt < p.k_tiles; ++kt) {
                if (!wait_bar_warp(empty(s), ph ^ 1u, abort, kSiteEmpty)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = lead_full0 + 8u * (uint32_t)s;
                const uint32_t sf = sbase + kOffSf + s * kSfStage;
                if (elect_one()) {
                    if (leader) bar_expect_tx(full(s), 2 * kStageTx);
                    tma_load_2d(sbase + s * kTileA, &p.tma_a, kt * kBK, m_tile * kBM, fb);
                    tma_load_2d(sbase + kOffB + s * kTileB, &p.tma_b, kt * kBK,
                                n_blk * kBN + (int)rank * (kBN / 2), fb);
                    tma_load_3d(sf, &p.tma_sfa, 0, kt, m_tile, fb);
                    tma_load_3d(sf + kSfTile, &p.tma_sfb, 0, kt, 2 * n_blk, fb);
                }
                __syncwarp();
                used |= 1u << s;
                last_par = (last_par & ~(1u << s)) | (ph << s);
                if (++s == kStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        if (ok) {
            // every stage's last release has arrived before the CTA may exit
            for (int i = 0; i < kStages; ++i) {
                if (!wait_bar_warp(empty(s), ph ^ 1u, abort, kSiteEmpty)) break;
                if (++s == kStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        } else if (leader) {
            // gave up: the pair's copies already issued land (the leader's full
            // barriers count both CTAs' bytes) before either CTA exits
            for (int i = 0; i < kStages; ++i)
                if ((used >> i) & 1u) drain_bar(full(i), (last_par >> i) & 1u);
        }
    } else if (warp == 1 && leader) {
        // ---------------------------------------------------- MMA issuer
        // One warp feeds the tensor pipe, so its loop is kept short. The whole
        // warp runs it (waits, stage counters, descriptors: values the same in
        // every lane) and one elected lane issues the MMAs and commits. The
        // descriptors of stage s and K offset k are precomputed words plus
        // constants (a descriptor's start field is the shared-memory address
        // >> 4 in its low bits; the other fields are the same for every tile
        // of a kind, and the addresses stay below 2^18, so adds never carry
        // out of the field).
        int s = 0;
        uint32_t ph = 0, local = 0;
        bool ok = true;
        const uint32_t acc = tmem;  // lane 0, column 0
        const uint64_t da = umma::kmajor_sw128_desc(sbase);
        const uint64_t db = umma::kmajor_sw128_desc(sbase + kOffB);
        const uint32_t a_lo0 = (uint32_t)da, op_hi = (uint32_t)(da >> 32);
        const uint32_t b_lo0 = (uint32_t)db;
        const uint32_t idesc0 = umma::idesc_mxf8(2 * kBM, kBN, 0, 0);
        const int full_steps = p.K / kBK;  // K steps with all four 32-element blocks
        const uint64_t dsf = umma::scale_tile_desc(sbase + kOffSf);
        const uint32_t sf_lo0 = (uint32_t)dsf, sf_hi = (uint32_t)(dsf >> 32);
        for (int tile = pair; ok && tile < p.num_tiles; tile += pairs, ++local) {
            if (!wait_bar_warp(tmem_empty, (local & 1u) ^ 1u, abort, kSiteTmemEmpty)) {
                ok = false;
                break;
            }
            tc_fence_after();
            for (int kt = 0; kt < p.k_tiles; ++kt) {
                if (!wait_bar_warp(full(s), ph, abort, kSiteFull)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t t_sfa = tmem + kColSfa + 4u * s;
                const uint32_t t_sfb = tmem + kColSfb + 8u * s;
                const uint32_t a_lo = a_lo0 + (uint32_t)s * (kTileA >> 4);
                const uint32_t b_lo = b_lo0 + (uint32_t)s * (kTileB >> 4);
                const uint32_t sf_lo = sf_lo0 + (uint32_t)s * (kSfStage >> 4);
                if (elect_one()) {
                    // scale slot s is free: the MMAs that last read it completed
                    // before the producer refilled stage s
                    tc_copy_scales(t_sfa, desc64(sf_lo, sf_hi));
                    tc_copy_scales(t_sfb, desc64(sf_lo + (kSfTile >> 4), sf_hi));
                    tc_copy_scales(t_sfb + 4u, desc64(sf_lo + 2 * (kSfTile >> 4), sf_hi));
                    if (kt < full_steps) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            tc_mma(acc, desc64(a_lo + 2u * k, op_hi),
                                   desc64(b_lo + 2u * k, op_hi),
                                   idesc0 | ((uint32_t)k << 29) | ((uint32_t)k << 4), t_sfa,
                                   t_sfb, (kt | k) != 0 ? 1u : 0u);
                    } else {
                        // the last, partial K step: only the 32-element blocks that exist
                        const int nk = (p.K - kt * kBK) / 32;
                        for (int k = 0; k < nk; ++k)
                            tc_mma(acc, desc64(a_lo + 2u * k, op_hi),
                                   desc64(b_lo + 2u * k, op_hi),
                                   idesc0 | ((uint32_t)k << 29) | ((uint32_t)k << 4), t_sfa,
                                   t_sfb, (kt | k) != 0 ? 1u : 0u);
                    }
                    tc_commit(empty(s), 3);
                }
                __syncwarp();
                if (++s == kStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            if (elect_one()) tc_commit(tmem_full, 3);
            __syncwarp();
        }
        if (!ok) {
            // gave up: let the pair's scale copies and MMAs finish first
            if (elect_one()) tc_commit(drain, 1);
            __syncwarp();
            drain_bar(drain, 0);
        }
    } else if (warp >= kEpilogueWarp0) {
        // ---------------------------------------------------- epilogue
        const int quarter = warp & 3;                   // TMEM lanes 32q .. 32q+31
        const int half = (warp - kEpilogueWarp0) >> 2;  // accumulator columns 128h ..
        const uint32_t lead_tmem_empty = peer_addr(tmem_empty, 0);
        const uint32_t buf = sbase + kOffEpi + (uint32_t)(warp - kEpilogueWarp0) * kEpiBuf;
        uint32_t local = 0;
        for (int tile = pair; tile < p.num_tiles; tile += pairs, ++local) {
            int m_pair, n_blk;
            tile_coords(p, tile, m_pair, n_blk);
            // every lane waits; the warp goes on (converged, as the .sync.aligned
            // tensor-memory loads need) only if all lanes saw the phase complete
            const bool ok = wait_bar(tmem_full, local & 1u, abort, kSiteTmemFull);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            // the CTA's last accumulator is complete: a GEMM launched after
            // this one as a programmatic dependent may start its set-up (it
            // reads and writes nothing before this grid has completed)
            if (tile + pairs >= p.num_tiles)
                asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            tc_fence_after();
            uint32_t packed[64];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tc_load32(umma::tmem_addr(tmem, 32u * quarter, 128u * half + 32u * c), r);
                tc_wait_load();
#pragma unroll
                for (int j = 0; j < 16; ++j) packed[16 * c + j] = bf16x2(r[2 * j], r[2 * j + 1]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) bar_arrive_cluster(lead_tmem_empty);
            // store: per 32-column chunk, the warp's 32 rows go to its staging
            // buffer (row `lane`: 64 bytes, 16-byte piece q at q ^ ((lane >> 1) & 3),
            // the 64-byte swizzle of the tensor map) and one lane issues a TMA
            // store of the 32 x 32 box; full lines reach L2, and the stores
            // run while the warp waits for the next tile
            // (coordinates compared in 64 bits: inside the tensor they fit in 32)
            const int64_t row0 = (int64_t)(2 * m_pair + (int)rank) * kBM + 32 * quarter;
            const int64_t col0 = (int64_t)n_blk * kBN + 128 * half;
            if (row0 < p.M) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (col0 + 32 * c >= p.N) break;
                    // the previous store has finished reading the buffer
                    if (lane == 0) bulk_wait_read<0>();
                    __syncwarp();
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        st_shared_v4(buf + 64u * lane + ((q ^ ((lane >> 1) & 3)) << 4),
                                     packed[16 * c + 4 * q], packed[16 * c + 4 * q + 1],
                                     packed[16 * c + 4 * q + 2], packed[16 * c + 4 * q + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&p.tma_out, buf, (int32_t)(col0 + 32 * c), (int32_t)row0);
                        bulk_commit();
                    }
                }
            }
        }
        // the output is written before the CTA exits
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    // both CTAs done with the pair's barriers and tensor memory
    tc_fence_before();
    cluster_sync();
    if (warp == 2) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// ----------------------------------------------------- kernel, skinny form ---

// Four 32-bit words into another CTA's shared memory (shared::cluster
// addresses), counted as 16 bytes on that CTA's barrier `bar`.
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                            uint32_t d, uint32_t bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, "
        "[%5];" ::"r"(addr),
        "r"(a), "r"(b), "r"(c), "r"(d), "r"(bar)
        : "memory");
}
// Four float32 from this CTA's shared memory.
__device__ __forceinline__ float4 ld_shared_f32x4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ uint16_t bf16_rn(float v) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(v));
    return r;
}

// out[M, N] for M <= kSkinnyMaxM. Cluster c takes the work tiles c,
// c + clusters, ... (tile t: 256-column output block t / m_blocks, activation
// rows mt (t % m_blocks) ..); pair j of the cluster (CTA ranks 2j, 2j + 1)
// accumulates the K steps [j * steps_per_split, ...) of the tile: weight
// rows 128 r .. of the block in CTA r's tensor-memory lanes, activation row m
// in column m of each accumulator (the 32-element blocks of a K step spread
// over kChains of them). With one pair the epilogue adds the accumulators and
// stores; with more, the CTAs of pairs 1, 2 send their float32 sums in turn
// into the receive area of pair 0's CTA with the same r, which adds them to
// its own, then stores.
template <int MT>
__global__ void __launch_bounds__(kSkThreads, 1)
    mxfp8_gemm_skinny_kernel(const __grid_constant__ SkinnyParams p) {
    using L = SkLayout<MT>;
    constexpr int kStages = L::kStages, kChains = L::kChains;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
    // bars[0, S): full; [S, 2S): empty; 2S: tmem_full; 2S+1: tmem_empty;
    // 2S+2: part_full (another pair's partials received, in pair 0);
    // 2S+3: part_free (pair 0's receive area free for this pair, in pairs >= 1);
    // 2S+4: drain (MMA issuer)
    const uint32_t bar0 = smem_u32(bars);
    auto full = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto empty = [&](int s) { return bar0 + 8u * (uint32_t)(kStages + s); };
    const uint32_t tmem_full = bar0 + 8u * (2 * kStages);
    const uint32_t tmem_empty = tmem_full + 8u;
    const uint32_t part_full = tmem_full + 16u;
    const uint32_t part_free = tmem_full + 24u;
    const uint32_t drain = tmem_full + 32u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffBar + 8 * L::kNumBars);
    volatile uint32_t* abort = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t crank = cluster_rank();
    const uint32_t r = crank & 1u;      // CTA of the pair
    const uint32_t pbase = crank & ~1u;  // the pair's leader
    const bool leader = r == 0;
    const int split = (int)(crank >> 1);
    const int csize = 2 * p.splits;
    const int cluster = (int)blockIdx.x / csize, clusters = (int)gridDim.x / csize;
    const uint16_t pair_mask = (uint16_t)(3u << pbase);
    const int k0 = split * p.steps_per_split;
    const int k1 = k0 + p.steps_per_split < p.k_tiles ? k0 + p.steps_per_split : p.k_tiles;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            bar_init(full(s), 1);  // the leader's producer; bytes from both CTAs
            bar_init(empty(s), 1);
        }
        bar_init(tmem_full, 1);
        bar_init(tmem_empty, 8);                  // the pair's 8 epilogue warps
        bar_init(part_full, 1);  // (pair 0) the expected bytes; one other pair's partials
        bar_init(part_free, 4);  // (pairs j >= 1) pair 0's CTA r's 4 warps: pair j's turn
        bar_init(drain, 1);
        *abort = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kSkTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t x_rows = (uint32_t)p.mt / 2;  // activation rows per CTA

    if (warp == 0) {
        // ---------------------------------------------------- producer
        const uint32_t lead_full0 = peer_addr(full(0), pbase);
        // both K steps of a stage are loaded (one past the range reads data
        // that is not multiplied, or zeros past K), so the byte count is fixed
        const uint32_t stage_tx = kSkSub * (kSkTileW + x_rows * kBK + kSkSf);
        int s = 0;
        uint32_t ph = 0;
        uint32_t used = 0, last_par = 0;  // per stage: filled at all; parity of its last fill
        bool ok = true;
        // the first tile's first stages of the weight when it may be read
        // before the wait (weight_early): the ring is empty, so these stages
        // need no wait, and their stage byte counts are announced here
        int early = 0;
        if (p.weight_early && cluster < p.num_tiles) {
            const int n_blk = cluster / p.m_blocks;
            const int stages = (k1 - k0 + kSkSub - 1) / kSkSub;
            early = stages < kStages ? stages : kStages;
            for (int i = 0; i < early; ++i) {
                const uint32_t fb = lead_full0 + 8u * (uint32_t)i;
                if (elect_one()) {
                    if (leader) bar_expect_tx(full(i), 2 * stage_tx);
#pragma unroll
                    for (int j = 0; j < kSkSub; ++j) {
                        const int kt = k0 + i * kSkSub + j;
                        tma_load_2d(sbase + i * L::kStageW + j * kSkTileW, &p.tma_w, kt * kBK,
                                    n_blk * 256 + (int)r * 128, fb);
                        tma_load_3d(sbase + L::kOffSf + i * L::kSfStage + j * kSkSf, &p.tma_sfw,
                                    0, kt, 2 * n_blk + (int)r, fb);
                    }
                }
                __syncwarp();
                used |= 1u << i;  // first fill: parity 0
            }
        }
        // launched as a programmatic dependent of the previous kernel on the
        // stream (which may have written A, B or their scales): nothing else
        // is read before it has completed; the set-up above overlapped its tail
        asm volatile("griddepcontrol.wait;" ::: "memory");
        for (int tile = cluster; ok && tile < p.num_tiles; tile += clusters) {
            const int n_blk = tile / p.m_blocks, mb = tile % p.m_blocks;
            for (int ks = k0; ks < k1; ks += kSkSub) {
                if (!wait_bar_warp(empty(s), ph ^ 1u, abort, kSiteEmpty)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = lead_full0 + 8u * (uint32_t)s;
                // the first tile's first `early` stages already hold their weight
                const bool w_done = tile == cluster && (ks - k0) / kSkSub < early;
                if (elect_one()) {
                    if (leader && !w_done) bar_expect_tx(full(s), 2 * stage_tx);
#pragma unroll
                    for (int j = 0; j < kSkSub; ++j) {
                        const int kt = ks + j;
                        const uint32_t sf = sbase + L::kOffSf + s * L::kSfStage + j * kSkSf;
                        if (!w_done) {
                            tma_load_2d(sbase + s * L::kStageW + j * kSkTileW, &p.tma_w,
                                        kt * kBK, n_blk * 256 + (int)r * 128, fb);
                            tma_load_3d(sf, &p.tma_sfw, 0, kt, 2 * n_blk + (int)r, fb);
                        }
                        tma_load_2d(sbase + L::kOffX + s * L::kStageX + j * L::kTileX, &p.tma_x,
                                    kt * kBK, mb * p.mt + (int)(r * x_rows), fb);
                        tma_load_3d(sf + 512, &p.tma_sfx, 0, kt, mb, fb);
                    }
                }
                __syncwarp();
                used |= 1u << s;
                last_par = (last_par & ~(1u << s)) | (ph << s);
                if (++s == kStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        if (ok) {
            // every stage's last release has arrived before the CTA may exit
            for (int i = 0; i < kStages; ++i) {
                if (!wait_bar_warp(empty(s), ph ^ 1u, abort, kSiteEmpty)) break;
                if (++s == kStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        } else if (leader) {
            // gave up: the pair's copies already issued land before either CTA exits
            for (int i = 0; i < kStages; ++i)
                if ((used >> i) & 1u) drain_bar(full(i), (last_par >> i) & 1u);
        }
    } else if (warp == 1 && leader) {
        // ---------------------------------------------------- MMA issuer
        // (as in the general form: the whole warp runs the loop, one elected
        // lane issues; per K step two scale copies and four 256 x mt x 32 MMAs)
        int s = 0;
        uint32_t ph = 0, local = 0;
        bool ok = true;
        const uint64_t dw = umma::kmajor_sw128_desc(sbase);
        const uint64_t dx = umma::kmajor_sw128_desc(sbase + L::kOffX);
        const uint32_t w_lo0 = (uint32_t)dw, op_hi = (uint32_t)(dw >> 32);
        const uint32_t x_lo0 = (uint32_t)dx;
        const uint32_t idesc0 = umma::idesc_mxf8(256, (uint32_t)p.mt, 0, 0);
        const int full_steps = p.K / kBK;  // K steps with all four 32-element blocks
        const uint64_t dsf = umma::scale_tile_desc(sbase + L::kOffSf);
        const uint32_t sf_lo0 = (uint32_t)dsf, sf_hi = (uint32_t)(dsf >> 32);
        for (int tile = cluster; ok && tile < p.num_tiles; tile += clusters, ++local) {
            if (!wait_bar_warp(tmem_empty, (local & 1u) ^ 1u, abort, kSiteTmemEmpty)) {
                ok = false;
                break;
            }
            tc_fence_after();
            for (int ks = k0; ks < k1; ks += kSkSub) {
                if (!wait_bar_warp(full(s), ph, abort, kSiteFull)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int j = 0; j < kSkSub; ++j) {
                        const int kt = ks + j;
                        if (kt >= k1) break;
                        const uint32_t w_lo = w_lo0 + (((uint32_t)s * L::kStageW + j * kSkTileW) >> 4);
                        const uint32_t x_lo = x_lo0 + (((uint32_t)s * L::kStageX + j * L::kTileX) >> 4);
                        const uint32_t sf_lo = sf_lo0 + (((uint32_t)s * L::kSfStage + j * kSkSf) >> 4);
                        const uint32_t t_sfw = tmem + L::kColSfw + 4u * (kSkSub * s + j);
                        const uint32_t t_sfx = tmem + L::kColSfx + 4u * (kSkSub * s + j);
                        tc_copy_scales(t_sfw, desc64(sf_lo, sf_hi));
                        tc_copy_scales(t_sfx, desc64(sf_lo + (512 >> 4), sf_hi));
                        // block k of the range's first K step starts its
                        // accumulator; every later block adds into it
                        const uint32_t en = kt != k0 ? 1u : 0u;
                        if (kt < full_steps) {
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                tc_mma(tmem + (uint32_t)(MT * (k % kChains)),
                                       desc64(w_lo + 2u * k, op_hi), desc64(x_lo + 2u * k, op_hi),
                                       idesc0 | ((uint32_t)k << 29) | ((uint32_t)k << 4), t_sfw,
                                       t_sfx, k >= kChains ? 1u : en);
                        } else {
                            // the last, partial K step: only the 32-element blocks that exist
                            const int nk = (p.K - kt * kBK) / 32;
                            for (int k = 0; k < nk; ++k)
                                tc_mma(tmem + (uint32_t)(MT * (k % kChains)),
                                       desc64(w_lo + 2u * k, op_hi), desc64(x_lo + 2u * k, op_hi),
                                       idesc0 | ((uint32_t)k << 29) | ((uint32_t)k << 4), t_sfw,
                                       t_sfx, k >= kChains ? 1u : en);
                        }
                    }
                    tc_commit(empty(s), pair_mask);
                }
                __syncwarp();
                if (++s == kStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            if (elect_one()) tc_commit(tmem_full, pair_mask);
            __syncwarp();
        }
        if (!ok) {
            // gave up: let the pair's scale copies and MMAs finish first
            if (elect_one()) tc_commit(drain, 1);
            __syncwarp();
            drain_bar(drain, 0);
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------- epilogue
        const int q = warp & 3;  // tensor-memory lanes 32q .. 32q + 31
        const uint32_t lead_tmem_empty = peer_addr(tmem_empty, pbase);
        const uint32_t adder_part_full = peer_addr(part_full, r);  // pair 0's CTA r
        const bool adder = split == 0;
        // the warp's region of the receive area (in pair 0's CTA r); this
        // lane's float4 group c at + 512 c
        const uint32_t region = smem_u32(smem + L::kOffP) + (uint32_t)q * (MT * 128u);
        const uint32_t my_part = region + 16u * (uint32_t)lane;
        const uint32_t adder_part = peer_addr(my_part, r);
        // accumulators that received an MMA: all of them, unless this pair's
        // whole K range is one partial step
        const int kend = k1 * kBK < p.K ? k1 * kBK : p.K;
        const int blocks = (kend - k0 * kBK) / 32;
        const int chains = blocks < kChains ? blocks : kChains;
        // the warp's bf16 staging buffer for its TMA store (row m of the
        // 32-column box at 64 m bytes): the start of its region, once read
        const uint32_t stage = region;
        // pair 0 receives the other pairs' partials in turn, one receive
        // phase each: phase local * (splits - 1) + j - 1 holds pair j's
        const uint32_t sends = (uint32_t)p.splits - 1u;
        uint32_t local = 0;
        uint32_t pending = 0;   // pair 0: the receive phase waited for next
        bool expected = false;  // pair 0: that phase's bytes announced
        int tile = cluster;
        for (; tile < p.num_tiles; tile += clusters, ++local) {
            pending = local * sends;
            expected = false;
            const bool ok = wait_bar(tmem_full, local & 1u, abort, kSiteTmemFull);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            // the CTA's last accumulator is complete: a dependent GEMM may
            // start its set-up (as in the general form)
            if (tile + clusters >= p.num_tiles)
                asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            tc_fence_after();
            // accumulator 0 straight into acc (all its loads in flight), the
            // others added 32 columns at a time (columns past mt are not read)
            float acc[MT];
#pragma unroll
            for (int c = 0; c < MT / 32; ++c)
                if (32 * c < p.mt)
                    tc_load32f(umma::tmem_addr(tmem, 32u * q, 32u * c),
                               *reinterpret_cast<float(*)[32]>(&acc[32 * c]));
            tc_wait_load();
            for (int k = 1; k < chains; ++k) {
#pragma unroll
                for (int c = 0; c < MT / 32; ++c) {
                    if (32 * c < p.mt) {
                        uint32_t v[32];
                        tc_load32(umma::tmem_addr(tmem, 32u * q, MT * k + 32u * c), v);
                        tc_wait_load();
#pragma unroll
                        for (int j = 0; j < 32; ++j) acc[32 * c + j] += __uint_as_float(v[j]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) bar_arrive_cluster(lead_tmem_empty);
            if (p.splits > 1) {
                if (!adder) {
                    // pair j >= 1: its turn has come (pair 1: pair 0's CTA r
                    // has stored the previous tile; pair j > 1: pair 0 has
                    // added pair j - 1's partials of this tile), then the
                    // partials go straight into pair 0's receive area
                    const uint32_t parity = split == 1 ? (local & 1u) ^ 1u : local & 1u;
                    const bool free_ok = wait_bar(part_free, parity, abort, kSiteTmemEmpty);
                    if (!__all_sync(0xFFFFFFFFu, free_ok)) break;
#pragma unroll
                    for (int m = 0; m < MT; m += 4)
                        if (m < p.mt)
                            st_async_v4(adder_part + 128u * (uint32_t)m, __float_as_uint(acc[m]),
                                        __float_as_uint(acc[m + 1]), __float_as_uint(acc[m + 2]),
                                        __float_as_uint(acc[m + 3]), adder_part_full);
                    continue;
                }
                bool got = true;
                for (int j = 1; j < p.splits; ++j) {
                    // pair 0: all of pair j's bytes for this tile have landed
                    if (warp == 4 && lane == 0) bar_expect_tx(part_full, 512u * (uint32_t)p.mt);
                    expected = true;
                    const bool full_ok = wait_bar(part_full, pending & 1u, abort, kSiteTmemFull);
                    if (!__all_sync(0xFFFFFFFFu, full_ok)) {
                        got = false;
                        break;
                    }
                    expected = false;
                    ++pending;
#pragma unroll
                    for (int m = 0; m < MT; m += 4) {
                        if (m < p.mt) {
                            const float4 v = ld_shared_f32x4(my_part + 128u * (uint32_t)m);
                            acc[m] += v.x;
                            acc[m + 1] += v.y;
                            acc[m + 2] += v.z;
                            acc[m + 3] += v.w;
                        }
                    }
                    // every lane has read the region before any overwrites it
                    __syncwarp();
                    if (j + 1 < p.splits && lane == 0)
                        bar_arrive_cluster(peer_addr(part_free, 2u * (uint32_t)(j + 1) + r));
                }
                if (!got) break;
            }
            // the warp's 32 output columns (the weight rows of its accumulator
            // lanes), all mt rows: bf16 into the staging buffer, then one TMA
            // store of the box, which the tensor map clips at M and N
            const int64_t n0 = (int64_t)(tile / p.m_blocks) * 256 + 128 * (int)r + 32 * q;
            const int32_t m0 = (tile % p.m_blocks) * p.mt;
            if (lane == 0) bulk_wait_read<0>();  // the previous tile's store has read it
            __syncwarp();
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (m < p.mt) st_shared_u16(stage + 64u * m + 2u * lane, bf16_rn(acc[m]));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && n0 < p.N) {
                tma_store_2d(&p.tma_out, stage, (int32_t)n0, m0);
                bulk_commit();
            }
            if (p.splits > 1 && lane == 0) {
                // the store has read the staging: pair 1 may send the next tile
                bulk_wait_read<0>();
                bar_arrive_cluster(peer_addr(part_free, 2u + r));
            }
        }
        // gave up with the pair whose turn it is possibly still sending its
        // partials (the others wait for a turn that does not come): they
        // land (bounded wait) before the CTA may exit
        if (tile < p.num_tiles && p.splits > 1 && adder && warp == 4) {
            if (lane == 0 && !expected) bar_expect_tx(part_full, 512u * (uint32_t)p.mt);
            __syncwarp();
            drain_bar(part_full, pending & 1u);
        }
        // the stores have completed before the CTA exits
        if (lane == 0) bulk_wait_all();
    }

    // every CTA of the cluster done with the barriers, the partials and tensor memory
    tc_fence_before();
    cluster_sync();
    if (warp == 2) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kSkTmemCols)
                     : "memory");
    }
}

// ------------------------------------------------------------------- host ---

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(f);
        else
            cudaGetLastError();
    });
    return fn;
}

// Tensor map of a K-major E4M3 operand [rows, K]: boxes of 128 bytes of K by
// 128 rows, 128-byte swizzle, zero fill outside the matrix.
int encode_operand(CUtensorMap* map, const void* base, int64_t rows, int64_t K,
                   uint32_t box_rows = 128) {
    EncodeTiled fn = encoder();
    if (fn == nullptr) return -1;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
    const cuuint32_t elem[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                          strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : (int)r;
}

// Tensor map of tiled scales (an operand with `rows` rows and K / 32 scale
// columns) as a 3-D array of 32-bit words: [128-row tiles][K steps][128 words],
// each innermost row one 512-byte scale tile; boxes of `tiles` 128-row tiles
// at one K step, zero fill past the last row tile.
int encode_scales(CUtensorMap* map, const void* base, int64_t rows, int64_t k_tiles,
                  uint32_t tiles) {
    EncodeTiled fn = encoder();
    if (fn == nullptr) return -1;
    const cuuint64_t dims[3] = {128, (cuuint64_t)k_tiles, (cuuint64_t)((rows + 127) / 128)};
    const cuuint64_t strides[2] = {kSfTile, (cuuint64_t)k_tiles * kSfTile};
    const cuuint32_t box[3] = {128, 1, tiles};
    const cuuint32_t elem[3] = {1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(base), dims,
                          strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : (int)r;
}

// Tensor map of the bf16 output [M, N] (row-major): boxes of 32 columns x
// box_rows rows, the staging layout of the epilogue: 64-byte swizzle (the
// general form) or none (the skinny form).
int encode_output(CUtensorMap* map, void* base, int64_t M, int64_t N, uint32_t box_rows = 32,
                  CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_64B) {
    EncodeTiled fn = encoder();
    if (fn == nullptr) return -1;
    const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)N * 2};
    const cuuint32_t box[2] = {32, box_rows};
    const cuuint32_t elem[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, elem,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : (int)r;
}

constexpr int kMaxDevices = 64;

int prepare_general(GemmParams* p, const uint8_t* a, const uint8_t* sfa, const uint8_t* b,
                    const uint8_t* sfb, uint16_t* out, int64_t M, int64_t N, int64_t K) {
    const int64_t k_tiles = (K + kBK - 1) / kBK;
    if (encode_operand(&p->tma_a, a, M, K) != 0 || encode_scales(&p->tma_sfa, sfa, M, k_tiles, 1))
        return -1;
    if (encode_operand(&p->tma_b, b, N, K) != 0 || encode_scales(&p->tma_sfb, sfb, N, k_tiles, 2))
        return -2;
    if (encode_output(&p->tma_out, out, M, N) != 0) return -3;
    p->M = (int32_t)M;
    p->N = (int32_t)N;
    p->K = (int32_t)K;
    p->m_tiles = (int32_t)((M + 2 * kBM - 1) / (2 * kBM));
    p->n_tiles = (int32_t)((N + kBN - 1) / kBN);
    p->k_tiles = (int32_t)k_tiles;
    p->num_tiles = p->m_tiles * p->n_tiles;
    return 0;
}

// SMs of the current device (cached per device), or 0 when it cannot be read.
int device_sms() {
    static int cache[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return 0;
    }
    if (cache[dev] == 0 &&
        cudaDeviceGetAttribute(&cache[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        cache[dev] = 0;
    }
    return cache[dev];
}

// Launch configuration of the skinny form's instance MT with clusters of
// 2 * splits CTAs.
template <int MT>
cudaLaunchConfig_t skinny_config(int splits, cudaLaunchAttribute* attr, void* stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kSkThreads, 1, 1);
    cfg.dynamicSmemBytes = SkLayout<MT>::kSmemBytes;
    cfg.stream = static_cast<cudaStream_t>(stream);
    attr->id = cudaLaunchAttributeClusterDimension;
    attr->val.clusterDim.x = (unsigned)(2 * splits);
    attr->val.clusterDim.y = 1;
    attr->val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// Clusters of 2 * splits CTAs of the skinny form's instance MT the current
// device holds at once (cached per device and split count), or 0 when that
// cannot be read.
template <int MT>
int skinny_resident(int splits) {
    static int cache[kMaxDevices][kSkMaxSplits + 1] = {};
    static bool sized[kMaxDevices] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices || splits < 1 ||
        splits > kSkMaxSplits) {
        cudaGetLastError();
        return 0;
    }
    if (cache[dev][splits] > 0) return cache[dev][splits];
    if (!sized[dev]) {
        if (cudaFuncSetAttribute(mxfp8_gemm_skinny_kernel<MT>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SkLayout<MT>::kSmemBytes) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        sized[dev] = true;
    }
    cudaLaunchAttribute attr;
    cudaLaunchConfig_t cfg = skinny_config<MT>(splits, &attr, nullptr);
    const int csize = 2 * splits;
    cfg.gridDim = dim3((unsigned)(device_sms() / csize * csize), 1, 1);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, mxfp8_gemm_skinny_kernel<MT>, &cfg) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cache[dev][splits] = clusters;
    return clusters;
}

// The instance for mt activation rows: 64 for mt <= 64, else 128.
int skinny_resident(int mt, int splits) {
    return mt <= 64 ? skinny_resident<64>(splits) : skinny_resident<128>(splits);
}

// The skinny form's shape, K split and cost estimate for M x N x K (no
// tensor maps): the split is the one with the fewest waves of work tiles
// times K steps per pair, each of the splits - 1 hand-overs of partial sums
// counted as K steps (measured on graph replays: about 8 at mt <= 64, 16 at
// mt = 128), ties to fewer pairs, every range non-empty.
void plan_skinny(SkinnyParams* p, int64_t M, int64_t N, int64_t K) {
    const int64_t k_tiles = (K + kBK - 1) / kBK;
    const int mt = M <= 32 ? 32 : M <= 64 ? 64 : 128;
    p->M = (int32_t)M;
    p->N = (int32_t)N;
    p->K = (int32_t)K;
    p->mt = mt;
    p->m_blocks = (int32_t)((M + mt - 1) / mt);
    p->n_tiles = (int32_t)((N + 255) / 256);
    p->k_tiles = (int32_t)k_tiles;
    p->num_tiles = p->n_tiles * p->m_blocks;
    const int64_t exchange = mt <= 64 ? 8 : 16;
    int best = 1;
    int64_t best_cost = -1;
    p->resident = 0;
    for (int splits = 1; splits <= kSkMaxSplits && splits <= k_tiles; ++splits) {
        const int resident = skinny_resident(mt, splits);
        if (resident < 1) break;
        const int64_t waves = (p->num_tiles + resident - 1) / resident;
        const int64_t cost = waves * ((k_tiles + splits - 1) / splits + (splits - 1) * exchange);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = splits;
            p->resident = resident;
        }
    }
    const int forced = hook_gemm_splits();
    if (forced > 0 && forced <= kSkMaxSplits) {
        const int f = forced < k_tiles ? forced : (int)k_tiles;
        const int resident = skinny_resident(mt, f);
        if (resident > 0) {
            best = f;
            p->resident = resident;
        }
    }
    const int64_t per = (k_tiles + best - 1) / best;
    p->steps_per_split = (int32_t)per;
    p->splits = (int32_t)((k_tiles + per - 1) / per);
    p->cost = best_cost < 0 ? 0 : best_cost;
}

// The tensor maps of a planned skinny form.
int encode_skinny(SkinnyParams* p, const uint8_t* a, const uint8_t* sfa, const uint8_t* b,
                  const uint8_t* sfb, uint16_t* out) {
    const int64_t M = p->M, N = p->N, K = p->K, k_tiles = p->k_tiles;
    if (encode_operand(&p->tma_x, a, M, K, (uint32_t)p->mt / 2) != 0 ||
        encode_scales(&p->tma_sfx, sfa, M, k_tiles, 1))
        return -1;
    if (encode_operand(&p->tma_w, b, N, K) != 0 || encode_scales(&p->tma_sfw, sfb, N, k_tiles, 1))
        return -2;
    if (encode_output(&p->tma_out, out, M, N, (uint32_t)p->mt, CU_TENSOR_MAP_SWIZZLE_NONE) != 0)
        return -3;
    return 0;
}

// Launch configuration of the general form (clusters of one CTA pair).
cudaLaunchConfig_t general_config(cudaLaunchAttribute* attrs, void* stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = static_cast<cudaStream_t>(stream);
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = 2;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    // programmatic dependent launch: set-up overlaps the previous kernel's tail
    attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 2;
    return cfg;
}

// CTA pairs of the general form the current device holds at once (cached per
// device), or a negative cudaError_t.
int general_resident() {
    static int resident[kMaxDevices] = {0};
    int dev = 0;
    int err = (int)cudaGetDevice(&dev);
    if (err != cudaSuccess) return -err;
    if (dev < 0 || dev >= kMaxDevices) return -(int)cudaErrorInvalidDevice;
    if (resident[dev] > 0) return resident[dev];
    err = (int)cudaFuncSetAttribute(mxfp8_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kSmemBytes);
    if (err != cudaSuccess) return -err;
    int sms = 0, clusters = 0;
    err = (int)cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return -err;
    cudaLaunchAttribute attrs[2];
    cudaLaunchConfig_t cfg = general_config(attrs, nullptr);
    cfg.gridDim = dim3((unsigned)(sms & ~1), 1, 1);
    err = (int)cudaOccupancyMaxActiveClusters(&clusters, mxfp8_gemm_kernel, &cfg);
    if (err != cudaSuccess) return -err;
    if (clusters < 1) return -(int)cudaErrorInvalidConfiguration;
    resident[dev] = clusters;
    return clusters;
}

int launch_general(const GemmParams& p, void* stream) {
    // pairs the device holds at once (the persistent grid: a pair that had to
    // wait for another to finish would run its whole share of tiles late)
    const int resident = general_resident();
    if (resident < 0) return -resident;
    const int pairs = p.num_tiles < resident ? p.num_tiles : resident;
    if (pairs <= 0) return cudaSuccess;
    cudaLaunchAttribute attrs[2];
    cudaLaunchConfig_t cfg = general_config(attrs, stream);
    cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
    return (int)cudaLaunchKernelEx(&cfg, mxfp8_gemm_kernel, p);
}

template <int MT>
int launch_skinny(const SkinnyParams& p, void* stream) {
    if (p.splits < 1 || p.splits > kSkMaxSplits) return (int)cudaErrorInvalidConfiguration;
    const int resident = skinny_resident<MT>(p.splits);
    if (resident < 1) {
        const int err = (int)cudaGetLastError();
        return err != cudaSuccess ? err : (int)cudaErrorInvalidConfiguration;
    }
    const int clusters = p.num_tiles < resident ? p.num_tiles : resident;
    if (clusters <= 0) return cudaSuccess;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = skinny_config<MT>(p.splits, attr, stream);
    // programmatic dependent launch: set-up overlaps the previous kernel's tail
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
    cfg.gridDim = dim3((unsigned)(clusters * 2 * p.splits), 1, 1);
    return (int)cudaLaunchKernelEx(&cfg, mxfp8_gemm_skinny_kernel<MT>, p);
}

int launch_skinny(const SkinnyParams& p, void* stream) {
    return p.mt <= 64 ? launch_skinny<64>(p, stream) : launch_skinny<128>(p, stream);
}

}  // namespace

int gemm_plan(GemmPlan* plan, const uint8_t* a, const uint8_t* sfa, const uint8_t* b,
              const uint8_t* sfb, uint16_t* out, int64_t M, int64_t N, int64_t K) {
    const int form = hook_gemm_form();
    if (form == 1 || M > kSkinnyMaxM) {
        plan->skinny = false;
        return prepare_general(&plan->general, a, sfa, b, sfb, out, M, N, K);
    }
    plan_skinny(&plan->thin, M, N, K);
    if (M <= 64 || form == 2) {
        plan->skinny = true;
        return encode_skinny(&plan->thin, a, sfa, b, sfb, out);
    }
    // 64 < M <= kSkinnyMaxM: the form with the smaller estimate. In cycles per
    // wave of tiles (measured on graph replays): general, 512 per 128-byte K
    // step and 3.3k for the tile switch; skinny at mt = 128, 330 per K step
    // (the split's hand-overs counted as K steps) and 2k for the epilogue.
    // Past 128 rows the skinny form is taken only when its tiles (activation
    // row blocks x weight blocks) fit in one wave: each further wave re-reads
    // the weight, and the estimate misses that (measured: 384 x 14336 x 4096
    // skinny in 3 waves 27.7 us, general in 2 waves 25.4 us).
    const int resident = general_resident();
    const int64_t k_tiles = (K + kBK - 1) / kBK;
    const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
    const int64_t general =
        resident > 0 ? (tiles + resident - 1) / resident * (512 * k_tiles + 3300) : -1;
    const int64_t thin_waves = (plan->thin.num_tiles + plan->thin.resident - 1) /
                               (plan->thin.resident > 0 ? plan->thin.resident : 1);
    const int64_t thin = 330 * plan->thin.cost + 2000 * thin_waves;
    plan->skinny = general < 0 || (thin < general && (M <= 128 || thin_waves == 1));
    return plan->skinny ? encode_skinny(&plan->thin, a, sfa, b, sfb, out)
                        : prepare_general(&plan->general, a, sfa, b, sfb, out, M, N, K);
}

int gemm_launch(const GemmPlan& plan, void* stream) {
    if (const int e = hook_launch_error()) return e;
    return plan.skinny ? launch_skinny(plan.thin, stream) : launch_general(plan.general, stream);
}

int gemm_status(bool clear, unsigned long long* out) {
    // every stream's work first: the copy below is ordered only after the
    // legacy default stream
    int err = (int)cudaDeviceSynchronize();
    if (err != cudaSuccess) return err;
    err = (int)cudaMemcpyFromSymbol(out, g_gemm_status, sizeof *out);
    if (err != cudaSuccess) return err;
    if (clear && *out != 0) {
        const unsigned long long zero = 0;
        err = (int)cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof zero);
    }
    return err;
}

}  // namespace mx
