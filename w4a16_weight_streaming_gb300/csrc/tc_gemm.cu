// tcgen05 tensor-core path of the W4A16 GEMM (any M), swap-AB orientation:
//
//   D[n][m] = sum_k W[k][n] * x[m][k]      A = W^T (128 output columns n = 128 TMEM lanes),
//                                          B = x tile (MT rows of x, K-major, shared memory),
//                                          D = fp32 accumulators in TMEM (128 lanes x MT columns).
//
// A never touches shared memory in fp16: dequantisation warps read the packed nibbles that TMA
// streamed into shared memory, dequantise in registers (exact fp16, common.cuh) and write the
// fp16 pairs straight into TMEM with tcgen05.st; the MMA reads A from TMEM (the "A in tensor
// memory" form of tcgen05.mma). Shared memory carries 0.5 B per weight instead of 2.
//
// Two rings:
//   shared-memory stages (s_stages): per stage ONE bulk copy of the 128-column tile's packed
//     weights for KC rows of K (contiguous in the streaming layout), ONE bulk copy of its scales,
//     ONE 3-D tensor copy of the x tile (KC/64 blocks of 64 k x MT rows, 128-byte swizzle, rows
//     beyond M zero-filled), all completing one mbarrier.
//   TMEM A stages (a_stages): KC/2 columns each (fp16 pairs).
//
// Warp roles:
//   warps 0-15 dequantise: warp w owns TMEM lanes 32*(w%4).. (column slice w%4) and part w/4 of
//              every stage's K range (KC/4 rows). All 16 run the epilogue.
//   warp 16    TMA producer (one thread); also allocates and frees TMEM.
// The stage's k-steps are split among NA fp32 accumulators D_0..D_{NA-1} (summed in order by
// the epilogue), so that NA threads issue tcgen05.mma: one thread issues one MMA only every
// ~45-55 cycles, slower than HBM delivers weights for the small-N MMAs of decode shapes. Two
// issue schemes (template GROUP_ISSUE):
//   dedicated (small tiles): warps 17.. issue, one per accumulator; the dequant warps arrive on
//     afull[a]; issuer 0 polls it and wakes the other issuers through a named barrier.
//   grouped (64-row tiles with 2 accumulators and the 256-row tile): the 16/NA dequant warps of the
//     parts feeding one accumulator meet at a named barrier once their A pieces are in TMEM, and the
//     group's first warp issues the group's k-steps itself. (Measured on GB300: the 256-row tile is
//     faster grouped, 81 against 86 us on 5120 x 34816 at M = 256; the 128-row tile is faster with
//     dedicated issuers, 57 against 63 us at M = 128.)
// Barriers: full[s] (TMA bytes landed; with dedicated issuers the x tile completes its own xfull[s],
// which only the issuers wait for, so that the dequantisation starts once the weights are in) ->
// A in TMEM -> MMAs -> tcgen05.commit by each issuer ->
// empty[s] (shared stage free; producer) and aempty[a] (TMEM A stage free; dequant warps). Every
// mbarrier wait is bounded; grouped warps leave their loop only through a barrier reduction, so a
// group leaves together.
//
// Split-K: the `split` CTAs of a thread-block cluster cover disjoint K ranges of the same
// 128 x MT output tile; after the mainloop each CTA writes its fp32 partial tile to shared
// memory and the cluster sums them through distributed shared memory in rank order, each CTA
// finishing 1/split of the tile. No global scratch memory is used.
//
// Work items: a launch covers the work items (column tile x row tile) [item0, item_end). A GEMM whose
// items overfill whole waves of resident CTAs can run as two launches on the same stream: the whole
// waves unsplit, then the remaining items split along K. An unsplit launch of the 128- or 256-row
// tile with more items than resident CTAs runs persistent (template PERSIST): one CTA per slot,
// each taking every slots-th item, its TMA ring and barrier phases running on from one item to the
// next, so that the copies for the next item overlap the last MMAs and the epilogue of the current
// one; the dequantisation warps meet at a barrier after each epilogue before the next item's MMAs
// overwrite the accumulator.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace w4a16 {
namespace {

// DW dequant warps = 4 lane quadrants x DW/4 K parts (16, or 8 for the two-CTAs-per-SM variant);
// warp DW is the TMA producer and TMEM allocator, warps DW+1.. the dedicated MMA issuers.
__host__ __device__ constexpr int threads_for(bool group_issue, int na, int dw) {
    return 32 * (dw + 1 + (group_issue ? 0 : na));
}
constexpr int kTileN = 128;  // output columns per CTA (= TMEM lanes)

struct SmemPlan {
    uint32_t x_off, x_stage;  // x tiles: s_stages x (MT * KC * 2)
    uint32_t w_off, w_stage;  // packed weights: s_stages x (128 * KC / 2)
    uint32_t s_off, s_stage;  // scales: s_stages x (ngs * 128 * 2)
    uint32_t red_off;         // split-K partial tile, MT * 128 * 4 (may overlap the x tiles)
    uint32_t bar_off;         // 3 * s_stages + 2 * a_stages + 1 mbarriers
    uint32_t misc_off;        // tmem address slot, abort flag, two issuer go flags, items committed
    uint32_t total;           // bytes from the 1024-aligned base
};

__host__ __device__ inline int groups_per_stage(int KC, int G) { return KC >= G ? KC / G : 1; }

__host__ __device__ inline SmemPlan make_plan(int MT, int KC, int s_stages, int a_stages, int G, int split) {
    SmemPlan p;
    p.x_stage = static_cast<uint32_t>(MT * KC * 2);
    p.w_stage = static_cast<uint32_t>(kTileN * KC / 2);
    p.s_stage = static_cast<uint32_t>(groups_per_stage(KC, G) * kTileN * 2);
    p.x_off = 0;
    p.w_off = p.x_off + s_stages * p.x_stage;
    p.s_off = p.w_off + s_stages * p.w_stage;
    uint32_t end = p.s_off + s_stages * p.s_stage;
    const uint32_t red_bytes = static_cast<uint32_t>(MT * kTileN * 4);
    if (split > 1 && red_bytes > s_stages * p.x_stage) {
        p.red_off = (end + 15u) & ~15u;
        end = p.red_off + red_bytes;
    } else {
        p.red_off = 0;
    }
    p.bar_off = (end + 7u) & ~7u;
    p.misc_off = p.bar_off + (3 * s_stages + 2 * a_stages + 1) * 8;
    p.total = p.misc_off + 20;
    return p;
}

__host__ __device__ inline int tmem_cols_needed(int MT, int KC, int a_stages, int accs) {
    return a_stages * (KC / 2) + accs * MT;
}

__host__ __device__ inline uint32_t tmem_alloc_cols(int MT, int KC, int a_stages, int accs) {
    const int need = tmem_cols_needed(MT, KC, a_stages, accs);
    uint32_t c = 32;
    while (static_cast<int>(c) < need) c <<= 1;
    return c;
}

__device__ __forceinline__ void tma_load_x_3d(uint32_t dst, const void* tmap, int k0, int m0, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            dst),
        "l"(tmap), "r"(0), "r"(m0), "r"(k0 / 64), "r"(bar)
        : "memory");
}

// Warp-wide wait with a fast path: when the phase is already complete (the usual case for a deep
// ring) one non-blocking test by every lane settles it; otherwise lane 0 polls (warp_wait).
__device__ __forceinline__ bool warp_wait_fast(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                               uint64_t timeout_ns, unsigned* status) {
    if (__all_sync(0xffffffffu, mbar_test_wait(bar, parity))) return true;
    return warp_wait(bar, parity, abort_flag, timeout_ns, status);
}

// Named barrier over `nthreads` threads that also ANDs a predicate across them.
__device__ __forceinline__ bool group_sync_and(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.and.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0u;
}

// FP4: NVFP4 weights (E2M1 codes in the canonical nibble order, G = 16 fp16 scales: two scale rows
// per 32-k block) instead of int4 with offset 8. tensor_scale multiplies every fp32 sum before
// the fp16 rounding (1 for int4); row_scale, when not null, then multiplies the sums of output row
// m by row_scale[m] (the int8 activations' per-token scale).
template <int MT, int KC, int NA, bool GROUP_ISSUE, int DW, bool FP4, bool PERSIST>
__global__ void __launch_bounds__(threads_for(GROUP_ISSUE, NA, DW), 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const uint4* __restrict__ wr,
                   const uint16_t* __restrict__ sr, uint16_t* __restrict__ y, int M, int N, int K, int G,
                   int split, int item0, int item_end, int s_stages, int a_stages, int x_3d, float tensor_scale,
                   const float* __restrict__ row_scale, unsigned* status, uint64_t timeout_ns) {
    static_assert(MT % 16 == 0 && MT >= 16 && MT <= 256, "MMA N must be a multiple of 16 in [16, 256]");
    static_assert(KC == 128 || KC == 256, "stage K must be 128 or 256");
    static_assert(NA == 1 || NA == 2 || NA == 4, "1, 2 or 4 accumulators");
    constexpr int kKB = KC / 32;                   // 32-k blocks per stage
    constexpr int kDequantWarps = DW;
    constexpr int kProducerWarp = DW;              // also the TMEM allocator
    constexpr int kIssuerWarp0 = DW + 1;           // first dedicated MMA issuer (dedicated scheme)
    constexpr int kParts = DW / 4;                 // K parts of a stage
    static_assert(DW == 8 || DW == 16, "8 or 16 dequant warps");
    static_assert(kKB % kParts == 0, "stage rows split evenly over the K parts");
    constexpr int kPartKB = kKB / kParts;          // 32-k blocks per dequant warp per stage (1 or 2)
    static_assert(kPartKB == 1 || kPartKB == 2, "1 or 2 blocks per warp per stage");
    constexpr int kACols = KC / 2;                 // TMEM columns of one A stage (fp16 pairs)
    constexpr int kGroupWarps = kDequantWarps / NA;  // warps feeding one accumulator
    constexpr int kGroupSteps = KC / 16 / NA;        // k-steps of 16 per accumulator per stage
    constexpr int kThreads = threads_for(GROUP_ISSUE, NA, DW);

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    const SmemPlan P = make_plan(MT, KC, s_stages, a_stages, G, split);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + P.bar_off;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (s_stages + s); };
    auto aempty_bar = [&](int a) { return bar0 + 8u * (2 * s_stages + a); };
    auto afull_bar = [&](int a) { return bar0 + 8u * (2 * s_stages + a_stages + a); };  // dedicated scheme
    const uint32_t dfull_bar = bar0 + 8u * (2 * s_stages + 2 * a_stages);
    // The x tile's own barrier (dedicated issuers: the dequantisation warps wait only for the weights
    // and scales, the issuers for x); the grouped scheme, whose issuing warp also dequantises, keeps
    // one barrier for all three copies.
    auto xfull_bar = [&](int s) {
        return GROUP_ISSUE ? full_bar(s) : bar0 + 8u * (2 * s_stages + 2 * a_stages + 1 + s);
    };
    constexpr uint32_t kXBytes = static_cast<uint32_t>(MT * KC * 2);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + P.misc_off);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P.misc_off + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t ncols = tmem_alloc_cols(MT, KC, a_stages, NA);

    if (threadIdx.x == 0) {
        for (int s = 0; s < s_stages; ++s) {
            mbar_init(full_bar(s), 1);  // weights and scales (and, grouped scheme, x) landed
            if (!GROUP_ISSUE) mbar_init(xfull_bar(s), 1);
            mbar_init(empty_bar(s), NA);  // one commit per accumulator group
        }
        for (int a = 0; a < a_stages; ++a) {
            mbar_init(aempty_bar(a), NA);
            mbar_init(afull_bar(a), kDequantWarps);  // one elected arrival per dequant warp
        }
        mbar_init(dfull_bar, NA);
        *abort_flag = 0;
        *reinterpret_cast<volatile int*>(smem + P.misc_off + 16) = 0;
        fence_barrier_init();
    }
    if (warp == kProducerWarp) {
        tmem_alloc(smem_u32(tmem_slot), ncols);
        tmem_relinquish();
        if (lane == 0) prefetch_tmap(&tmap_x);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t d_tmem = tmem + static_cast<uint32_t>(a_stages * kACols);

    // Work items (column tile, row tile) in [item0, item_end), the row tile varying fastest: cluster
    // cl of the launch (`split` consecutive CTAs) takes items item0 + cl, item0 + cl + ncl, ... One
    // item per cluster when the grid covers them all; several, back to back, for a persistent grid
    // of unsplit CTAs, whose copies for the next item then overlap the current item's last MMAs and
    // epilogue. Consecutive items run side by side, so the CTAs that stream one weight tile for
    // different rows of x all but the first find it in L2.
    const int mtiles = (M + MT - 1) / MT;
    const int rank = static_cast<int>(blockIdx.x) % split;
    const int cl = static_cast<int>(blockIdx.x) / split;
    const int ncl = static_cast<int>(gridDim.x) / split;
    const int first_item = item0 + cl;
    const int KB = K / 32;
    const int NG = K / G;
    const int ngs = groups_per_stage(KC, G);
    const int C = K / KC;
    const int c_begin = static_cast<int>((static_cast<int64_t>(rank) * C) / split);
    const int c_end = static_cast<int>((static_cast<int64_t>(rank + 1) * C) / split);
    const int niter = c_end - c_begin;  // stages per item, the same for every item of this CTA
    struct Item {
        int tile, n0, wt, m0;  // wt: columns of the tile (32, 64, 96 or 128)
    };
    auto item_at = [&](int rest) {
        Item it;
        it.tile = rest / mtiles;
        it.n0 = it.tile * kTileN;
        it.wt = min(kTileN, N - it.n0);
        it.m0 = (rest % mtiles) * MT;
        return it;
    };
    // items whose accumulator the issuers committed (dfull phases), for the drain at exit
    volatile int* items_committed = reinterpret_cast<volatile int*>(smem + P.misc_off + 16);
    const Item it1 = item_at(first_item);  // the first (with split > 1 the only) item of this cluster

    if (warp == kProducerWarp) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            // (debug-bounds build: every copy's source range inside its buffer; a copy that is not
            // issued leaves its stage incomplete, so the kernel also reports the wait's timeout)
            const int64_t w_bytes_all = static_cast<int64_t>(N) * K / 2, s_bytes_all = static_cast<int64_t>(NG) * N * 2;
            int issued = 0;  // stage uses of the ring issued, over all items of this CTA
            if constexpr (!PERSIST) {  // one work item (this straight form measured faster than the loop)
                const uint4* w_tile = wr + static_cast<int64_t>(it1.tile) * kTileN * KB;     // [K/32][wt] vectors
                const uint16_t* s_tile = sr + static_cast<int64_t>(it1.tile) * kTileN * NG;  // [K/G][wt]
                const int wt = it1.wt, m0 = it1.m0;
                const uint32_t wbytes = static_cast<uint32_t>(kKB * wt * 16);
                const uint32_t sbytes = static_cast<uint32_t>(ngs * wt * 2);
                const uint32_t bytes = wbytes + sbytes + (GROUP_ISSUE ? kXBytes : 0u);
                auto issue_w = [&](int i) {  // weights and scales of stage use i (no dependence on x)
                    const int s = i % s_stages;
                    const int k0 = (c_begin + i) * KC;
                    const uint32_t fb = full_bar(s);
                    const uint4* wsrc = w_tile + static_cast<int64_t>(k0 / 32) * wt;
                    const uint16_t* ssrc = s_tile + static_cast<int64_t>(k0 / G) * wt;
                    mbar_arrive_expect_tx(fb, bytes);
                    if (in_bounds((wsrc - wr) * 16 + wbytes <= w_bytes_all, status))
                        bulk_g2s(sbase + P.w_off + s * P.w_stage, wsrc, wbytes, fb, pol);
                    if (in_bounds((ssrc - sr) * 2 + sbytes <= s_bytes_all, status))
                        bulk_g2s(sbase + P.s_off + s * P.s_stage, ssrc, sbytes, fb, pol);
                };
                auto issue_x = [&](int i) {
                    const int s = i % s_stages;
                    const int k0 = (c_begin + i) * KC;
                    in_bounds(k0 + KC <= K && m0 < M, status);  // rows >= M of the box are zero-filled by the copy
                    const uint32_t xs = sbase + P.x_off + s * P.x_stage;
                    if (!GROUP_ISSUE) mbar_arrive_expect_tx(xfull_bar(s), kXBytes);
                    if (x_3d) {
                        tma_load_x_3d(xs, &tmap_x, k0, m0, xfull_bar(s));
                    } else {
#pragma unroll
                        for (int a = 0; a < KC / 64; ++a)
                            tma_load_2d(xs + a * MT * 128, &tmap_x, k0 + 64 * a, m0, xfull_bar(s));
                    }
                };
                // Programmatic dependent launch: the first ring fill of weights goes out before the
                // previous grid on the stream has finished; x (possibly its output) only after.
                const int pre = niter < s_stages ? niter : s_stages;
                for (int i = 0; i < pre; ++i) issue_w(i);
                griddep_wait();
                for (int i = 0; i < pre; ++i) issue_x(i);
                issued = pre;
                for (int i = pre; i < niter; ++i) {
                    // far ahead of the consumers: a suspending wait costs no issue slots and no latency here
                    const uint32_t ph = static_cast<uint32_t>(i / s_stages) & 1u;  // parity of this use of the stage
                    if (!mbar_wait(empty_bar(i % s_stages), ph ^ 1u, abort_flag, timeout_ns, status)) break;
                    issue_w(i);
                    issue_x(i);
                    issued = i + 1;
                }
            } else {  // every item of this CTA, the ring continuing from one item to the next
                bool go_on = true;
                for (int rest = first_item;; rest += ncl) {
                    const Item it = item_at(rest);
                    const uint4* w_tile = wr + static_cast<int64_t>(it.tile) * kTileN * KB;     // [K/32][wt] vectors
                    const uint16_t* s_tile = sr + static_cast<int64_t>(it.tile) * kTileN * NG;  // [K/G][wt]
                    const uint32_t wbytes = static_cast<uint32_t>(kKB * it.wt * 16);
                    const uint32_t sbytes = static_cast<uint32_t>(ngs * it.wt * 2);
                        const uint32_t bytes = wbytes + sbytes + (GROUP_ISSUE ? kXBytes : 0u);
                    auto issue_w = [&](int i, int u) {  // weights and scales of stage i, ring use u (no x)
                        const int s = u % s_stages;
                        const int k0 = (c_begin + i) * KC;
                        const uint32_t fb = full_bar(s);
                        const uint4* wsrc = w_tile + static_cast<int64_t>(k0 / 32) * it.wt;
                        const uint16_t* ssrc = s_tile + static_cast<int64_t>(k0 / G) * it.wt;
                        mbar_arrive_expect_tx(fb, bytes);
                        if (in_bounds((wsrc - wr) * 16 + wbytes <= w_bytes_all, status))
                            bulk_g2s(sbase + P.w_off + s * P.w_stage, wsrc, wbytes, fb, pol);
                        if (in_bounds((ssrc - sr) * 2 + sbytes <= s_bytes_all, status))
                            bulk_g2s(sbase + P.s_off + s * P.s_stage, ssrc, sbytes, fb, pol);
                    };
                    auto issue_x = [&](int i, int u) {
                        const int s = u % s_stages;
                        const int k0 = (c_begin + i) * KC;
                        in_bounds(k0 + KC <= K && it.m0 < M, status);  // rows >= M of the box are zero-filled
                        const uint32_t xs = sbase + P.x_off + s * P.x_stage;
                        if (!GROUP_ISSUE) mbar_arrive_expect_tx(xfull_bar(s), kXBytes);
                        if (x_3d) {
                            tma_load_x_3d(xs, &tmap_x, k0, it.m0, xfull_bar(s));
                        } else {
#pragma unroll
                            for (int a = 0; a < KC / 64; ++a)
                                tma_load_2d(xs + a * MT * 128, &tmap_x, k0 + 64 * a, it.m0, xfull_bar(s));
                        }
                    };
                    int i = 0;
                    if (rest == first_item) {  // the first ring fill, as above
                        const int pre = niter < s_stages ? niter : s_stages;
                        for (int k = 0; k < pre; ++k) issue_w(k, k);
                        griddep_wait();
                        for (int k = 0; k < pre; ++k) issue_x(k, k);
                        issued = i = pre;
                    }
                    for (; i < niter; ++i) {
                        const int u = issued;
                        const uint32_t ph = static_cast<uint32_t>(u / s_stages) & 1u;  // parity of this use of the slot
                        if (u >= s_stages && !mbar_wait(empty_bar(u % s_stages), ph ^ 1u, abort_flag, timeout_ns, status)) {
                            go_on = false;
                            break;
                        }
                        issue_w(i, u);
                        issue_x(i, u);
                        ++issued;
                    }
                    if (!PERSIST || !go_on || rest + ncl >= item_end) break;
                }
            }
            griddep_launch_dependents();
            // Let the copies still in flight land before shared memory can be released.
            int dummy_abort = 0;
            for (int i = issued > s_stages ? issued - s_stages : 0; i < issued; ++i) {  // (only after the loop)
                mbar_wait(full_bar(i % s_stages), static_cast<uint32_t>(i / s_stages) & 1u, &dummy_abort, timeout_ns,
                          status);
                if (!GROUP_ISSUE)
                    mbar_wait(xfull_bar(i % s_stages), static_cast<uint32_t>(i / s_stages) & 1u, &dummy_abort,
                              timeout_ns, status);
            }
        }
        __syncwarp();
    } else if (!GROUP_ISSUE && warp >= kIssuerWarp0) {
        // ---------------- dedicated MMA issuers, one per accumulator
        const int j = warp - kIssuerWarp0;
        constexpr uint32_t idesc = idesc_f16_f32(128, MT);
        const uint32_t d_j = d_tmem + static_cast<uint32_t>(j * MT);
        const uint64_t desc0 = smem_desc_sw128(sbase + P.x_off);
        const uint32_t stage_step = P.x_stage >> 4;
        // go[i & 1]: issuer 0's verdict for stage i, double-buffered so that one named barrier per
        // stage suffices (every reader has read go[(i - 1) & 1] before it reaches barrier i).
        volatile int* go = reinterpret_cast<volatile int*>(smem + P.misc_off + 8);
        int s = 0, a = 0;
        uint32_t sph = 0, aph = 0;
        int u = 0;  // stage uses consumed, over all items
        int n_done = 0;
        bool go_on = true;
        for (int rest = first_item;; rest += ncl) {
            for (int i = 0; i < niter; ++i, ++u) {
                const int gu = PERSIST ? u : i;  // this stage's use of the ring, over all items
                if (j == 0 && lane == 0)
                    go[gu & 1] = (mbar_spin(afull_bar(a), aph, abort_flag, timeout_ns, status) &&
                                 mbar_spin(xfull_bar(s), sph, abort_flag, timeout_ns, status))
                                    ? 1
                                    : 0;
                if (NA > 1) asm volatile("bar.sync 5, %0;" ::"n"(32 * NA) : "memory");
                else __syncwarp();
                if (go[gu & 1] == 0) {
                    go_on = false;
                    break;
                }
                if (lane == 0) {
                    tc_fence_after();
                    const uint32_t a_tmem = tmem + static_cast<uint32_t>(a * kACols);
                    const uint64_t dstage = desc0 + static_cast<uint64_t>(s * stage_step);
#pragma unroll
                    for (int t = 0; t < kGroupSteps; ++t) {
                        const int ks = j + t * NA;  // interleaved k-steps keep the issuers evenly busy
                        const uint32_t koff = static_cast<uint32_t>(((ks / 4) * MT * 128 + (ks % 4) * 32) >> 4);
                        umma_f16_ts(d_j, a_tmem + ks * 8, dstage + koff, idesc, (i > 0) || (t > 0));
                    }
                    umma_commit(empty_bar(s));
                    umma_commit(aempty_bar(a));
                }
                __syncwarp();
                if (++s == s_stages) {
                    s = 0;
                    sph ^= 1u;
                }
                if (++a == a_stages) {
                    a = 0;
                    aph ^= 1u;
                }
            }
            if (lane == 0) umma_commit(dfull_bar);
            ++n_done;
            __syncwarp();
            if (!PERSIST || !go_on || rest + ncl >= item_end) break;
        }
        if (j == 0 && lane == 0) *items_committed = n_done;
        __syncwarp();
    } else {
        // ---------------- dequantisation warps (and, grouped scheme, per group one MMA issuer)
        const int q = warp & 3;
        const int part = warp >> 2;
        const int grp = warp / kGroupWarps;               // accumulator group
        const bool issuer = (warp % kGroupWarps) == 0;    // first warp of the group issues its MMAs
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        // scale row (within a stage's scale block) of each of this warp's 32-k blocks
        int srow[kPartKB];
#pragma unroll
        for (int u = 0; u < kPartKB; ++u) srow[u] = KC >= G ? (32 * (part * kPartKB + u)) / G : 0;
        const uint32_t sst0 = sbase + P.s_off + 2u * static_cast<uint32_t>(32 * q + lane);
        const uint32_t a_base = tmem + lane_base + static_cast<uint32_t>(part * kPartKB * 16);
        // MMA operands of this group: k-steps grp*kGroupSteps .. +kGroupSteps of each stage
        constexpr uint32_t idesc = idesc_f16_f32(128, MT);
        const uint32_t d_g = d_tmem + static_cast<uint32_t>(grp * MT);
        const uint64_t desc0 = smem_desc_sw128(sbase + P.x_off);
        const uint32_t stage_step = P.x_stage >> 4;
        int s = 0, a = 0;
        uint32_t sph = 0, aph = 0;
        int u = 0;      // stage uses consumed, over all items
        int jdone = 0;  // items entered (each commits the accumulator once)
        for (int rest = first_item;; rest += ncl) {
            const Item it = item_at(rest);
            const int wt = it.wt, n0 = it.n0, m0 = it.m0;
            const bool valid = 32 * q < wt;
            // shared address of this lane's first vector in stage 0 (explicit shared loads)
            const uint32_t wst0 = sbase + P.w_off + 16u * static_cast<uint32_t>(32 * q + lane + part * kPartKB * wt);
            for (int i = 0; i < niter; ++i, ++u) {
                bool ok = warp_wait_fast(full_bar(s), sph, abort_flag, timeout_ns, status);
                if (ok && (PERSIST ? u : i) >= a_stages)
                    ok = warp_wait_fast(aempty_bar(a), aph ^ 1u, abort_flag, timeout_ns, status);
                if (ok && valid) {
                    const uint32_t wst = wst0 + static_cast<uint32_t>(s) * P.w_stage;
                    const uint32_t sst = sst0 + static_cast<uint32_t>(s) * P.s_stage;
                    uint32_t regs[kPartKB * 16];
                    uint4 v[kPartKB];
                    uint32_t sb[kPartKB], sb2[kPartKB];
#pragma unroll
                    for (int u = 0; u < kPartKB; ++u) {
                        v[u] = lds128(wst + 16u * static_cast<uint32_t>(u * wt));
                        sb[u] = lds16(sst + 2u * static_cast<uint32_t>(srow[u] * wt));
                        // NVFP4: the block's second 16-k half has the next scale row
                        sb2[u] = FP4 ? lds16(sst + 2u * static_cast<uint32_t>((srow[u] + 1) * wt)) : sb[u];
                    }
#pragma unroll
                    for (int u = 0; u < kPartKB; ++u) {
                        const uint32_t s2 = sb[u] | (sb[u] << 16);
                        if (FP4) {
                            const uint32_t s2b = sb2[u] | (sb2[u] << 16);
                            dequant8_nvfp4(v[u].x, s2, &regs[u * 16 + 0]);
                            dequant8_nvfp4(v[u].y, s2, &regs[u * 16 + 4]);
                            dequant8_nvfp4(v[u].z, s2b, &regs[u * 16 + 8]);
                            dequant8_nvfp4(v[u].w, s2b, &regs[u * 16 + 12]);
                        } else {
                            dequant8(v[u].x, s2, &regs[u * 16 + 0]);
                            dequant8(v[u].y, s2, &regs[u * 16 + 4]);
                            dequant8(v[u].z, s2, &regs[u * 16 + 8]);
                            dequant8(v[u].w, s2, &regs[u * 16 + 12]);
                        }
                    }
                    tmem_st<kPartKB * 16>(a_base + static_cast<uint32_t>(a * kACols), regs);
                    tmem_wait_st();
                }
                tc_fence_before();
                if (!GROUP_ISSUE) {
                    __syncwarp();
                    if (!ok) break;
                    if (lane == 0) mbar_arrive(afull_bar(a));
                } else {
                // the group's A pieces for this stage are in TMEM (or some warp gave up a wait)
                if (!group_sync_and(1 + grp, 32 * kGroupWarps, ok)) break;
                if (issuer && lane == 0) {
                    tc_fence_after();
                    const uint32_t a_tmem = tmem + static_cast<uint32_t>(a * kACols);
                    const uint64_t dstage = desc0 + static_cast<uint64_t>(s * stage_step);
#pragma unroll
                    for (int t = 0; t < kGroupSteps; ++t) {
                        const int ks = grp * kGroupSteps + t;  // k-step of 16 within the stage
                        const uint32_t koff = static_cast<uint32_t>(((ks / 4) * MT * 128 + (ks % 4) * 32) >> 4);
                        umma_f16_ts(d_g, a_tmem + ks * 8, dstage + koff, idesc, (i > 0) || (t > 0));
                    }
                    umma_commit(empty_bar(s));
                    umma_commit(aempty_bar(a));
                }
                }
                __syncwarp();
                if (++s == s_stages) {
                    s = 0;
                    sph ^= 1u;
                }
                if (++a == a_stages) {
                    a = 0;
                    aph ^= 1u;
                }
            }
            if (GROUP_ISSUE && issuer && lane == 0) umma_commit(dfull_bar);
            __syncwarp();

            // ---------------- epilogue: TMEM -> registers -> y (or the split-K partial tile)
            griddep_wait();  // y may still be read or written by the previous grid on the stream
            const bool have_d = warp_wait(dfull_bar, static_cast<uint32_t>(jdone) & 1u, abort_flag, timeout_ns, status);
            tc_fence_after();
            if (have_d) {
                constexpr int kPartCols = MT / kParts;  // accumulator columns (activation rows) per K part
                constexpr int kCols = kPartCols < 8 ? kPartCols : 8;  // columns per TMEM load
                const int mbase = part * kPartCols;
                float* red = reinterpret_cast<float*>(smem + P.red_off);
                const int n = n0 + 32 * q + lane;
#pragma unroll 1
                for (int c = 0; c < kPartCols; c += kCols) {
                    uint32_t r[kCols];
                    tmem_ld<kCols>(tmem + lane_base + static_cast<uint32_t>(a_stages * kACols + mbase + c), r);
                    tmem_wait_ld();
#pragma unroll
                    for (int g = 1; g < NA; ++g) {  // fixed order: D_0 + D_1 + ...
                        uint32_t r2[kCols];
                        tmem_ld<kCols>(tmem + lane_base + static_cast<uint32_t>(a_stages * kACols + g * MT + mbase + c), r2);
                        tmem_wait_ld();
#pragma unroll
                        for (int t = 0; t < kCols; ++t) r[t] = __float_as_uint(__uint_as_float(r[t]) + __uint_as_float(r2[t]));
                    }
                    if (split == 1) {
                        if (valid) {
#pragma unroll
                            for (int j = 0; j < kCols; ++j) {
                                const int m = m0 + mbase + c + j;
                                if (m < M && in_bounds(static_cast<int64_t>(m) * N + n < static_cast<int64_t>(M) * N, status)) {
                                    float v = __uint_as_float(r[j]) * tensor_scale;
                                    if (row_scale != nullptr) v *= row_scale[m];
                                    y[static_cast<int64_t>(m) * N + n] = __half_as_ushort(__float2half_rn(v));
                                }
                            }
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < kCols; ++j)
                            red[(mbase + c + j) * kTileN + 32 * q + lane] = __uint_as_float(r[j]);
                    }
                }
            }
            tc_fence_before();
            ++jdone;
            if (!PERSIST) break;
            // every dequantisation warp has read the accumulator before an issuer starts the next
            // item's MMAs into it; after an abort all leave together
            if (!group_sync_and(6, 32 * kDequantWarps, *abort_flag == 0) || rest + ncl >= item_end) break;
        }
        if (GROUP_ISSUE && warp == 0 && lane == 0) *items_committed = jdone;
        __syncwarp();
    }

    if (split > 1) {  // (one work item per cluster)
        const int m0 = it1.m0, n0 = it1.n0, wt = it1.wt;
        __syncwarp();
        griddep_wait();  // every thread of the reduction writes y
        cluster_sync_all();
        const int E4 = MT * kTileN / 4;
        const int beg = static_cast<int>((static_cast<int64_t>(rank) * E4) / split);
        const int end = static_cast<int>((static_cast<int64_t>(rank + 1) * E4) / split);
        const uint32_t red_s = sbase + P.red_off;
        for (int e4 = beg + static_cast<int>(threadIdx.x); e4 < end; e4 += kThreads) {  // all warps
            float4 acc = cluster_sum_f4(red_s + 16u * e4, split);
            acc.x *= tensor_scale;
            acc.y *= tensor_scale;
            acc.z *= tensor_scale;
            acc.w *= tensor_scale;
            const int e = 4 * e4;
            const int m = m0 + e / kTileN;
            const int c = e % kTileN;
            if (m < M && c < wt &&
                in_bounds(static_cast<int64_t>(m) * N + n0 + c + 4 <= static_cast<int64_t>(M) * N, status)) {
                if (row_scale != nullptr) {
                    const float rs = row_scale[m];
                    acc.x *= rs;
                    acc.y *= rs;
                    acc.z *= rs;
                    acc.w *= rs;
                }
                const uint32_t lo = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc.x))) |
                                    (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc.y))) << 16);
                const uint32_t hi = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc.z))) |
                                    (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc.w))) << 16);
                *reinterpret_cast<uint2*>(y + static_cast<int64_t>(m) * N + n0 + c) = make_uint2(lo, hi);
            }
        }
        __syncwarp();
        cluster_sync_all();
    }

    __syncthreads();
    if (warp == kProducerWarp) {
        // Every issuer commits dfull after its loop, also when it left early, so this phase
        // completes once the MMAs in flight (reading the x stages and writing TMEM) have drained.
        // After an abort the epilogue did not wait for it; wait here, with a private abort flag and
        // still bounded, before shared memory and TMEM are released.
        if (lane == 0) {
            int drain_abort = 0;
            const int n = *items_committed;  // the last committed phase: n - 1
            if (n > 0) mbar_wait(dfull_bar, static_cast<uint32_t>(n - 1) & 1u, &drain_abort, timeout_ns, status);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

// ------------------------------------------------------------------------------------ host
// Dynamic shared memory for a config: the plan, plus padding so that no more CTAs share an SM
// than its TMEM can hold (no CTA ever waits in tcgen05.alloc for a CTA of another cluster).
size_t launch_smem(int MT, int KC, int G, const TcConfig& c) {
    const SmemPlan P = make_plan(MT, KC, c.stages, c.tmem_stages, G, c.split);
    size_t smem = P.total + 1024;  // + alignment slack for the 1024-byte base
    const int per_sm_tmem = 512 / static_cast<int>(tmem_alloc_cols(MT, KC, c.tmem_stages, c.issuers));
    const size_t min_smem = 233472 / (per_sm_tmem + 1) - 1024 + 16;
    return smem < min_smem ? min_smem : smem;
}

template <typename Kern>
cudaError_t prepare_kernel(Kern kern, size_t smem, int split) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (split > 8) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

template <int MT, int KC, int NI, bool GI, int DW>
cudaLaunchConfig_t make_config(const TcConfig& c, int items, size_t smem, cudaStream_t stream,
                               cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(c.split) * static_cast<unsigned>(items), 1, 1);
    cfg.blockDim = dim3(threads_for(GI, NI, DW), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (c.split > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = c.split;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cfg;
}

// The kernel for a launch: the persistent form (several work items per CTA) exists for the 128-
// and 256-row tiles, whose one-CTA-per-SM grids span several waves at large M.
template <int MT, int KC, int NI, bool GI, int DW>
auto tc_kernel_for(bool fp4, bool persist) {
    if constexpr (MT >= 128) {
        if (persist)
            return fp4 ? tc_gemm_kernel<MT, KC, NI, GI, DW, true, true> : tc_gemm_kernel<MT, KC, NI, GI, DW, false, true>;
    }
    return fp4 ? tc_gemm_kernel<MT, KC, NI, GI, DW, true, false> : tc_gemm_kernel<MT, KC, NI, GI, DW, false, false>;
}

template <int MT, int KC, int NI, bool GI, int DW>
cudaError_t launch_tc_t(const CUtensorMap& tmap, bool three_d, const uint32_t* qweight_r, const uint16_t* scales_r,
                        uint16_t* y, int M, int N, int K, int G, const TcConfig& c, const LaunchCtx& ctx) {
    const int items = ((N + kTileN - 1) / kTileN) * ((M + MT - 1) / MT);
    const int tail = c.tail_items;
    // the work items of the full waves, then those of the last partial wave, split further along K
    for (int part = 0; part < 2; ++part) {
        TcConfig cp = c;
        if (part == 1) cp.split = c.tail_split;
        const int n = part == 0 ? items - tail : tail;
        if (n <= 0) continue;
        const int first = part == 0 ? 0 : items - tail;
        const bool persist = MT >= 128 && cp.split == 1 && c.persist_ctas > 0 && n > c.persist_ctas;
        const int clusters = persist ? c.persist_ctas : n;
        auto kern = tc_kernel_for<MT, KC, NI, GI, DW>(ctx.nvfp4 != 0, persist);
        const size_t smem = launch_smem(MT, KC, G, cp);
        cudaError_t e = prepare_kernel(kern, smem, cp.split);
        if (e != cudaSuccess) return e;
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg = make_config<MT, KC, NI, GI, DW>(cp, clusters, smem, ctx.stream, attr);
        e = cudaLaunchKernelEx(&cfg, kern, tmap, reinterpret_cast<const uint4*>(qweight_r), scales_r, y, M, N, K, G,
                               cp.split, first, first + n, cp.stages, cp.tmem_stages, three_d ? 1 : 0,
                               ctx.tensor_scale, ctx.row_scale, ctx.status, ctx.timeout_ns);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// CTAs of this config the device keeps resident at once (clusters x cluster size), or 0.
template <int MT, int KC, int NI, bool GI, int DW>
int resident_ctas_t(const TcConfig& c, int G) {
    auto kern = tc_gemm_kernel<MT, KC, NI, GI, DW, false, false>;  // (the other variants: the same resources)
    const size_t smem = launch_smem(MT, KC, G, c);
    if (prepare_kernel(kern, smem, c.split) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c.split, 1, 1);
    cfg.blockDim = dim3(threads_for(GI, NI, DW), 1, 1);
    cfg.dynamicSmemBytes = smem;
    attr[0].id = cudaLaunchAttributeClusterDimension;  // the cluster shape, also for split 1
    attr[0].val.clusterDim.x = c.split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return clusters * c.split;
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// x viewed as [K/64 blocks][M rows][64 k] (strides 128 B and 2K B): one box = the whole stage
// tile [KC/64][MT][64], laid out in shared memory exactly as the MMA's 128-byte-swizzle K-major
// operand atoms expect. Falls back to a 2-D map ([M][K], box 64 x MT, KC/64 copies per stage)
// if the driver refuses the 3-D one.
bool encode_x_map(CUtensorMap* map, const uint16_t* x, int M, int K, int MT, int KC, bool* three_d) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode == nullptr) return false;
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    {
        const cuuint64_t dims[3] = {64u, static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(K / 64)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 128u};
        const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(MT), static_cast<cuuint32_t>(KC / 64)};
        if (encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<uint16_t*>(x), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS) {
            *three_d = true;
            return true;
        }
    }
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(MT)};
    *three_d = false;
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// (m_tile, k_chunk, issuers, group issue, dequant warps) of every instantiated kernel.
#define W4A16_TC_COMBOS(X)                                                                              \
    X(16, 128, 4, false, 16) X(16, 256, 4, false, 16) X(32, 128, 4, false, 16) X(32, 256, 4, false, 16) \
    X(64, 128, 4, false, 16) X(64, 256, 4, false, 16) X(64, 256, 2, true, 16) X(128, 128, 2, false, 16)  \
    X(128, 128, 1, false, 16) X(256, 128, 1, true, 16) X(16, 128, 4, false, 8) X(32, 128, 4, false, 8)    \
    X(64, 128, 2, false, 8)

bool tc_instantiated(int m_tile, int k_chunk, int issuers, int dequant_warps) {
#define W4A16_TC_IS(MT_, KC_, NI_, GI_, DW_) \
    if (m_tile == MT_ && k_chunk == KC_ && issuers == NI_ && dequant_warps == DW_) return true;
    W4A16_TC_COMBOS(W4A16_TC_IS)
#undef W4A16_TC_IS
    return false;
}

bool tc_config_valid(const TcConfig& c, int M, int N, int K, int G) {
    if (c.m_tile != 16 && c.m_tile != 32 && c.m_tile != 64 && c.m_tile != 128 && c.m_tile != 256) return false;
    // grid.x = split x column tiles x row tiles must stay below 2^31
    if (static_cast<int64_t>(c.split) * ((N + 127) / 128) * ((M + c.m_tile - 1) / c.m_tile) > 0x7fffffffLL)
        return false;
    if (c.k_chunk != 128 && c.k_chunk != 256) return false;
    if (K % c.k_chunk != 0) return false;
    if (c.stages < 2 || c.stages > 16) return false;
    if (c.tmem_stages < 2 || c.tmem_stages > 8) return false;
    if (c.split < 1 || c.split > 16 || c.split > K / c.k_chunk) return false;
    if (!tc_instantiated(c.m_tile, c.k_chunk, c.issuers, c.dequant_warps)) return false;
    if (tmem_cols_needed(c.m_tile, c.k_chunk, c.tmem_stages, c.issuers) > 512) return false;
    if (c.k_chunk < G && G % c.k_chunk != 0) return false;
    if (c.k_chunk >= G && c.k_chunk % G != 0) return false;
    const SmemPlan P = make_plan(c.m_tile, c.k_chunk, c.stages, c.tmem_stages, G, c.split);
    if (P.total + 1024 > 232448) return false;
    if (c.tail_items < 0) return false;
    if (c.tail_items > 0) {  // a second launch for the last partial wave's items, split 2..16 ways
        const int64_t items = static_cast<int64_t>((N + 127) / 128) * ((M + c.m_tile - 1) / c.m_tile);
        if (c.tail_items >= items) return false;
        if (c.tail_split < 2 || c.tail_split > 16 || c.tail_split > K / c.k_chunk) return false;
        if (static_cast<int64_t>(c.tail_split) * c.tail_items > 0x7fffffffLL) return false;
        if (make_plan(c.m_tile, c.k_chunk, c.stages, c.tmem_stages, G, c.tail_split).total + 1024 > 232448)
            return false;
    }
    return true;
}

size_t tc_smem_bytes(const TcConfig& c, int G) {
    return make_plan(c.m_tile, c.k_chunk, c.stages, c.tmem_stages, G, c.split).total + 1024;
}

int tc_tmem_cols(const TcConfig& c) {
    return static_cast<int>(tmem_alloc_cols(c.m_tile, c.k_chunk, c.tmem_stages, c.issuers));
}

int tc_resident_ctas(const TcConfig& c, int G) {
#define W4A16_TC_RES(MT_, KC_, NI_, GI_, DW_)                                                           \
    if (c.m_tile == MT_ && c.k_chunk == KC_ && c.issuers == NI_ && c.dequant_warps == DW_) \
        return resident_ctas_t<MT_, KC_, NI_, GI_, DW_>(c, G);
    W4A16_TC_COMBOS(W4A16_TC_RES)
#undef W4A16_TC_RES
    return 0;
}

cudaError_t launch_tc(const uint16_t* x, const uint32_t* qweight_r, const uint16_t* scales_r, uint16_t* y, int M,
                      int N, int K, int G, const TcConfig& c, const LaunchCtx& ctx) {
    CUtensorMap tmap;
    bool three_d = false;
    if (!encode_x_map(&tmap, x, M, K, c.m_tile, c.k_chunk, &three_d)) return cudaErrorInvalidValue;
#define W4A16_TC_CASE(MT_, KC_, NI_, GI_, DW_)                                                          \
    if (c.m_tile == MT_ && c.k_chunk == KC_ && c.issuers == NI_ && c.dequant_warps == DW_)               \
        return launch_tc_t<MT_, KC_, NI_, GI_, DW_>(tmap, three_d, qweight_r, scales_r, y, M, N, K, G, c, ctx);
    W4A16_TC_COMBOS(W4A16_TC_CASE)
#undef W4A16_TC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace w4a16
