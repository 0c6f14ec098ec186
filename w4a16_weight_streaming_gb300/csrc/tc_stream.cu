// Persistent tcgen05 streaming kernel for the bandwidth-bound shapes (M <= 64 activation rows):
// the decode and speculative-verify GEMMs whose cost is one read of the packed weights ("Qwen3.8-27B
// at 764, 1,035 and 1,623 tok/s", section "One weight read, shared by every stream").
//
//   D[n][m] = sum_k W[k][n] * x[m][k]   swap-AB as in tc_gemm.cu: A = dequantised W^T in TMEM
//                                        (128 output columns = 128 TMEM lanes), B = x in shared
//                                        memory, D = fp32 in TMEM.
//
// What differs from tc_gemm.cu, and why (all measured on GB300):
//  * For MMA N <= 64 every tcgen05.mma (M = 128, K = 16) costs ~40 cycles of the SM's tensor pipe
//    whatever its N, i.e. the pipe consumes 1 KB of packed weights per ~40 cycles, about one SM's
//    share of HBM bandwidth, while one thread issues an MMA only every ~110 cycles. The MMAs must
//    run back to back: NA issuer threads (own accumulators, interleaved k-steps), all woken through
//    one named barrier per TMEM A stage (no polling, ~20-cycle wake-up), commit per stage.
//  * TMA moves ~23 B/clk per SM from DRAM, again about one SM's share of HBM: the x operand is made
//    resident in shared memory once per launch instead of being copied with every weight stage,
//    so the TMA carries only packed weights and scales.
//  * Grids of short-lived CTAs paid a ~2,600-cycle prologue and a pipeline drain per tile, plus a
//    tail wave: here each cluster is persistent and walks its share of the 128-column tiles with
//    one continuous shared-memory ring; the accumulator is double-buffered in TMEM so that the
//    epilogue of tile j overlaps the main loop of tile j + 1.
//
// Grid: (split, clusters). The `split` CTAs of a cluster own disjoint K slices [r*C/split,
// (r+1)*C/split) of the K/KC chunks, the same for every tile; cluster c processes tiles c,
// c + clusters, ... Partial tiles are summed through distributed shared memory in rank order.
//
// Waiting: a thread suspended in mbarrier.try_wait wakes up hundreds to thousands of cycles after the
// phase completes (measured), so no warp on the critical path suspends: single threads poll with
// test_wait, and the 16 dequant warps are released per stage through a named barrier by one
// scheduler warp that polls the TMA and TMEM phases for them.
//
// Warp roles (32 * (22 + NA) threads):
//   0-15  dequantise: warp w owns TMEM lanes 32*(w%4) (column slice w%4) and K part w/4 of every
//         stage; reads the packed stage from shared memory, writes exact fp16 A with tcgen05.st.
//   16    TMA producer (one thread): resident x slice once, then weights + scales per stage; also
//         allocates and frees TMEM.
//   17..  NA MMA issuers (one thread each), issuer j owning accumulator D_j and k-steps j, j+NA, ...
//   next 4: epilogue: TMEM -> registers (D_0 + D_1 + ... in order) -> y, or -> partial tile ->
//         cluster reduction -> y. The accumulators are double-buffered when TMEM has room.
//   last: scheduler: per stage, polls full[s] and aempty[a], then releases the dequant warps.
// Barriers: full[s] (TMA landed) and aempty[a] (TMEM A stage free) -> scheduler -> named barrier
// 8+a (go) -> dequant warps -> empty[s] (stage reusable, producer) and named barrier 1+a (A stage a
// in TMEM, issuers) -> MMAs -> aempty[a] (commit) ...
// last stage of a tile -> dfull[b] (commit; epilogue) -> dempty[b] (epilogue read D[b]; issuer).
// Split-K: redfull[b] / redempty[b] count one arrival per cluster rank. Every wait is bounded.
#include "common.cuh"
#include "internal.h"

namespace w4a16 {
namespace {

constexpr int kTileN = 128;
constexpr int kDqWarps = 16;
constexpr int kProdWarp = 16;
constexpr int kMmaWarp0 = 17;
constexpr int kEpiWarps = 4;
__host__ __device__ constexpr int stream_threads(int na) { return 32 * (kDqWarps + 1 + na + kEpiWarps + 1); }
constexpr int kEpiBarId = 15;
constexpr int kGoBar0 = 8;          // named barriers 8..14: stage released to the dequant warps
constexpr int kMaxAStages = 7;      // A-ready barriers 1..7, go barriers 8..14
constexpr int kGoBarThreads = 32 * (kDqWarps + 1);

__host__ __device__ inline int stream_groups_per_stage(int KC, int G) { return KC >= G ? KC / G : 1; }

struct StreamSmem {
    uint32_t x_off, x_chunk;  // resident x slice: nck chunks of MT * KC * 2 bytes
    uint32_t w_off, w_stage;  // packed weights ring
    uint32_t s_off, s_stage;  // scales ring
    uint32_t red_off, red_buf;  // split > 1: two partial tiles MT * 128 fp32
    uint32_t bar_off;         // 2 * stages + a_stages + 10 mbarriers
    uint32_t misc_off;        // TMEM address slot, abort flag
    uint32_t total;
};

__host__ __device__ inline StreamSmem stream_smem_plan(int MT, int KC, int nck, int stages, int a_stages, int G,
                                                       int split) {
    StreamSmem p;
    p.x_chunk = static_cast<uint32_t>(MT * KC * 2);
    p.x_off = 0;
    p.w_stage = static_cast<uint32_t>(kTileN * KC / 2);
    p.w_off = p.x_off + static_cast<uint32_t>(nck) * p.x_chunk;
    p.s_stage = static_cast<uint32_t>(stream_groups_per_stage(KC, G) * kTileN * 2);
    p.s_off = p.w_off + static_cast<uint32_t>(stages) * p.w_stage;
    uint32_t end = p.s_off + static_cast<uint32_t>(stages) * p.s_stage;
    p.red_buf = static_cast<uint32_t>(MT * kTileN * 4);
    p.red_off = (end + 15u) & ~15u;
    if (split > 1) end = p.red_off + 2u * p.red_buf;
    p.bar_off = (end + 7u) & ~7u;
    p.misc_off = p.bar_off + static_cast<uint32_t>(2 * stages + a_stages + 10) * 8u;
    p.total = p.misc_off + 16u;
    return p;
}

__host__ __device__ inline int stream_tmem_cols(int MT, int KC, int a_stages, int na, int dbuf) {
    return a_stages * (KC / 2) + dbuf * na * MT;
}

__device__ __forceinline__ void tma_load_x_3d_s(uint32_t dst, const void* tmap, int k0, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            dst),
        "l"(tmap), "r"(0), "r"(0), "r"(k0 / 64), "r"(bar)
        : "memory");
}

// Barrier over the four epilogue warps (named barrier 15) that also ANDs a predicate across them.
__device__ __forceinline__ bool epi_sync_and(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "barrier.red.and.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "n"(kEpiBarId), "n"(32 * kEpiWarps)
        : "memory");
    return r != 0u;
}

// Warp-wide bounded wait on a phase completed by cluster peers: lane 0 polls, then every lane takes
// the cluster-scope acquire of the completed phase.
__device__ __forceinline__ bool warp_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                  uint64_t timeout_ns, unsigned* status) {
    int ok = 1;
    if ((threadIdx.x & 31u) == 0u) ok = mbar_wait_cluster(bar, parity, abort_flag, timeout_ns, status) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) mbar_test_wait_cluster(bar, parity);
    return ok != 0;
}

template <int MT, int KC, int NA>
__global__ void __launch_bounds__(stream_threads(NA), 1)
    tc_stream_kernel(const __grid_constant__ CUtensorMap tmap_x, const uint4* __restrict__ wr,
                     const uint16_t* __restrict__ sr, uint16_t* __restrict__ y, int M, int N, int K, int G,
                     int stages, int a_stages, int dbuf, int x_3d, unsigned* status, uint64_t timeout_ns) {
    static_assert(MT == 16 || MT == 32 || MT == 64, "streaming tiles hold 16, 32 or 64 activation rows");
    static_assert(KC == 128 || KC == 256, "stage K must be 128 or 256");
    static_assert(NA == 2 || NA == 4, "2 or 4 MMA issuers");
    constexpr int kEpiWarp0 = kMmaWarp0 + NA;
    constexpr int kSchedWarp = kEpiWarp0 + kEpiWarps;
    constexpr int kAStageBarThreads = 32 * (kDqWarps + NA);  // dequant warps + the issuer warps
    constexpr int kKB = KC / 32;      // 32-k blocks per stage
    constexpr int kPartKB = kKB / 4;  // 32-k blocks per dequant warp per stage (1 or 2)
    constexpr int kACols = KC / 2;    // TMEM columns of one A stage (fp16 pairs)
    constexpr int kSteps = KC / 16;   // MMAs per stage
    constexpr int kIssSteps = kSteps / NA;  // MMAs per stage per issuer

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    const int split = gridDim.x;
    const int rank = blockIdx.x;
    const int C = K / KC;
    const int c_begin = static_cast<int>((static_cast<int64_t>(rank) * C) / split);
    const int c_end = static_cast<int>((static_cast<int64_t>(rank + 1) * C) / split);
    const int nck = c_end - c_begin;              // chunks of this CTA's K slice
    const int nck_max = (C + split - 1) / split;  // sizes the resident x region
    const StreamSmem P = stream_smem_plan(MT, KC, nck_max, stages, a_stages, G, split);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + P.bar_off;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (stages + s); };
    auto aempty_bar = [&](int a) { return bar0 + 8u * (2 * stages + a); };
    const uint32_t xfull_bar = bar0 + 8u * (2 * stages + a_stages);
    auto dfull_bar = [&](int b) { return xfull_bar + 8u * (1 + b); };
    auto dempty_bar = [&](int b) { return xfull_bar + 8u * (3 + b); };
    auto redfull_bar = [&](int b) { return xfull_bar + 8u * (5 + b); };
    auto redempty_bar = [&](int b) { return xfull_bar + 8u * (7 + b); };
    const uint32_t drain_bar = xfull_bar + 8u * 9;  // every MMA of this CTA has completed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + P.misc_off);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P.misc_off + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t ncols = 512;  // one CTA per SM

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kDqWarps);  // one elected arrival per dequant warp
        }
        for (int a = 0; a < a_stages; ++a) mbar_init(aempty_bar(a), NA);  // one commit per issuer
        mbar_init(xfull_bar, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(dfull_bar(b), NA);
            mbar_init(dempty_bar(b), kEpiWarps);
            mbar_init(redfull_bar(b), split);
            mbar_init(redempty_bar(b), split);
        }
        mbar_init(drain_bar, NA);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kProdWarp) {
        tmem_alloc(smem_u32(tmem_slot), ncols);
        tmem_relinquish();
        if (lane == 0) prefetch_tmap(&tmap_x);
    }
    tc_fence_before();
    __syncthreads();
    if (split > 1) cluster_sync_all();  // peers' barriers are initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t d_tmem = tmem + static_cast<uint32_t>(a_stages * kACols);  // D[b][j] at + (b * NA + j) * MT

    const int n_tiles = (N + kTileN - 1) / kTileN;
    const int n_clusters = gridDim.y;
    const int KB = K / 32;
    const int NG = K / G;
    const int ngs = stream_groups_per_stage(KC, G);

    if (warp == kProdWarp) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint32_t xbytes = static_cast<uint32_t>(nck) * P.x_chunk;
            mbar_arrive_expect_tx(xfull_bar, xbytes);
            for (int c = 0; c < nck; ++c) {
                const uint32_t dst = sbase + P.x_off + static_cast<uint32_t>(c) * P.x_chunk;
                const int k0 = (c_begin + c) * KC;
                if (x_3d) {
                    tma_load_x_3d_s(dst, &tmap_x, k0, xfull_bar);
                } else {
#pragma unroll
                    for (int a = 0; a < KC / 64; ++a) tma_load_2d(dst + a * MT * 128, &tmap_x, k0 + 64 * a, 0, xfull_bar);
                }
            }
            const uint64_t pol = policy_evict_first();
            int s = 0;
            uint32_t ph = 0;
            int64_t it = 0;
            bool ok = true;
            for (int tile = blockIdx.y; ok && tile < n_tiles; tile += n_clusters) {
                const int wt = min(kTileN, N - tile * kTileN);
                const uint32_t wbytes = static_cast<uint32_t>(kKB * wt * 16);
                const uint32_t sbytes = static_cast<uint32_t>(ngs * wt * 2);
                const uint4* w_tile = wr + static_cast<int64_t>(tile) * kTileN * KB;
                const uint16_t* s_tile = sr + static_cast<int64_t>(tile) * kTileN * NG;
                for (int c = c_begin; c < c_end; ++c, ++it) {
                    if (it >= stages && !mbar_spin(empty_bar(s), ph ^ 1u, abort_flag, timeout_ns, status)) {
                        ok = false;
                        break;
                    }
                    const int k0 = c * KC;
                    const uint32_t fb = full_bar(s);
                    mbar_arrive_expect_tx(fb, wbytes + sbytes);
                    bulk_g2s(sbase + P.w_off + s * P.w_stage, w_tile + static_cast<int64_t>(k0 / 32) * wt, wbytes, fb,
                             pol);
                    bulk_g2s(sbase + P.s_off + s * P.s_stage, s_tile + static_cast<int64_t>(k0 / G) * wt, sbytes, fb,
                             pol);
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // Copies still in flight land before this CTA may exit: wait for the last `stages` fills
            // (their full phases) and for the resident x.
            int dummy_abort = 0;
            const int64_t first = it > stages ? it - stages : 0;
            for (int64_t i = first; i < it; ++i)
                mbar_wait(full_bar(static_cast<int>(i % stages)), static_cast<uint32_t>((i / stages) & 1),
                          &dummy_abort, timeout_ns, status);
            mbar_wait(xfull_bar, 0, &dummy_abort, timeout_ns, status);
        }
        __syncwarp();
    } else if (warp >= kMmaWarp0 && warp < kEpiWarp0) {
        // ------------------------------------------------------------ MMA issuers
        const int jn = warp - kMmaWarp0;  // this issuer's accumulator and k-step phase
        constexpr uint32_t idesc = idesc_f16_f32(128, MT);
        bool ok = warp_wait(xfull_bar, 0, abort_flag, timeout_ns, status);
        tc_fence_after();
        // Every issuer takes part in every stage's named barrier, also after a failed wait or an abort
        // (then it only stops issuing): issuers that left the loop early would hang the others.
        int a = 0;
        int j = 0;
        for (int tile = blockIdx.y; tile < n_tiles; tile += n_clusters, ++j) {
            const int b = j % dbuf;
            const int use = j / dbuf;  // uses of buffer b so far
            if (ok && use >= 1)
                ok = warp_spin(dempty_bar(b), static_cast<uint32_t>((use - 1) & 1), abort_flag, timeout_ns, status);
            tc_fence_after();
            const uint32_t d = d_tmem + static_cast<uint32_t>((b * NA + jn) * MT);
            for (int cl = 0; cl < nck; ++cl) {
                named_sync(1 + a, kAStageBarThreads);  // A stage a written by all dequant warps
                if (*abort_flag) ok = false;
                if (ok && lane == 0) {
                    tc_fence_after();
                    const uint32_t a_tmem = tmem + static_cast<uint32_t>(a * kACols);
                    const uint64_t desc = smem_desc_sw128(sbase + P.x_off + static_cast<uint32_t>(cl) * P.x_chunk);
#pragma unroll
                    for (int t = 0; t < kIssSteps; ++t) {
                        const int ks = jn + t * NA;  // interleaved k-steps keep the issuers evenly busy
                        const uint32_t koff = static_cast<uint32_t>(((ks / 4) * MT * 128 + (ks % 4) * 32) >> 4);
                        umma_f16_ts(d, a_tmem + ks * 8, desc + koff, idesc, (cl > 0) || (t > 0));
                    }
                    umma_commit(aempty_bar(a));
                }
                __syncwarp();
                if (++a == a_stages) a = 0;
            }
            if (ok && lane == 0) umma_commit(dfull_bar(b));
            __syncwarp();
        }
        // No MMA may still be writing TMEM when it is freed (matters only after an abort).
        if (lane == 0) {
            umma_commit(drain_bar);
            int dummy_abort = 0;
            mbar_wait(drain_bar, 0, &dummy_abort, timeout_ns, status);
        }
        __syncwarp();
    } else if (warp < kDqWarps) {
        // ------------------------------------------------------------ dequantisation warps
        const int q = warp & 3;
        const int part = warp >> 2;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        int srow[kPartKB];
#pragma unroll
        for (int u = 0; u < kPartKB; ++u) srow[u] = KC >= G ? (32 * (part * kPartKB + u)) / G : 0;
        const uint32_t a_base = tmem + lane_base + static_cast<uint32_t>(part * kPartKB * 16);
        int s = 0, a = 0;
        bool ok = true;
        // Every dequant warp takes part in every stage's named barriers, also after an abort (then it
        // skips its work), so that the scheduler and the issuers, which do the same, never hang.
        for (int tile = blockIdx.y; tile < n_tiles; tile += n_clusters) {
            const int wt = min(kTileN, N - tile * kTileN);
            const bool valid = 32 * q < wt;
            // shared addresses of this lane's first vector / scale in stage 0
            const uint32_t wst0 = sbase + P.w_off + 16u * static_cast<uint32_t>(32 * q + lane + part * kPartKB * wt);
            const uint32_t sst0 = sbase + P.s_off + 2u * static_cast<uint32_t>(32 * q + lane);
            for (int cl = 0; cl < nck; ++cl) {
                named_sync(kGoBar0 + a, kGoBarThreads);  // stage s landed and A stage a is free
                tc_fence_after();                          // the MMAs that read A stage a are complete
                if (*abort_flag) ok = false;
                if (ok && valid) {
                    const uint32_t wst = wst0 + static_cast<uint32_t>(s) * P.w_stage;
                    const uint32_t sst = sst0 + static_cast<uint32_t>(s) * P.s_stage;
                    uint32_t regs[kPartKB * 16];
                    uint4 v[kPartKB];
                    uint32_t sb[kPartKB];
#pragma unroll
                    for (int u = 0; u < kPartKB; ++u) {
                        v[u] = lds128(wst + 16u * static_cast<uint32_t>(u * wt));
                        sb[u] = lds16(sst + 2u * static_cast<uint32_t>(srow[u] * wt));
                    }
#pragma unroll
                    for (int u = 0; u < kPartKB; ++u) {
                        const uint32_t s2 = sb[u] | (sb[u] << 16);
                        dequant8(v[u].x, s2, &regs[u * 16 + 0]);
                        dequant8(v[u].y, s2, &regs[u * 16 + 4]);
                        dequant8(v[u].z, s2, &regs[u * 16 + 8]);
                        dequant8(v[u].w, s2, &regs[u * 16 + 12]);
                    }
                    tmem_st<kPartKB * 16>(a_base + static_cast<uint32_t>(a * kACols), regs);
                    tmem_wait_st();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar(s));  // this warp's reads of stage s are done
                named_arrive(1 + a, kAStageBarThreads);    // always arrive: the issuer never hangs
                if (++s == stages) s = 0;
                if (++a == a_stages) a = 0;
            }
        }
    } else if (warp == kSchedWarp) {
        // ------------------------------------------------------------ scheduler
        int s = 0, a = 0;
        uint32_t sph = 0, aph = 0;
        int64_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.y; tile < n_tiles; tile += n_clusters) {
            for (int cl = 0; cl < nck; ++cl, ++it) {
                if (lane == 0) {
                    if (ok) ok = mbar_spin(full_bar(s), sph, abort_flag, timeout_ns, status);
                    if (ok && it >= a_stages) ok = mbar_spin(aempty_bar(a), aph ^ 1u, abort_flag, timeout_ns, status);
                }
                __syncwarp();
                named_arrive(kGoBar0 + a, kGoBarThreads);  // always: the dequant warps never hang
                if (++s == stages) {
                    s = 0;
                    sph ^= 1u;
                }
                if (++a == a_stages) {
                    a = 0;
                    aph ^= 1u;
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        float* red0 = reinterpret_cast<float*>(smem + P.red_off);
        constexpr int kCols = 8;
        int j = 0;
        for (int tile = blockIdx.y; tile < n_tiles; tile += n_clusters, ++j) {
            const int b = j % dbuf;  // accumulator buffer
            const int rb = j & 1;    // partial-tile buffer
            const uint32_t par = static_cast<uint32_t>((j / dbuf) & 1);
            const uint32_t rpar = static_cast<uint32_t>((j >> 1) & 1);
            const int n0 = tile * kTileN;
            const int wt = min(kTileN, N - n0);
            bool ok = warp_spin(dfull_bar(b), par, abort_flag, timeout_ns, status);
            // the peers have finished reading this CTA's partial tile of tile j - 2 (same buffer)
            if (ok && split > 1 && j >= 2)
                ok = warp_wait_cluster(redempty_bar(rb), rpar ^ 1u, abort_flag, timeout_ns, status);
            // the four warps leave together or not at all (they meet at named barriers below)
            if (!epi_sync_and(ok)) break;
            tc_fence_after();
            float* red = red0 + rb * (MT * kTileN);
            const int n = n0 + 32 * q + lane;
            const bool col_ok = 32 * q + lane < wt;
#pragma unroll 1
            for (int c = 0; c < MT; c += kCols) {
                uint32_t r[kCols];
                tmem_ld<kCols>(d_tmem + lane_base + static_cast<uint32_t>(b * NA * MT + c), r);
                tmem_wait_ld();
#pragma unroll
                for (int g = 1; g < NA; ++g) {  // fixed order: D_0 + D_1 + ...
                    uint32_t r2[kCols];
                    tmem_ld<kCols>(d_tmem + lane_base + static_cast<uint32_t>((b * NA + g) * MT + c), r2);
                    tmem_wait_ld();
#pragma unroll
                    for (int u = 0; u < kCols; ++u) r[u] = __float_as_uint(__uint_as_float(r[u]) + __uint_as_float(r2[u]));
                }
                if (split == 1) {
                    if (col_ok) {
#pragma unroll
                        for (int t = 0; t < kCols; ++t)
                            if (c + t < M)
                                y[static_cast<int64_t>(c + t) * N + n] =
                                    __half_as_ushort(__float2half_rn(__uint_as_float(r[t])));
                    }
                } else {
#pragma unroll
                    for (int t = 0; t < kCols; ++t) red[(c + t) * kTileN + 32 * q + lane] = __uint_as_float(r[t]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dempty_bar(b));  // D[b] may be overwritten (tile j + dbuf)
            if (split > 1) {
                named_sync(kEpiBarId, 32 * kEpiWarps);  // this CTA's partial tile is complete
                if (warp == kEpiWarp0 && lane == 0) {
                    asm volatile("fence.acq_rel.cluster;" ::: "memory");
                    for (int p = 0; p < split; ++p) mbar_arrive_remote(redfull_bar(rb), static_cast<uint32_t>(p));
                }
                if (!epi_sync_and(warp_wait_cluster(redfull_bar(rb), rpar, abort_flag, timeout_ns, status))) break;
                const int E4 = MT * kTileN / 4;
                const int beg = static_cast<int>((static_cast<int64_t>(rank) * E4) / split);
                const int end = static_cast<int>((static_cast<int64_t>(rank + 1) * E4) / split);
                const uint32_t red_s = sbase + P.red_off + static_cast<uint32_t>(rb) * P.red_buf;
                for (int e4 = beg + (warp - kEpiWarp0) * 32 + lane; e4 < end; e4 += 32 * kEpiWarps) {
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int p = 0; p < split; ++p) {  // fixed order: rank 0, 1, ...
                        const float4 v = ld_dsmem_f4(map_peer(red_s + 16u * e4, static_cast<uint32_t>(p)));
                        acc.x += v.x;
                        acc.y += v.y;
                        acc.z += v.z;
                        acc.w += v.w;
                    }
                    const int e = 4 * e4;
                    const int m = e / kTileN;
                    const int cc = e % kTileN;
                    if (m < M && cc < wt) {
                        const uint32_t lo = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc.x))) |
                                            (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc.y))) << 16);
                        const uint32_t hi = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc.z))) |
                                            (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc.w))) << 16);
                        *reinterpret_cast<uint2*>(y + static_cast<int64_t>(m) * N + n0 + cc) = make_uint2(lo, hi);
                    }
                }
                named_sync(kEpiBarId, 32 * kEpiWarps);  // this CTA is done reading the peers' partials
                if (warp == kEpiWarp0 && lane == 0) {
                    asm volatile("fence.acq_rel.cluster;" ::: "memory");
                    for (int p = 0; p < split; ++p) mbar_arrive_remote(redempty_bar(rb), static_cast<uint32_t>(p));
                }
            }
        }
    }

    __syncwarp();
    if (split > 1) cluster_sync_all();  // no CTA leaves while a peer may still read its partials
    __syncthreads();
    if (warp == kProdWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

size_t stream_launch_smem(int MT, int KC, int G, const StreamConfig& c, int K) {
    const int C = K / KC;
    const int nck_max = (C + c.split - 1) / c.split;
    return stream_smem_plan(MT, KC, nck_max, c.stages, c.tmem_stages, G, c.split).total + 1024;
}

template <int MT, int KC, int NA>
cudaError_t prepare_stream(size_t smem, int split) {
    auto kern = tc_stream_kernel<MT, KC, NA>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (split > 8) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

template <int MT, int KC, int NA>
cudaLaunchConfig_t stream_config(const StreamConfig& c, size_t smem, cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c.split, c.clusters, 1);
    cfg.blockDim = dim3(stream_threads(NA), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c.split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = c.split > 1 ? 1 : 0;
    return cfg;
}

template <int MT, int KC, int NA>
cudaError_t launch_stream_t(const CUtensorMap& tmap, bool three_d, const uint32_t* qweight_r,
                            const uint16_t* scales_r, uint16_t* y, int M, int N, int K, int G, const StreamConfig& c,
                            const LaunchCtx& ctx) {
    const size_t smem = stream_launch_smem(MT, KC, G, c, K);
    cudaError_t e = prepare_stream<MT, KC, NA>(smem, c.split);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = stream_config<MT, KC, NA>(c, smem, ctx.stream, attr);
    return cudaLaunchKernelEx(&cfg, tc_stream_kernel<MT, KC, NA>, tmap, reinterpret_cast<const uint4*>(qweight_r),
                              scales_r, y, M, N, K, G, c.stages, c.tmem_stages, c.dbuf, three_d ? 1 : 0, ctx.status,
                              ctx.timeout_ns);
}

template <int MT, int KC, int NA>
int stream_max_clusters_t(const StreamConfig& c, int G, int K) {
    const size_t smem = stream_launch_smem(MT, KC, G, c, K);
    if (prepare_stream<MT, KC, NA>(smem, c.split) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchAttribute attr[1];
    StreamConfig one = c;
    one.clusters = 1;
    cudaLaunchConfig_t cfg = stream_config<MT, KC, NA>(one, smem, nullptr, attr);
    cfg.numAttrs = 1;  // query with the cluster shape even for split 1
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, tc_stream_kernel<MT, KC, NA>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return clusters;
}

}  // namespace

// Instantiated (m_tile, k_chunk, issuers) combinations.
bool stream_instantiated(int m_tile, int k_chunk, int issuers) {
    static const int kCombos[][3] = {{16, 128, 4}, {16, 256, 4}, {32, 128, 4}, {32, 256, 4},
                                     {64, 128, 2}, {64, 256, 2}, {64, 128, 4}, {64, 256, 4}};
    for (const auto& t : kCombos)
        if (t[0] == m_tile && t[1] == k_chunk && t[2] == issuers) return true;
    return false;
}

int stream_tmem_columns(const StreamConfig& c) {
    return stream_tmem_cols(c.m_tile, c.k_chunk, c.tmem_stages, c.issuers, c.dbuf);
}

bool stream_config_valid(const StreamConfig& c, int M, int N, int K, int G) {
    (void)N;
    if (!stream_instantiated(c.m_tile, c.k_chunk, c.issuers)) return false;
    if (M > c.m_tile) return false;  // one activation block: x is resident
    if (K % c.k_chunk != 0) return false;
    if (c.k_chunk < G && G % c.k_chunk != 0) return false;
    if (c.k_chunk >= G && c.k_chunk % G != 0) return false;
    if (c.stages < 2 || c.stages > 16) return false;
    if (c.tmem_stages < 2 || c.tmem_stages > kMaxAStages) return false;
    if (c.dbuf != 1 && c.dbuf != 2) return false;
    if (stream_tmem_columns(c) > 512) return false;
    if (c.split < 1 || c.split > 16 || c.split > K / c.k_chunk) return false;
    if (c.clusters < 1) return false;
    if (stream_launch_smem(c.m_tile, c.k_chunk, G, c, K) > 232448) return false;
    return true;
}

size_t stream_smem_bytes(const StreamConfig& c, int G, int K) { return stream_launch_smem(c.m_tile, c.k_chunk, G, c, K); }

#define W4A16_ST_COMBOS(X) X(16, 128, 4) X(16, 256, 4) X(32, 128, 4) X(32, 256, 4) \
    X(64, 128, 2) X(64, 256, 2) X(64, 128, 4) X(64, 256, 4)

int stream_max_clusters(const StreamConfig& c, int G, int K) {
#define W4A16_ST_OCC(MT_, KC_, NA_) \
    if (c.m_tile == MT_ && c.k_chunk == KC_ && c.issuers == NA_) return stream_max_clusters_t<MT_, KC_, NA_>(c, G, K);
    W4A16_ST_COMBOS(W4A16_ST_OCC)
#undef W4A16_ST_OCC
    return 0;
}

cudaError_t launch_stream(const uint16_t* x, const uint32_t* qweight_r, const uint16_t* scales_r, uint16_t* y, int M,
                          int N, int K, int G, const StreamConfig& c, const LaunchCtx& ctx) {
    CUtensorMap tmap;
    bool three_d = false;
    if (!encode_x_map(&tmap, x, M, K, c.m_tile, c.k_chunk, &three_d)) return cudaErrorInvalidValue;
#define W4A16_ST_CASE(MT_, KC_, NA_)                    \
    if (c.m_tile == MT_ && c.k_chunk == KC_ && c.issuers == NA_) \
        return launch_stream_t<MT_, KC_, NA_>(tmap, three_d, qweight_r, scales_r, y, M, N, K, G, c, ctx);
    W4A16_ST_COMBOS(W4A16_ST_CASE)
#undef W4A16_ST_CASE
    return cudaErrorInvalidValue;
}

}  // namespace w4a16
