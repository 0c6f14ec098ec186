// Persistent stream-K tcgen05 kernel of the W4A16 GEMM for M <= 64 (one row tile of MT = 16, 32 or
// 64 activation rows). Swap-AB as in the tile kernel:
//
//   D[n][m] = sum_k W[k][n] * x[m][k]   A = dequantised W^T in TMEM (128 output columns = 128 lanes),
//                                       B = x tile in shared memory (K-major, 128-byte swizzle),
//                                       D = fp32 accumulators in TMEM.
//
// Work split (stream-K): the (128-column tile, KC-row chunk) units of the whole matrix, in
// tile-major order, are cut into gridDim.x contiguous ranges of equal length, one per CTA, so every
// SM streams the same number of weight bytes in one long run and no SM idles in a last wave. A
// CTA's range falls into segments, one per tile it touches. A segment that covers its whole tile
// writes y directly. A partial segment writes its fp32 partial tile to the workspace and adds one to
// the tile's counter; the CTA that brings the counter to the number of the tile's CTAs sums every
// partial of the tile in CTA order (deterministic), writes y and resets the counter. No CTA ever
// waits for another one.
//
// Warp roles (21 warps, one CTA per SM):
//   warps 0-15  four dequantisation groups of four warps; warp w is in group w/4 and owns the TMEM
//               lane quadrant w%4 (32 output columns, lane = column). Unit j of the CTA's range
//               belongs to group j%4: the group's warps read the stage's packed nibbles from shared
//               memory, dequantise them exactly (common.cuh) and store fp16 A into the group's own
//               TMEM ring, 64 k at a time; lane 0 of the group's first warp issues the group's MMAs
//               into the group's own accumulator. Groups wait on different stages, so they drift
//               apart, and one group's shared-memory reads, TMEM stores and hand-offs overlap the
//               others' arithmetic instead of every warp passing each stage in lockstep.
//   warp 16     TMA producer (one thread): per unit ONE bulk copy of the tile's packed weights (KC
//               rows are one contiguous block of the streaming layout), one of its scales, one 3-D
//               tensor copy of the x tile (rows >= M zero-filled); it also allocates and frees TMEM.
//   warps 17-20 epilogue: per segment, the sum of the groups' accumulators in group order, then y or
//               the partial tile. Accumulators are double-buffered where TMEM has room, so a
//               segment's epilogue overlaps the next segment's MMAs.
//
// Programmatic dependent launch: the producer issues the weight and scale copies of its first
// stages before griddepcontrol.wait (weights never depend on an earlier kernel), and the x copies
// after it; the epilogue waits before its first global write. Every mbarrier wait is bounded.
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace w4a16 {
namespace {

constexpr int kTileN = 128;
constexpr int kGroups = 4;
constexpr int kProducerWarp = 16;
constexpr int kEpiWarp0 = 17;
constexpr int kThreads = 21 * 32;
constexpr int kSubK = 64;      // k per TMEM A stage
constexpr int kSubCols = 32;   // TMEM columns of one A stage (fp16 pairs)
constexpr int kEpiBarrier = 1; // named barrier of the four epilogue warps

__host__ __device__ inline int sk_groups_per_stage(int KC, int G) { return KC >= G ? KC / G : 1; }

struct SkPlan {
    uint32_t x_off, x_stage;  // x tiles (1024-aligned for the 128-byte swizzle)
    uint32_t w_off, w_stage;  // packed weights
    uint32_t s_off, s_stage;  // scales
    uint32_t bar_off;         // mbarriers
    uint32_t misc_off;        // TMEM address, abort flag, fixup flag
    uint32_t total;           // bytes from the 1024-aligned base
};

__host__ __device__ inline int sk_num_barriers(int S, int SA, int NBUF) {
    return 2 * S + 2 * kGroups * SA + kGroups * NBUF + NBUF + 1;
}

__host__ __device__ inline SkPlan sk_plan(int MT, int KC, int S, int SA, int NBUF, int G) {
    SkPlan p;
    p.x_stage = static_cast<uint32_t>(MT * KC * 2);
    p.w_stage = static_cast<uint32_t>(kTileN * KC / 2);
    p.s_stage = static_cast<uint32_t>(sk_groups_per_stage(KC, G) * kTileN * 2);
    p.x_off = 0;
    p.w_off = p.x_off + S * p.x_stage;
    p.s_off = p.w_off + S * p.w_stage;
    const uint32_t end = p.s_off + S * p.s_stage;
    p.bar_off = (end + 7u) & ~7u;
    p.misc_off = p.bar_off + sk_num_barriers(S, SA, NBUF) * 8;
    p.total = p.misc_off + 16;
    return p;
}

// First unit of CTA b when U units are cut into nb equal contiguous ranges.
__device__ __forceinline__ long long range_begin(long long U, int nb, int b) { return U * b / nb; }

// The CTA whose range holds unit u.
__device__ __forceinline__ int cta_of_unit(long long U, int nb, long long u) {
    int b = static_cast<int>((u * nb) / U);
    while (b + 1 < nb && range_begin(U, nb, b + 1) <= u) ++b;
    while (b > 0 && range_begin(U, nb, b) > u) --b;
    return b;
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void tma_x_3d(uint32_t dst, const void* tmap, int k0, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            dst),
        "l"(tmap), "r"(0), "r"(0), "r"(k0 / 64), "r"(bar)
        : "memory");
}

// Warp-wide wait: every lane tests the phase once; if it is not yet complete, lane 0 waits (bounded).
__device__ __forceinline__ bool sk_warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             uint64_t timeout_ns, unsigned* status) {
    if (__all_sync(0xffffffffu, mbar_test_wait(bar, parity))) return true;
    return warp_wait(bar, parity, abort_flag, timeout_ns, status);
}

// Named barrier over the epilogue warps that also ANDs a predicate across them.
__device__ __forceinline__ bool epi_sync_and(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.and.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "n"(kEpiBarrier), "n"(128)
        : "memory");
    return r != 0u;
}

__device__ __forceinline__ void st_cg_f32(float* p, float v) {
    asm volatile("st.global.cg.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
__device__ __forceinline__ float ld_cg_f32(const float* p) {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// One segment of a CTA's range: units [j0, j0 + len) of the range, tile t, chunks [cb, cb + len).
struct Segment {
    int t, cb, len, j0;
};

template <int MT, int KC, int NBUF, int SA>
__global__ void __launch_bounds__(kThreads, 1)
    tc_streamk_kernel(const __grid_constant__ CUtensorMap tmap_x, const uint4* __restrict__ wr,
                      const uint16_t* __restrict__ sr, uint16_t* __restrict__ y, float* __restrict__ ws_part,
                      unsigned* __restrict__ ws_cnt, int M, int N, int K, int G, int S, unsigned* status,
                      uint64_t timeout_ns) {
    static_assert(MT == 16 || MT == 32 || MT == 64, "row tile of 16, 32 or 64");
    static_assert(KC == 128 || KC == 256, "stage of 128 or 256 k");
    static_assert(kGroups * SA * kSubCols + kGroups * NBUF * MT <= 512, "TMEM columns");
    constexpr int kSubs = KC / kSubK;   // TMEM A stages per unit
    constexpr uint32_t kAccBase = kGroups * SA * kSubCols;

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    const SkPlan P = sk_plan(MT, KC, S, SA, NBUF, G);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + P.bar_off;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto afull_bar = [&](int g, int a) { return bar0 + 8u * (2 * S + g * SA + a); };
    auto aempty_bar = [&](int g, int a) { return bar0 + 8u * (2 * S + kGroups * SA + g * SA + a); };
    auto dfull_bar = [&](int g, int b) { return bar0 + 8u * (2 * S + 2 * kGroups * SA + g * NBUF + b); };
    auto accfree_bar = [&](int b) { return bar0 + 8u * (2 * S + 2 * kGroups * SA + kGroups * NBUF + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * S + 2 * kGroups * SA + kGroups * NBUF + NBUF);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + P.misc_off);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P.misc_off + 4);
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + P.misc_off + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int g = 0; g < kGroups; ++g) {
            for (int a = 0; a < SA; ++a) {
                mbar_init(afull_bar(g, a), 4);  // one elected arrival per warp of the group
                mbar_init(aempty_bar(g, a), 1);
            }
            for (int b = 0; b < NBUF; ++b) mbar_init(dfull_bar(g, b), 1);
        }
        for (int b = 0; b < NBUF; ++b) mbar_init(accfree_bar(b), 4);  // the four epilogue warps
        mbar_init(drain_bar, kGroups);
        *abort_flag = 0;
        *last_flag = 0;
        fence_barrier_init();
    }
    if (warp == kProducerWarp) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
        if (lane == 0) prefetch_tmap(&tmap_x);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int nb = static_cast<int>(gridDim.x);
    const int cta = static_cast<int>(blockIdx.x);
    const int tiles = (N + kTileN - 1) / kTileN;
    const int C = K / KC;
    const int KB = K / 32;
    const int NG = K / G;
    const int ngs = sk_groups_per_stage(KC, G);
    const long long U = static_cast<long long>(tiles) * C;
    const long long u0 = range_begin(U, nb, cta);
    const long long u1 = range_begin(U, nb, cta + 1);
    const int nunits = static_cast<int>(u1 - u0);

    // the s-th segment of this CTA's range, walked identically by every role
    auto first_segment = [&]() {
        Segment sg;
        sg.t = static_cast<int>(u0 / C);
        sg.cb = static_cast<int>(u0 - static_cast<long long>(sg.t) * C);
        sg.len = static_cast<int>(min(u1, static_cast<long long>(sg.t + 1) * C) - u0);
        sg.j0 = 0;
        return sg;
    };
    auto next_segment = [&](const Segment& p) {
        Segment sg;
        sg.t = p.t + 1;
        sg.cb = 0;
        sg.j0 = p.j0 + p.len;
        sg.len = static_cast<int>(min(static_cast<long long>(nunits - sg.j0), static_cast<long long>(C)));
        return sg;
    };

    if (warp == kProducerWarp) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0 && nunits > 0) {
            const uint64_t pol = policy_evict_first();
            const uint32_t xbytes = static_cast<uint32_t>(MT * KC * 2);
            auto unit_tile = [&](int j) { return static_cast<int>((u0 + j) / C); };
            auto issue_w = [&](int j) {
                const long long u = u0 + j;
                const int t = static_cast<int>(u / C);
                const int c = static_cast<int>(u - static_cast<long long>(t) * C);
                const int wt = min(kTileN, N - kTileN * t);
                const int s = j % S;
                const uint32_t wbytes = static_cast<uint32_t>((KC / 32) * wt * 16);
                const uint32_t sbytes = static_cast<uint32_t>(ngs * wt * 2);
                const uint4* w_tile = wr + static_cast<int64_t>(t) * kTileN * KB;
                const uint16_t* s_tile = sr + static_cast<int64_t>(t) * kTileN * NG;
                mbar_arrive_expect_tx(full_bar(s), wbytes + sbytes + xbytes);
                bulk_g2s(sbase + P.w_off + s * P.w_stage, w_tile + static_cast<int64_t>(c) * (KC / 32) * wt, wbytes,
                         full_bar(s), pol);
                bulk_g2s(sbase + P.s_off + s * P.s_stage, s_tile + static_cast<int64_t>((c * KC) / G) * wt, sbytes,
                         full_bar(s), pol);
            };
            auto issue_x = [&](int j) {
                const long long u = u0 + j;
                const int c = static_cast<int>(u - static_cast<long long>(unit_tile(j)) * C);
                const int s = j % S;
                tma_x_3d(sbase + P.x_off + s * P.x_stage, &tmap_x, c * KC, full_bar(s));
            };
            const int pre = min(S, nunits);
            for (int j = 0; j < pre; ++j) issue_w(j);  // independent of any earlier kernel
            griddep_wait();                             // x may be an earlier kernel's output
            for (int j = 0; j < pre; ++j) issue_x(j);
            int issued = pre;
            for (int j = pre; j < nunits; ++j) {
                const int s = j % S;
                if (!mbar_wait(empty_bar(s), static_cast<uint32_t>((j / S) - 1) & 1u, abort_flag, timeout_ns, status))
                    break;
                issue_w(j);
                issue_x(j);
                issued = j + 1;
            }
            griddep_launch_dependents();
            // let the copies still in flight land before shared memory can be released
            int dummy_abort = 0;
            for (int i = issued > S ? issued - S : 0; i < issued; ++i)
                mbar_wait(full_bar(i % S), static_cast<uint32_t>(i / S) & 1u, &dummy_abort, timeout_ns, status);
        }
        __syncwarp();
    } else if (warp < kProducerWarp) {
        // ---------------------------------------------------------------- dequantisation groups
        const int g = warp >> 2;
        const int q = warp & 3;
        const bool issuer_warp = q == 0;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        const uint32_t a_ring = tmem + static_cast<uint32_t>(g * SA * kSubCols);
        constexpr uint32_t idesc = idesc_f16_f32(128, MT);
        const uint64_t xdesc0 = smem_desc_sw128(sbase + P.x_off);
        int subc = 0;  // uses of this group's A ring
        bool ok = true;
        int sidx = 0;
        for (Segment sg = first_segment(); nunits > 0 && ok && sg.j0 < nunits; sg = next_segment(sg), ++sidx) {
            const int wt = min(kTileN, N - kTileN * sg.t);
            const bool valid = 32 * q < wt;
            const int buf = NBUF == 1 ? 0 : (sidx % NBUF);
            const uint32_t d_g = tmem + kAccBase + static_cast<uint32_t>((buf * kGroups + g) * MT);
            const uint32_t acc_parity = static_cast<uint32_t>((sidx / NBUF) - 1) & 1u;
            bool first = true;
            const int jstart = sg.j0 + ((g - (sg.j0 & 3)) & 3);
            for (int j = jstart; j < sg.j0 + sg.len; j += kGroups) {
                const int s = j % S;
                ok = sk_warp_wait(full_bar(s), static_cast<uint32_t>(j / S) & 1u, abort_flag, timeout_ns, status);
                if (!ok) break;
                // this lane's vectors and scales of sub-chunk `sub` (two 32-k vectors), read one
                // sub-chunk ahead of the dequantisation
                const uint32_t wst = sbase + P.w_off + s * P.w_stage + 16u * static_cast<uint32_t>(32 * q + lane);
                const uint32_t sst = sbase + P.s_off + s * P.s_stage + 2u * static_cast<uint32_t>(32 * q + lane);
                uint4 vn[2];
                uint32_t sn[2];
                auto load_sub = [&](int sub) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int kb = 2 * sub + h;
                        vn[h] = lds128(wst + 16u * static_cast<uint32_t>(kb * wt));
                        const int srow = KC >= G ? (32 * kb) / G : 0;
                        const uint32_t sb = lds16(sst + 2u * static_cast<uint32_t>(srow * wt));
                        sn[h] = sb | (sb << 16);
                    }
                };
                if (valid) load_sub(0);
#pragma unroll
                for (int sub = 0; sub < kSubs; ++sub) {
                    const int a = subc % SA;
                    const uint32_t aph = static_cast<uint32_t>(subc / SA) & 1u;
                    uint32_t regs[32];
                    if (valid) {
                        const uint4 v0 = vn[0], v1 = vn[1];
                        const uint32_t s0 = sn[0], s1 = sn[1];
                        if (sub + 1 < kSubs) load_sub(sub + 1);
                        dequant8(v0.x, s0, &regs[0]);
                        dequant8(v0.y, s0, &regs[4]);
                        dequant8(v0.z, s0, &regs[8]);
                        dequant8(v0.w, s0, &regs[12]);
                        dequant8(v1.x, s1, &regs[16]);
                        dequant8(v1.y, s1, &regs[20]);
                        dequant8(v1.z, s1, &regs[24]);
                        dequant8(v1.w, s1, &regs[28]);
                    }
                    if (subc >= SA) {  // the MMAs that read this A stage last time have completed
                        ok = sk_warp_wait(aempty_bar(g, a), aph ^ 1u, abort_flag, timeout_ns, status);
                        if (!ok) break;
                        tc_fence_after();
                    }
                    const uint32_t a_stage = a_ring + static_cast<uint32_t>(a * kSubCols);
                    if (valid) {
                        tmem_st<32>(a_stage + lane_base, regs);
                        tmem_wait_st();
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(afull_bar(g, a));
                    if (issuer_warp) {
                        int iok = 1;
                        if (lane == 0) {
                            iok = mbar_wait(afull_bar(g, a), aph, abort_flag, timeout_ns, status) ? 1 : 0;
                            if (iok && first && sub == 0 && sidx >= NBUF)
                                iok = mbar_wait(accfree_bar(buf), acc_parity, abort_flag, timeout_ns, status) ? 1 : 0;
                            if (iok) {
                                tc_fence_after();
                                const uint64_t xd = xdesc0 + static_cast<uint64_t>((s * P.x_stage) >> 4);
#pragma unroll
                                for (int i = 0; i < kSubK / 16; ++i) {
                                    const int ks = sub * (kSubK / 16) + i;  // k-step of 16 within the stage
                                    const uint32_t koff =
                                        static_cast<uint32_t>(((ks / 4) * MT * 128 + (ks % 4) * 32) >> 4);
                                    umma_f16_ts(d_g, a_stage + static_cast<uint32_t>(8 * i), xd + koff, idesc,
                                                !(first && sub == 0 && i == 0));
                                }
                                umma_commit(aempty_bar(g, a));
                                if (sub == kSubs - 1) umma_commit(empty_bar(s));
                            }
                        }
                        iok = __shfl_sync(0xffffffffu, iok, 0);
                        if (!iok) {
                            ok = false;
                            break;
                        }
                    }
                    ++subc;
                }
                if (!ok) break;
                first = false;
            }
            if (!ok) break;
            // End of the segment for this group: its accumulator is complete once its MMAs drain.
            // A group without units in this segment still waits for the buffer's release, so that
            // no group runs two segments ahead of the epilogue.
            if (issuer_warp) {
                int iok = 1;
                if (lane == 0) {
                    if (first && sidx >= NBUF)
                        iok = mbar_wait(accfree_bar(buf), acc_parity, abort_flag, timeout_ns, status) ? 1 : 0;
                    umma_commit(dfull_bar(g, buf));
                }
                iok = __shfl_sync(0xffffffffu, iok, 0);
                if (!iok) ok = false;
            }
        }
        if (issuer_warp && lane == 0) umma_commit(drain_bar);
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- epilogue warps
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        const int nl = 32 * q + lane;  // column within the tile
        griddep_wait();                // y and the workspace may be in use by an earlier kernel
        int sidx = 0;
        for (Segment sg = first_segment(); nunits > 0 && sg.j0 < nunits; sg = next_segment(sg), ++sidx) {
            const int wt = min(kTileN, N - kTileN * sg.t);
            const int n0 = kTileN * sg.t;
            const int buf = NBUF == 1 ? 0 : (sidx % NBUF);
            const uint32_t parity = static_cast<uint32_t>(sidx / NBUF) & 1u;
            bool ok = true;
#pragma unroll
            for (int g = 0; g < kGroups; ++g)
                if (ok) ok = warp_wait(dfull_bar(g, buf), parity, abort_flag, timeout_ns, status);
            if (!epi_sync_and(ok)) break;
            tc_fence_after();
            const bool whole = sg.cb == 0 && sg.len == C;
            // group g accumulated in this segment iff one of its units falls in [j0, j0 + len)
            bool has[kGroups];
#pragma unroll
            for (int g = 0; g < kGroups; ++g) has[g] = sg.len >= kGroups || ((g - (sg.j0 & 3)) & 3) < sg.len;
            const int slot = sg.t == static_cast<int>(u0 / C) ? 0 : 1;
            float* part = ws_part + static_cast<size_t>(2 * cta + slot) * MT * kTileN;
#pragma unroll 1
            for (int mc = 0; mc < MT; mc += 8) {
                float acc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
                for (int g = 0; g < kGroups; ++g) {  // fixed order: D_0 + D_1 + D_2 + D_3
                    if (!has[g]) continue;
                    uint32_t r[8];
                    tmem_ld<8>(tmem + kAccBase + static_cast<uint32_t>((buf * kGroups + g) * MT + mc) + lane_base, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i] += __uint_as_float(r[i]);
                }
                if (whole) {
                    if (nl < wt) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            if (mc + i < M)
                                y[static_cast<int64_t>(mc + i) * N + n0 + nl] = __half_as_ushort(__float2half_rn(acc[i]));
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) st_cg_f32(part + (mc + i) * kTileN + nl, acc[i]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(accfree_bar(buf));
            if (whole) continue;
            // ---- partial tile: count in, and the last of the tile's CTAs sums the partials
            __threadfence();
            named_sync(kEpiBarrier, 128);
            const long long tu0 = static_cast<long long>(sg.t) * C;
            const int bf = cta_of_unit(U, nb, tu0);
            const int bl = cta_of_unit(U, nb, tu0 + C - 1);
            if (warp == kEpiWarp0 && lane == 0) {
                const unsigned old = atom_add_acq_rel(ws_cnt + sg.t, 1u);
                const bool last = old == static_cast<unsigned>(bl - bf);
                if (last) ws_cnt[sg.t] = 0u;  // ready for the next call
                *last_flag = last ? 1 : 0;
            }
            named_sync(kEpiBarrier, 128);
            const bool last = *last_flag != 0;
            named_sync(kEpiBarrier, 128);  // every warp has read the flag before it is reused
            if (!last) continue;
            __threadfence();
            if (nl < wt) {
#pragma unroll 1
                for (int m = 0; m < M; ++m) {
                    float acc = 0.f;
                    for (int b = bf; b <= bl; ++b) {  // fixed order: CTA bf, bf + 1, ..., bl
                        const int sl = sg.t == static_cast<int>(range_begin(U, nb, b) / C) ? 0 : 1;
                        acc += ld_cg_f32(ws_part + static_cast<size_t>(2 * b + sl) * MT * kTileN + m * kTileN + nl);
                    }
                    y[static_cast<int64_t>(m) * N + n0 + nl] = __half_as_ushort(__float2half_rn(acc));
                }
            }
        }
    }

    __syncthreads();
    if (warp == kProducerWarp) {
        // every group's issuer commits drain_bar after its last MMA, also when it left early
        if (lane == 0 && nunits > 0) {
            int drain_abort = 0;
            mbar_wait(drain_bar, 0, &drain_abort, timeout_ns, status);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------------------------ host
template <int MT, int KC, int NBUF, int SA>
cudaError_t launch_sk_t(const CUtensorMap& tmap, const uint32_t* qweight_r, const uint16_t* scales_r, uint16_t* y,
                        float* ws_part, unsigned* ws_cnt, int M, int N, int K, int G, const StreamKConfig& c,
                        const LaunchCtx& ctx) {
    auto kern = tc_streamk_kernel<MT, KC, NBUF, SA>;
    // at least 120 KB: one CTA per SM, so that no CTA waits in tcgen05.alloc for another one's TMEM
    const size_t smem = std::max<size_t>(sk_plan(MT, KC, c.stages, SA, NBUF, G).total + 1024, 120 * 1024);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(c.ctas), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmap, reinterpret_cast<const uint4*>(qweight_r), scales_r, y, ws_part, ws_cnt,
                              M, N, K, G, c.stages, ctx.status, ctx.timeout_ns);
}

// (m_tile, k_chunk, accumulator buffers, TMEM A stages per group) of every instantiated kernel:
// 4 x SA x 32 + 4 x NBUF x MT = 512 TMEM columns.
#define W4A16_SK_COMBOS(X) \
    X(16, 128, 2, 3) X(16, 256, 2, 3) X(32, 128, 2, 2) X(32, 256, 2, 2) X(64, 128, 1, 2) X(64, 256, 1, 2)

}  // namespace

bool streamk_instantiated(int m_tile, int k_chunk) {
#define W4A16_SK_IS(MT_, KC_, NB_, SA_) \
    if (m_tile == MT_ && k_chunk == KC_) return true;
    W4A16_SK_COMBOS(W4A16_SK_IS)
#undef W4A16_SK_IS
    return false;
}

size_t streamk_smem_bytes(const StreamKConfig& c, int G) {
#define W4A16_SK_SM(MT_, KC_, NB_, SA_) \
    if (c.m_tile == MT_ && c.k_chunk == KC_) return sk_plan(MT_, KC_, c.stages, SA_, NB_, G).total + 1024;
    W4A16_SK_COMBOS(W4A16_SK_SM)
#undef W4A16_SK_SM
    return 0;
}

// Workspace layout: a fixed zone of one counter per 128-column tile (room for the widest supported
// N, so that calls of any shape and plan find their counters at the same place and no partial tile
// of any call ever lands on one), then the fp32 partial tiles [ctas][2][m_tile][128].
size_t streamk_workspace_bytes(const StreamKConfig& c, int N) {
    (void)N;
    return kStreamKCounterBytes + static_cast<size_t>(c.ctas) * 2 * c.m_tile * kTileN * 4;
}

bool streamk_config_valid(const StreamKConfig& c, int M, int N, int K, int G) {
    if (!streamk_instantiated(c.m_tile, c.k_chunk)) return false;
    if (M < 1 || M > c.m_tile) return false;
    if (K % c.k_chunk != 0) return false;
    if (c.k_chunk >= G ? c.k_chunk % G != 0 : G % c.k_chunk != 0) return false;
    if (c.stages < 2 || c.stages > 16) return false;
    const long long units = static_cast<long long>((N + kTileN - 1) / kTileN) * (K / c.k_chunk);
    if (c.ctas < 1 || c.ctas > 65535 || c.ctas > units) return false;
    return streamk_smem_bytes(c, G) <= 232448;
}

cudaError_t launch_streamk(const uint16_t* x, const uint32_t* qweight_r, const uint16_t* scales_r, uint16_t* y,
                           void* workspace, int M, int N, int K, int G, const StreamKConfig& c, const LaunchCtx& ctx) {
    CUtensorMap tmap;
    bool three_d = false;
    if (!encode_x_map(&tmap, x, M, K, c.m_tile, c.k_chunk, &three_d) || !three_d) return cudaErrorInvalidValue;
    unsigned* ws_cnt = static_cast<unsigned*>(workspace);
    float* ws_part = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + kStreamKCounterBytes);
#define W4A16_SK_CASE(MT_, KC_, NB_, SA_)                                                                      \
    if (c.m_tile == MT_ && c.k_chunk == KC_)                                                                   \
        return launch_sk_t<MT_, KC_, NB_, SA_>(tmap, qweight_r, scales_r, y, ws_part, ws_cnt, M, N, K, G, c, ctx);
    W4A16_SK_COMBOS(W4A16_SK_CASE)
#undef W4A16_SK_CASE
    return cudaErrorInvalidValue;
}

}  // namespace w4a16
