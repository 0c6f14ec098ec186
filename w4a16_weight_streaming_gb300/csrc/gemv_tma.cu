// TMA-fed CUDA-core GEMV for the smallest decode batches (M <= 4).
//
// Measured on GB300: a GEMV whose warps load a batch of weights and then compute on it runs in
// about (memory time + compute time) — the dequantisation and fma work of a warp does not overlap
// its own loads, and there are too few warps per SM to hide it. Here the loads leave the warps
// entirely: one producer thread streams the column tile's rows through a shared-memory ring with
// 1-D TMA bulk copies (one contiguous copy per stage in the 128-column-tile layout), and eight
// consumer warps dequantise and accumulate from shared memory as the stages land, each at its own
// pace (a per-stage mbarrier, no lockstep). Memory streaming and arithmetic then overlap, and the
// kernel runs at about the larger of the two.
//
// CTA = (128-column tile, K-slice); consumer warp (q, h) = (w % 4, w / 4) owns columns 32q..32q+31
// (lane = column) and half h of every stage's rows. x of the K-slice is staged in shared memory
// as fp16; products are fp16 x fp16 rounded once into fp32 accumulators. The K-slices of a tile
// form a thread-block cluster and are summed through distributed shared memory in rank order.
// Every mbarrier wait is bounded; consumers never leave their loop early (they skip work after a
// failed wait), so the producer never waits on a warp that has gone.
#include "common.cuh"
#include "internal.h"

namespace w4a16 {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kConsBarId = 1;  // named barrier over the consumer warps

struct GtSmem {
    uint32_t x_off;            // x slice: MR x klen_max fp16
    uint32_t w_off, w_stage;   // weight ring: stages x (rows x 128 x 16 B)
    uint32_t s_off, s_stage;   // scale ring: stages x (groups x 128 x 2 B)
    uint32_t red_off;          // consumer partial sums: kConsumerWarps x MR x 32 fp32, then MR x 128 fp32
    uint32_t bar_off;          // full[stages], empty[stages]
    uint32_t misc_off;         // abort flag
    uint32_t total;
};

__host__ __device__ inline int gt_rows_per_stage(int KC) { return KC / 32; }
// scale rows one stage can touch: KC consecutive k starting anywhere inside a group span at most
// (KC - 1) / G + 2 groups (G need not divide KC, e.g. G = 96)
__host__ __device__ inline int gt_groups_per_stage(int KC, int G) { return (KC - 1) / G + 2; }

__host__ __device__ inline GtSmem gt_plan(int MR, int KC, int G, int stages, int klen_max) {
    GtSmem p;
    p.x_off = 0;
    p.w_stage = static_cast<uint32_t>(gt_rows_per_stage(KC) * 128 * 16);
    p.w_off = (static_cast<uint32_t>(MR * klen_max * 2) + 127u) & ~127u;
    p.s_stage = static_cast<uint32_t>(gt_groups_per_stage(KC, G) * 128 * 2);
    p.s_off = p.w_off + static_cast<uint32_t>(stages) * p.w_stage;
    p.red_off = (p.s_off + static_cast<uint32_t>(stages) * p.s_stage + 15u) & ~15u;
    const uint32_t red_bytes = static_cast<uint32_t>((kConsumerWarps * MR * 32 + MR * 128) * 4);
    p.bar_off = (p.red_off + red_bytes + 7u) & ~7u;
    p.misc_off = p.bar_off + static_cast<uint32_t>(2 * stages) * 8u;
    p.total = p.misc_off + 16u;
    return p;
}

template <int MR, int KC>
__global__ void __launch_bounds__(kThreads) gemv_tma_kernel(const uint16_t* __restrict__ x,
                                                            const uint4* __restrict__ wr,
                                                            const uint16_t* __restrict__ sr,
                                                            uint16_t* __restrict__ y, int N, int K, int G,
                                                            int stages, unsigned* status, uint64_t timeout_ns) {
    constexpr int kR = KC / 32;  // 32-k rows per stage
    constexpr int kHalf = kR / 2;
    extern __shared__ __align__(128) unsigned char smem[];
    const int KB = K / 32;
    const int NG = K / G;
    const int split = gridDim.x;
    const int rank = blockIdx.x;
    const int tile = blockIdx.y;
    const int wt = min(128, N - 128 * tile);
    // K-slice of this CTA, in stages of kR rows (the last stage of the matrix may be shorter)
    const int C = (KB + kR - 1) / kR;
    const int c_begin = static_cast<int>((static_cast<int64_t>(rank) * C) / split);
    const int c_end = static_cast<int>((static_cast<int64_t>(rank + 1) * C) / split);
    const int kb_begin = c_begin * kR;
    const int kb_end = min(KB, c_end * kR);
    const int klen = (kb_end - kb_begin) * 32;
    const int klen_max = ((C + split - 1) / split) * kR * 32;
    const GtSmem P = gt_plan(MR, KC, G, stages, klen_max);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + P.bar_off;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (stages + s); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P.misc_off);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int gb = G / 32;  // rows per scale group

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kConsumerWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kProducerWarp) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            const uint4* w_tile = wr + static_cast<int64_t>(tile) * 128 * KB;
            const uint16_t* s_tile = sr + static_cast<int64_t>(tile) * 128 * NG;
            int s = 0;
            uint32_t ph = 0;
            int issued = 0;
            for (int c = c_begin; c < c_end; ++c, ++issued) {
                if (issued >= stages && !mbar_spin(empty_bar(s), ph ^ 1u, abort_flag, timeout_ns, status)) break;
                const int b0 = c * kR, b1 = min(KB, b0 + kR);
                const int g0 = b0 / gb, g1 = (b1 - 1) / gb;
                const uint32_t wbytes = static_cast<uint32_t>((b1 - b0) * wt * 16);
                const uint32_t sbytes = static_cast<uint32_t>((g1 - g0 + 1) * wt * 2);
                const uint32_t fb = full_bar(s);
                mbar_arrive_expect_tx(fb, wbytes + sbytes);
                bulk_g2s(sbase + P.w_off + s * P.w_stage, w_tile + static_cast<int64_t>(b0) * wt, wbytes, fb, pol);
                bulk_g2s(sbase + P.s_off + s * P.s_stage, s_tile + static_cast<int64_t>(g0) * wt, sbytes, fb, pol);
                if (++s == stages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            // copies still in flight land before the CTA may exit
            int dummy_abort = 0;
            for (int i = issued > stages ? issued - stages : 0; i < issued; ++i)
                mbar_wait(full_bar(i % stages), static_cast<uint32_t>((i / stages) & 1), &dummy_abort, timeout_ns,
                          status);
        }
        __syncwarp();
    } else {
        // ---- stage x[0:MR][slice] (consumers only), fp16, 16-byte copies
        __half* xs = reinterpret_cast<__half*>(smem + P.x_off);
        {
            const int vec_per_row = klen / 8;
            for (int i = threadIdx.x; i < MR * vec_per_row; i += 32 * kConsumerWarps) {
                const int m = i / vec_per_row;
                const int c = i % vec_per_row;
                const uint4 xv =
                    *reinterpret_cast<const uint4*>(x + static_cast<int64_t>(m) * K + kb_begin * 32 + 8 * c);
                *reinterpret_cast<uint4*>(xs + m * klen + 8 * c) = xv;
            }
        }
        named_sync(kConsBarId, 32 * kConsumerWarps);

        const int q = warp & 3;   // column quadrant
        const int h = warp >> 2;  // half of each stage's rows
        const bool valid = 32 * q < wt;
        const uint32_t xs_s = sbase + P.x_off;
        float acc[2][MR][2];
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int m = 0; m < MR; ++m) acc[c][m][0] = acc[c][m][1] = 0.f;

        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int c = c_begin; c < c_end; ++c) {
            if (ok) ok = warp_spin(full_bar(s), ph, abort_flag, timeout_ns, status);
            const int b0 = c * kR, b1 = min(KB, b0 + kR);
            const int g0 = b0 / gb;
            if (ok && valid) {
                const uint32_t wst = sbase + P.w_off + s * P.w_stage + 16u * static_cast<uint32_t>(32 * q + lane);
                const uint32_t sst = sbase + P.s_off + s * P.s_stage + 2u * static_cast<uint32_t>(32 * q + lane);
                uint4 v[kHalf];
                uint32_t sb[kHalf];
#pragma unroll
                for (int u = 0; u < kHalf; ++u) {
                    const int b = b0 + h * kHalf + u;
                    if (b < b1) {
                        v[u] = lds128(wst + 16u * static_cast<uint32_t>((b - b0) * wt));
                        sb[u] = lds16(sst + 2u * static_cast<uint32_t>((b / gb - g0) * wt));
                    }
                }
#pragma unroll
                for (int u = 0; u < kHalf; ++u) {
                    const int b = b0 + h * kHalf + u;
                    if (b < b1) {
                        const uint32_t s2 = sb[u] | (sb[u] << 16);
                        const uint32_t words[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                        const uint32_t xblk = xs_s + 64u * static_cast<uint32_t>(b - kb_begin);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            uint32_t w2[4];
                            dequant8(words[i], s2, w2);
#pragma unroll
                            for (int m = 0; m < MR; ++m) {
                                const uint4 xv = lds128(xblk + 2u * static_cast<uint32_t>(m * klen + 8 * i));
                                fma2_mixed(acc[i & 1][m][0], acc[i & 1][m][1], w2[0], xv.x);
                                fma2_mixed(acc[i & 1][m][0], acc[i & 1][m][1], w2[1], xv.y);
                                fma2_mixed(acc[i & 1][m][0], acc[i & 1][m][1], w2[2], xv.z);
                                fma2_mixed(acc[i & 1][m][0], acc[i & 1][m][1], w2[3], xv.w);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(s));  // this warp's reads of stage s are consumed
            if (++s == stages) {
                s = 0;
                ph ^= 1u;
            }
        }

        float* red = reinterpret_cast<float*>(smem + P.red_off);  // [warp][MR][32]
        float* part = red + kConsumerWarps * MR * 32;              // [MR][128]
#pragma unroll
        for (int m = 0; m < MR; ++m)
            red[(warp * MR + m) * 32 + lane] = (acc[0][m][0] + acc[0][m][1]) + (acc[1][m][0] + acc[1][m][1]);
        named_sync(kConsBarId, 32 * kConsumerWarps);
        // element e = (m, c), c = 32 * quadrant + lane; the two row halves in order
        for (int e = threadIdx.x; e < MR * 128; e += 32 * kConsumerWarps) {
            const int m = e / 128, cc = e % 128;
            const int qq = cc / 32, l = cc % 32;
            part[e] = red[(qq * MR + m) * 32 + l] + red[((4 + qq) * MR + m) * 32 + l];
        }
        named_sync(kConsBarId, 32 * kConsumerWarps);
        if (split == 1) {
            for (int e = threadIdx.x; e < MR * 128; e += 32 * kConsumerWarps) {
                const int m = e / 128, cc = e % 128;
                if (cc < wt) y[static_cast<int64_t>(m) * N + 128 * tile + cc] = __half_as_ushort(__float2half_rn(part[e]));
            }
        }
    }

    if (split > 1) {
        __syncwarp();
        cluster_sync_all();  // every rank's partial tile is in its shared memory
        if (warp < kConsumerWarps) {
            const uint32_t part_s = sbase + P.red_off + static_cast<uint32_t>(kConsumerWarps * MR * 32 * 4);
            for (int e = threadIdx.x; e < MR * 128; e += 32 * kConsumerWarps) {
                if ((e % split) != rank) continue;
                const int m = e / 128, cc = e % 128;
                if (cc >= wt) continue;
                float acc = 0.f;
                for (int p = 0; p < split; ++p) acc += ld_dsmem_f1(map_peer(part_s + 4u * e, p));  // rank order
                y[static_cast<int64_t>(m) * N + 128 * tile + cc] = __half_as_ushort(__float2half_rn(acc));
            }
        }
        __syncwarp();
        cluster_sync_all();  // no CTA leaves while a peer may still read its partial tile
    }
}

int gt_klen_max(int K, int KC, int split) {
    const int KB = K / 32;
    const int R = gt_rows_per_stage(KC);
    const int C = (KB + R - 1) / R;
    return ((C + split - 1) / split) * R * 32;
}

template <int MR, int KC>
cudaError_t prepare_gt(size_t smem, int split) {
    auto kern = gemv_tma_kernel<MR, KC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (split > 8) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

template <int MR, int KC>
cudaLaunchConfig_t gt_config(int split, int N, size_t smem, cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(split, (N + 127) / 128, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = split > 1 ? 1 : 0;
    return cfg;
}

template <int MR, int KC>
cudaError_t launch_gt_t(const uint16_t* x, const uint32_t* qweight_r, const uint16_t* scales_r, uint16_t* y, int N,
                        int K, int G, int split, int stages, const LaunchCtx& ctx) {
    const size_t smem = gt_plan(MR, KC, G, stages, gt_klen_max(K, KC, split)).total;
    cudaError_t e = prepare_gt<MR, KC>(smem, split);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = gt_config<MR, KC>(split, N, smem, ctx.stream, attr);
    return cudaLaunchKernelEx(&cfg, gemv_tma_kernel<MR, KC>, x, reinterpret_cast<const uint4*>(qweight_r), scales_r, y,
                              N, K, G, stages, ctx.status, ctx.timeout_ns);
}

template <int MR, int KC>
int gt_resident_ctas_t(int N, int K, int G, int split, int stages) {
    const size_t smem = gt_plan(MR, KC, G, stages, gt_klen_max(K, KC, split)).total;
    if (prepare_gt<MR, KC>(smem, split) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = gt_config<MR, KC>(split, 128, smem, nullptr, attr);
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, gemv_tma_kernel<MR, KC>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return clusters * split;
}

}  // namespace

size_t gemv_tma_smem_bytes(int M, int K, int G, int KC, int split, int stages) {
    return gt_plan(M, KC, G, stages, gt_klen_max(K, KC, split)).total;
}

#define W4A16_GT_DISPATCH(CALL)                       \
    switch (M * 1000 + KC) {                          \
        case 1128: return CALL(1, 128);               \
        case 1256: return CALL(1, 256);               \
        case 2128: return CALL(2, 128);               \
        case 2256: return CALL(2, 256);               \
        case 3128: return CALL(3, 128);               \
        case 3256: return CALL(3, 256);               \
        case 4128: return CALL(4, 128);               \
        case 4256: return CALL(4, 256);               \
        default: break;                               \
    }

int gemv_tma_resident_ctas(int M, int N, int K, int G, int KC, int split, int stages) {
#define W4A16_GT_RES(MR_, KC_) gt_resident_ctas_t<MR_, KC_>(N, K, G, split, stages)
    W4A16_GT_DISPATCH(W4A16_GT_RES)
#undef W4A16_GT_RES
    return 0;
}

cudaError_t launch_gemv_tma(const uint16_t* x, const uint32_t* qweight_r, const uint16_t* scales_r, uint16_t* y,
                            int M, int N, int K, int G, int KC, int split, int stages, const LaunchCtx& ctx) {
#define W4A16_GT_LAUNCH(MR_, KC_) launch_gt_t<MR_, KC_>(x, qweight_r, scales_r, y, N, K, G, split, stages, ctx)
    W4A16_GT_DISPATCH(W4A16_GT_LAUNCH)
#undef W4A16_GT_LAUNCH
    return cudaErrorInvalidValue;
}

#undef W4A16_GT_DISPATCH

}  // namespace w4a16
