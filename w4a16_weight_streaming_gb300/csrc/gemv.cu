// CUDA-core split-K GEMV for the smallest decode batches (M <= 8).
//
// One CTA = 4 warps on one 32-column slice of W and one K-slice. Lane l owns one column and
// streams its 16-byte vectors (32 k each, 512 contiguous bytes per warp per 32-k block in the
// 128-column-tile layout); the 4 warps interleave over the K-slice's 32-k blocks
// and combine through shared memory. The K-slices of one column tile form a thread-block
// cluster and are summed through distributed shared memory, in a fixed rank order, by the CTA
// that owns each output element. Activations of the K-slice are staged once in shared memory as
// fp16 and read as broadcasts; products are fp16 x fp16 rounded once into fp32 accumulators.
//
// Per weight: ~1.6 instructions of exact dequantisation (common.cuh) + M fused multiply-adds.
#include "common.cuh"
#include "internal.h"

namespace w4a16 {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint16_t ldg_u16(const uint16_t* p) {
    uint16_t v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

struct GemvSlice {
    int kb_begin, kb_end, klen;  // 32-k blocks [kb_begin, kb_end), klen = K elements in slice
};

__device__ __forceinline__ GemvSlice slice_of(int rank, int split, int KB) {
    GemvSlice s;
    s.kb_begin = static_cast<int>((static_cast<int64_t>(rank) * KB) / split);
    s.kb_end = static_cast<int>((static_cast<int64_t>(rank + 1) * KB) / split);
    s.klen = (s.kb_end - s.kb_begin) * 32;
    return s;
}

// acc[c][m][h]: chain c (word parity), row m, half h (even / odd k of a pair). sbits: the scale of
// the block's 32 k (int4), or the scales of its two 16-k halves (NVFP4: lo16 = k 0..15).
// NVFP4 codes of one word as fp16 pairs (k offsets 2i, 2i + 1 in out[i]): exact, unscaled.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t word, uint32_t out[4]) {
    asm("{\n\t.reg .b8 a0, a1, a2, a3;\n\t"
        "mov.b32 {a0, a1, a2, a3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, a0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, a1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, a2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, a3;\n\t}"
        : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
        : "r"(word));
}

// NVFP4: e2m1 * s is exact in fp16, so the block scale can leave the inner product: each 16-k half
// sums x * e2m1 in fp32 and is added to acc scaled once by its scale (one FFMA per half and row
// instead of four fp16 multiplies per 8 weights). The same products, rounded in another order.
template <int MR>
__device__ __forceinline__ void gemv_block_fp4(const uint4 v, uint32_t sbits, const __half* xs_blk, int klen,
                                               float (&acc)[2][MR][2]) {
    const float sh[2] = {__half2float(__ushort_as_half(static_cast<uint16_t>(sbits & 0xFFFFu))),
                         __half2float(__ushort_as_half(static_cast<uint16_t>(sbits >> 16)))};
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float blk[MR][2];
#pragma unroll
        for (int m = 0; m < MR; ++m) blk[m][0] = blk[m][1] = 0.f;
#pragma unroll
        for (int i = 2 * h; i < 2 * h + 2; ++i) {
            uint32_t e2[4];
            e2m1x8_to_f16x2(words[i], e2);
#pragma unroll
            for (int m = 0; m < MR; ++m) {
                const uint4 xv = *reinterpret_cast<const uint4*>(xs_blk + m * klen + 8 * i);
                fma2_mixed(blk[m][0], blk[m][1], e2[0], xv.x);
                fma2_mixed(blk[m][0], blk[m][1], e2[1], xv.y);
                fma2_mixed(blk[m][0], blk[m][1], e2[2], xv.z);
                fma2_mixed(blk[m][0], blk[m][1], e2[3], xv.w);
            }
        }
#pragma unroll
        for (int m = 0; m < MR; ++m) {
            acc[h][m][0] = fmaf(sh[h], blk[m][0], acc[h][m][0]);
            acc[h][m][1] = fmaf(sh[h], blk[m][1], acc[h][m][1]);
        }
    }
}

template <int MR, bool FP4>
__device__ __forceinline__ void gemv_block(const uint4 v, uint32_t sbits, const __half* xs_blk, int klen,
                                           float (&acc)[2][MR][2]) {
    if (FP4) {
        gemv_block_fp4<MR>(v, sbits, xs_blk, klen, acc);
        return;
    }
    const uint32_t slo = sbits & 0xFFFFu, shi = FP4 ? (sbits >> 16) : slo;
    const uint32_t s2a = slo | (slo << 16), s2b = shi | (shi << 16);
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t w2[4];
        if (FP4)
            dequant8_nvfp4(words[i], i < 2 ? s2a : s2b, w2);
        else
            dequant8(words[i], s2a, w2);
#pragma unroll
        for (int m = 0; m < MR; ++m) {
            const uint4 xv = *reinterpret_cast<const uint4*>(xs_blk + m * klen + 8 * i);
            fma2_mixed(acc[i & 1][m][0], acc[i & 1][m][1], w2[0], xv.x);
            fma2_mixed(acc[i & 1][m][0], acc[i & 1][m][1], w2[1], xv.y);
            fma2_mixed(acc[i & 1][m][0], acc[i & 1][m][1], w2[2], xv.z);
            fma2_mixed(acc[i & 1][m][0], acc[i & 1][m][1], w2[3], xv.w);
        }
    }
}

// U: 32-k blocks in flight per warp: 4, or 8 at one and two rows when the grid fits in one wave of
// the larger-register kernel (fewer load round trips for short K-slices).
template <int MR, bool FP4, int U>
__global__ void __launch_bounds__(kThreads) gemv_kernel(const uint16_t* __restrict__ x,
                                                        const uint4* __restrict__ wr,
                                                        const uint16_t* __restrict__ sr, uint16_t* __restrict__ y,
                                                        int N, int K, int G, int split, float tensor_scale,
                                                        unsigned* status) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int KB = K / 32;
    const int NG = K / G;
    // grid.x = slices x split, one cluster of `split` consecutive CTAs per 32-column slice
    const int rank = static_cast<int>(blockIdx.x) % split;
    const int t = static_cast<int>(blockIdx.x) / split;  // 32-column slice: columns 32t .. 32t + 31
    const int tile = t / 4;             // 128-column tile of the streaming layout
    const int wt = min(128, N - 128 * tile);
    const int cofs = 32 * (t % 4);      // slice offset inside the tile
    const GemvSlice sl = slice_of(rank, split, KB);
    const int klen_max = ((KB + split - 1) / split) * 32;

    __half* xs = reinterpret_cast<__half*>(smem);
    float* red = reinterpret_cast<float*>(smem + static_cast<size_t>(MR) * klen_max * 2);  // [kWarps][MR][32]
    float* part = red + kWarps * MR * 32;                                                  // [MR][32]

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint4* wcol = wr + static_cast<int64_t>(tile) * 128 * KB + cofs + lane;      // + kb * wt
    const uint16_t* scol = sr + static_cast<int64_t>(tile) * 128 * NG + cofs + lane;  // + g * wt

    // scale row of 32-k block b: b / (G / 32), a shift when G / 32 is a power of two (int4; NVFP4
    // has two scale rows per block, 2b and 2b + 1)
    const int gb = FP4 ? 1 : G / 32;
    const int gshift = (gb & (gb - 1)) == 0 ? __ffs(gb) - 1 : -1;
    auto group_of = [&](int b) { return gshift >= 0 ? (b >> gshift) : b / gb; };

    // index checks of the debug-bounds build: vector and scale indices within the whole buffers
    const int64_t w_total = static_cast<int64_t>(N) * KB, s_total = static_cast<int64_t>(NG) * N;
    const int64_t w_base = wcol - wr, s_base = scol - sr;
    auto load_w = [&](int b) {
        return in_bounds(w_base + static_cast<int64_t>(b) * wt < w_total, status)
                   ? ldg_stream(wcol + static_cast<int64_t>(b) * wt)
                   : make_uint4(0u, 0u, 0u, 0u);
    };
    auto load_s = [&](int b) -> uint32_t {
        if (FP4) {
            const int64_t r = 2 * static_cast<int64_t>(b);
            if (!in_bounds(s_base + (r + 1) * wt < s_total, status)) return 0u;
            return static_cast<uint32_t>(ldg_u16(scol + r * wt)) |
                   (static_cast<uint32_t>(ldg_u16(scol + (r + 1) * wt)) << 16);
        }
        return in_bounds(s_base + static_cast<int64_t>(group_of(b)) * wt < s_total, status)
                   ? static_cast<uint32_t>(ldg_u16(scol + static_cast<int64_t>(group_of(b)) * wt))
                   : 0u;
    };

    // Programmatic dependent launch: the warp's first batch of weights and scales is loaded while the
    // previous grid on the stream finishes; x (possibly its output) is read only after it completed.
    int kb = sl.kb_begin + warp;
    const bool first = kb + kWarps * (U - 1) < sl.kb_end;
    uint4 v0[U];
    uint32_t s0[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        v0[u] = first ? load_w(kb + kWarps * u) : make_uint4(0u, 0u, 0u, 0u);
        s0[u] = first ? load_s(kb + kWarps * u) : 0u;
    }
    griddep_wait();

    // Stage x[0:MR][slice] as fp16 (16-byte copies).
    {
        const int vec_per_row = sl.klen / 8;
        for (int i = threadIdx.x; i < MR * vec_per_row; i += kThreads) {
            const int m = i / vec_per_row;
            const int c = i % vec_per_row;
            const int64_t xi = static_cast<int64_t>(m) * K + sl.kb_begin * 32 + 8 * c;
            const uint4 v = in_bounds(xi + 8 <= static_cast<int64_t>(MR) * K, status)
                                ? *reinterpret_cast<const uint4*>(x + xi)
                                : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(xs + m * sl.klen + 8 * c) = v;
        }
    }
    __syncthreads();

    float acc[2][MR][2];
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int m = 0; m < MR; ++m) acc[c][m][0] = acc[c][m][1] = 0.f;

    if (first) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = kb + kWarps * u;
            gemv_block<MR, FP4>(v0[u], s0[u], xs + (b - sl.kb_begin) * 32, sl.klen, acc);
        }
        kb += kWarps * U;
    }
    for (; kb + kWarps * (U - 1) < sl.kb_end; kb += kWarps * U) {
        uint4 v[U];
        uint32_t sb[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = kb + kWarps * u;
            v[u] = load_w(b);
            sb[u] = load_s(b);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = kb + kWarps * u;
            gemv_block<MR, FP4>(v[u], sb[u], xs + (b - sl.kb_begin) * 32, sl.klen, acc);
        }
    }
    if (kb < sl.kb_end) {  // the last (< U) blocks: their loads issued together as well
        uint4 v[U];
        uint32_t sb[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = kb + kWarps * u;
            v[u] = b < sl.kb_end ? load_w(b) : make_uint4(0u, 0u, 0u, 0u);
            sb[u] = b < sl.kb_end ? load_s(b) : 0u;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = kb + kWarps * u;
            if (b < sl.kb_end) gemv_block<MR, FP4>(v[u], sb[u], xs + (b - sl.kb_begin) * 32, sl.klen, acc);
        }
    }

    griddep_launch_dependents();
#pragma unroll
    for (int m = 0; m < MR; ++m)
        red[(warp * MR + m) * 32 + lane] = (acc[0][m][0] + acc[0][m][1]) + (acc[1][m][0] + acc[1][m][1]);
    __syncthreads();

    // element e = (m, lane) = (e / 32, e % 32); MR * 32 may exceed the CTA's 128 threads
    if (split == 1) {
        for (int e = threadIdx.x; e < MR * 32; e += kThreads) {
            const int m = e / 32, l = e % 32;
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) s += red[(w * MR + m) * 32 + l];
            const int64_t yi = static_cast<int64_t>(m) * N + 32 * t + l;
            if (in_bounds(yi < static_cast<int64_t>(MR) * N, status)) y[yi] = __half_as_ushort(__float2half_rn(s * tensor_scale));
        }
        return;
    }
    for (int e = threadIdx.x; e < MR * 32; e += kThreads) {
        const int m = e / 32, l = e % 32;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += red[(w * MR + m) * 32 + l];
        part[e] = s;
    }
    cluster_sync_all();
    for (int e = threadIdx.x; e < MR * 32; e += kThreads) {
        if ((e % split) != rank) continue;
        const uint32_t local = smem_u32(part + e);
        const float s = cluster_sum_f1(local, split);
        const int m = e / 32, l = e % 32;
        const int64_t yi = static_cast<int64_t>(m) * N + 32 * t + l;
        if (in_bounds(yi < static_cast<int64_t>(MR) * N, status)) y[yi] = __half_as_ushort(__float2half_rn(s * tensor_scale));
    }
    cluster_sync_all();
}

template <int MR>
auto gemv_kernel_for(bool fp4, int unroll) {
    if constexpr (MR <= 2) {
        if (unroll == 8) return fp4 ? gemv_kernel<MR, true, 8> : gemv_kernel<MR, false, 8>;
    }
    return fp4 ? gemv_kernel<MR, true, 4> : gemv_kernel<MR, false, 4>;
}

template <int MR>
cudaError_t launch_gemv_m(const uint16_t* x, const uint32_t* qweight_r, const uint16_t* scales_r, uint16_t* y,
                          int N, int K, int G, int split, int unroll, size_t smem, const LaunchCtx& ctx) {
    const cudaStream_t s = ctx.stream;
    unsigned* status = ctx.status;
    auto kern = gemv_kernel_for<MR>(ctx.nvfp4 != 0, unroll);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (split > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(split) * static_cast<unsigned>(N / 32), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (split > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = split;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, x, reinterpret_cast<const uint4*>(qweight_r), scales_r, y, N, K, G, split,
                              ctx.tensor_scale, status);
}

}  // namespace

size_t gemv_smem_bytes(int M, int N, int K, int split) {
    (void)N;
    const int KB = K / 32;
    const size_t klen_max = static_cast<size_t>((KB + split - 1) / split) * 32;
    return static_cast<size_t>(M) * klen_max * 2 + static_cast<size_t>(kWarps + 1) * M * 32 * 4;
}

// CTAs of the M-row GEMV with `unroll` blocks in flight that the device keeps resident at once
// (both weight formats; the smaller of the two), 0 if the query fails.
int gemv_resident_ctas(int M, int unroll, size_t smem, int sm_count) {
    if (M != 1 && M != 2) return 0;
    int best = -1;
    for (int f = 0; f < 2; ++f) {
        const void* kern = M == 1 ? reinterpret_cast<const void*>(gemv_kernel_for<1>(f != 0, unroll))
                                  : reinterpret_cast<const void*>(gemv_kernel_for<2>(f != 0, unroll));
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
            cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        int blocks = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kern, kThreads, smem) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        best = best < 0 || blocks < best ? blocks : best;
    }
    return best < 0 ? 0 : best * sm_count;
}

cudaError_t launch_gemv(const uint16_t* x, const uint32_t* qweight_r, const uint16_t* scales_r, uint16_t* y, int M,
                        int N, int K, int G, int split, int unroll, const LaunchCtx& ctx) {
    const size_t smem = gemv_smem_bytes(M, N, K, split);
    switch (M) {
        case 1: return launch_gemv_m<1>(x, qweight_r, scales_r, y, N, K, G, split, unroll, smem, ctx);
        case 2: return launch_gemv_m<2>(x, qweight_r, scales_r, y, N, K, G, split, unroll, smem, ctx);
        case 3: return launch_gemv_m<3>(x, qweight_r, scales_r, y, N, K, G, split, unroll, smem, ctx);
        case 4: return launch_gemv_m<4>(x, qweight_r, scales_r, y, N, K, G, split, unroll, smem, ctx);
        case 5: return launch_gemv_m<5>(x, qweight_r, scales_r, y, N, K, G, split, unroll, smem, ctx);
        case 6: return launch_gemv_m<6>(x, qweight_r, scales_r, y, N, K, G, split, unroll, smem, ctx);
        case 7: return launch_gemv_m<7>(x, qweight_r, scales_r, y, N, K, G, split, unroll, smem, ctx);
        case 8: return launch_gemv_m<8>(x, qweight_r, scales_r, y, N, K, G, split, unroll, smem, ctx);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace w4a16
