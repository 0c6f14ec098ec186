// W4A8: int8 activations with the int4 weights of the W4A16 device layout.
//
// "Qwen3.8-27B at 764, 1,035 and 1,623 tok/s" (ai.satyajit.si), section "Where the line bends",
// runs the MLP GEMMs with int8 activations. Reading taken (per-token symmetric int8):
//   sx[m] = fl32(max_k |x[m][k]| / 127), xq[m][k] = rne(fl32(x[m][k] / sx[m])) in [-127, 127]
//   (all 0 for a zero row), y[m][n] = sx[m] * sum_g s[g][n] * sum_{k in g} (q[k][n] - 8) * xq[m][k].
//
// quantize_x_int8_kernel: one CTA per activation row. The scale is an IEEE binary32 division; each
//   code is rne(fl32(x / sx)), reached through the reciprocal product with the IEEE division
//   wherever the product lies near a half-integer (quantize1 gives the argument), so the integers
//   are exactly those of the binary32 steps above. It writes xq as int8 and, optionally, the same
//   integers as fp16 (exact, |xq| <= 127) for the tensor-core tiles.
// gemv_w4a8_kernel (M <= 8): a CUDA-core split-K GEMV with integer arithmetic (one CTA per
//   128-column tile and K-slice, one warp per 32-column slice of it). The
//   unsigned nibbles of a weight word are split into two words of four bytes (one AND, one shift
//   and AND) and multiplied with the int8 activations by dp4a (four products and their sum per
//   instruction); the offset 8 is folded in as -8 * sum(xq) of the 32-k block, staged with x. Per
//   32-k block the exact int32 sum is scaled by the block's group scale into an fp32 accumulator;
//   y = fp16(sx * sum). Per weight at M = 1 the inner loop spends ~0.4 instructions on unpacking
//   and a quarter of a dp4a, against ~1.6 of dequantisation and one FMA on the fp16 path.
// The tensor-core tiles (M > 8) are the W4A16 tile kernel fed with the fp16 copy of xq (the MMA
// of fp16 operands is exact on integers) and a per-row output scale sx: sm_103a has no int8 MMA
// (tcgen05 kind::i8 is not available on this target).
#include "common.cuh"
#include "internal.h"

namespace w4a16 {
namespace {

// ------------------------------------------------------------------------------------ quantisation
constexpr int kQThreads = 1024;
constexpr int kQCache = 4;  // 16-byte vectors of the row kept in registers per thread (K <= 32768)

__device__ __forceinline__ float absmax8(const uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
    return m;
}

// One activation to its int8 code: rne(fl32(f / s)), clamped; 0 for a zero row (amax = 0). r is
// fl32(1 / s). The quotient estimate qa = fl32(f * r) is within 2^-23 |f / s| <= 1.6e-5 of f / s
// (two roundings of 2^-24 each), and fl32(f / s) within 2^-24 |f / s| <= 7.6e-6 of it (|f / s| <=
// 127 + 2^-16), so the two differ by less than 2.3e-5: wherever qa is at least 1e-4 away from a
// half-integer, both round to the same integer (and fl32(f / s) is not a tie). Only the remaining
// cases take the exact IEEE division.
__device__ __forceinline__ int quantize1(float f, float s, float r, bool nonzero) {
    if (!nonzero) return 0;
    const float qa = f * r;
    const float frac = qa - floorf(qa);
    const float q = fabsf(frac - 0.5f) < 1e-4f ? __fdiv_rn(f, s) : qa;
    return min(127, max(-127, __float2int_rn(q)));
}

__global__ void __launch_bounds__(kQThreads) quantize_x_int8_kernel(const uint4* __restrict__ x, uint2* __restrict__ xq,
                                                                    uint4* __restrict__ xh, float* __restrict__ sx,
                                                                    int M, int K, unsigned* status) {
    // the GEMM that follows may start streaming its weights now; it waits for xq before reading it
    griddep_launch_dependents();
    griddep_wait();  // x may be the previous kernel's output
    __shared__ float wmax[kQThreads / 32];
    const int m = blockIdx.x;
    const int V = K / 8;  // 16-byte vectors (8 fp16) per row
    const int64_t base = static_cast<int64_t>(m) * V;
    const int64_t total = static_cast<int64_t>(M) * V;
    auto load = [&](int v) {
        return in_bounds(base + v < total, status) ? x[base + v] : make_uint4(0u, 0u, 0u, 0u);
    };
    uint4 cache[kQCache];
    float amax = 0.f;
#pragma unroll
    for (int u = 0; u < kQCache; ++u) {
        const int v = static_cast<int>(threadIdx.x) + u * kQThreads;
        cache[u] = v < V ? load(v) : make_uint4(0u, 0u, 0u, 0u);
        amax = fmaxf(amax, absmax8(cache[u]));
    }
    for (int v = static_cast<int>(threadIdx.x) + kQCache * kQThreads; v < V; v += kQThreads)
        amax = fmaxf(amax, absmax8(load(v)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = 0.f;
#pragma unroll 8
    for (int w = 0; w < kQThreads / 32; ++w) amax = fmaxf(amax, wmax[w]);
    const float s = __fdiv_rn(amax, 127.0f);
    const float rs = __frcp_rn(s);
    if (threadIdx.x == 0 && in_bounds(m < M, status)) sx[m] = s;

    auto emit = [&](int v, const uint4 val) {
        const uint32_t w[4] = {val.x, val.y, val.z, val.w};
        uint32_t q8[2] = {0u, 0u};
        uint32_t h2[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
            const int a = quantize1(f.x, s, rs, amax > 0.f), b = quantize1(f.y, s, rs, amax > 0.f);
            q8[i >> 1] |= ((static_cast<uint32_t>(a) & 0xFFu) | ((static_cast<uint32_t>(b) & 0xFFu) << 8))
                          << (16 * (i & 1));
            const __half2 hq = __halves2half2(__int2half_rn(a), __int2half_rn(b));
            h2[i] = *reinterpret_cast<const uint32_t*>(&hq);
        }
        if (!in_bounds(base + v < total, status)) return;
        xq[base + v] = make_uint2(q8[0], q8[1]);
        if (xh != nullptr) xh[base + v] = make_uint4(h2[0], h2[1], h2[2], h2[3]);
    };
#pragma unroll
    for (int u = 0; u < kQCache; ++u) {
        const int v = static_cast<int>(threadIdx.x) + u * kQThreads;
        if (v < V) emit(v, cache[u]);
    }
    for (int v = static_cast<int>(threadIdx.x) + kQCache * kQThreads; v < V; v += kQThreads) emit(v, load(v));
}

// ------------------------------------------------------------------------------------ integer GEMV
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kUnroll = 4;  // 32-k blocks in flight per warp

// d + sum_{i<4} a.byte[i] * b.byte[i], a's bytes unsigned, b's signed.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int d) {
    int r;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(d));
    return r;
}

__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int d) {
    int r;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(d));
    return r;
}

// One 32-k block of one lane's column: v = its 4 weight words (word i = k 8i .. 8i + 7, nibble
// order of the device layout), xw = the block's staged activations per row (lo words, then hi
// words), ofs = -8 * sum of the block's activations per row.
template <int MR>
__device__ __forceinline__ void w4a8_block(const uint4 v, float s, const uint4* xw, const int* ofs, int row_stride,
                                           float (&acc)[MR]) {
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
    uint32_t lo[4], hi[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        lo[i] = words[i] & 0x0F0F0F0Fu;          // nibbles 0, 2, 4, 6: k offsets 0, 4, 1, 5
        hi[i] = (words[i] >> 4) & 0x0F0F0F0Fu;   // nibbles 1, 3, 5, 7: k offsets 2, 6, 3, 7
    }
#pragma unroll
    for (int m = 0; m < MR; ++m) {
        const uint4 xl = xw[2 * m * row_stride];
        const uint4 xh = xw[2 * m * row_stride + 1];
        int d = ofs[m * row_stride];
        d = dp4a_us(lo[0], xl.x, d);
        d = dp4a_us(hi[0], xh.x, d);
        d = dp4a_us(lo[1], xl.y, d);
        d = dp4a_us(hi[1], xh.y, d);
        d = dp4a_us(lo[2], xl.z, d);
        d = dp4a_us(hi[2], xh.z, d);
        d = dp4a_us(lo[3], xl.w, d);
        d = dp4a_us(hi[3], xh.w, d);
        acc[m] = fmaf(s, static_cast<float>(d), acc[m]);
    }
}

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

// CTAs per SM the register budget must allow: the grids are a few waves of 128-thread CTAs, and
// one CTA fewer per SM can add a whole wave (8 per SM = at most 64 registers per thread).
__host__ __device__ constexpr int gemv_w4a8_min_ctas(int mr) { return mr <= 2 ? 8 : mr <= 4 ? 6 : 5; }

// One CTA = one 128-column weight tile and one K-slice: warp w owns the tile's column slice w and
// runs the whole K-slice, so the four warps read each 2 KB row of the tile (32 k of 128 columns)
// together. (With the four column slices in four CTAs, each row was fetched in 512-byte parts at
// different times: measured 20 % slower once the weights in flight exceed ~2 GB, as in a decode
// step.) The K-slices of a tile form a cluster summed through DSMEM in rank order.
template <int MR>
__global__ void __launch_bounds__(kThreads, gemv_w4a8_min_ctas(MR))
    gemv_w4a8_kernel(const uint4* __restrict__ xq, const float* __restrict__ sx, const uint4* __restrict__ wr,
                     const uint16_t* __restrict__ sr, uint16_t* __restrict__ y, int N, int K, int G, int split,
                     unsigned* status) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int KB = K / 32;
    const int NG = K / G;
    const int rank = static_cast<int>(blockIdx.x) % split;
    const int tile = static_cast<int>(blockIdx.x) / split;
    const int wt = min(128, N - 128 * tile);  // columns of this tile (32, 64, 96 or 128)
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int col = 32 * warp + lane;         // column within the tile
    const bool valid = 32 * warp < wt;        // (warps past a ragged last tile only take part in the syncs)
    const int kb_begin = static_cast<int>((static_cast<int64_t>(rank) * KB) / split);
    const int kb_end = static_cast<int>((static_cast<int64_t>(rank + 1) * KB) / split);
    const int nblk = kb_end - kb_begin;
    const int nblk_max = (KB + split - 1) / split;

    uint4* xw = reinterpret_cast<uint4*>(smem);                                              // [MR][nblk_max][2]
    int* ofs = reinterpret_cast<int*>(smem + static_cast<size_t>(MR) * nblk_max * 32);        // [MR][nblk_max]
    float* part = reinterpret_cast<float*>(smem + static_cast<size_t>(MR) * nblk_max * 36);   // [MR][128]

    const uint4* wcol = wr + static_cast<int64_t>(tile) * 128 * KB + col;
    const uint16_t* scol = sr + static_cast<int64_t>(tile) * 128 * NG + col;

    const int gb = G / 32;
    const int gshift = (gb & (gb - 1)) == 0 ? __ffs(gb) - 1 : -1;
    auto group_of = [&](int b) { return gshift >= 0 ? (b >> gshift) : b / gb; };
    const int64_t w_total = static_cast<int64_t>(N) * KB, s_total = static_cast<int64_t>(NG) * N;
    const int64_t w_base = wcol - wr, s_base = scol - sr;
    auto load_w = [&](int b) {
        return in_bounds(w_base + static_cast<int64_t>(b) * wt < w_total, status)
                   ? ldg_stream(wcol + static_cast<int64_t>(b) * wt)
                   : make_uint4(0u, 0u, 0u, 0u);
    };
    auto load_s = [&](int b) -> float {
        const int64_t r = group_of(b);
        return in_bounds(s_base + r * wt < s_total, status) ? __half2float(__ushort_as_half(ldg_u16(scol + r * wt)))
                                                            : 0.f;
    };

    // Programmatic dependent launch: the warp's first batch of weights and scales is loaded while
    // the previous grid on the stream (typically the quantisation of x) finishes; xq only after it.
    int kb = kb_begin;
    const bool first = valid && kb + kUnroll - 1 < kb_end;
    uint4 v0[kUnroll];
    float s0[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        v0[u] = first ? load_w(kb + u) : make_uint4(0u, 0u, 0u, 0u);
        s0[u] = first ? load_s(kb + u) : 0.f;
    }
    griddep_wait();

    // Stage the K-slice of xq: per row and 32-k block, the activations in the byte order of the
    // weight nibbles (per 8 k: (k0, k4, k1, k5) and (k2, k6, k3, k7)) and -8 * their sum.
    {
        const int64_t xq_total = static_cast<int64_t>(MR) * K / 16;  // 16-byte vectors
        for (int i = threadIdx.x; i < MR * nblk; i += kThreads) {
            const int m = i / nblk, jb = i % nblk;
            const int64_t src = (static_cast<int64_t>(m) * K + static_cast<int64_t>(kb_begin + jb) * 32) / 16;
            uint4 a = make_uint4(0u, 0u, 0u, 0u), b = make_uint4(0u, 0u, 0u, 0u);
            if (in_bounds(src + 2 <= xq_total, status)) {
                a = xq[src];
                b = xq[src + 1];
            }
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            uint32_t lo[4], hi[4];
            int sum = 0;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                lo[g] = __byte_perm(w[2 * g], w[2 * g + 1], 0x5140);
                hi[g] = __byte_perm(w[2 * g], w[2 * g + 1], 0x7362);
                sum = dp4a_ss(w[2 * g], 0x01010101u, sum);
                sum = dp4a_ss(w[2 * g + 1], 0x01010101u, sum);
            }
            xw[2 * (m * nblk_max + jb)] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            xw[2 * (m * nblk_max + jb) + 1] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            ofs[m * nblk_max + jb] = -8 * sum;
        }
    }
    __syncthreads();

    float acc[MR];
#pragma unroll
    for (int m = 0; m < MR; ++m) acc[m] = 0.f;
    if (valid) {
        if (first) {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int jb = kb + u - kb_begin;
                w4a8_block<MR>(v0[u], s0[u], xw + 2 * jb, ofs + jb, nblk_max, acc);
            }
            kb += kUnroll;
        }
        for (; kb + kUnroll - 1 < kb_end; kb += kUnroll) {
            uint4 v[kUnroll];
            float sb[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                v[u] = load_w(kb + u);
                sb[u] = load_s(kb + u);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int jb = kb + u - kb_begin;
                w4a8_block<MR>(v[u], sb[u], xw + 2 * jb, ofs + jb, nblk_max, acc);
            }
        }
        if (kb < kb_end) {  // the last (< kUnroll) blocks: their loads issued together as well
            uint4 v[kUnroll];
            float sb[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                v[u] = kb + u < kb_end ? load_w(kb + u) : make_uint4(0u, 0u, 0u, 0u);
                sb[u] = kb + u < kb_end ? load_s(kb + u) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (kb + u < kb_end) w4a8_block<MR>(v[u], sb[u], xw + 2 * (kb + u - kb_begin), ofs + (kb + u - kb_begin),
                                                    nblk_max, acc);
        }
    }

    griddep_launch_dependents();
    auto row_scale = [&](int m) { return in_bounds(m < MR, status) ? sx[m] : 0.f; };
    if (split == 1) {
        if (valid) {
#pragma unroll
            for (int m = 0; m < MR; ++m) {
                const int64_t yi = static_cast<int64_t>(m) * N + 128 * tile + col;
                if (in_bounds(yi < static_cast<int64_t>(MR) * N, status))
                    y[yi] = __half_as_ushort(__float2half_rn(acc[m] * row_scale(m)));
            }
        }
        return;
    }
#pragma unroll
    for (int m = 0; m < MR; ++m) part[m * 128 + col] = acc[m];
    cluster_sync_all();
    for (int e = threadIdx.x; e < MR * 128; e += kThreads) {
        if ((e % split) != rank) continue;
        const uint32_t local = smem_u32(part + e);
        const float s = cluster_sum_f1(local, split);
        const int m = e / 128, c = e % 128;
        const int64_t yi = static_cast<int64_t>(m) * N + 128 * tile + c;
        if (c < wt && in_bounds(yi < static_cast<int64_t>(MR) * N, status))
            y[yi] = __half_as_ushort(__float2half_rn(s * row_scale(m)));
    }
    cluster_sync_all();
}

template <int MR>
cudaError_t launch_gemv_w4a8_m(const int8_t* xq, const float* sx, const uint32_t* qweight_r, const uint16_t* scales_r,
                               uint16_t* y, int N, int K, int G, int split, size_t smem, const LaunchCtx& ctx) {
    auto kern = gemv_w4a8_kernel<MR>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (split > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(split) * static_cast<unsigned>((N + 127) / 128), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = ctx.stream;
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
    return cudaLaunchKernelEx(&cfg, kern, reinterpret_cast<const uint4*>(xq), sx,
                              reinterpret_cast<const uint4*>(qweight_r), scales_r, y, N, K, G, split, ctx.status);
}

}  // namespace

cudaError_t launch_quantize_x_int8(const uint16_t* x, int8_t* xq, uint16_t* xq_f16, float* sx, int M, int K,
                                   cudaStream_t s, unsigned* status) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(M), 1, 1);
    cfg.blockDim = dim3(kQThreads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quantize_x_int8_kernel, reinterpret_cast<const uint4*>(x),
                              reinterpret_cast<uint2*>(xq), reinterpret_cast<uint4*>(xq_f16), sx, M, K, status);
}

int gemv_w4a8_ctas_per_sm(int M) { return gemv_w4a8_min_ctas(M); }

size_t gemv_w4a8_smem_bytes(int M, int K, int split) {
    const size_t nblk_max = static_cast<size_t>((K / 32 + split - 1) / split);
    return static_cast<size_t>(M) * nblk_max * 36 + static_cast<size_t>(M) * 128 * 4;
}

cudaError_t launch_gemv_w4a8(const int8_t* xq, const float* sx, const uint32_t* qweight_r, const uint16_t* scales_r,
                             uint16_t* y, int M, int N, int K, int G, int split, const LaunchCtx& ctx) {
    const size_t smem = gemv_w4a8_smem_bytes(M, K, split);
    switch (M) {
        case 1: return launch_gemv_w4a8_m<1>(xq, sx, qweight_r, scales_r, y, N, K, G, split, smem, ctx);
        case 2: return launch_gemv_w4a8_m<2>(xq, sx, qweight_r, scales_r, y, N, K, G, split, smem, ctx);
        case 3: return launch_gemv_w4a8_m<3>(xq, sx, qweight_r, scales_r, y, N, K, G, split, smem, ctx);
        case 4: return launch_gemv_w4a8_m<4>(xq, sx, qweight_r, scales_r, y, N, K, G, split, smem, ctx);
        case 5: return launch_gemv_w4a8_m<5>(xq, sx, qweight_r, scales_r, y, N, K, G, split, smem, ctx);
        case 6: return launch_gemv_w4a8_m<6>(xq, sx, qweight_r, scales_r, y, N, K, G, split, smem, ctx);
        case 7: return launch_gemv_w4a8_m<7>(xq, sx, qweight_r, scales_r, y, N, K, G, split, smem, ctx);
        case 8: return launch_gemv_w4a8_m<8>(xq, sx, qweight_r, scales_r, y, N, K, G, split, smem, ctx);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace w4a16
