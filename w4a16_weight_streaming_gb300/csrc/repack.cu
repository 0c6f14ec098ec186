// One-time re-layout of the canonical W4A16 matrix into the streaming layout, and its inverse.
// Pure integer bit moves; both are bijections on the bytes.
#include "common.cuh"
#include "internal.h"

namespace w4a16 {
namespace {

// Nibble position inside a repacked word for canonical nibble j (k offset j within 8):
// even k offsets in positions 0..3, odd ones in 4..7, so one AND with 0x000F000F yields an
// fp16-ready (k, k+1) pair.
__device__ __forceinline__ uint32_t interleave_word(uint32_t w) {
    uint32_t out = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int pos = (j & 1) ? 4 + (j >> 1) : (j >> 1);
        out |= ((w >> (4 * j)) & 0xFu) << (4 * pos);
    }
    return out;
}

__device__ __forceinline__ uint32_t deinterleave_word(uint32_t w) {
    uint32_t out = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int pos = (j & 1) ? 4 + (j >> 1) : (j >> 1);
        out |= ((w >> (4 * pos)) & 0xFu) << (4 * j);
    }
    return out;
}

// One thread per 16-byte output vector (tile t, k-block b, lane l): reads the four canonical
// words qweight[4b + i][32t + l] (consecutive l -> consecutive addresses) and writes the vector.
__global__ void repack_weights_kernel(const uint32_t* __restrict__ qw, uint4* __restrict__ out, int N, int K) {
    const int64_t total = static_cast<int64_t>(N) * (K / 32);
    const int KB = K / 32;
    for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < total;
         v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int l = static_cast<int>(v % 32);
        const int64_t tb = v / 32;
        const int b = static_cast<int>(tb % KB);
        const int t = static_cast<int>(tb / KB);
        const int n = 32 * t + l;
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = interleave_word(qw[static_cast<int64_t>(4 * b + i) * N + n]);
        out[v] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

__global__ void unrepack_weights_kernel(const uint4* __restrict__ in, uint32_t* __restrict__ qw, int N, int K) {
    const int64_t total = static_cast<int64_t>(N) * (K / 32);
    const int KB = K / 32;
    for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < total;
         v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int l = static_cast<int>(v % 32);
        const int64_t tb = v / 32;
        const int b = static_cast<int>(tb % KB);
        const int t = static_cast<int>(tb / KB);
        const int n = 32 * t + l;
        const uint4 x = in[v];
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) qw[static_cast<int64_t>(4 * b + i) * N + n] = deinterleave_word(w[i]);
    }
}

// scales [K/G][N] <-> scales_r [N/32][K/G][32]; one thread per element, indexed by the
// canonical position when `to_tiles`, by the tiled position otherwise (so writes coalesce).
__global__ void scales_kernel(const uint16_t* __restrict__ in, uint16_t* __restrict__ out, int N, int NG,
                              bool to_tiles) {
    const int64_t total = static_cast<int64_t>(N) * NG;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        if (to_tiles) {
            // i = (t * NG + g) * 32 + l  (output order)
            const int l = static_cast<int>(i % 32);
            const int64_t tg = i / 32;
            const int g = static_cast<int>(tg % NG);
            const int t = static_cast<int>(tg / NG);
            out[i] = in[static_cast<int64_t>(g) * N + 32 * t + l];
        } else {
            // i = g * N + n  (output order)
            const int n = static_cast<int>(i % N);
            const int g = static_cast<int>(i / N);
            out[i] = in[(static_cast<int64_t>(n / 32) * NG + g) * 32 + (n % 32)];
        }
    }
}

int grid_for(int64_t total, int block) {
    const int64_t blocks = (total + block - 1) / block;
    return static_cast<int>(blocks < 65535 * 16 ? blocks : 65535 * 16);
}

}  // namespace

cudaError_t launch_repack(const int32_t* qweight, const uint16_t* scales, uint32_t* qweight_r, uint16_t* scales_r,
                          int N, int K, int G, cudaStream_t s) {
    const int64_t vec = static_cast<int64_t>(N) * (K / 32);
    repack_weights_kernel<<<grid_for(vec, 256), 256, 0, s>>>(reinterpret_cast<const uint32_t*>(qweight),
                                                              reinterpret_cast<uint4*>(qweight_r), N, K);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t ns = static_cast<int64_t>(N) * (K / G);
    scales_kernel<<<grid_for(ns, 256), 256, 0, s>>>(scales, scales_r, N, K / G, true);
    return cudaGetLastError();
}

cudaError_t launch_unrepack(const uint32_t* qweight_r, const uint16_t* scales_r, int32_t* qweight, uint16_t* scales,
                            int N, int K, int G, cudaStream_t s) {
    const int64_t vec = static_cast<int64_t>(N) * (K / 32);
    unrepack_weights_kernel<<<grid_for(vec, 256), 256, 0, s>>>(reinterpret_cast<const uint4*>(qweight_r),
                                                                reinterpret_cast<uint32_t*>(qweight), N, K);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t ns = static_cast<int64_t>(N) * (K / G);
    scales_kernel<<<grid_for(ns, 256), 256, 0, s>>>(scales_r, scales, N, K / G, false);
    return cudaGetLastError();
}

}  // namespace w4a16
