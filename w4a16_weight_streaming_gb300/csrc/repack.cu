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

// Tile geometry of the streaming layout: 128-column tiles, the last one w_t = N - 128t wide.
__device__ __forceinline__ int tile_width(int N, int t) { return min(128, N - 128 * t); }

// One thread per 16-byte vector (k-block b, column n), v = b * N + n: reads the four canonical
// words qweight[4b + i][n] (consecutive n -> consecutive addresses) and writes the vector at
// tile t = n / 128, position b * w_t + (n - 128t) of that tile's [K/32][w_t] block.
// PERMUTE: int4 words get the fp16-ready nibble order; NVFP4 words keep the canonical order (byte i
// = codes of k offsets 2i, 2i + 1, the operand of the hardware E2M1 pair conversion).
template <bool PERMUTE>
__global__ void repack_weights_kernel(const uint32_t* __restrict__ qw, uint4* __restrict__ out, int N, int K,
                                      unsigned* status) {
    const int64_t total = static_cast<int64_t>(N) * (K / 32);
    for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < total;
         v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int n = static_cast<int>(v % N);
        const int b = static_cast<int>(v / N);
        const int t = n / 128;
        const int64_t o = static_cast<int64_t>(t) * 128 * (K / 32) + static_cast<int64_t>(b) * tile_width(N, t) + (n - 128 * t);
        if (!in_bounds(o < total && static_cast<int64_t>(4 * b + 3) * N + n < 4 * total, status)) continue;
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t cw = qw[static_cast<int64_t>(4 * b + i) * N + n];
            w[i] = PERMUTE ? interleave_word(cw) : cw;
        }
        out[o] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <bool PERMUTE>
__global__ void unrepack_weights_kernel(const uint4* __restrict__ in, uint32_t* __restrict__ qw, int N, int K,
                                        unsigned* status) {
    const int64_t total = static_cast<int64_t>(N) * (K / 32);
    for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < total;
         v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int n = static_cast<int>(v % N);
        const int b = static_cast<int>(v / N);
        const int t = n / 128;
        const int64_t o = static_cast<int64_t>(t) * 128 * (K / 32) + static_cast<int64_t>(b) * tile_width(N, t) + (n - 128 * t);
        if (!in_bounds(o < total && static_cast<int64_t>(4 * b + 3) * N + n < 4 * total, status)) continue;
        const uint4 x = in[o];
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) qw[static_cast<int64_t>(4 * b + i) * N + n] = PERMUTE ? deinterleave_word(w[i]) : w[i];
    }
}

// scales [K/G][N] <-> scales_r (tile t: [K/G][w_t] at element 128t * K/G); one thread per
// canonical element i = g * N + n.
__global__ void scales_kernel(const uint16_t* __restrict__ in, uint16_t* __restrict__ out, int N, int NG,
                              bool to_tiles, unsigned* status) {
    const int64_t total = static_cast<int64_t>(N) * NG;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int n = static_cast<int>(i % N);
        const int g = static_cast<int>(i / N);
        const int t = n / 128;
        const int64_t tiled = static_cast<int64_t>(t) * 128 * NG + static_cast<int64_t>(g) * tile_width(N, t) + (n - 128 * t);
        if (!in_bounds(tiled < total, status)) continue;
        if (to_tiles)
            out[tiled] = in[i];
        else
            out[i] = in[tiled];
    }
}

// NVFP4 scales: E4M3 bytes [K/16][N] <-> fp16 of equal value in the tiled layout (group 16). Every
// E4M3 value is exactly an fp16 number, so both directions are exact for the values that occur.
__global__ void scales_e4m3_kernel(const uint8_t* __restrict__ in8, uint16_t* __restrict__ out16, int N, int NG,
                                   unsigned* status) {
    const int64_t total = static_cast<int64_t>(N) * NG;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int n = static_cast<int>(i % N);
        const int g = static_cast<int>(i / N);
        const int t = n / 128;
        const int64_t tiled = static_cast<int64_t>(t) * 128 * NG + static_cast<int64_t>(g) * tile_width(N, t) + (n - 128 * t);
        if (!in_bounds(tiled < total, status)) continue;
        uint32_t h2;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(in8[i])));
        out16[tiled] = static_cast<uint16_t>(h2 & 0xFFFFu);  // the low byte converts into the low half
    }
}

__global__ void scales_to_e4m3_kernel(const uint16_t* __restrict__ in16, uint8_t* __restrict__ out8, int N, int NG,
                                      unsigned* status) {
    const int64_t total = static_cast<int64_t>(N) * NG;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int n = static_cast<int>(i % N);
        const int g = static_cast<int>(i / N);
        const int t = n / 128;
        const int64_t tiled = static_cast<int64_t>(t) * 128 * NG + static_cast<int64_t>(g) * tile_width(N, t) + (n - 128 * t);
        if (!in_bounds(tiled < total, status)) continue;
        uint16_t b2;
        asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(b2) : "r"(static_cast<uint32_t>(in16[tiled])));
        out8[i] = static_cast<uint8_t>(b2 & 0xFFu);
    }
}

int grid_for(int64_t total, int block) {
    const int64_t blocks = (total + block - 1) / block;
    return static_cast<int>(blocks < 65535 * 16 ? blocks : 65535 * 16);
}

}  // namespace

cudaError_t launch_repack(const int32_t* qweight, const uint16_t* scales, uint32_t* qweight_r, uint16_t* scales_r,
                          int N, int K, int G, cudaStream_t s, unsigned* status) {
    const int64_t vec = static_cast<int64_t>(N) * (K / 32);
    repack_weights_kernel<true><<<grid_for(vec, 256), 256, 0, s>>>(reinterpret_cast<const uint32_t*>(qweight),
                                                              reinterpret_cast<uint4*>(qweight_r), N, K, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t ns = static_cast<int64_t>(N) * (K / G);
    scales_kernel<<<grid_for(ns, 256), 256, 0, s>>>(scales, scales_r, N, K / G, true, status);
    return cudaGetLastError();
}

cudaError_t launch_unrepack(const uint32_t* qweight_r, const uint16_t* scales_r, int32_t* qweight, uint16_t* scales,
                            int N, int K, int G, cudaStream_t s, unsigned* status) {
    const int64_t vec = static_cast<int64_t>(N) * (K / 32);
    unrepack_weights_kernel<true><<<grid_for(vec, 256), 256, 0, s>>>(reinterpret_cast<const uint4*>(qweight_r),
                                                                reinterpret_cast<uint32_t*>(qweight), N, K, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t ns = static_cast<int64_t>(N) * (K / G);
    scales_kernel<<<grid_for(ns, 256), 256, 0, s>>>(scales_r, scales, N, K / G, false, status);
    return cudaGetLastError();
}

cudaError_t launch_repack_nvfp4(const int32_t* qweight, const uint8_t* scales8, uint32_t* qweight_r, uint16_t* scales_r,
                                int N, int K, cudaStream_t s, unsigned* status) {
    const int64_t vec = static_cast<int64_t>(N) * (K / 32);
    repack_weights_kernel<false><<<grid_for(vec, 256), 256, 0, s>>>(reinterpret_cast<const uint32_t*>(qweight),
                                                                     reinterpret_cast<uint4*>(qweight_r), N, K, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t ns = static_cast<int64_t>(N) * (K / 16);
    scales_e4m3_kernel<<<grid_for(ns, 256), 256, 0, s>>>(scales8, scales_r, N, K / 16, status);
    return cudaGetLastError();
}

cudaError_t launch_unrepack_nvfp4(const uint32_t* qweight_r, const uint16_t* scales_r, int32_t* qweight,
                                  uint8_t* scales8, int N, int K, cudaStream_t s, unsigned* status) {
    const int64_t vec = static_cast<int64_t>(N) * (K / 32);
    unrepack_weights_kernel<false><<<grid_for(vec, 256), 256, 0, s>>>(reinterpret_cast<const uint4*>(qweight_r),
                                                                       reinterpret_cast<uint32_t*>(qweight), N, K, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t ns = static_cast<int64_t>(N) * (K / 16);
    scales_to_e4m3_kernel<<<grid_for(ns, 256), 256, 0, s>>>(scales_r, scales8, N, K / 16, status);
    return cudaGetLastError();
}

}  // namespace w4a16
