// SwiGLU activation between the fused gate+up GEMM and the down projection of a dense layer:
//   act[m][i] = fp16_rne(silu(g) * u),  g = gu[m][i], u = gu[m][I + i],  silu(g) = g / (1 + e^-g),
// evaluated in fp32 from the fp16 inputs. One thread per 8 consecutive outputs (16-byte loads and
// stores); launched with programmatic dependent launch after the GEMM that writes gu.
#include "common.cuh"
#include "internal.h"

namespace w4a16 {
namespace {

__device__ __forceinline__ float silu_f32(float g) { return g / (1.0f + expf(-g)); }

__global__ void __launch_bounds__(256) silu_mul_kernel(const uint4* __restrict__ gu, uint4* __restrict__ act, int M,
                                                       int I, unsigned* status) {
    // The next kernel (the down projection) may start now: its weight copies do not depend on act,
    // and it waits for this grid to complete before it reads act.
    griddep_launch_dependents();
    griddep_wait();  // gu is the previous kernel's output
    const int v_per_row = I / 8;
    const int64_t total = static_cast<int64_t>(M) * v_per_row;
    for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < total;
         v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = v / v_per_row;
        const int64_t c = v - m * v_per_row;
        if (!in_bounds(m * 2 * v_per_row + v_per_row + c < 2 * total && v < total, status)) continue;
        const uint4 g4 = gu[m * 2 * v_per_row + c];
        const uint4 u4 = gu[m * 2 * v_per_row + v_per_row + c];
        const uint32_t g2[4] = {g4.x, g4.y, g4.z, g4.w};
        const uint32_t u2[4] = {u4.x, u4.y, u4.z, u4.w};
        uint32_t o2[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 g = *reinterpret_cast<const __half2*>(&g2[i]);
            const __half2 u = *reinterpret_cast<const __half2*>(&u2[i]);
            const float lo = silu_f32(__low2float(g)) * __low2float(u);
            const float hi = silu_f32(__high2float(g)) * __high2float(u);
            const __half2 r = __floats2half2_rn(lo, hi);
            o2[i] = *reinterpret_cast<const uint32_t*>(&r);
        }
        act[v] = make_uint4(o2[0], o2[1], o2[2], o2[3]);
    }
}

}  // namespace

cudaError_t launch_silu_mul(const uint16_t* gu, uint16_t* act, int M, int I, int sm_count, cudaStream_t s,
                            unsigned* status) {
    const int64_t total = static_cast<int64_t>(M) * (I / 8);
    const int64_t blocks_needed = (total + 255) / 256;
    const int blocks = static_cast<int>(blocks_needed < 8LL * sm_count ? blocks_needed : 8LL * sm_count);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks > 0 ? blocks : 1), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, silu_mul_kernel, reinterpret_cast<const uint4*>(gu), reinterpret_cast<uint4*>(act),
                              M, I, status);
}

}  // namespace w4a16
