// Host-side interface between the C-ABI layer (w4a16_api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace w4a16 {

// Everything a kernel launch needs besides its data pointers.
struct LaunchCtx {
    cudaStream_t stream;
    unsigned* status;     // device address of this device's status word
    uint64_t timeout_ns;  // limit of every bounded wait
    int sm_count;
    // Weight format: 0 = int4 with offset 8 and fp16 group scales; 1 = NVFP4 (E2M1 codes in the
    // canonical nibble order, fp16 scales per 16 k converted from E4M3, group passed as 16).
    int nvfp4 = 0;
    float tensor_scale = 1.0f;  // multiplies every fp32 sum before the fp16 rounding (1 for int4)
    // Tile kernel only: when not null, the sums of output row m are then multiplied by row_scale[m]
    // (the per-token scale of int8 activations, W4A8).
    const float* row_scale = nullptr;
};

// ---- repack.cu
cudaError_t launch_repack(const int32_t* qweight, const uint16_t* scales, uint32_t* qweight_r, uint16_t* scales_r,
                          int N, int K, int G, cudaStream_t s, unsigned* status);
cudaError_t launch_unrepack(const uint32_t* qweight_r, const uint16_t* scales_r, int32_t* qweight, uint16_t* scales,
                            int N, int K, int G, cudaStream_t s, unsigned* status);

// NVFP4: E2M1 codes keep the canonical nibble order; E4M3 scales [K/16][N] become fp16 of equal value.
cudaError_t launch_repack_nvfp4(const int32_t* qweight, const uint8_t* scales8, uint32_t* qweight_r, uint16_t* scales_r,
                                int N, int K, cudaStream_t s, unsigned* status);
cudaError_t launch_unrepack_nvfp4(const uint32_t* qweight_r, const uint16_t* scales_r, int32_t* qweight,
                                  uint8_t* scales8, int N, int K, cudaStream_t s, unsigned* status);

// ---- gemv.cu: CUDA-core split-K GEMV, M <= 8.
constexpr int kGemvMaxM = 8;
size_t gemv_smem_bytes(int M, int N, int K, int split);
// unroll: 32-k blocks in flight per warp, 4 (any M) or 8 (M <= 2).
cudaError_t launch_gemv(const uint16_t* x, const uint32_t* qweight_r, const uint16_t* scales_r, uint16_t* y, int M,
                        int N, int K, int G, int split, int unroll, const LaunchCtx& ctx);
// CTAs of the M-row GEMV (M <= 2) with `unroll` blocks in flight resident at once, 0 if unknown.
int gemv_resident_ctas(int M, int unroll, size_t smem, int sm_count);

// ---- tc_gemm.cu: the x operand's tensor map. x viewed as
// [K/64 blocks][M rows][64 k]; one box = one stage tile [KC/64][MT][64] in the MMA's 128-byte-swizzle
// K-major layout; rows >= M read as zero. Falls back to a 2-D map when the driver refuses the 3-D one.
bool encode_x_map(CUtensorMap* map, const uint16_t* x, int M, int K, int MT, int KC, bool* three_d);

// ---- tc_gemm.cu: tcgen05 tensor-core path.
struct TcConfig {
    int m_tile;       // 16, 32, 64, 128, 256
    int k_chunk;      // K per stage: 64, 128 or 256
    int stages;       // shared-memory ring depth, 2..16
    int split;        // CTAs per cluster along K, 1..16
    int tmem_stages;  // TMEM A ring depth, 2..8
    int issuers;      // MMA-issuing threads (1, 2 or 4), each with its own accumulator
    int dequant_warps;  // 16, or 8 (small tiles that fit two CTAs per SM)
    // Work items (column tile x row tile) of the last, partial wave of a split-1 launch, run as a
    // second launch whose clusters split each item `tail_split` ways along K (0: no second launch).
    int tail_items = 0;
    int tail_split = 0;
    // > 0: a launch of unsplit CTAs with more work items than this runs this many CTAs, each taking
    // every persist_ctas-th item (persistent grid); 0: one CTA (cluster) per item
    int persist_ctas = 0;
};
bool tc_instantiated(int m_tile, int k_chunk, int issuers, int dequant_warps);
bool tc_config_valid(const TcConfig& c, int M, int N, int K, int G);
size_t tc_smem_bytes(const TcConfig& c, int G);
int tc_tmem_cols(const TcConfig& c);
// CTAs of this config resident on the current device at once (cluster occupancy), 0 if unknown.
int tc_resident_ctas(const TcConfig& c, int G);
cudaError_t launch_tc(const uint16_t* x, const uint32_t* qweight_r, const uint16_t* scales_r, uint16_t* y, int M,
                      int N, int K, int G, const TcConfig& c, const LaunchCtx& ctx);

// ---- w4a8.cu: int8 activations (W4A8).
// Per-token symmetric quantisation: sx[m] = amax / 127, xq = rne(x / sx) (binary32), optionally
// also written as fp16 integers (xq_f16 may be null).
cudaError_t launch_quantize_x_int8(const uint16_t* x, int8_t* xq, uint16_t* xq_f16, float* sx, int M, int K,
                                   cudaStream_t s, unsigned* status);
// Integer (dp4a) split-K GEMV, M <= 8: y = fp16(sx[m] * sum_blocks s * sum (q - 8) xq).
size_t gemv_w4a8_smem_bytes(int M, int K, int split);
int gemv_w4a8_ctas_per_sm(int M);  // CTAs per SM its register bound guarantees
cudaError_t launch_gemv_w4a8(const int8_t* xq, const float* sx, const uint32_t* qweight_r, const uint16_t* scales_r,
                             uint16_t* y, int M, int N, int K, int G, int split, const LaunchCtx& ctx);

// ---- act.cu: SwiGLU activation of a fused gate+up output, act = silu(gate) * up.
cudaError_t launch_silu_mul(const uint16_t* gu, uint16_t* act, int M, int I, int sm_count, cudaStream_t s,
                            unsigned* status);

}  // namespace w4a16
