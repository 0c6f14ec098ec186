/*
 * libw4a16: the W4A16 weight-streaming GEMM on one GB300 (sm_103a).
 *
 *   y[M,N] = x[M,K] . W[K,N]      W stored as 4-bit integers with fp16 group scales,
 *                                 w[k][n] = fp16_rne((q[k][n] - 8) * s[k/G][n]),
 *                                 fp16 x, fp32 accumulation, fp16 y (round to nearest even).
 *
 * The operation: a weight matrix stored in 4 bits multiplied by 16-bit activations ("RTX 3090
 * Tested: Qwen's 381 tok/s Myth Busted", kongchang.com, section "What Exactly Is This Stack"),
 * with one read of the weights shared by all M activation rows of a decode or verify step
 * ("Qwen3.8-27B at 764, 1,035 and 1,623 tok/s", ai.satyajit.si, sections "One weight read,
 * shared by every stream" and "Speculation spends the same arithmetic": M = streams x verified
 * positions). The canonical packed format is the workload's (the pages do not print one):
 *
 *   qweight int32 [K/8][N]   nibble j (bits 4j..4j+3 of the word taken as unsigned) of
 *                            qweight[k/8][n] is q[k][n] with j = k mod 8 (low nibble first)
 *   scales  fp16  [K/G][N]   (passed as uint16_t bit patterns)
 *
 * Conventions shared by every entry point:
 *   - Every data pointer is a DEVICE pointer owned by the caller; the library never frees or
 *     keeps it. Host pointers are rejected where the CUDA runtime can tell (see each call).
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream). Calls that
 *     launch work are asynchronous on it and return once the work is queued.
 *   - The library allocates no device or host memory on any call. Its only device state is one
 *     status word per device (see w4a16_device_status).
 *   - Every call returns a w4a16_status. Argument checks happen before any launch; a rejected
 *     call launches nothing and leaves every buffer untouched.
 *   - Supported shapes: N % 32 == 0, K % 64 == 0, group % 32 == 0, K % group == 0,
 *     1 <= M <= 2^20, N <= 2^23, K <= 2^22. x, y, qweight and scales 16-byte aligned.
 *     x and y must not overlap. The tensor-core path (M > 8, or M >= 2 with automatic plans)
 *     also needs K % 128 == 0 and group dividing 128 or a multiple of it (32, 64, 128, 256,
 *     384, ...). Shapes that miss that condition run on the CUDA-core GEMV, which needs M <= 8
 *     and stages its slice of x in shared memory: M*K <= 1,500,000 always fits. Any other
 *     shape in the set above gets an automatic plan.
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    W4A16_OK = 0,
    W4A16_ERR_INVALID_ARG = 1,       /* null pointer, non-positive size, overlap, host pointer */
    W4A16_ERR_UNSUPPORTED_SHAPE = 2, /* shape outside the supported set above */
    W4A16_ERR_MISALIGNED = 3,        /* a pointer is not 16-byte aligned */
    W4A16_ERR_CUDA = 4,              /* the CUDA runtime refused a launch or query */
    W4A16_ERR_DEVICE_TIMEOUT = 5,    /* a kernel gave up a bounded wait (reported by w4a16_device_status) */
    W4A16_ERR_BOUNDS = 6             /* a kernel index check failed: the debug-bounds build only (see below) */
} w4a16_status;

/* Which kernel family runs a GEMM. */
typedef enum {
    W4A16_PATH_AUTO = 0, /* the dispatcher decides from (M, N, K) */
    W4A16_PATH_GEMV = 1, /* CUDA-core split-K GEMV, M <= 8 */
    W4A16_PATH_TC = 2    /* tcgen05 tensor-core tiles, any M */
} w4a16_path;

/* A launch plan. Zero fields mean "choose automatically". */
typedef struct {
    int path;        /* w4a16_path */
    int split_k;     /* CTAs of one thread-block cluster splitting K (1..16) */
    int m_tile;      /* TC: activation rows per tile: 16, 32, 64, 128, 256 */
    int k_chunk;     /* TC: K per pipeline stage, 128 or 256 */
    int stages;      /* TC: shared-memory pipeline depth, 2..16 */
    int tmem_stages; /* TC: tensor-memory (dequantised A) pipeline depth, 2..8 */
    int mma_issuers; /* TC: threads issuing tensor-core MMAs, each with its own accumulator: 1, 2, 4 */
    int clusters;    /* reserved, must be 0 */
    int dequant_warps; /* TC: 16, or 8 (m_tile <= 64, k_chunk 128: half-size CTAs, two per SM) */
    int tail_split;  /* TC: when the work items (128 output columns x m_tile rows), split_k CTAs
                        each (0 taken as 1), do not fill whole waves of resident CTAs, the items of
                        the last, partial wave run as a second launch on the same stream, each split
                        this many ways along K (2..16). 0: none in an explicit plan, the dispatcher's
                        choice in an automatic one (all fields 0); other values:
                        W4A16_ERR_INVALID_ARG. */
} w4a16_plan;

/* Library version: major*10000 + minor*100 + patch. */
int w4a16_version(void);

/*
 * 1 in the debug-bounds build of the library (libw4a16_debug.so, compiled with W4A16_DEBUG_BOUNDS),
 * 0 in the normal one. In the debug-bounds build every kernel checks each global-memory index (and
 * each bulk-copy source range) against the size of its buffer before the access; a bad index is
 * not accessed and records W4A16_ERR_BOUNDS in the device status word, which w4a16_device_status
 * reports (the first error of a launch is kept). Nothing traps: the context stays usable. It
 * stands in for a memory checker on hardware where none can be run. Same entry points, slower.
 */
int w4a16_debug_bounds(void);

/* Human-readable name of a w4a16_status value (static string; never NULL). */
const char* w4a16_status_string(int code);

/* Bytes of the repacked weight / scale buffers for an N x K matrix with group size `group`;
 * 0 when the shape is unsupported. They equal the canonical sizes, K*N/2 and (K/group)*N*2. */
size_t w4a16_repacked_qweight_bytes(int N, int K, int group);
size_t w4a16_repacked_scales_bytes(int N, int K, int group);

/*
 * One-time re-layout of a canonical matrix into the device layout the GEMM streams
 * (a bijection of the bytes; not part of the timed step):
 *   Columns are grouped in tiles of 128 (the last one w_t = N - 128t wide, t = n / 128).
 *   qweight_r: tile t occupies bytes [64*t*K, 64*t*K + w_t*K/2), laid out [K/32][w_t] of
 *              16-byte vectors; a vector holds 32 consecutive k of one column as 4 words of 8 k,
 *              and inside a word q[k][n] sits in nibble position p = 0,4,1,5,2,6,3,7 for
 *              k mod 8 = 0..7. One tile's rows k0..k0+KC are therefore one contiguous block.
 *   scales_r:  tile t occupies elements [128*t*(K/group), ...), laid out [K/group][w_t].
 * In: qweight int32 [K/8][N], scales uint16 [K/group][N] (device). Out: qweight_r
 * (w4a16_repacked_qweight_bytes), scales_r (w4a16_repacked_scales_bytes) (device, caller
 * allocated, must not overlap the inputs). Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED,
 * CUDA.
 */
int w4a16_repack(const int32_t* qweight, const uint16_t* scales, void* qweight_r, void* scales_r, int N, int K,
                 int group, void* stream);

/* Exact inverse of w4a16_repack (used to check the round trip bit for bit). */
int w4a16_unrepack(const void* qweight_r, const void* scales_r, int32_t* qweight, uint16_t* scales, int N, int K,
                   int group, void* stream);

/*
 * y[M][N] = x[M][K] . dequant(W), the hot path of a decode or speculative-verify step.
 *   x:         fp16 [M][K] row-major (uint16_t bit patterns), device
 *   qweight_r: repacked weights from w4a16_repack, device
 *   scales_r:  repacked scales from w4a16_repack, device
 *   y:         fp16 [M][N] row-major, device, written in full (every element)
 * The dispatcher picks the kernel family and launch plan from (M, N, K, group); w4a16_last_dispatch
 * reports what ran. A call is one kernel launch on `stream`, or two when the tile plan splits off the
 * last, partial wave of work items (w4a16_plan.tail_split); unsplit 128- and 256-row tile launches
 * with more work items than resident CTAs run one CTA per SM over several items. Accuracy: every element is within 2^-10*|y_exact| + 2^-10*sum_k|x*w| of the
 * exact result (fp32 accumulation chains are kept short enough for that bound).
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, CUDA (launch refused).
 */
int w4a16_gemm(const uint16_t* x, const void* qweight_r, const void* scales_r, uint16_t* y, int M, int N, int K,
               int group, void* stream);

/* As w4a16_gemm with an explicit plan (NULL or zero fields = automatic). An invalid plan
 * (e.g. GEMV with M > 8, split_k larger than the K chunks) returns UNSUPPORTED_SHAPE; a tail_split
 * outside {0, 2..16}, INVALID_ARG. */
int w4a16_gemm_ex(const uint16_t* x, const void* qweight_r, const void* scales_r, uint16_t* y, int M, int N, int K,
                  int group, const w4a16_plan* plan, void* stream);

/*
 * w4a16_gemm for activations and results in HOST memory, queued on `stream` as three operations:
 * copy x_host -> x_dev (M*K fp16), the GEMM into y_dev (automatic plan), copy y_dev -> y_host
 * (M*N fp16). The step of the paths above that a serving loop runs each decode step, with its
 * host<->device copies; one call instead of three keeps the host cost of a step low.
 *   x_host, y_host: host buffers (pinned, for the copies to be asynchronous), caller-owned; they
 *                   must not overlap. y_host is valid once `stream` has been synchronised.
 *   x_dev, y_dev:   caller-owned device buffers of M*K and M*N fp16 (16-byte aligned); the
 *                   library allocates nothing.
 *   qweight_r, scales_r, M, N, K, group, stream: as w4a16_gemm.
 * Every check of w4a16_gemm (on x_dev, y_dev and the weights) runs before anything is queued, and
 * x_host / y_host are rejected (INVALID_ARG) when null, overlapping or known to the runtime as
 * device memory. A rejected call queues nothing. Errors: INVALID_ARG, UNSUPPORTED_SHAPE,
 * MISALIGNED, CUDA (a copy or launch refused; operations queued before it stay queued).
 */
int w4a16_gemm_host(const uint16_t* x_host, uint16_t* x_dev, const void* qweight_r, const void* scales_r,
                    uint16_t* y_dev, uint16_t* y_host, int M, int N, int K, int group, void* stream);

/* The plan w4a16_gemm would use for this shape (host only; launches nothing).
 * Automatic plans (w4a16_gemm, w4a16_gemm_host, w4a16_gemm_ex with NULL or all-zero plan, this
 * call) can be overridden without rebuilding: the environment variable W4A16_PLAN, read once per
 * process, holds "field=value[,field=value...]" with the w4a16_plan field names, no spaces
 * (e.g. "path=2,m_tile=64,split_k=3"). It is then used as the plan of every such call. A malformed
 * W4A16_PLAN makes them return INVALID_ARG; a plan invalid for a shape, UNSUPPORTED_SHAPE. */
int w4a16_plan_for(int M, int N, int K, int group, w4a16_plan* out);

/*
 * The activation between the fused gate+up projection and the down projection of a dense layer
 * (the 17,408-wide MLPs of "Qwen3.8-27B at 764, 1,035 and 1,623 tok/s", ai.satyajit.si, section
 * "Where the line bends"; read as SwiGLU, the plainest reading for that model family):
 *   act[m][i] = fp16_rne(silu(g) * u),  g = gu[m][i], u = gu[m][I + i],  silu(g) = g / (1 + e^-g),
 * evaluated in fp32 from the fp16 inputs (error about one fp16 rounding of the result).
 *   gu:  fp16 [M][2I] row-major, device: the output of w4a16_gemm with the fused 2I-column
 *        gate+up matrix, gate columns first.
 *   act: fp16 [M][I] row-major, device, written in full; must not overlap gu.
 * Supported: I % 8 == 0, 1 <= M <= 2^20, I <= 2^22; both pointers 16-byte aligned. Asynchronous on
 * `stream`, launched with programmatic dependent launch: it is scheduled while the GEMM before it
 * finishes and reads gu only after that GEMM completed. Allocates nothing.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, CUDA.
 */
int w4a16_silu_mul(const uint16_t* gu, uint16_t* act, int M, int I, void* stream);

/*
 * NVFP4 weights (the RTX 5090 runs of "Qwen3.8-27B at 764, 1,035 and 1,623 tok/s", section "One
 * weight read, shared by every stream", keep their weights in NVFP4; the pages print no format, so
 * the published NVFP4 definition is the reading). Activations stay fp16, as for every call here:
 *   qweight  int32 [K/8][N]: nibble (k mod 8) of qweight[k/8][n] is the 4-bit E2M1 code of w[k][n]
 *            (sign bit 3; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6);
 *   scales8  uint8 [K/16][N]: E4M3 bit patterns (bias 7, subnormals, no infinities), one per 16
 *            consecutive k of a column;
 *   tensor_scale: one fp32 per matrix;
 *   y[m][n] = fp16_rne(tensor_scale * sum_k x[m][k] * e2m1(q[k][n]) * e4m3(s[k/16][n])),
 *            fp32 accumulation. e2m1 * e4m3 is exact in fp16, so the dequantised weight is exact.
 * Acceptance bound per element, as for int4: |y - y_ref| <= 2^-10 |y_ref| + 2^-10 sum_k |x g w|.
 * Shapes: N % 32 == 0, K % 64 == 0, N <= 2^23, K <= 2^22 (K % 128 for the tensor-core tiles; the
 * CUDA-core GEMV takes M <= 8 for the other K). Errors as for w4a16_gemm; a non-finite
 * tensor_scale is W4A16_ERR_INVALID_ARG.
 */

/* Bytes of the repacked NVFP4 scale buffer: (K/16) * N * 2 (fp16); the repacked weights take
 * K * N / 2 bytes. 0 for an unsupported shape. */
size_t w4a16_repacked_nvfp4_scales_bytes(int N, int K);

/* One-time re-layout of canonical NVFP4 weights into the device layout: the weight words move as
 * in w4a16_repack but keep the canonical nibble order (byte i of a word = codes of k offsets 2i
 * and 2i+1); every E4M3 scale becomes the fp16 number of equal value (exact) in the tiled
 * [K/16][w_t] layout of w4a16_repack. Device pointers, 16-byte aligned, no overlaps. */
int w4a16_repack_nvfp4(const int32_t* qweight, const uint8_t* scales8, void* qweight_r, void* scales_r, int N, int K,
                       void* stream);

/* Exact inverse of w4a16_repack_nvfp4 (each fp16 scale back to its E4M3 pattern). */
int w4a16_unrepack_nvfp4(const void* qweight_r, const void* scales_r, int32_t* qweight, uint8_t* scales8, int N,
                         int K, void* stream);

/* y[M,N] = x[M,K] . dequant(W) for repacked NVFP4 weights; the same kernels, dispatcher and
 * plans as w4a16_gemm (x, y fp16 device buffers). */
int w4a16_gemm_nvfp4(const uint16_t* x, const void* qweight_r, const void* scales_r, float tensor_scale, uint16_t* y,
                     int M, int N, int K, void* stream);

/* As w4a16_gemm_nvfp4 with an explicit plan (the fields of w4a16_gemm_ex). */
int w4a16_gemm_nvfp4_ex(const uint16_t* x, const void* qweight_r, const void* scales_r, float tensor_scale,
                        uint16_t* y, int M, int N, int K, const w4a16_plan* plan, void* stream);

/* The automatic plan of w4a16_gemm_nvfp4 for this shape (host only). */
int w4a16_plan_for_nvfp4(int M, int N, int K, w4a16_plan* out);

/*
 * W4A8: int8 activations with the int4 weights of w4a16_repack ("Qwen3.8-27B at 764, 1,035 and
 * 1,623 tok/s" (ai.satyajit.si), section "Where the line bends": the MLP GEMMs run with int8
 * activations past the bend; the pages print no quantisation, so the reading is per-token
 * symmetric int8):
 *   sx[m]    = fl32(max_k |x[m][k]| / 127)               IEEE binary32 division, ties to even
 *   xq[m][k] = rne(fl32(x[m][k] / sx[m])), in [-127, 127]; 0 for every k when the row is all 0
 *   y[m][n]  = fp16_rne(sx[m] * sum_g s[g][n] * sum_{k in g} (q[k][n] - 8) * xq[m][k])
 * The group sums are exact integers (int32 dp4a in the GEMV for M <= 8); the tensor-core tiles
 * (M > 8) multiply the fp16 copy of xq (exact) by the fp16 W4A16 weights fp16_rne((q - 8) s) and
 * scale row m by sx[m] at the end. Acceptance bound per element: |y - y_ref| <= 2^-10 |y_ref| +
 * 2^-10 sum_k |sx xq (q - 8) s| (the weights' fp16 rounding on the tile path is within it). sm_103a
 * has no int8 tensor-core MMA, so W4A8 is not a faster tensor path on this GPU; its int8 arithmetic
 * pays in the CUDA-core GEMV.
 */

/* Per-token symmetric int8 quantisation of x (fp16 [M][K], device): writes xq (int8 [M][K]),
 * optionally xq_f16 (fp16 [M][K], the same integers; NULL to skip; the tensor-core path of
 * w4a16_gemm_w4a8 needs it) and sx (fp32 [M]). x must be finite. K % 8 == 0, M <= 2^20,
 * K <= 2^22. x, xq, xq_f16 16-byte aligned, sx 4-byte aligned, device pointers, no overlaps.
 * Asynchronous on `stream` (with programmatic dependent launch). Errors: INVALID_ARG, MISALIGNED,
 * UNSUPPORTED_SHAPE, CUDA. */
int w4a16_quantize_x_int8(const uint16_t* x, int8_t* xq, uint16_t* xq_f16, float* sx, int M, int K, void* stream);

/* y[M,N] (fp16, device) for int8 activations (xq, xq_f16, sx as written by w4a16_quantize_x_int8)
 * and repacked int4 weights (w4a16_repack, group `group`). The automatic plan takes the integer
 * GEMV for M <= 2, for M = 3 when its grid fits in one wave, and the tensor-core tiles otherwise
 * (w4a16_plan_for_w4a8 tells which); xq_f16 may be NULL when the plan is the GEMV
 * (W4A16_ERR_INVALID_ARG if the tiles would need it). Shapes and errors as w4a16_gemm. */
int w4a16_gemm_w4a8(const int8_t* xq, const uint16_t* xq_f16, const float* sx, const void* qweight_r,
                    const void* scales_r, uint16_t* y, int M, int N, int K, int group, void* stream);

/* As w4a16_gemm_w4a8 with an explicit plan (the fields of w4a16_gemm_ex). */
int w4a16_gemm_w4a8_ex(const int8_t* xq, const uint16_t* xq_f16, const float* sx, const void* qweight_r,
                       const void* scales_r, uint16_t* y, int M, int N, int K, int group, const w4a16_plan* plan,
                       void* stream);

/* w4a16_quantize_x_int8 then w4a16_gemm_w4a8 in one call (two kernels on `stream`, the GEMM with
 * programmatic dependent launch): writes xq, xq_f16 (may be NULL when the plan is the GEMV) and sx,
 * which stay valid for other GEMMs of the same x, and y. Outputs overlap neither each other nor an
 * input. Errors as the two calls. */
int w4a16_quantize_gemm_w4a8(const uint16_t* x, int8_t* xq, uint16_t* xq_f16, float* sx, const void* qweight_r,
                              const void* scales_r, uint16_t* y, int M, int N, int K, int group,
                              const w4a16_plan* plan, void* stream);

/* The automatic plan of w4a16_gemm_w4a8 for this shape (host only). */
int w4a16_plan_for_w4a8(int M, int N, int K, int group, w4a16_plan* out);

/* Describes the last GEMM this process launched (path, tile, split, grid) into buf (NUL
 * terminated, truncated to len). Host only. Returns W4A16_OK or INVALID_ARG. */
int w4a16_last_dispatch(char* buf, size_t len);

/*
 * Reads and clears the current device's status word, after the work queued on `stream` before the
 * call. Kernels set the word when a bounded wait runs out (W4A16_ERR_DEVICE_TIMEOUT) instead of
 * hanging; the CUDA context stays usable. The word is per DEVICE, not per stream: a timeout of a
 * kernel on any stream of the device is reported by the next read. The read and the clear are one
 * atomic exchange on the device (queued on `stream`), so a timeout recorded concurrently by a
 * kernel on another stream is never lost: it is either returned now or by the next call. The call
 * then synchronises `stream`. Returns W4A16_OK, W4A16_ERR_DEVICE_TIMEOUT, W4A16_ERR_BOUNDS (debug-bounds
 * build), or W4A16_ERR_CUDA if the launch, copy or synchronisation failed.
 */
int w4a16_device_status(void* stream);

/* Limit for every bounded wait inside the kernels, in nanoseconds (default 2e9; minimum 1e5).
 * Host-side setting applied to launches made after the call. */
int w4a16_set_wait_timeout_ns(uint64_t ns);

/*
 * Exercises the failure-reporting path without a fault: launches (asynchronously, on `stream`) a
 * one-warp kernel whose bounded wait can never complete (an mbarrier phase nothing arrives on),
 * using the kernels' own wait routine: mode 0 = the suspending wait, mode 1 = the polling wait.
 * The wait gives up after the current wait limit (w4a16_set_wait_timeout_ns), so a following
 * w4a16_device_status(stream) returns W4A16_ERR_DEVICE_TIMEOUT and clears it; the CUDA context
 * stays usable. (The pages' engine died of an allocation failure inside its GEMM: this library
 * reports failures as status codes instead.) Allocates nothing.
 * Errors: INVALID_ARG (mode not 0 or 1), CUDA (launch refused).
 */
int w4a16_selftest_wait_timeout(int mode, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
