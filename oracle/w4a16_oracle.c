/*
 * W4A16 GEMM oracle: a plain, slow, fp64 CPU statement of what the GPU path computes.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline
 * leg may load or run this code. The product path (libw4a16 and its Python binding) never
 * touches it, and this file shares no code, header or table with the CUDA sources.
 *
 * What is computed (each function below cites the passage it follows):
 *
 *   W4A16 ("weights stored in 4-bit, activations remain 16-bit"):
 *     "RTX 3090 Tested: Qwen's 381 tok/s Myth Busted" (kongchang.com), section
 *     "What Exactly Is This Stack".
 *   One weight read shared by B activation rows (y = x . W with x of B rows):
 *     "Qwen3.8-27B at 764, 1,035 and 1,623 tok/s" (ai.satyajit.si), section
 *     "One weight read, shared by every stream".
 *   Canonical packed format of the workload (the pages are silent on it; this is the plainest
 *   reading the workload definition gives):
 *     qweight int32 [K/8][N]: nibble j (bits 4j..4j+3, read as an unsigned 32-bit word) of
 *       qweight[k/8][n] is q[k][n] with j = k mod 8 (low nibble first);
 *     scales fp16 [K/G][N];
 *     w[k][n] = fp16_rne((q[k][n] - 8) * scales[k/G][n]);
 *     y[m][n] = sum_k x[m][k] * w[k][n], summed here in fp64 in ascending k.
 *   NVFP4 weights and int8 activations (W4A8): the sections of those names below.
 *
 * The fp16 codec is written out bit by bit (sign, exponent, mantissa, subnormals, overflow to
 * infinity, round-to-nearest-even); no compiler half type is used.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- fp16 codec (IEEE binary16) */

/* binary16 bits -> exact double. Subnormal: m * 2^-24; normal: (1024 + m) * 2^(e - 25). */
double w4o_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return sign ? -v : v;
}

/* double -> binary16 bits, one rounding to nearest, ties to even. NaN -> 0x7e00 (quiet). */
uint16_t w4o_double_to_half(double v) {
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    if (isnan(v)) return 0x7e00;
    double a = fabs(v);
    if (isinf(a)) return (uint16_t)(sign | 0x7c00);
    if (a == 0.0) return sign;
    int e2;
    frexp(a, &e2);           /* a = f * 2^e2, f in [0.5, 1)  =>  a in [2^(e2-1), 2^e2) */
    int ex = e2 - 1;         /* a in [2^ex, 2^(ex+1)) */
    if (ex < -14) ex = -14;  /* below the normal range the spacing stays 2^-24 */
    /* the spacing of binary16 values around a is 2^(ex-10); a / spacing is exact in double */
    double n = ldexp(a, 10 - ex);
    /* round n to an integer, ties to even, without relying on the FP rounding mode */
    double fl = floor(n);
    double diff = n - fl;
    double r;
    if (diff > 0.5)
        r = fl + 1.0;
    else if (diff < 0.5)
        r = fl;
    else
        r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    /* r * 2^(ex-10) is the rounded magnitude; r in [0, 2048] */
    if (r >= 2048.0) { /* carried into the next binade */
        r = 1024.0;
        ex += 1;
    }
    if (r < 1024.0) {
        /* only possible when ex == -14: subnormal (or zero), mantissa = r */
        return (uint16_t)(sign | (uint16_t)r);
    }
    int field = ex + 15;
    if (field >= 31) return (uint16_t)(sign | 0x7c00); /* overflow */
    return (uint16_t)(sign | (uint16_t)(field << 10) | (uint16_t)((int)r - 1024));
}

void w4o_half_to_double_array(const uint16_t* h, double* out, int64_t count) {
    for (int64_t i = 0; i < count; ++i) out[i] = w4o_half_to_double(h[i]);
}

void w4o_double_to_half_array(const double* v, uint16_t* out, int64_t count) {
    for (int64_t i = 0; i < count; ++i) out[i] = w4o_double_to_half(v[i]);
}

/* ---------------------------------------------------------------- canonical format */

/* q[k][n]: nibble (k mod 8) of qweight[k/8][n], the word taken as unsigned. */
int w4o_nibble(const int32_t* qweight, int N, int k, int n) {
    uint32_t word = (uint32_t)qweight[(size_t)(k / 8) * (size_t)N + (size_t)n];
    return (int)((word >> (4 * (k % 8))) & 0xFu);
}

/* w[k][n] = fp16_rne((q - 8) * s). (q - 8) * s has at most 4 + 11 significant bits, so the
 * double product is exact and w4o_double_to_half applies the only rounding. */
double w4o_weight(const int32_t* qweight, const uint16_t* scales, int N, int G, int k, int n) {
    int q = w4o_nibble(qweight, N, k, n);
    double s = w4o_half_to_double(scales[(size_t)(k / G) * (size_t)N + (size_t)n]);
    double prod = (double)(q - 8) * s;
    return w4o_half_to_double(w4o_double_to_half(prod));
}

void w4o_unpack(const int32_t* qweight, int K, int N, uint8_t* q_out) {
    for (int k = 0; k < K; ++k)
        for (int n = 0; n < N; ++n) q_out[(size_t)k * N + n] = (uint8_t)w4o_nibble(qweight, N, k, n);
}

void w4o_dequant(const int32_t* qweight, const uint16_t* scales, int K, int N, int G, double* w_out) {
    for (int k = 0; k < K; ++k)
        for (int n = 0; n < N; ++n) w_out[(size_t)k * N + n] = w4o_weight(qweight, scales, N, G, k, n);
}

static int shape_ok(int M, int N, int K, int G) {
    if (M < 0 || N <= 0 || K <= 0 || G <= 0) return 0;
    if (K % 8 != 0 || G % 8 != 0 || K % G != 0) return 0;
    return 1;
}

/* ---------------------------------------------------------------- the GEMM */

/* One output column n: w[:, n] is dequantised into col (K doubles), then every requested row m
 * is summed in ascending k. y and absy receive sum_k x*w and sum_k |x*w|. */
static void column_dot(const double* xrow, int K, const double* col, double* y, double* absy) {
    double acc = 0.0, aacc = 0.0;
    for (int k = 0; k < K; ++k) {
        double p = xrow[k] * col[k];
        acc += p;
        aacc += fabs(p);
    }
    *y = acc;
    *absy = aacc;
}

static void dequant_column(const int32_t* qweight, const uint16_t* scales, int N, int K, int G, int n,
                           double* col) {
    for (int k = 0; k < K; ++k) col[k] = w4o_weight(qweight, scales, N, G, k, n);
}

/* y[m][n] (fp64) for x given as double [M][K]. Rows of x are used as given. */
int w4o_gemm_xf64(const double* x, const int32_t* qweight, const uint16_t* scales, int M, int N, int K,
                  int G, double* y, double* absy, int nthreads) {
    if (!shape_ok(M, N, K, G)) return 1;
    if (nthreads < 1) nthreads = 1;
    int failed = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double* col = (double*)malloc(sizeof(double) * (size_t)K);
        if (!col) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 8)
#endif
            for (int n = 0; n < N; ++n) {
                dequant_column(qweight, scales, N, K, G, n, col);
                for (int m = 0; m < M; ++m)
                    column_dot(x + (size_t)m * K, K, col, &y[(size_t)m * N + n], &absy[(size_t)m * N + n]);
            }
            free(col);
        }
    }
    return failed ? 2 : 0;
}

/* y[m][n] for x given as fp16 bits [M][K]: x is decoded exactly to double, then as above. */
int w4o_gemm(const uint16_t* x, const int32_t* qweight, const uint16_t* scales, int M, int N, int K, int G,
             double* y, double* absy, int nthreads) {
    if (!shape_ok(M, N, K, G)) return 1;
    double* xd = (double*)malloc(sizeof(double) * ((size_t)M * K + 1));
    if (!xd) return 2;
    w4o_half_to_double_array(x, xd, (int64_t)M * K);
    int rc = w4o_gemm_xf64(xd, qweight, scales, M, N, K, G, y, absy, nthreads);
    free(xd);
    return rc;
}

/* The same sum for a list of (m, n) pairs only: used where the full product is too large. */
int w4o_gemm_sampled(const uint16_t* x, const int32_t* qweight, const uint16_t* scales, int M, int N, int K,
                     int G, const int64_t* ms, const int64_t* ns, int64_t count, double* y, double* absy,
                     int nthreads) {
    if (!shape_ok(M, N, K, G)) return 1;
    for (int64_t i = 0; i < count; ++i)
        if (ms[i] < 0 || ms[i] >= M || ns[i] < 0 || ns[i] >= N) return 1;
    if (nthreads < 1) nthreads = 1;
    int failed = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double* col = (double*)malloc(sizeof(double) * (size_t)K);
        double* xr = (double*)malloc(sizeof(double) * (size_t)K);
        if (!col || !xr) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t i = 0; i < count; ++i) {
                int m = (int)ms[i], n = (int)ns[i];
                dequant_column(qweight, scales, N, K, G, n, col);
                for (int k = 0; k < K; ++k) xr[k] = w4o_half_to_double(x[(size_t)m * K + k]);
                column_dot(xr, K, col, &y[i], &absy[i]);
            }
        }
        free(col);
        free(xr);
    }
    return failed ? 2 : 0;
}

/* ---------------------------------------------------------------- the device layout
 *
 * The one-time re-layout the GPU path streams from (a bijection of the canonical bytes). This is
 * the library's own format, stated here independently of the CUDA code.
 *
 * Columns are grouped in tiles of 128: tile t holds columns [128t, 128t + w_t) with
 * w_t = min(128, N - 128t) (N is a multiple of 32, so w_t is 32, 64, 96 or 128).
 *
 *   weights: tile t occupies the 4-byte words [16t*K, 16t*K + w_t*K/8) (a column holds K/8
 *            words; all earlier tiles are full). Inside it, column n (c = n - 128t) and k
 *            (block b = k/32, word w = (k mod 32)/8, j = k mod 8) address the word
 *            16t*K + (b*w_t + c)*4 + w, and q[k][n] sits in nibble position p of that word with
 *            p = 0,4,1,5,2,6,3,7 for j = 0..7 (positions 0..3 hold the even k, 4..7 the odd k).
 *   scales:  tile t occupies the elements [128t*(K/G), ...), laid out [K/G][w_t]:
 *            scales[g][n] sits at 128t*(K/G) + g*w_t + c.
 */
static const int kPosOfJ[8] = {0, 4, 1, 5, 2, 6, 3, 7};

static int layout_ok(int N, int K, int G) {
    return N > 0 && K > 0 && G > 0 && N % 32 == 0 && K % 32 == 0 && K % G == 0 && G % 8 == 0;
}

static size_t weight_word_index(int K, int N, int k, int n) {
    int t = n / 128, c = n % 128;
    int wt = N - 128 * t < 128 ? N - 128 * t : 128;
    int b = k / 32, w = (k % 32) / 8;
    return (size_t)16 * t * K + ((size_t)b * wt + c) * 4 + w;
}

static size_t scale_index(int K, int N, int G, int g, int n) {
    int t = n / 128, c = n % 128;
    int wt = N - 128 * t < 128 ? N - 128 * t : 128;
    return (size_t)128 * t * (K / G) + (size_t)g * wt + c;
}

int w4o_repack(const int32_t* qweight, const uint16_t* scales, int K, int N, int G, uint32_t* wr, uint16_t* sr) {
    if (!layout_ok(N, K, G)) return 1;
    size_t nwords = (size_t)N * K / 8;
    memset(wr, 0, nwords * sizeof(uint32_t));
    for (int k = 0; k < K; ++k) {
        for (int n = 0; n < N; ++n) {
            uint32_t q = (uint32_t)w4o_nibble(qweight, N, k, n);
            wr[weight_word_index(K, N, k, n)] |= q << (4 * kPosOfJ[k % 8]);
        }
    }
    for (int g = 0; g < K / G; ++g)
        for (int n = 0; n < N; ++n) sr[scale_index(K, N, G, g, n)] = scales[(size_t)g * N + n];
    return 0;
}

int w4o_unrepack(const uint32_t* wr, const uint16_t* sr, int K, int N, int G, int32_t* qweight, uint16_t* scales) {
    if (!layout_ok(N, K, G)) return 1;
    size_t nwords = (size_t)N * K / 8;
    memset(qweight, 0, nwords * sizeof(int32_t));
    for (int k = 0; k < K; ++k) {
        for (int n = 0; n < N; ++n) {
            uint32_t q = (wr[weight_word_index(K, N, k, n)] >> (4 * kPosOfJ[k % 8])) & 0xFu;
            uint32_t* dst = (uint32_t*)&qweight[(size_t)(k / 8) * N + n];
            *dst |= q << (4 * (k % 8));
        }
    }
    for (int g = 0; g < K / G; ++g)
        for (int n = 0; n < N; ++n) scales[(size_t)g * N + n] = sr[scale_index(K, N, G, g, n)];
    return 0;
}

/* ---------------------------------------------------------------- the dense layer's activation
 *
 * act[m][i] = silu(g) * u with g = gu[m][i], u = gu[m][I + i] and silu(g) = g / (1 + e^-g), in
 * double, plus its fp16 rounding: the activation between the fused gate+up projection and the down
 * projection of the 17,408-wide MLPs of "Qwen3.8-27B at 764, 1,035 and 1,623 tok/s"
 * (ai.satyajit.si), section "Where the line bends". The pages do not print the activation;
 * SwiGLU (gate columns first in the fused matrix) is the plainest reading for that model family. */
void w4o_silu_mul(const uint16_t* gu, int M, int I, double* act_exact, uint16_t* act_half) {
    for (int m = 0; m < M; ++m) {
        for (int i = 0; i < I; ++i) {
            const double g = w4o_half_to_double(gu[(size_t)m * 2 * I + i]);
            const double u = w4o_half_to_double(gu[(size_t)m * 2 * I + I + i]);
            const double v = g / (1.0 + exp(-g)) * u;
            act_exact[(size_t)m * I + i] = v;
            act_half[(size_t)m * I + i] = w4o_double_to_half(v);
        }
    }
}

int w4o_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

int w4o_has_openmp(void) {
#ifdef _OPENMP
    return 1;
#else
    return 0;
#endif
}

/* ---------------------------------------------------------------- NVFP4 weights
 *
 * The RTX 5090 runs of "Qwen3.8-27B at 764, 1,035 and 1,623 tok/s" (ai.satyajit.si), section
 * "One weight read, shared by every stream", store the weights as NVFP4; the pages print no
 * format. Reading taken (the published NVFP4 definition): every weight is a 4-bit E2M1 code, every
 * 16 consecutive weights along K share one E4M3 scale, and the tensor has one fp32 scale g.
 * Activations stay fp16 (the W4A16 contract of this library):
 *
 *   qweight int32 [K/8][N]: nibble (k mod 8) of qweight[k/8][n] is the E2M1 code of w[k][n]
 *     (the container of the 4-bit format above);
 *   scales8 uint8 [K/16][N]: E4M3 bit patterns;
 *   w[k][n] = e2m1(code) * e4m3(scales8[k/16][n])   (at most 2 x 4 significant bits: exact in
 *     double, and exact in fp16 for every finite scale);
 *   y[m][n] = g * sum_k x[m][k] * w[k][n], summed here in fp64 in ascending k.
 */

/* E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0; exponent 0 is subnormal
 * (m * 2^-1). Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double w4o_e2m1_to_double(int code) {
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* E4M3: sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0; exponent 0 is subnormal
 * (m/8 * 2^-6); exponent 15 with mantissa 7 is NaN (no infinities). Largest finite value 448. */
double w4o_e4m3_to_double(uint8_t b) {
    int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp(m / 8.0, -6);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

void w4o_e4m3_to_double_array(const uint8_t* b, double* out, int64_t count) {
    for (int64_t i = 0; i < count; ++i) out[i] = w4o_e4m3_to_double(b[i]);
}

double w4o_weight_nvfp4(const int32_t* qweight, const uint8_t* scales8, int N, int k, int n) {
    return w4o_e2m1_to_double(w4o_nibble(qweight, N, k, n)) *
           w4o_e4m3_to_double(scales8[(size_t)(k / 16) * (size_t)N + (size_t)n]);
}

void w4o_dequant_nvfp4(const int32_t* qweight, const uint8_t* scales8, int K, int N, double* w_out) {
    for (int k = 0; k < K; ++k)
        for (int n = 0; n < N; ++n) w_out[(size_t)k * N + n] = w4o_weight_nvfp4(qweight, scales8, N, k, n);
}

/* y = g * sum_k x w and absy = |g| * sum_k |x w| (the tolerance scale of the effective weights
 * g * w), for x given as fp16 bits [M][K]. */
int w4o_gemm_nvfp4(const uint16_t* x, const int32_t* qweight, const uint8_t* scales8, double g, int M, int N,
                   int K, double* y, double* absy, int nthreads) {
    if (M < 0 || N <= 0 || K <= 0 || K % 16 != 0) return 1;
    if (nthreads < 1) nthreads = 1;
    double* xd = (double*)malloc(sizeof(double) * ((size_t)M * K + 1));
    if (!xd) return 2;
    w4o_half_to_double_array(x, xd, (int64_t)M * K);
    int failed = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double* col = (double*)malloc(sizeof(double) * (size_t)K);
        if (!col) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 8)
#endif
            for (int n = 0; n < N; ++n) {
                for (int k = 0; k < K; ++k) col[k] = w4o_weight_nvfp4(qweight, scales8, N, k, n);
                for (int m = 0; m < M; ++m) {
                    double s = 0.0, a = 0.0;
                    column_dot(xd + (size_t)m * K, K, col, &s, &a);
                    y[(size_t)m * N + n] = g * s;
                    absy[(size_t)m * N + n] = fabs(g) * a;
                }
            }
            free(col);
        }
    }
    free(xd);
    return failed ? 2 : 0;
}

/* The same for a list of (m, n) pairs. */
int w4o_gemm_nvfp4_sampled(const uint16_t* x, const int32_t* qweight, const uint8_t* scales8, double g, int M,
                           int N, int K, const int64_t* ms, const int64_t* ns, int64_t count, double* y,
                           double* absy) {
    if (M < 0 || N <= 0 || K <= 0 || K % 16 != 0) return 1;
    for (int64_t i = 0; i < count; ++i) {
        if (ms[i] < 0 || ms[i] >= M || ns[i] < 0 || ns[i] >= N) return 1;
        double s = 0.0, a = 0.0;
        for (int k = 0; k < K; ++k) {
            double p = w4o_half_to_double(x[(size_t)ms[i] * K + k]) *
                       w4o_weight_nvfp4(qweight, scales8, N, k, (int)ns[i]);
            s += p;
            a += fabs(p);
        }
        y[i] = g * s;
        absy[i] = fabs(g) * a;
    }
    return 0;
}

/* The library's NVFP4 device layout: the weight words sit where the int4 layout puts them
 * (weight_word_index) but keep the canonical nibble order (k mod 8 at nibble k mod 8), and each
 * E4M3 scale is stored as the fp16 number of equal value (exact: an E4M3 value has 4 significant
 * bits and lies within the fp16 range) at scale_index with a group of 16. */
int w4o_repack_nvfp4(const int32_t* qweight, const uint8_t* scales8, int K, int N, uint32_t* wr, uint16_t* sr) {
    if (!layout_ok(N, K, 16)) return 1;
    size_t nwords = (size_t)N * K / 8;
    memset(wr, 0, nwords * sizeof(uint32_t));
    for (int k = 0; k < K; ++k) {
        for (int n = 0; n < N; ++n) {
            uint32_t q = (uint32_t)w4o_nibble(qweight, N, k, n);
            wr[weight_word_index(K, N, k, n)] |= q << (4 * (k % 8));
        }
    }
    for (int g = 0; g < K / 16; ++g)
        for (int n = 0; n < N; ++n)
            sr[scale_index(K, N, 16, g, n)] = w4o_double_to_half(w4o_e4m3_to_double(scales8[(size_t)g * N + n]));
    return 0;
}

/* Inverse of w4o_repack_nvfp4. An fp16 scale maps back to the E4M3 pattern of equal value (the
 * positive pattern for zero); a value no E4M3 pattern has is an error (rc 2). */
int w4o_unrepack_nvfp4(const uint32_t* wr, const uint16_t* sr, int K, int N, int32_t* qweight, uint8_t* scales8) {
    if (!layout_ok(N, K, 16)) return 1;
    size_t nwords = (size_t)N * K / 8;
    memset(qweight, 0, nwords * sizeof(int32_t));
    for (int k = 0; k < K; ++k) {
        for (int n = 0; n < N; ++n) {
            uint32_t q = (wr[weight_word_index(K, N, k, n)] >> (4 * (k % 8))) & 0xFu;
            uint32_t* dst = (uint32_t*)&qweight[(size_t)(k / 8) * N + n];
            *dst |= q << (4 * (k % 8));
        }
    }
    for (int g = 0; g < K / 16; ++g) {
        for (int n = 0; n < N; ++n) {
            double v = w4o_half_to_double(sr[scale_index(K, N, 16, g, n)]);
            int found = -1;
            for (int b = 0; b < 256 && found < 0; ++b)
                if (w4o_e4m3_to_double((uint8_t)b) == v && !(v == 0.0 && b != 0)) found = b;
            if (found < 0) return 2;
            scales8[(size_t)g * N + n] = (uint8_t)found;
        }
    }
    return 0;
}

/* ---------------------------------------------------------------- W4A8: int8 activations
 *
 * "Qwen3.8-27B at 764, 1,035 and 1,623 tok/s" (ai.satyajit.si), section "Where the line bends",
 * runs the MLP GEMMs with int8 activations past the bend (a W4A8 path: 4-bit weights, 8-bit
 * activations), and the technobrother.ru news page on the same project names INT8 arithmetic;
 * neither prints the quantisation. Reading taken (the plainest one: per-token symmetric int8; the
 * weights are the W4A16 weights before their fp16 rounding, i.e. integer codes and group scales as
 * an integer GEMM consumes them):
 *
 *   amax[m]  = max_k |x[m][k]|                  (fp16 -> binary32, exact)
 *   sx[m]    = fl32(amax[m] / 127)              (one IEEE binary32 division, ties to even)
 *   xq[m][k] = rne(fl32(x[m][k] / sx[m]))       (binary32 division, then to the nearest integer,
 *                                                ties to even; clamped to [-127, 127], which the
 *                                                division never leaves); all 0 when amax[m] = 0
 *   y[m][n]  = sx[m] * sum_g scales[g][n] * sum_{k in group g} (q[k][n] - 8) * xq[m][k]
 *
 * The quantisation is a decision taken in floating point: it is written in binary32 exactly as
 * above so that any implementation taking the same binary32 steps reaches the same integers. The
 * group sums are integers, exact here in 64 bits; the rest is fp64.
 */
int w4o_quantize_x_int8(const uint16_t* x, int M, int K, int8_t* xq, float* sx) {
    if (M < 0 || K <= 0) return 1;
    for (int m = 0; m < M; ++m) {
        const uint16_t* row = x + (size_t)m * K;
        float amax = 0.0f;
        for (int k = 0; k < K; ++k) {
            float v = fabsf((float)w4o_half_to_double(row[k]));
            if (v > amax) amax = v;
        }
        float s = amax / 127.0f;
        sx[m] = s;
        for (int k = 0; k < K; ++k) {
            int v = 0;
            if (amax > 0.0f) {
                float r = (float)w4o_half_to_double(row[k]) / s;
                float t = nearbyintf(r);
                if (t > 127.0f) t = 127.0f;
                if (t < -127.0f) t = -127.0f;
                v = (int)t;
            }
            xq[(size_t)m * K + k] = (int8_t)v;
        }
    }
    return 0;
}

/* One output column n for the rows listed in ms (count rows): the codes of column n are unpacked
 * once into qcol (K ints), then per row and group the exact integer sum and its absolute value. */
static void w4a8_column(const int8_t* xq, const float* sx, const uint16_t* scales, int N, int K, int G,
                        const int* qcol, int n, int m, double* y, double* absy) {
    double acc = 0.0, aacc = 0.0;
    for (int g = 0; g < K / G; ++g) {
        int64_t isum = 0, iabs = 0;
        for (int k = g * G; k < (g + 1) * G; ++k) {
            const int64_t d = (int64_t)(qcol[k] - 8) * (int64_t)xq[(size_t)m * K + k];
            isum += d;
            iabs += d < 0 ? -d : d;
        }
        const double s = w4o_half_to_double(scales[(size_t)g * (size_t)N + (size_t)n]);
        acc += s * (double)isum;
        aacc += fabs(s) * (double)iabs;
    }
    const double sxm = (double)sx[m];
    *y = sxm * acc;
    *absy = fabs(sxm) * aacc;
}

/* y[m][n] and absy[m][n] = sum_k |(sx[m] xq[m][k]) (q[k][n] - 8) scales[k/G][n]| (the tolerance
 * scale, with the dequantised activations and unrounded weights) for every m, n. */
int w4o_gemm_w4a8(const int8_t* xq, const float* sx, const int32_t* qweight, const uint16_t* scales, int M, int N,
                  int K, int G, double* y, double* absy, int nthreads) {
    if (M < 0 || N <= 0 || K <= 0 || G <= 0 || K % G != 0 || K % 8 != 0) return 1;
    if (nthreads < 1) nthreads = 1;
    int failed = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(nthreads)
#endif
    {
        int* qcol = (int*)malloc(sizeof(int) * (size_t)K);
        if (!qcol) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 8)
#endif
            for (int n = 0; n < N; ++n) {
                for (int k = 0; k < K; ++k) qcol[k] = w4o_nibble(qweight, N, k, n);
                for (int m = 0; m < M; ++m) {
                    const size_t at = (size_t)m * (size_t)N + (size_t)n;
                    w4a8_column(xq, sx, scales, N, K, G, qcol, n, m, y + at, absy + at);
                }
            }
            free(qcol);
        }
    }
    return failed ? 2 : 0;
}

/* The same for a list of (m, n) pairs. */
int w4o_gemm_w4a8_sampled(const int8_t* xq, const float* sx, const int32_t* qweight, const uint16_t* scales, int M,
                          int N, int K, int G, const int64_t* ms, const int64_t* ns, int64_t count, double* y,
                          double* absy) {
    if (M < 0 || N <= 0 || K <= 0 || G <= 0 || K % G != 0 || K % 8 != 0) return 1;
    int* qcol = (int*)malloc(sizeof(int) * (size_t)K);
    if (!qcol) return 2;
    for (int64_t i = 0; i < count; ++i) {
        if (ms[i] < 0 || ms[i] >= M || ns[i] < 0 || ns[i] >= N) {
            free(qcol);
            return 1;
        }
        for (int k = 0; k < K; ++k) qcol[k] = w4o_nibble(qweight, N, k, (int)ns[i]);
        w4a8_column(xq, sx, scales, N, K, G, qcol, (int)ns[i], (int)ms[i], &y[i], &absy[i]);
    }
    free(qcol);
    return 0;
}
