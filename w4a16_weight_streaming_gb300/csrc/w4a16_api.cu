// C-ABI entry points of libw4a16 (declared in include/w4a16.h): argument checks, the per-shape
// dispatcher, and the per-device status word. Allocates nothing.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <cmath>
#include <mutex>
#include <string>
#include <tuple>

#include "common.cuh"
#include "internal.h"
#include "w4a16.h"

namespace w4a16 {

// The device state: a status word per device, set by kernels whose bounded waits ran out, and
// the word w4a16_device_status copies its value through (read and cleared in one atomic step).
__device__ unsigned g_status_word;
__device__ unsigned g_status_taken;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    unsigned* status = nullptr;
    unsigned* taken = nullptr;
    int sm_count = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
std::atomic<uint64_t> g_timeout_ns{2000000000ull};
char g_last[320] = "none";

// Resolves (once per device, with that device current) the status word's device address and
// the SM count. Returns false if the runtime refuses.
bool device_info(DeviceInfo* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        void* p = nullptr;
        void* t = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return false;
        if (cudaGetSymbolAddress(&t, g_status_taken) != cudaSuccess) return false;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
        d.status = static_cast<unsigned*>(p);
        d.taken = static_cast<unsigned*>(t);
        d.sm_count = sms;
        d.ready = true;
    }
    *out = d;
    return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Rejects pointers the runtime knows to be host memory (pageable host pointers are unknown to
// it and are reported as unregistered; those cannot be told apart from device pointers of
// another runtime and pass).
bool is_host_pointer(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

// True for pointers the runtime knows to be device (or managed) memory.
bool is_device_pointer(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

int check_matrix_shape(int N, int K, int G) {
    if (N <= 0 || K <= 0 || G <= 0) return W4A16_ERR_INVALID_ARG;
    if (N % 32 != 0 || K % 64 != 0 || G % 32 != 0 || K % G != 0) return W4A16_ERR_UNSUPPORTED_SHAPE;
    if (N > (1 << 23) || K > (1 << 22)) return W4A16_ERR_UNSUPPORTED_SHAPE;
    return W4A16_OK;
}

// NVFP4 weights: the same limits, with the format's fixed block of 16 rows per scale.
int check_matrix_shape_nvfp4(int N, int K) {
    if (N <= 0 || K <= 0) return W4A16_ERR_INVALID_ARG;
    if (N % 32 != 0 || K % 64 != 0) return W4A16_ERR_UNSUPPORTED_SHAPE;
    if (N > (1 << 23) || K > (1 << 22)) return W4A16_ERR_UNSUPPORTED_SHAPE;
    return W4A16_OK;
}
constexpr int kNvfp4Block = 16;

// ----------------------------------------------------------------------------- dispatcher
struct Choice {
    int path;
    TcConfig tc;
    int gemv_split;
    int gemv_unroll = 4;  // 32-k blocks in flight per warp (fp16 GEMV)
};

// Split along K for the CUDA-core GEMV: enough 128-thread CTAs to cover every SM about four
// times over (measured best for the decode shapes), each keeping at least 16 blocks of 32 k.
int gemv_pick_split(int M, int N, int K, int sm_count) {
    const int KB = K / 32;
    const int tiles = N / 32;
    int split = 2;
    while (split < 16 && tiles * split < 4 * sm_count && KB / (split * 2) >= 16) split *= 2;
    while (split < 16 && gemv_smem_bytes(M, N, K, split) > 96 * 1024) split *= 2;
    return std::min(split, std::max(1, KB));
}

// Split along K for the integer GEMV (one CTA per 128-column tile and K-slice): the largest power of
// two up to 16 whose grid still fits in one wave of resident CTAs, with at least two 32-k blocks per
// rank. Measured on GB300 at M = 1: 5120 x 34816 (272 tiles) 18.4 us at split 4 (one wave), 22.4 at
// 8 (1.8 waves); 17408 x 5120 (40 tiles) 16.0 us at 16, 22.1 at 8.
int gemv_w4a8_pick_split(int M, int N, int K, int sm_count) {
    const int64_t tiles = (N + 127) / 128;
    const int64_t slots = static_cast<int64_t>(gemv_w4a8_ctas_per_sm(M)) * sm_count;
    int split = 1;
    while (split < 16 && 2 * split <= K / 64 && tiles * 2 * split <= slots) split *= 2;
    return split;
}

constexpr size_t kGemvMaxSmem = 200 * 1024;  // the GEMV's dynamic shared memory limit

bool group_fits(int KC, int G) { return KC >= G ? KC % G == 0 : G % KC == 0; }

// Largest shared-memory ring that fits `budget` bytes for a tile shape.
int fill_stages(const TcConfig& base, int G, size_t budget, int max_stages) {
    TcConfig c = base;
    int best = 2;
    for (int s = 2; s <= max_stages; ++s) {
        c.stages = s;
        if (tc_smem_bytes(c, G) <= budget) best = s;
    }
    return best;
}

// MMA issuers: one thread issues a tcgen05.mma only every ~45-55 cycles, while an N = 16..32 MMA
// executes in 8-16; small tiles need several issuers, N >= 128 tiles are bound by the math.
int default_issuers(int m_tile) { return m_tile <= 64 ? 4 : m_tile <= 128 ? 2 : 1; }

int default_tmem_stages(int m_tile, int k_chunk, int issuers) {
    return std::min(4, (512 - issuers * m_tile) / (k_chunk / 2));
}

// Split along K that minimises (waves) x (stages of work per CTA + fixed cost) + a small cost per
// cluster rank. Waves use the device's cluster occupancy for each split (clusters must fit inside
// one GPC, so large clusters leave SMs idle); without a device, the SM count.
// CTAs of config c resident at once: the driver's cluster occupancy, or without a device an
// estimate from TMEM columns and shared memory per SM.
int resident_slots(const TcConfig& c, int G, int sm_count, bool have_device) {
    int slots = have_device ? tc_resident_ctas(c, G) : 0;
    if (slots <= 0) {
        const int per_sm =
            std::max(1, std::min(512 / tc_tmem_cols(c), static_cast<int>(233472 / (tc_smem_bytes(c, G) + 1024))));
        slots = (sm_count * per_sm / c.split) * c.split;
    }
    return slots;
}

int pick_split(const TcConfig& base, int M, int N, int K, int G, int sm_count, bool have_device) {
    const int tiles = ((N + 127) / 128) * ((M + base.m_tile - 1) / base.m_tile);
    const int C = K / base.k_chunk;
    double best = 1e30;
    int split = 1;
    for (int s = 1; s <= 16 && s <= C; ++s) {
        if (static_cast<int64_t>(tiles) * s > 0x7fffffffLL) break;  // the grid's x extent
        TcConfig c = base;
        c.split = s;
        const int slots = resident_slots(c, G, sm_count, have_device);
        if (slots <= 0) continue;
        const int ctas = tiles * s;
        const int waves = (ctas + slots - 1) / slots;
        const int per_cta = (C + s - 1) / s;
        // In stages of the CTA's own K loop. 128- and 256-row tiles (one CTA per SM), fitted to
        // GB300 timings at M = 128..1024: ~0.71 us per 128-k stage (256 rows), plus ~12 us per
        // wave (prologue, ring fill, epilogue) and a cluster reduction that grows with the split.
        const double cost = base.m_tile >= 128 ? static_cast<double>(waves) * (per_cta + 17.0 + s)
                                               : static_cast<double>(waves) * (per_cta + 2.0) + 0.25 * s;
        if (cost < best - 1e-9) {
            best = cost;
            split = s;
        }
    }
    return split;
}

// Work items (column tile x row tile) of the last, partial wave when config c runs unsplit; 0 when
// the items fill whole waves or fit in one.
int partial_wave_items(const TcConfig& c, int M, int N, int G, int sm_count, bool have_device) {
    TcConfig cw = c;  // the whole waves run at c.split (clusters of c.split CTAs per item)
    cw.tail_items = cw.tail_split = 0;
    const int items = ((N + 127) / 128) * ((M + c.m_tile - 1) / c.m_tile);
    const int per_wave = resident_slots(cw, G, sm_count, have_device) / c.split;
    return per_wave <= 0 || items <= per_wave ? 0 : items % per_wave;
}

// Whole waves of unsplit work items, then a second launch for the items of the last, partial wave,
// each split along K so that together they fill one wave: taken when pick_split's cost model (128-
// and 256-row tiles) rates it below the single launch. Measured on GB300 at M = 1024: 5120 x 5120
// 79.2 -> 56.6 us, 17408 x 5120 194.7 -> 144.5 us, 5120 x 7168 79.9 -> 67.7 us, 5120 x 34816
// 323.7 -> 304 us; the model's splits were within 3 % of the best forced one.
void pick_tail(TcConfig& c, int M, int N, int K, int G, int sm_count, bool have_device) {
    const int items = ((N + 127) / 128) * ((M + c.m_tile - 1) / c.m_tile);
    const int C = K / c.k_chunk;
    const int slots = resident_slots(c, G, sm_count, have_device);
    if (slots <= 0) return;
    const int waves = static_cast<int>((static_cast<int64_t>(items) * c.split + slots - 1) / slots);
    double best = static_cast<double>(waves) * ((C + c.split - 1) / c.split + 17.0 + c.split);
    int main_split = 0, tail_split = 0, tail_items = 0;
    // The whole waves run unsplit. (Split whole waves, which explicit plans may ask for, were rated
    // cheaper for 17408 x 5120 at M = 512, split 3 then a tail split 4: 95.0 -> 90.3 us alone, but the
    // dense-layer sweep step measured 1.717 -> 1.743 ms: the full tail wave leaves the next GEMM no
    // idle SMs to start on.)
    for (int s1 = 1; s1 <= 1; ++s1) {
        TcConfig cm = c;
        cm.split = s1;
        const int r = partial_wave_items(cm, M, N, G, sm_count, have_device);
        if (r <= 0) continue;
        const int full_waves = items / (resident_slots(cm, G, sm_count, have_device) / s1);
        for (int s = s1 + 1; s <= 16 && s <= C; ++s) {
            TcConfig ct = c;
            ct.split = s;
            if (r * s > resident_slots(ct, G, sm_count, have_device)) continue;  // the tail in one wave
            const double cost =
                full_waves * ((C + s1 - 1) / s1 + 17.0 + s1) + ((C + s - 1) / s + 17.0 + s);
            if (cost < best - 1e-9) {
                best = cost;
                main_split = s1;
                tail_split = s;
                tail_items = r;
            }
        }
    }
    if (tail_split > 0) {
        c.split = main_split;
        c.tail_items = tail_items;
        c.tail_split = tail_split;
    }
}

TcConfig tc_default(int M, int N, int K, int G, int sm_count, bool have_device) {
    TcConfig c;
    c.m_tile = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
    c.split = 1;
    // Wide matrices at small M (at least one 128-column tile per SM): half-size CTAs, two per SM,
    // whose stages interleave (measured ~6% faster on 5120 x 34816); narrower ones keep the
    // 16-warp CTA, whose deeper K chunks suit their split-K.
    if (c.m_tile <= 64 && (N + 127) / 128 >= sm_count && K % 128 == 0 && group_fits(128, G)) {
        c.k_chunk = 128;
        c.dequant_warps = 8;
        c.issuers = c.m_tile <= 32 ? 4 : 2;
        c.tmem_stages = std::min(4, (256 - c.issuers * c.m_tile) / (c.k_chunk / 2));
        c.stages = fill_stages(c, G, 110 * 1024, 8);
        c.split = pick_split(c, M, N, K, G, sm_count, have_device);
        return c;
    }
    const bool kc256 = c.m_tile <= 64 && K % 256 == 0 && group_fits(256, G);
    c.k_chunk = kc256 ? 256 : 128;
    c.issuers = default_issuers(c.m_tile);
    c.dequant_warps = 16;
    c.tmem_stages = default_tmem_stages(c.m_tile, c.k_chunk, c.issuers);
    c.stages = fill_stages(c, G, 225 * 1024, 8);
    c.split = pick_split(c, M, N, K, G, sm_count, have_device);
    if (c.m_tile >= 128) pick_tail(c, M, N, K, G, sm_count, have_device);
    return c;
}

int resolve_plan_uncached(int M, int N, int K, int G, const w4a16_plan* plan, int sm_count, bool have_device,
                          Choice* out, bool w4a8);

// Automatic plans are resolved once per (device, M, N, K, group, activation type) and cached: the
// resolution queries the driver's cluster occupancy for every candidate split.
std::map<std::tuple<int, int, int, int, int, int>, Choice> g_plan_cache;

// W4A16_PLAN: an override of every automatic plan, read once per process. Its value is
// "field=value[,field=value...]" with the w4a16_plan field names, e.g. "path=2,m_tile=64,split_k=3",
// no spaces. A malformed value fails every automatic call with INVALID_ARG instead of being ignored.
struct EnvPlan {
    bool present = false;
    bool valid = true;
    w4a16_plan plan = {};
};

const EnvPlan& env_plan() {
    static const EnvPlan e = [] {
        EnvPlan r;
        const char* v = std::getenv("W4A16_PLAN");
        if (!v || !*v) return r;
        r.present = true;
        const std::string s(v);
        size_t pos = 0;
        while (r.valid && pos <= s.size()) {
            size_t end = s.find(',', pos);
            if (end == std::string::npos) end = s.size();
            const std::string item = s.substr(pos, end - pos);
            const size_t eq = item.find('=');
            const std::string key = eq == std::string::npos ? item : item.substr(0, eq);
            const std::string val = eq == std::string::npos ? std::string() : item.substr(eq + 1);
            char* stop = nullptr;
            const long n = val.empty() ? -1 : std::strtol(val.c_str(), &stop, 10);
            int* field = key == "path"            ? &r.plan.path
                         : key == "split_k"       ? &r.plan.split_k
                         : key == "m_tile"        ? &r.plan.m_tile
                         : key == "k_chunk"       ? &r.plan.k_chunk
                         : key == "stages"        ? &r.plan.stages
                         : key == "tmem_stages"   ? &r.plan.tmem_stages
                         : key == "mma_issuers"   ? &r.plan.mma_issuers
                         : key == "clusters"      ? &r.plan.clusters
                         : key == "dequant_warps" ? &r.plan.dequant_warps
                         : key == "tail_split"    ? &r.plan.tail_split
                                                  : nullptr;
            if (!field || n < 0 || n > 4096 || (stop && *stop != '\0')) {
                r.valid = false;
                break;
            }
            *field = static_cast<int>(n);
            pos = end + 1;
        }
        return r;
    }();
    return e;
}

// (w4a8: int8 activations; the GEMV path is then the integer GEMV of w4a8.cu.)
int resolve_plan(int M, int N, int K, int G, const w4a16_plan* plan, int sm_count, bool have_device, Choice* out,
                 bool w4a8 = false) {
    bool automatic = plan == nullptr || (plan->path == 0 && plan->split_k == 0 && plan->m_tile == 0 &&
                                         plan->k_chunk == 0 && plan->stages == 0 && plan->tmem_stages == 0 &&
                                         plan->mma_issuers == 0 && plan->clusters == 0 && plan->dequant_warps == 0 &&
                                         plan->tail_split == 0);
    if (automatic && env_plan().present) {
        if (!env_plan().valid) return W4A16_ERR_INVALID_ARG;
        plan = &env_plan().plan;
        automatic = false;
    }
    if (!automatic || !have_device) return resolve_plan_uncached(M, N, K, G, plan, sm_count, have_device, out, w4a8);
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(dev, M, N, K, G, w4a8 ? 1 : 0);
    {
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_plan_cache.find(key);
        if (it != g_plan_cache.end()) {
            *out = it->second;
            return W4A16_OK;
        }
    }
    const int rc = resolve_plan_uncached(M, N, K, G, plan, sm_count, have_device, out, w4a8);
    if (rc == W4A16_OK) {
        std::lock_guard<std::mutex> lock(g_mu);
        if (g_plan_cache.size() < 4096) g_plan_cache[key] = *out;
    }
    return rc;
}

int resolve_plan_uncached(int M, int N, int K, int G, const w4a16_plan* plan, int sm_count, bool have_device,
                          Choice* out, bool w4a8) {
    w4a16_plan p = {};
    if (plan) p = *plan;
    if (p.path < 0 || p.path > 2) return W4A16_ERR_INVALID_ARG;
    int path = p.path;
    if (path == W4A16_PATH_AUTO && w4a8) {
        // int8 activations, measured on GB300 (the four dense-layer matrices): the integer GEMV is
        // faster than the tiles at one and two rows on every matrix (5120 x 34816 at M = 2: 21.0
        // against 34.0 us); at three rows only while its grid fits in one wave at 5 CTAs per SM
        // (17408 x 5120: 19.2 against 21.6 us; 5120 x 7168, with 896 CTAs, loses); from four rows
        // the tiles. The tiles need whole 128-k stages.
        const bool tc_ok = K % 128 == 0 && group_fits(128, G);
        if (M <= 2) {
            path = W4A16_PATH_GEMV;
        } else if (M == 3) {
            const int64_t ctas = static_cast<int64_t>((N + 127) / 128) * gemv_w4a8_pick_split(M, N, K, sm_count);
            path = ctas <= 5 * static_cast<int64_t>(sm_count) ? W4A16_PATH_GEMV : W4A16_PATH_TC;
        } else {
            path = W4A16_PATH_TC;
        }
        if (path == W4A16_PATH_TC && !tc_ok && M <= kGemvMaxM) path = W4A16_PATH_GEMV;
        if (path == W4A16_PATH_GEMV && tc_ok && gemv_w4a8_smem_bytes(M, K, 16) > kGemvMaxSmem) path = W4A16_PATH_TC;
    } else if (path == W4A16_PATH_AUTO) {
        // Measured on GB300: the CUDA-core GEMV streams faster than the tensor-core tiles for one
        // activation row; from 3 rows on the tcgen05 tiles.
        // At two rows the GEMV wins only on the smaller matrices (5120 x 5120, 5120 x 7168); on
        // 5120 x 34816 and 17408 x 5120 the tiles are 1-2 us faster.
        const bool small = static_cast<int64_t>(K) * N < (int64_t{64} << 20);
        path = (M == 1 || (M == 2 && small)) ? W4A16_PATH_GEMV : W4A16_PATH_TC;
        // The tile kernels run whole 128-k stages and stage whole scale groups per stage; a K that
        // is not a multiple of 128, or a group that neither divides nor is a multiple of 128
        // (96, 160, ...), goes to the GEMV, which works in 32-k rows with one scale each.
        const bool tc_ok = K % 128 == 0 && group_fits(128, G);
        if (path == W4A16_PATH_TC && !tc_ok && M <= kGemvMaxM) path = W4A16_PATH_GEMV;
        // The GEMV stages its K-slice of x in shared memory: for very long K (even at the largest
        // split) the tiles, which stream x per stage, take over when they can.
        if (path == W4A16_PATH_GEMV && tc_ok && gemv_smem_bytes(M, N, K, 16) > kGemvMaxSmem) path = W4A16_PATH_TC;
    }
    out->path = path;
    if (path == W4A16_PATH_GEMV) {
        if (M > kGemvMaxM) return W4A16_ERR_UNSUPPORTED_SHAPE;
        int split = p.split_k > 0 ? p.split_k
                    : w4a8 ? gemv_w4a8_pick_split(M, N, K, sm_count)
                           : gemv_pick_split(M, N, K, sm_count);
        if (split < 1 || split > 16 || split > K / 32) return W4A16_ERR_UNSUPPORTED_SHAPE;
        const size_t smem = w4a8 ? gemv_w4a8_smem_bytes(M, K, split) : gemv_smem_bytes(M, N, K, split);
        if (smem > kGemvMaxSmem) return W4A16_ERR_UNSUPPORTED_SHAPE;
        out->gemv_split = split;
        out->gemv_unroll = 4;
        // fp16 GEMV at one or two rows: 8 blocks in flight per warp when the grid still fits in one
        // wave of that kernel (it holds more registers: 5 CTAs per SM against 9), so that short
        // K-slices take fewer load round trips. Measured on GB300 at M = 1: 5120 x 5120 (640 CTAs)
        // 7.78 -> 7.30 us, 17408 x 5120 (640) 17.33 -> 16.78 us, at M = 2 5120 x 5120 9.3 -> 8.9 us;
        // 5120 x 7168 (896 CTAs, two waves) 8.70 -> 11.29 us, which therefore keeps 4.
        // At one row with an automatic split, a smaller split whose grid fits that wave is taken when
        // there is one above 2 (5120 x 7168: split 4, 896 CTAs, 8.69 us -> split 3, 672 CTAs, 8.28 us).
        if (!w4a8 && M <= 2) {
            const int64_t slices = N / 32;
            const int slots = have_device ? gemv_resident_ctas(M, 8, smem, sm_count) : 5 * sm_count;
            if (slots > 0 && split * slices <= slots) {
                out->gemv_unroll = 8;
            } else if (slots > 0 && M == 1 && p.split_k <= 0) {
                for (int s = split - 1; s > 2; --s) {
                    if (s * slices > slots) continue;
                    const size_t smem_s = gemv_smem_bytes(M, N, K, s);
                    const int slots_s = have_device ? gemv_resident_ctas(M, 8, smem_s, sm_count) : 5 * sm_count;
                    if (smem_s <= kGemvMaxSmem && slots_s > 0 && s * slices <= slots_s) {
                        out->gemv_split = s;
                        out->gemv_unroll = 8;
                    }
                    break;
                }
            }
        }
        return W4A16_OK;
    }
    TcConfig c = tc_default(M, N, K, G, sm_count, have_device);
    const bool custom = p.m_tile > 0 || p.k_chunk > 0 || p.stages > 0 || p.split_k > 0 || p.tmem_stages > 0 ||
                        p.mma_issuers > 0 || p.dequant_warps > 0;
    if (custom) {
        if (p.m_tile > 0) c.m_tile = p.m_tile;
        if (p.k_chunk > 0) {
            c.k_chunk = p.k_chunk;
        } else {
            if (c.m_tile > 64) c.k_chunk = 128;
            // shrink the stage until every cluster rank gets at least one stage
            if (p.split_k > 0 && K / c.k_chunk < p.split_k) c.k_chunk = 128;
        }
        c.dequant_warps = p.dequant_warps > 0 ? p.dequant_warps : 16;
        if (c.dequant_warps == 8) {
            // two CTAs per SM: half the TMEM and at most ~110 KB of shared memory each
            if (p.k_chunk <= 0) c.k_chunk = 128;
            c.issuers = p.mma_issuers > 0 ? p.mma_issuers : (c.m_tile <= 32 ? 4 : 2);
            c.tmem_stages = p.tmem_stages > 0 ? p.tmem_stages
                                              : std::min(4, (256 - c.issuers * c.m_tile) / (c.k_chunk / 2));
            c.stages = p.stages > 0 ? p.stages : fill_stages(c, G, 110 * 1024, 8);
        } else {
            c.issuers = p.mma_issuers > 0 ? p.mma_issuers : default_issuers(c.m_tile);
            c.tmem_stages = p.tmem_stages > 0 ? p.tmem_stages : default_tmem_stages(c.m_tile, c.k_chunk, c.issuers);
            c.stages = p.stages > 0 ? p.stages : fill_stages(c, G, 225 * 1024, 8);
        }
        c.split = p.split_k > 0 ? p.split_k : std::min(pick_split(c, M, N, K, G, sm_count, have_device), K / c.k_chunk);
        c.tail_items = c.tail_split = 0;
    }
    if (p.tail_split != 0) {  // the last partial wave's items as a second launch, split tail_split ways
        if (p.tail_split < 2 || p.tail_split > 16) return W4A16_ERR_INVALID_ARG;
        c.split = p.split_k > 0 ? p.split_k : 1;
        c.tail_items = partial_wave_items(c, M, N, G, sm_count, have_device);
        c.tail_split = c.tail_items > 0 ? p.tail_split : 0;
    }
    // Unsplit 128- and 256-row tiles (one CTA per SM) with more work items than resident CTAs: a
    // persistent grid, one CTA per slot taking every slots-th item, so that each CTA's copies for
    // its next item overlap the MMAs and epilogue of the current one instead of a new wave's ramp.
    // Measured on GB300 (5120 x 34816): M = 256 80.2 -> 77.4 us, M = 512 160.0 -> 151.3 us, M = 1024
    // 300 -> 282 us.
    c.persist_ctas = c.m_tile >= 128 && c.split == 1 ? resident_slots(c, G, sm_count, have_device) : 0;
    if (!tc_config_valid(c, M, N, K, G)) return W4A16_ERR_UNSUPPORTED_SHAPE;
    out->tc = c;
    return W4A16_OK;
}

}  // namespace
}  // namespace w4a16

namespace w4a16 {
namespace {

// A one-warp kernel whose bounded wait can never complete: nothing arrives on its mbarrier. The
// wait gives up after `timeout_ns`, records kErrTimeout in the status word and the kernel returns.
// mode 0: the suspending wait (mbar_wait); mode 1: the polling wait (mbar_spin).
__global__ void wait_timeout_selftest_kernel(unsigned* status, uint64_t timeout_ns, int mode) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) {
        if (mode == 0)
            mbar_wait(b, 0, &abort_flag, timeout_ns, status);
        else
            mbar_spin(b, 0, &abort_flag, timeout_ns, status);
    }
    __syncwarp();
}

// Moves the status word into `taken` and clears it in one atomic exchange, so that a timeout
// recorded concurrently by a kernel on another stream is either taken now or left for the next read.
__global__ void take_status_kernel(unsigned* status, unsigned* taken) { *taken = atomicExch(status, 0u); }

}  // namespace
}  // namespace w4a16

using namespace w4a16;

namespace w4a16 {
namespace {

// Every argument check of a GEMM on device buffers, then the plan; launches nothing.
// (nvfp4: NVFP4 weights, group = 16.)
int prepare_gemm(const uint16_t* x, const void* qweight_r, const void* scales_r, uint16_t* y, int M, int N, int K,
                 int group, const w4a16_plan* plan, DeviceInfo* d, Choice* ch, bool nvfp4 = false) {
    if (!x || !qweight_r || !scales_r || !y) return W4A16_ERR_INVALID_ARG;
    if (M <= 0) return W4A16_ERR_INVALID_ARG;
    const int sh = nvfp4 ? check_matrix_shape_nvfp4(N, K) : check_matrix_shape(N, K, group);
    if (sh != W4A16_OK) return sh;
    if (M > (1 << 20)) return W4A16_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(x) || !aligned16(qweight_r) || !aligned16(scales_r) || !aligned16(y)) return W4A16_ERR_MISALIGNED;
    const size_t xb = static_cast<size_t>(M) * K * 2, yb = static_cast<size_t>(M) * N * 2;
    const size_t qb = static_cast<size_t>(N) * K / 2, sb = static_cast<size_t>(K / group) * N * 2;
    if (overlaps(x, xb, y, yb) || overlaps(qweight_r, qb, y, yb) || overlaps(scales_r, sb, y, yb))
        return W4A16_ERR_INVALID_ARG;
    if (is_host_pointer(x) || is_host_pointer(qweight_r) || is_host_pointer(scales_r) || is_host_pointer(y))
        return W4A16_ERR_INVALID_ARG;
    if (!device_info(d)) return W4A16_ERR_CUDA;
    return resolve_plan(M, N, K, group, plan, d->sm_count, true, ch);
}

// W4A8 (sx not null): x is the fp16 copy of the int8 activations (tile path), xq the int8 ones
// (GEMV path) and sx their per-token scales.
int launch_gemm(const Choice& ch, const uint16_t* x, const void* qweight_r, const void* scales_r, uint16_t* y, int M,
                int N, int K, int group, const DeviceInfo& d, void* stream, bool nvfp4 = false,
                float tensor_scale = 1.0f, const int8_t* xq = nullptr, const float* sx = nullptr) {
    LaunchCtx ctx;
    ctx.stream = static_cast<cudaStream_t>(stream);
    ctx.status = d.status;
    ctx.timeout_ns = g_timeout_ns.load();
    ctx.sm_count = d.sm_count;
    ctx.nvfp4 = nvfp4 ? 1 : 0;
    ctx.tensor_scale = tensor_scale;
    ctx.row_scale = sx;
    const char* fmt = nvfp4 ? " weights=nvfp4" : sx != nullptr ? " activations=int8" : "";
    cudaError_t e;
    char desc[256];
    if (ch.path == W4A16_PATH_GEMV) {
        if (sx != nullptr)
            e = launch_gemv_w4a8(xq, sx, static_cast<const uint32_t*>(qweight_r), static_cast<const uint16_t*>(scales_r),
                                 y, M, N, K, group, ch.gemv_split, ctx);
        else
            e = launch_gemv(x, static_cast<const uint32_t*>(qweight_r), static_cast<const uint16_t*>(scales_r), y, M, N,
                            K, group, ch.gemv_split, ch.gemv_unroll, ctx);
        const long long ctas = static_cast<long long>(ch.gemv_split) * (sx != nullptr ? (N + 127) / 128 : N / 32);
        snprintf(desc, sizeof(desc), "path=gemv M=%d N=%d K=%d group=%d split_k=%d grid=(%lld,1,1) block=128%s%s", M,
                 N, K, group, ch.gemv_split, ctas, sx == nullptr && ch.gemv_unroll == 8 ? " unroll=8" : "", fmt);
    } else {
        const long long items = static_cast<long long>((N + 127) / 128) * ((M + ch.tc.m_tile - 1) / ch.tc.m_tile);
        const long long main_items = items - ch.tc.tail_items;
        const bool persistent = ch.tc.split == 1 && ch.tc.persist_ctas > 0 && main_items > ch.tc.persist_ctas;
        char tail[80] = "";
        if (ch.tc.tail_items > 0)
            snprintf(tail, sizeof(tail), " tail_items=%d tail_split=%d tail_grid=(%lld,1,1)", ch.tc.tail_items,
                     ch.tc.tail_split, static_cast<long long>(ch.tc.tail_items) * ch.tc.tail_split);
        e = launch_tc(x, static_cast<const uint32_t*>(qweight_r), static_cast<const uint16_t*>(scales_r), y, M, N, K,
                      group, ch.tc, ctx);
        snprintf(desc, sizeof(desc),
                 "path=tc M=%d N=%d K=%d group=%d m_tile=%d k_chunk=%d stages=%d tmem_stages=%d issuers=%d "
                 "dequant_warps=%d split_k=%d grid=(%lld,1,1)%s%s tmem_cols=%d smem=%zu%s",
                 M, N, K, group, ch.tc.m_tile, ch.tc.k_chunk, ch.tc.stages, ch.tc.tmem_stages, ch.tc.issuers,
                 ch.tc.dequant_warps, ch.tc.split,
                 persistent ? static_cast<long long>(ch.tc.persist_ctas) : ch.tc.split * main_items,
                 persistent ? " persistent" : "", tail, tc_tmem_cols(ch.tc), tc_smem_bytes(ch.tc, group), fmt);
    }
    {
        std::lock_guard<std::mutex> lock(g_mu);
        snprintf(g_last, sizeof(g_last), "%s%s", desc, e == cudaSuccess ? "" : " (launch failed)");
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return W4A16_ERR_CUDA;
    }
    return W4A16_OK;
}

}  // namespace
}  // namespace w4a16

extern "C" {

int w4a16_version(void) { return 300; }

int w4a16_debug_bounds(void) {
#ifdef W4A16_DEBUG_BOUNDS
    return 1;
#else
    return 0;
#endif
}

const char* w4a16_status_string(int code) {
    switch (code) {
        case W4A16_OK: return "W4A16_OK";
        case W4A16_ERR_INVALID_ARG: return "W4A16_ERR_INVALID_ARG: null pointer, bad size, overlap or host pointer";
        case W4A16_ERR_UNSUPPORTED_SHAPE: return "W4A16_ERR_UNSUPPORTED_SHAPE: shape or plan outside the supported set";
        case W4A16_ERR_MISALIGNED: return "W4A16_ERR_MISALIGNED: a pointer is not 16-byte aligned";
        case W4A16_ERR_CUDA: return "W4A16_ERR_CUDA: the CUDA runtime refused the call";
        case W4A16_ERR_DEVICE_TIMEOUT: return "W4A16_ERR_DEVICE_TIMEOUT: a kernel gave up a bounded wait";
        case W4A16_ERR_BOUNDS: return "W4A16_ERR_BOUNDS: a kernel index check failed (debug-bounds build)";
        default: return "W4A16_ERR_UNKNOWN";
    }
}

size_t w4a16_repacked_qweight_bytes(int N, int K, int group) {
    if (check_matrix_shape(N, K, group) != W4A16_OK) return 0;
    return static_cast<size_t>(N) * static_cast<size_t>(K) / 2;
}

size_t w4a16_repacked_scales_bytes(int N, int K, int group) {
    if (check_matrix_shape(N, K, group) != W4A16_OK) return 0;
    return static_cast<size_t>(K / group) * static_cast<size_t>(N) * 2;
}

static int repack_common_checks(const void* a, const void* b, const void* c, const void* d, int N, int K, int group) {
    if (!a || !b || !c || !d) return W4A16_ERR_INVALID_ARG;
    const int sh = check_matrix_shape(N, K, group);
    if (sh != W4A16_OK) return sh;
    if (!aligned16(a) || !aligned16(b) || !aligned16(c) || !aligned16(d)) return W4A16_ERR_MISALIGNED;
    const size_t qb = static_cast<size_t>(N) * K / 2, sb = static_cast<size_t>(K / group) * N * 2;
    if (overlaps(a, qb, c, qb) || overlaps(a, qb, d, sb) || overlaps(b, sb, c, qb) || overlaps(b, sb, d, sb) ||
        overlaps(c, qb, d, sb))
        return W4A16_ERR_INVALID_ARG;
    if (is_host_pointer(a) || is_host_pointer(b) || is_host_pointer(c) || is_host_pointer(d))
        return W4A16_ERR_INVALID_ARG;
    return W4A16_OK;
}

int w4a16_repack(const int32_t* qweight, const uint16_t* scales, void* qweight_r, void* scales_r, int N, int K,
                 int group, void* stream) {
    const int rc = repack_common_checks(qweight, scales, qweight_r, scales_r, N, K, group);
    if (rc != W4A16_OK) return rc;
    DeviceInfo d;
    if (!device_info(&d)) return W4A16_ERR_CUDA;
    const cudaError_t e = launch_repack(qweight, scales, static_cast<uint32_t*>(qweight_r),
                                        static_cast<uint16_t*>(scales_r), N, K, group,
                                        static_cast<cudaStream_t>(stream), d.status);
    return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}

int w4a16_unrepack(const void* qweight_r, const void* scales_r, int32_t* qweight, uint16_t* scales, int N, int K,
                   int group, void* stream) {
    const int rc = repack_common_checks(qweight_r, scales_r, qweight, scales, N, K, group);
    if (rc != W4A16_OK) return rc;
    DeviceInfo d;
    if (!device_info(&d)) return W4A16_ERR_CUDA;
    const cudaError_t e = launch_unrepack(static_cast<const uint32_t*>(qweight_r),
                                          static_cast<const uint16_t*>(scales_r), qweight, scales, N, K, group,
                                          static_cast<cudaStream_t>(stream), d.status);
    return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}

static int plan_for_group(int M, int N, int K, int group, w4a16_plan* out, bool w4a8 = false);

int w4a16_plan_for(int M, int N, int K, int group, w4a16_plan* out) {
    if (!out) return W4A16_ERR_INVALID_ARG;
    if (M <= 0) return W4A16_ERR_INVALID_ARG;
    const int sh = check_matrix_shape(N, K, group);
    if (sh != W4A16_OK) return sh;
    if (M > (1 << 20)) return W4A16_ERR_UNSUPPORTED_SHAPE;
    return plan_for_group(M, N, K, group, out);
}

// The automatic plan of a checked shape (also for NVFP4 weights, group 16; w4a8: int8 activations).
static int plan_for_group(int M, int N, int K, int group, w4a16_plan* out, bool w4a8) {
    DeviceInfo d;
    const bool dev = device_info(&d);
    const int sms = dev ? d.sm_count : 152;
    Choice ch;
    const int rc = resolve_plan(M, N, K, group, nullptr, sms, dev, &ch, w4a8);
    if (rc != W4A16_OK) return rc;
    out->path = ch.path;
    out->clusters = 0;
    out->dequant_warps = 0;
    out->tail_split = ch.path == W4A16_PATH_TC ? ch.tc.tail_split : 0;
    if (ch.path == W4A16_PATH_GEMV) {
        out->split_k = ch.gemv_split;
        out->m_tile = out->k_chunk = out->stages = out->tmem_stages = out->mma_issuers = 0;
    } else {
        out->split_k = ch.tc.split;
        out->m_tile = ch.tc.m_tile;
        out->k_chunk = ch.tc.k_chunk;
        out->stages = ch.tc.stages;
        out->tmem_stages = ch.tc.tmem_stages;
        out->mma_issuers = ch.tc.issuers;
        out->dequant_warps = ch.tc.dequant_warps;
    }
    return W4A16_OK;
}

int w4a16_gemm_ex(const uint16_t* x, const void* qweight_r, const void* scales_r, uint16_t* y, int M, int N, int K,
                  int group, const w4a16_plan* plan, void* stream) {
    DeviceInfo d;
    Choice ch;
    const int rc = prepare_gemm(x, qweight_r, scales_r, y, M, N, K, group, plan, &d, &ch);
    if (rc != W4A16_OK) return rc;
    return launch_gemm(ch, x, qweight_r, scales_r, y, M, N, K, group, d, stream);
}

int w4a16_gemm_host(const uint16_t* x_host, uint16_t* x_dev, const void* qweight_r, const void* scales_r,
                    uint16_t* y_dev, uint16_t* y_host, int M, int N, int K, int group, void* stream) {
    if (!x_host || !y_host) return W4A16_ERR_INVALID_ARG;
    DeviceInfo d;
    Choice ch;
    const int rc = prepare_gemm(x_dev, qweight_r, scales_r, y_dev, M, N, K, group, nullptr, &d, &ch);
    if (rc != W4A16_OK) return rc;
    const size_t xb = static_cast<size_t>(M) * K * 2, yb = static_cast<size_t>(M) * N * 2;
    if (overlaps(x_host, xb, y_host, yb) || is_device_pointer(x_host) || is_device_pointer(y_host))
        return W4A16_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(x_dev, x_host, xb, cudaMemcpyHostToDevice, st) != cudaSuccess) {
        cudaGetLastError();
        return W4A16_ERR_CUDA;
    }
    const int lr = launch_gemm(ch, x_dev, qweight_r, scales_r, y_dev, M, N, K, group, d, stream);
    if (lr != W4A16_OK) return lr;
    if (cudaMemcpyAsync(y_host, y_dev, yb, cudaMemcpyDeviceToHost, st) != cudaSuccess) {
        cudaGetLastError();
        return W4A16_ERR_CUDA;
    }
    return W4A16_OK;
}

int w4a16_gemm(const uint16_t* x, const void* qweight_r, const void* scales_r, uint16_t* y, int M, int N, int K,
               int group, void* stream) {
    return w4a16_gemm_ex(x, qweight_r, scales_r, y, M, N, K, group, nullptr, stream);
}

// ---------------------------------------------------------------------------- NVFP4 weights
size_t w4a16_repacked_nvfp4_scales_bytes(int N, int K) {
    if (check_matrix_shape_nvfp4(N, K) != W4A16_OK) return 0;
    return static_cast<size_t>(K / kNvfp4Block) * N * 2;
}

static int nvfp4_repack_checks(const void* a, const void* b, const void* c, const void* d, int N, int K,
                               bool canonical_first) {
    if (!a || !b || !c || !d) return W4A16_ERR_INVALID_ARG;
    const int sh = check_matrix_shape_nvfp4(N, K);
    if (sh != W4A16_OK) return sh;
    if (!aligned16(a) || !aligned16(b) || !aligned16(c) || !aligned16(d)) return W4A16_ERR_MISALIGNED;
    const size_t qb = static_cast<size_t>(N) * K / 2;
    const size_t s8 = static_cast<size_t>(K / kNvfp4Block) * N, s16 = 2 * s8;
    // (a, b) = (qweight, scales) of the source, (c, d) of the destination
    const size_t sb_src = canonical_first ? s8 : s16, sb_dst = canonical_first ? s16 : s8;
    if (overlaps(a, qb, c, qb) || overlaps(a, qb, d, sb_dst) || overlaps(b, sb_src, c, qb) ||
        overlaps(b, sb_src, d, sb_dst) || overlaps(c, qb, d, sb_dst))
        return W4A16_ERR_INVALID_ARG;
    if (is_host_pointer(a) || is_host_pointer(b) || is_host_pointer(c) || is_host_pointer(d))
        return W4A16_ERR_INVALID_ARG;
    return W4A16_OK;
}

int w4a16_repack_nvfp4(const int32_t* qweight, const uint8_t* scales8, void* qweight_r, void* scales_r, int N, int K,
                       void* stream) {
    const int rc = nvfp4_repack_checks(qweight, scales8, qweight_r, scales_r, N, K, true);
    if (rc != W4A16_OK) return rc;
    DeviceInfo d;
    if (!device_info(&d)) return W4A16_ERR_CUDA;
    const cudaError_t e = launch_repack_nvfp4(qweight, scales8, static_cast<uint32_t*>(qweight_r),
                                              static_cast<uint16_t*>(scales_r), N, K,
                                              static_cast<cudaStream_t>(stream), d.status);
    return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}

int w4a16_unrepack_nvfp4(const void* qweight_r, const void* scales_r, int32_t* qweight, uint8_t* scales8, int N,
                         int K, void* stream) {
    const int rc = nvfp4_repack_checks(qweight_r, scales_r, qweight, scales8, N, K, false);
    if (rc != W4A16_OK) return rc;
    DeviceInfo d;
    if (!device_info(&d)) return W4A16_ERR_CUDA;
    const cudaError_t e = launch_unrepack_nvfp4(static_cast<const uint32_t*>(qweight_r),
                                                static_cast<const uint16_t*>(scales_r), qweight, scales8, N, K,
                                                static_cast<cudaStream_t>(stream), d.status);
    return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}

int w4a16_gemm_nvfp4_ex(const uint16_t* x, const void* qweight_r, const void* scales_r, float tensor_scale,
                        uint16_t* y, int M, int N, int K, const w4a16_plan* plan, void* stream) {
    if (!std::isfinite(tensor_scale)) return W4A16_ERR_INVALID_ARG;
    DeviceInfo d;
    Choice ch;
    const int rc = prepare_gemm(x, qweight_r, scales_r, y, M, N, K, kNvfp4Block, plan, &d, &ch, true);
    if (rc != W4A16_OK) return rc;
    return launch_gemm(ch, x, qweight_r, scales_r, y, M, N, K, kNvfp4Block, d, stream, true, tensor_scale);
}

int w4a16_gemm_nvfp4(const uint16_t* x, const void* qweight_r, const void* scales_r, float tensor_scale, uint16_t* y,
                     int M, int N, int K, void* stream) {
    return w4a16_gemm_nvfp4_ex(x, qweight_r, scales_r, tensor_scale, y, M, N, K, nullptr, stream);
}

int w4a16_plan_for_nvfp4(int M, int N, int K, w4a16_plan* out) {
    if (!out) return W4A16_ERR_INVALID_ARG;
    if (M <= 0) return W4A16_ERR_INVALID_ARG;
    const int sh = check_matrix_shape_nvfp4(N, K);
    if (sh != W4A16_OK) return sh;
    if (M > (1 << 20)) return W4A16_ERR_UNSUPPORTED_SHAPE;
    return plan_for_group(M, N, K, kNvfp4Block, out);
}

// ---------------------------------------------------------------------------- W4A8 (int8 activations)
int w4a16_quantize_x_int8(const uint16_t* x, int8_t* xq, uint16_t* xq_f16, float* sx, int M, int K, void* stream) {
    if (!x || !xq || !sx || M <= 0 || K <= 0) return W4A16_ERR_INVALID_ARG;
    if (K % 8 != 0 || M > (1 << 20) || K > (1 << 22)) return W4A16_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(x) || !aligned16(xq) || (xq_f16 && !aligned16(xq_f16)) || (reinterpret_cast<uintptr_t>(sx) & 3u))
        return W4A16_ERR_MISALIGNED;
    const size_t xb = static_cast<size_t>(M) * K * 2, qb = static_cast<size_t>(M) * K, sb = static_cast<size_t>(M) * 4;
    if (overlaps(x, xb, xq, qb) || overlaps(x, xb, sx, sb) || overlaps(xq, qb, sx, sb) ||
        (xq_f16 && (overlaps(xq_f16, xb, x, xb) || overlaps(xq_f16, xb, xq, qb) || overlaps(xq_f16, xb, sx, sb))))
        return W4A16_ERR_INVALID_ARG;
    if (is_host_pointer(x) || is_host_pointer(xq) || is_host_pointer(sx) || (xq_f16 && is_host_pointer(xq_f16)))
        return W4A16_ERR_INVALID_ARG;
    DeviceInfo d;
    if (!device_info(&d)) return W4A16_ERR_CUDA;
    if (launch_quantize_x_int8(x, xq, xq_f16, sx, M, K, static_cast<cudaStream_t>(stream), d.status) != cudaSuccess) {
        cudaGetLastError();
        return W4A16_ERR_CUDA;
    }
    return W4A16_OK;
}

int w4a16_gemm_w4a8_ex(const int8_t* xq, const uint16_t* xq_f16, const float* sx, const void* qweight_r,
                       const void* scales_r, uint16_t* y, int M, int N, int K, int group, const w4a16_plan* plan,
                       void* stream) {
    if (!xq || !sx || !qweight_r || !scales_r || !y || M <= 0) return W4A16_ERR_INVALID_ARG;
    const int sh = check_matrix_shape(N, K, group);
    if (sh != W4A16_OK) return sh;
    if (M > (1 << 20)) return W4A16_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(xq) || (xq_f16 && !aligned16(xq_f16)) || (reinterpret_cast<uintptr_t>(sx) & 3u) ||
        !aligned16(qweight_r) || !aligned16(scales_r) || !aligned16(y))
        return W4A16_ERR_MISALIGNED;
    const size_t qxb = static_cast<size_t>(M) * K, hb = qxb * 2, sb = static_cast<size_t>(M) * 4;
    const size_t yb = static_cast<size_t>(M) * N * 2, wb = static_cast<size_t>(N) * K / 2;
    const size_t scb = static_cast<size_t>(K / group) * N * 2;
    if (overlaps(xq, qxb, y, yb) || (xq_f16 && overlaps(xq_f16, hb, y, yb)) || overlaps(sx, sb, y, yb) ||
        overlaps(qweight_r, wb, y, yb) || overlaps(scales_r, scb, y, yb))
        return W4A16_ERR_INVALID_ARG;
    if (is_host_pointer(xq) || (xq_f16 && is_host_pointer(xq_f16)) || is_host_pointer(sx) ||
        is_host_pointer(qweight_r) || is_host_pointer(scales_r) || is_host_pointer(y))
        return W4A16_ERR_INVALID_ARG;
    DeviceInfo d;
    if (!device_info(&d)) return W4A16_ERR_CUDA;
    Choice ch;
    const int rc = resolve_plan(M, N, K, group, plan, d.sm_count, true, &ch, true);
    if (rc != W4A16_OK) return rc;
    if (ch.path == W4A16_PATH_TC && xq_f16 == nullptr) return W4A16_ERR_INVALID_ARG;  // the tiles read fp16
    return launch_gemm(ch, xq_f16, qweight_r, scales_r, y, M, N, K, group, d, stream, false, 1.0f, xq, sx);
}

int w4a16_gemm_w4a8(const int8_t* xq, const uint16_t* xq_f16, const float* sx, const void* qweight_r,
                    const void* scales_r, uint16_t* y, int M, int N, int K, int group, void* stream) {
    return w4a16_gemm_w4a8_ex(xq, xq_f16, sx, qweight_r, scales_r, y, M, N, K, group, nullptr, stream);
}

int w4a16_quantize_gemm_w4a8(const uint16_t* x, int8_t* xq, uint16_t* xq_f16, float* sx, const void* qweight_r,
                              const void* scales_r, uint16_t* y, int M, int N, int K, int group,
                              const w4a16_plan* plan, void* stream) {
    if (!x || !xq || !sx || !qweight_r || !scales_r || !y || M <= 0) return W4A16_ERR_INVALID_ARG;
    const int sh = check_matrix_shape(N, K, group);
    if (sh != W4A16_OK) return sh;
    if (M > (1 << 20)) return W4A16_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(x) || !aligned16(xq) || (xq_f16 && !aligned16(xq_f16)) || (reinterpret_cast<uintptr_t>(sx) & 3u) ||
        !aligned16(qweight_r) || !aligned16(scales_r) || !aligned16(y))
        return W4A16_ERR_MISALIGNED;
    const size_t xb = static_cast<size_t>(M) * K * 2, qxb = static_cast<size_t>(M) * K, sb = static_cast<size_t>(M) * 4;
    const size_t yb = static_cast<size_t>(M) * N * 2, wb = static_cast<size_t>(N) * K / 2;
    const size_t scb = static_cast<size_t>(K / group) * N * 2;
    const void* outs[4] = {xq, xq_f16, sx, y};
    const size_t out_bytes[4] = {qxb, xb, sb, yb};
    for (int i = 0; i < 4; ++i) {  // the outputs overlap neither each other nor any input
        if (!outs[i]) continue;
        if (overlaps(outs[i], out_bytes[i], x, xb) || overlaps(outs[i], out_bytes[i], qweight_r, wb) ||
            overlaps(outs[i], out_bytes[i], scales_r, scb) || is_host_pointer(outs[i]))
            return W4A16_ERR_INVALID_ARG;
        for (int j = i + 1; j < 4; ++j)
            if (outs[j] && overlaps(outs[i], out_bytes[i], outs[j], out_bytes[j])) return W4A16_ERR_INVALID_ARG;
    }
    if (is_host_pointer(x) || is_host_pointer(qweight_r) || is_host_pointer(scales_r)) return W4A16_ERR_INVALID_ARG;
    DeviceInfo d;
    if (!device_info(&d)) return W4A16_ERR_CUDA;
    Choice ch;
    const int rc = resolve_plan(M, N, K, group, plan, d.sm_count, true, &ch, true);
    if (rc != W4A16_OK) return rc;
    if (ch.path == W4A16_PATH_TC && xq_f16 == nullptr) return W4A16_ERR_INVALID_ARG;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (launch_quantize_x_int8(x, xq, xq_f16, sx, M, K, st, d.status) != cudaSuccess) {
        cudaGetLastError();
        return W4A16_ERR_CUDA;
    }
    return launch_gemm(ch, xq_f16, qweight_r, scales_r, y, M, N, K, group, d, stream, false, 1.0f, xq, sx);
}

int w4a16_plan_for_w4a8(int M, int N, int K, int group, w4a16_plan* out) {
    if (!out) return W4A16_ERR_INVALID_ARG;
    if (M <= 0) return W4A16_ERR_INVALID_ARG;
    const int sh = check_matrix_shape(N, K, group);
    if (sh != W4A16_OK) return sh;
    if (M > (1 << 20)) return W4A16_ERR_UNSUPPORTED_SHAPE;
    return plan_for_group(M, N, K, group, out, true);
}

int w4a16_silu_mul(const uint16_t* gu, uint16_t* act, int M, int I, void* stream) {
    if (!gu || !act || M <= 0 || I <= 0) return W4A16_ERR_INVALID_ARG;
    if (I % 8 != 0 || M > (1 << 20) || I > (1 << 22)) return W4A16_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(gu) || !aligned16(act)) return W4A16_ERR_MISALIGNED;
    const size_t gb = static_cast<size_t>(M) * I * 4, ab = static_cast<size_t>(M) * I * 2;
    if (overlaps(gu, gb, act, ab) || is_host_pointer(gu) || is_host_pointer(act)) return W4A16_ERR_INVALID_ARG;
    DeviceInfo d;
    if (!device_info(&d)) return W4A16_ERR_CUDA;
    if (launch_silu_mul(gu, act, M, I, d.sm_count, static_cast<cudaStream_t>(stream), d.status) != cudaSuccess) {
        cudaGetLastError();
        return W4A16_ERR_CUDA;
    }
    return W4A16_OK;
}

int w4a16_last_dispatch(char* buf, size_t len) {
    if (!buf || len == 0) return W4A16_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    snprintf(buf, len, "%s", g_last);
    return W4A16_OK;
}

int w4a16_device_status(void* stream) {
    DeviceInfo d;
    if (!device_info(&d)) return W4A16_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    take_status_kernel<<<1, 1, 0, s>>>(d.status, d.taken);
    if (cudaGetLastError() != cudaSuccess) return W4A16_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpyAsync(&v, d.taken, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) {
        cudaGetLastError();
        return W4A16_ERR_CUDA;
    }
    if (cudaStreamSynchronize(s) != cudaSuccess) return W4A16_ERR_CUDA;
    return v == 0 ? W4A16_OK : static_cast<int>(v);
}

int w4a16_selftest_wait_timeout(int mode, void* stream) {
    if (mode != 0 && mode != 1) return W4A16_ERR_INVALID_ARG;
    DeviceInfo d;
    if (!device_info(&d)) return W4A16_ERR_CUDA;
    wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(d.status, g_timeout_ns.load(), mode);
    if (cudaGetLastError() != cudaSuccess) return W4A16_ERR_CUDA;
    return W4A16_OK;
}

int w4a16_set_wait_timeout_ns(uint64_t ns) {
    if (ns < 100000ull) return W4A16_ERR_INVALID_ARG;
    g_timeout_ns.store(ns);
    return W4A16_OK;
}

}  // extern "C"
