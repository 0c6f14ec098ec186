// Device-side building blocks shared by the libw4a16 kernels (sm_103a only):
// mbarrier waits with a time limit, TMA bulk / tensor copies, tcgen05 (TMEM + UMMA) wrappers,
// cluster / DSMEM helpers and the exact 4-bit -> fp16 dequantisation.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "libw4a16 kernels target sm_103a (tcgen05 / TMA); build with -gencode arch=compute_103a,code=sm_103a"
#endif

namespace w4a16 {

// Status codes written into the per-device status word (mirror w4a16_status).
constexpr unsigned kErrTimeout = 5u;
constexpr unsigned kErrBounds = 6u;

// Records an error code in the status word unless an earlier error is already there (the first
// error of a launch is the one reported).
__device__ __forceinline__ void record_error(unsigned* status, unsigned code) { atomicCAS(status, 0u, code); }

// Index checks of the debug-bounds build (compiled with W4A16_DEBUG_BOUNDS): the kernels test
// every global-memory index against the size of its buffer before the access; a bad index records
// kErrBounds and the access is skipped (no trap: the context stays usable). In the normal build the
// test compiles away.
#ifdef W4A16_DEBUG_BOUNDS
__device__ __forceinline__ bool in_bounds(bool ok, unsigned* status) {
    if (!ok) record_error(status, kErrBounds);
    return ok;
}
#else
__device__ __forceinline__ bool in_bounds(bool, unsigned*) { return true; }
#endif

// ------------------------------------------------------------------------------------ misc
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------------------------ PDL
// Programmatic dependent launch. griddep_wait blocks until the grids this one depends on have
// completed and their writes are visible (a no-op when launched without the attribute);
// griddep_launch_dependents lets the next grid on the stream start launching (the first call by any
// thread of the CTA counts).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0u;
}

// Waits for the phase of `bar` with parity `parity` to complete. Gives up when `abort_flag`
// (CTA shared) is raised by another thread, or after `timeout_ns`, in which case it records
// kErrTimeout in the device status word and raises the abort flag. Returns false on give-up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t timeout_ns, unsigned* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 31u) == 0u) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > timeout_ns) {
                record_error(status, kErrTimeout);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// Same contract as mbar_wait, for single-thread roles on the critical path (producer, MMA
// issuer): polls with the non-suspending test_wait so the thread reacts as soon as the phase
// completes instead of after a suspension time slice.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0u;
}

__device__ __forceinline__ bool mbar_spin(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t timeout_ns, unsigned* status) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_test_wait(bar, parity)) return true;
        if ((spin & 255u) == 0u) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > timeout_ns) {
                record_error(status, kErrTimeout);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// Non-blocking test of a phase with acquire semantics at cluster scope: for phases completed by
// arrivals of other CTAs of the cluster (mbar_arrive_remote), so that their prior shared-memory
// writes are seen. (Measured: a thread suspended in try_wait is not woken promptly by a remote
// arrival, so these phases are polled.)
__device__ __forceinline__ bool mbar_test_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0u;
}

// Bounded wait of mbar_wait's contract on a phase completed by cluster peers (polled).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                  uint64_t timeout_ns, unsigned* status) {
    if (mbar_test_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_test_wait_cluster(bar, parity)) return true;
        if ((spin & 255u) == 0u) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > timeout_ns) {
                record_error(status, kErrTimeout);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// Arrives once, with release semantics at cluster scope, on the mbarrier at shared address `bar`
// in the CTA of cluster rank `rank` (may be this CTA).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar, uint32_t rank) {
    asm volatile(
        "{\n\t.reg .b32 ra;\n\t"
        "mapa.shared::cluster.u32 ra, %0, %1;\n\t"
        "mbarrier.arrive.release.cluster.shared::cluster.b64 _, [ra];\n\t}" ::"r"(bar),
        "r"(rank)
        : "memory");
}

// Named barriers (ids 1..15; id 0 is __syncthreads). `nthreads` counts every participating
// thread, a multiple of 32. arrive does not wait; sync waits for the generation to complete.
__device__ __forceinline__ void named_arrive(int id, int nthreads) {
    asm volatile("barrier.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Warp-wide wait: lane 0 polls (so a warp puts one poller, not 32, on the barrier), the warp
// reconverges, then every lane performs its own (now immediate) acquiring test of the phase.
// Returns the same verdict in all lanes. Must be called by all 32 lanes.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t timeout_ns, unsigned* status) {
    int ok = 1;
    if ((threadIdx.x & 31u) == 0u) ok = mbar_wait(bar, parity, abort_flag, timeout_ns, status) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) mbar_try_wait(bar, parity);
    return ok != 0;
}

// Warp-wide bounded wait that never suspends: lane 0 polls with test_wait (a thread suspended in
// try_wait wakes up hundreds to thousands of cycles after the phase completes), then every lane
// takes the acquire of the completed phase. Returns the same verdict in all lanes.
__device__ __forceinline__ bool warp_spin(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint64_t timeout_ns,
                                          unsigned* status) {
    int ok = 1;
    if ((threadIdx.x & 31u) == 0u) ok = mbar_spin(bar, parity, abort_flag, timeout_ns, status) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) mbar_test_wait(bar, parity);
    return ok != 0;
}

// ------------------------------------------------------------------------------------ shared memory
// Explicit shared-space loads by 32-bit shared address (a generic pointer into dynamic shared
// memory is not always recognised as shared and would take the generic load path).
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

// ------------------------------------------------------------------------------------ TMA
// 1-D bulk copy global -> this CTA's shared memory, completing `bytes` on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// 2-D tiled tensor copy global -> shared through a tensor map (box given by the map).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(tmap), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// One warp stores N consecutive 32-bit TMEM columns of its 32 lanes (lane i <- thread i).
template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const uint32_t (&r)[N]);

template <>
__device__ __forceinline__ void tmem_st<16>(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

template <>
__device__ __forceinline__ void tmem_st<32>(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// One warp loads N consecutive 32-bit TMEM columns of its 32 lanes (thread i <- lane i).
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[N]);

template <>
__device__ __forceinline__ void tmem_ld<4>(uint32_t taddr, uint32_t (&r)[4]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr)
                 : "memory");
}

template <>
__device__ __forceinline__ void tmem_ld<8>(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
}

// D[tmem] (+)= A[tmem] . B[smem]^T, kind::f16, one CTA. `accumulate` false overwrites D.
__device__ __forceinline__ void umma_f16_ts(uint32_t d_taddr, uint32_t a_taddr, uint64_t b_desc, uint32_t idesc,
                                            bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_taddr),
        "r"(a_taddr), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzle layout
// (8 rows x 128 B atoms, atoms 1024 B apart). Start address advances by 32 B per K step of 16.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
    d |= static_cast<uint64_t>(1u) << 16;                  // leading byte offset (unused for SW128 K-major)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;          // stride byte offset: 8-row group pitch
    d |= static_cast<uint64_t>(1u) << 46;                  // descriptor version for tcgen05
    d |= static_cast<uint64_t>(2u) << 61;                  // swizzle mode: 128 B
    return d;
}

// Instruction descriptor, kind::f16: fp16 A and B (both K-major), fp32 D, shape M x N x 16.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4)                                   // D format: f32
           | (0u << 7) | (0u << 10)                   // A, B format: f16
           | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// ------------------------------------------------------------------------------------ cluster
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_peer(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ float ld_dsmem_f1(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Sum over the cluster's first `split` CTAs (split <= 16) of the value at shared address `local`,
// added in rank order 0, 1, ... Groups of four remote loads are issued before their adds, so their
// latencies overlap instead of following one another (same sum, same order as a plain loop).
__device__ __forceinline__ float cluster_sum_f1(uint32_t local, int split) {
    float s = 0.f;
    for (int p0 = 0; p0 < split; p0 += 4) {
        float v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = p0 + u < split ? ld_dsmem_f1(map_peer(local, p0 + u)) : 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (p0 + u < split) s += v[u];
    }
    return s;
}

__device__ __forceinline__ float4 cluster_sum_f4(uint32_t local, int split) {
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p0 = 0; p0 < split; p0 += 4) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            v[u] = p0 + u < split ? ld_dsmem_f4(map_peer(local, p0 + u)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (p0 + u < split) {
                s.x += v[u].x;
                s.y += v[u].y;
                s.z += v[u].z;
                s.w += v[u].w;
            }
        }
    }
    return s;
}

// ------------------------------------------------------------------------------------ dequant
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t mask, uint32_t bits) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(bits));  // (a & mask) | bits
    return d;
}
__device__ __forceinline__ uint32_t hadd2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// One repacked 32-bit word holds 8 consecutive k of one column with nibble positions
// 0,4,1,5,2,6,3,7 for k offsets 0..7. Produces four fp16 pairs in k order,
// out[i] = (w[2i], w[2i+1]) with w = fp16_rne((q - 8) * s), s2 = (s, s).
//   (word & 0x000F000F) | 0x6400_6400  -> fp16 (1024 + q) for k offsets 0,1
//   (word & 0x00F000F0) | 0x6400_6400  -> fp16 (1024 + 16 q) for k offsets 2,3
//   the same on word >> 8                 for k offsets 4,5 and 6,7
// q - 8 is then exact: (1024 + q) - 1032, or (1024 + 16 q) * 2^-4 - 72 in one fused step whose
// exact value is a small integer; the product with s is the single rounding.
__device__ __forceinline__ void dequant8(uint32_t word, uint32_t s2, uint32_t out[4]) {
    constexpr uint32_t kMagic = 0x64006400u;     // (1024, 1024)
    constexpr uint32_t kNeg1032 = 0xE408E408u;   // (-1032, -1032)
    constexpr uint32_t kSixteenth = 0x2C002C00u; // (1/16, 1/16)
    constexpr uint32_t kNeg72 = 0xD480D480u;     // (-72, -72)
    const uint32_t hi = word >> 8;
    const uint32_t a = and_or(word, 0x000F000Fu, kMagic);
    const uint32_t b = and_or(word, 0x00F000F0u, kMagic);
    const uint32_t c = and_or(hi, 0x000F000Fu, kMagic);
    const uint32_t d = and_or(hi, 0x00F000F0u, kMagic);
    out[0] = hmul2(hadd2(a, kNeg1032), s2);
    out[1] = hmul2(hfma2(b, kSixteenth, kNeg72), s2);
    out[2] = hmul2(hadd2(c, kNeg1032), s2);
    out[3] = hmul2(hfma2(d, kSixteenth, kNeg72), s2);
}

// NVFP4 weights: out[i] = (w[2i], w[2i+1]) with w = e2m1(code) * s, s2 = (s, s) the fp16 value of
// the block's E4M3 scale. The word keeps the canonical nibble order (code of k offset j in nibble
// j), so byte i holds the codes of k offsets 2i and 2i+1 and one hardware conversion turns it into
// that fp16 pair (E2M1 values are exact in fp16). e2m1 * s has at most 2 + 4 significant bits and
// lies within the fp16 normal range for every finite E4M3 scale: the multiply is exact.
__device__ __forceinline__ void dequant8_nvfp4(uint32_t word, uint32_t s2, uint32_t out[4]) {
    uint32_t h[4];
    asm("{\n\t.reg .b8 a0, a1, a2, a3;\n\t"
        "mov.b32 {a0, a1, a2, a3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, a0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, a1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, a2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, a3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(word));
#pragma unroll
    for (int i = 0; i < 4; ++i) out[i] = hmul2(h[i], s2);
}

// Two fp32 accumulations acc0 += lo(w2) * lo(x2), acc1 += hi(w2) * hi(x2): fp16 operands, the
// exact product rounded once into fp32.
__device__ __forceinline__ void fma2_mixed(float& acc0, float& acc1, uint32_t w2, uint32_t x2) {
    asm("{\n\t.reg .f16 wl, wh, xl, xh;\n\t"
        "mov.b32 {wl, wh}, %2;\n\t"
        "mov.b32 {xl, xh}, %3;\n\t"
        "fma.rn.f32.f16 %0, wl, xl, %0;\n\t"
        "fma.rn.f32.f16 %1, wh, xh, %1;\n\t}"
        : "+f"(acc0), "+f"(acc1)
        : "r"(w2), "r"(x2));
}

}  // namespace w4a16
