// ngr_ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarrier, TMA bulk
// tensor copies, tcgen05 (TMEM allocation, UMMA, commit, TMEM loads), proxy
// fences and programmatic dependent launch.  Every spin on an mbarrier is
// bounded in time; a wait that runs out records an error word and returns.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace ngr {

// Device error word values (kept in the first 4 bytes of the workspace).
enum : int { kDevErrTimeout = 1 };

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar,
                                                      uint32_t bytes)
{
    asm volatile(
        "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
            smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Where a bounded wait reports to: `abort` is a per-CTA flag in shared
// memory (zeroed at kernel start) that tells the CTA's other roles to stop;
// `err` is the device error word of the call, which kernels only ever set.
struct WaitCtx {
    int *abort;                 // shared memory
    int *err;                   // global memory
    unsigned long long timeout_ns;
};

// Wait for the phase of `bar` with parity `parity` to complete.  Gives up
// after `timeout_ns` of global time, or as soon as another role of this CTA
// has given up; on giving up it raises the CTA's abort flag, records
// kDevErrTimeout in the error word and returns false.
static __device__ __noinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, const WaitCtx &w)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*reinterpret_cast<volatile int *>(w.abort) != 0) return false;
            if (global_timer_ns() - t0 > w.timeout_ns) {
                *reinterpret_cast<volatile int *>(w.abort) = 1;
                atomicExch(w.err, kDevErrTimeout);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same bounded wait for the pipeline roles whose wake-up latency sits
// on every stage's round trip (the MMA issuers, the decode producer): it
// polls with the non-blocking test instead of the potentially suspending
// try, so that the thread resumes as soon as the phase completes (a
// suspended thread without a time hint was measured to resume late enough
// to slow the tile kernels by 14-20 % at LayerNorm 1024 x 8192 -> 8192 and
// RMSNorm 512 x 14336 -> 49152).  NGR_SPIN_WAIT=0 selects the suspending
// form.
#ifndef NGR_SPIN_WAIT
#define NGR_SPIN_WAIT 1
#endif
__device__ __forceinline__ bool mbar_wait_spin(uint64_t *bar, uint32_t parity, const WaitCtx &w)
{
#if NGR_SPIN_WAIT == 0
    return mbar_wait(bar, parity, w);
#else
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_test_wait(bar, parity)) return true;
        if ((it & 1023u) == 0) {
            if (*reinterpret_cast<volatile int *>(w.abort) != 0) return false;
            if (global_timer_ns() - t0 > w.timeout_ns) {
                *reinterpret_cast<volatile int *>(w.abort) = 1;
                atomicExch(w.err, kDevErrTimeout);
                return false;
            }
        }
    }
#endif
}

// The wait of the roles that run ahead of the tensor core (the transform
// warps, the TMA producers of the tile kernels): up to NGR_POLLS_FIRST
// non-blocking tests, then try_wait with a suspend-time hint of
// NGR_WAIT_HINT_NS, so that the thread may sleep until the phase completes
// or the hint runs out.  Measured against polling alone on GB300: 2.4-3.2 %
// faster with RMSNorm (512 x 14336 -> 49152 fp16 and bf16, 1024 x 8192 ->
// 8192), 0.4 % with LayerNorm; a try_wait without the polls first, or with
// a 500-ns hint, was slower.
#ifndef NGR_POLLS_FIRST
#define NGR_POLLS_FIRST 64
#endif
#ifndef NGR_WAIT_HINT_NS
#define NGR_WAIT_HINT_NS 200
#endif
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(static_cast<uint32_t>(NGR_WAIT_HINT_NS))
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_ahead(uint64_t *bar, uint32_t parity, const WaitCtx &w)
{
    for (int i = 0; i < NGR_POLLS_FIRST; ++i)
        if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_hint(bar, parity)) return true;
        if ((it & 15u) == 0) {
            if (*reinterpret_cast<volatile int *>(w.abort) != 0) return false;
            if (global_timer_ns() - t0 > w.timeout_ns) {
                *reinterpret_cast<volatile int *>(w.abort) = 1;
                atomicExch(w.err, kDevErrTimeout);
                return false;
            }
        }
    }
}

// Warp-uniform form of mbar_wait_ahead (lane 0 waits).
__device__ __forceinline__ bool mbar_wait_warp_ahead(uint64_t *bar, uint32_t parity, const WaitCtx &w)
{
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_ahead(bar, parity, w) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) (void)mbar_try_wait(bar, parity);
    return ok != 0;
}

// Warp-uniform form of mbar_wait_spin (lane 0 polls).
__device__ __forceinline__ bool mbar_wait_warp_spin(uint64_t *bar, uint32_t parity, const WaitCtx &w)
{
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_spin(bar, parity, w) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) (void)mbar_try_wait(bar, parity);
    return ok != 0;
}

// The bounded wait for phases that take long to come (a tile's accumulator
// for the epilogue, the last commit before a kernel exits): a test, then a
// short sleep, repeated.  A waiting warp costs few issue slots, and it
// resumes within about NGR_NAP_NS of the phase completing, whereas a
// try_wait may suspend the thread for microseconds past it (measured:
// four such waits in a row added about 20 us to a kernel's tail).
// NGR_LONG_WAIT_NAP=0 selects the suspending form.
#ifndef NGR_NAP_NS
#define NGR_NAP_NS 128
#endif
#ifndef NGR_LONG_WAIT_NAP
#define NGR_LONG_WAIT_NAP 1
#endif
__device__ __forceinline__ bool mbar_wait_long(uint64_t *bar, uint32_t parity, const WaitCtx &w)
{
#if NGR_LONG_WAIT_NAP == 0
    return mbar_wait(bar, parity, w);
#else
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        __nanosleep(NGR_NAP_NS);
        if (mbar_test_wait(bar, parity)) return true;
        if ((it & 15u) == 0) {
            if (*reinterpret_cast<volatile int *>(w.abort) != 0) return false;
            if (global_timer_ns() - t0 > w.timeout_ns) {
                *reinterpret_cast<volatile int *>(w.abort) = 1;
                atomicExch(w.err, kDevErrTimeout);
                return false;
            }
        }
    }
#endif
}

// Warp-uniform form of mbar_wait_long (lane 0 waits).
__device__ __forceinline__ bool mbar_wait_warp_long(uint64_t *bar, uint32_t parity, const WaitCtx &w)
{
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_long(bar, parity, w) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) (void)mbar_try_wait(bar, parity);
    return ok != 0;
}

// Warp-uniform form for roles whose next step is warp-collective: lane 0
// waits, the verdict is broadcast, and every lane then acquires the
// completed phase itself.  All 32 lanes must call it.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity, const WaitCtx &w)
{
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, w) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) (void)mbar_try_wait(bar, parity);
    return ok != 0;
}

// ------------------------------------------------------------- TMA copies
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *m)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m))
                 : "memory");
}

// 2-D tiled load of the box at coordinates (c0 = innermost, c1) into shared
// memory; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *m,
                                            uint64_t *bar, int c0, int c1,
                                            uint64_t cache_hint)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1),
        "l"(cache_hint)
        : "memory");
}

__device__ __forceinline__ void tma_load_1d(void *dst, const CUtensorMap *m,
                                            uint64_t *bar, int c0,
                                            uint64_t cache_hint)
{
    asm volatile(
        "cp.async.bulk.tensor.1d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3}], [%2], %4;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0),
        "l"(cache_hint)
        : "memory");
}

// The same load delivered to every CTA of the cluster whose bit is set in
// `cta_mask`, at the same shared-memory offset in each, with completion
// signalled on the mbarrier at the same offset in each destination CTA.
__device__ __forceinline__ void tma_load_2d_mc(void *dst, const CUtensorMap *m, uint64_t *bar,
                                               int c0, int c1, uint16_t cta_mask,
                                               uint64_t cache_hint)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5, %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "h"(cta_mask),
        "l"(cache_hint)
        : "memory");
}

// L2 eviction-priority policies for the cache_hint operand.
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Make this thread's generic-proxy writes to shared memory visible to the
// async proxy (the tensor core reads operands through it).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier among `nthreads` threads (a multiple of 32).
// Bring the 128-byte line holding `p` into L1 (no data returned).
__device__ __forceinline__ void prefetch_l1(const void *p)
{
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}


// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t *smem_dst, uint32_t ncols)
{
    asm volatile(
        "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
            smem_u32(smem_dst)),
        "r"(ncols)
        : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::
                     : "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(
                     taddr),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] . B[smem]^T, both operands K-major, issued by one
// thread.  `accumulate` = 0 overwrites D.
__device__ __forceinline__ void umma_f16_ss(uint32_t d_tmem, uint64_t a_desc,
                                            uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Warp-collective load of 32 consecutive 32-bit TMEM columns: lane l of the
// warp receives row (lane base + l), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
        "%30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
          "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]),
          "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

// 16 consecutive columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
        "[%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
          "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]),
          "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored in the
// 128-byte swizzle layout the TMA writes: rows of 128 bytes, 8-row groups
// 1024 bytes apart, tile base 1024-byte aligned.  Fields: start address >> 4
// (bits 0-13), leading byte offset >> 4 (16-29; unused for this layout, set
// to 1), stride byte offset >> 4 (32-45), descriptor version 1 (46-48),
// swizzle mode 2 = 128-byte (61-63).  Advancing K by 16 elements inside the
// 128-byte row adds 32 bytes to the start address.
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor for kind::f16 with FP32 accumulation, both operands
// K-major, dense: D format F32 (bits 4-5 = 1), A and B format F16 = 0 or
// BF16 = 1 (bits 7-9, 10-12), N >> 3 (bits 17-22), M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, int M, int N)
{
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// ------------------------------------------------- programmatic dependent launch
// Wait until the grids this one depends on have completed and their memory
// is visible (a no-op when launched without the attribute).
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Allow the dependent grid to begin launching.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace ngr

namespace ngr {

// ------------------------------------------------- CTA pairs (clusters of 2)
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank)
{
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
    return d;
}

// Arrive on an mbarrier that may live in another CTA of the cluster
// (default semantics; an explicit cluster-scope release here costs a full
// fence per arrival and throttles a per-stage handshake).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Full barrier across all threads of both CTAs of the cluster.
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release;\n\t"
                 "barrier.cluster.wait.acquire;" ::
                     : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t *smem_dst, uint32_t ncols)
{
    asm volatile(
        "tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
            smem_u32(smem_dst)),
        "r"(ncols)
        : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(ncols)
                 : "memory");
}

// D (both CTAs' tensor memory, 128 rows each) (+)= A . B^T with A split by
// rows and B split by columns over the two CTAs' shared memory (same
// offsets in both).  Issued by one thread of the even CTA.
__device__ __forceinline__ void umma_f16_ss_pair(uint32_t d_tmem, uint64_t a_desc,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the mbarrier at this shared-memory offset in every CTA of
// `cta_mask` when all tcgen05 operations issued so far by this thread are
// complete.
__device__ __forceinline__ void umma_commit_pair(uint64_t *bar, uint16_t cta_mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
        "[%0], %1;" ::"r"(smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

}  // namespace ngr

namespace ngr {

// 2-D tiled load into this CTA's shared memory whose completion (transaction
// bytes) is signalled on an mbarrier of either CTA of the pair, given by its
// shared::cluster address.
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *m,
                                                 uint32_t bar_cluster_addr, int c0, int c1,
                                                 uint64_t cache_hint)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster_addr), "r"(c0), "r"(c1),
        "l"(cache_hint)
        : "memory");
}

}  // namespace ngr
