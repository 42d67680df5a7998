// pi_async.cuh -- bulk asynchronous copies, mbarriers, L2 prefetch and a bounded grid barrier (sm_103a).
//
// Every wait here is bounded by the global nanosecond timer: on expiry the
// caller gets `false`, records PI_ERR_TIMEOUT in the status word and leaves.
#pragma once

#include "pi_common.cuh"

namespace pi {

constexpr unsigned long long WAIT_LIMIT_NS = 200ull * 1000 * 1000;   // 200 ms

__device__ __forceinline__ unsigned long long globaltimer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

// ---------------------------------------------------------------- mbarrier -------------------

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_inval(uint64_t *bar)
{
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Make initialised barriers visible to the async proxy (bulk copies complete on them).
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory accesses (and, after a CTA barrier,
// those of the threads it synchronised with) before its later async-proxy ones.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
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

// Wait for phase `parity` of the barrier to complete; false after WAIT_LIMIT_NS.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) return false;
    return true;
}

// ---------------------------------------------------------------- named barriers -------------

// Barrier `id` (1..15; 0 is __syncthreads) over `count` threads (a multiple of 32).
__device__ __forceinline__ void bar_sync(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// bar_sync that also returns the AND of v over the participating threads.
__device__ __forceinline__ bool bar_and(int id, int count, bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// ---------------------------------------------------------------- bulk copies ----------------

// global -> shared, `bytes` (multiple of 16, both addresses 16-byte aligned); completion
// is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 4-byte global -> shared copy (cp.async); the issuing thread waits with cp_async_wait_all.
__device__ __forceinline__ void cp_async4(void *dst_smem, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst_smem)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Bring `bytes` (multiple of 16, 16-byte aligned) of global memory into L2 without waiting.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// One 128-byte line into L2 (a hint: no completion, no fault on a valid address).
__device__ __forceinline__ void prefetch_line_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void prefetch_l2_range(const void *src, size_t bytes)
{
    const char *p = (const char *)src;
    bytes &= ~(size_t)15;
    while (bytes > 0) {
        const uint32_t n = bytes > (64u << 10) ? (64u << 10) : (uint32_t)bytes;
        prefetch_l2(p, n);
        p += n;
        bytes -= n;
    }
}

// ---------------------------------------------------------------- grid barrier ---------------

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Wait (bounded) until *p >= v (a value another CTA of the same launch publishes with a release
// store); false after WAIT_LIMIT_NS.
__device__ __forceinline__ bool wait_flag_ge(const unsigned long long *p, unsigned long long v)
{
    if ((long long)(ld_acquire_u64(p) - v) >= 0) return true;
    const unsigned long long t0 = globaltimer_ns();
    while ((long long)(ld_acquire_u64(p) - v) < 0) {
        if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) return false;
        __nanosleep(32);
    }
    return true;
}

__device__ __forceinline__ void red_release_add_u64(unsigned long long *p, unsigned long long v)
{
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Monotonic grid barrier: every arrival adds 1 to a 64-bit counter (no reply awaited),
// and the k-th barrier of a launch completes when the counter reaches base + k * nblocks.
// A launch that passes all its barriers leaves the counter at a multiple of
// (barriers per launch * nblocks), which is how the next launch finds its base.
__device__ __forceinline__ unsigned long long barrier_base(const unsigned long long *cnt, unsigned long long per_launch)
{
    const unsigned long long c = ld_acquire_u64(cnt);
    return c - c % per_launch;
}

// Bulk copies a CTA may have in flight at a grid barrier: phase tile_par[k] of tiles[k] for
// k < ntiles (where >= 0), and phase *many_par of each of many[0..nmany) (if >= 0). The
// parities live in shared memory.
struct PendingCopies {
    uint64_t *tiles;
    const int *tile_par;
    int ntiles;
    uint64_t *many;
    int nmany;
    const int *many_par;
};

struct NoWork {
    __device__ void operator()() const {}
};

// Returns false in every thread of a CTA that gave up waiting (after recording PI_ERR_TIMEOUT
// and waiting, bounded, for the copies `pc` names to land). Every thread runs `work` between
// the CTA's arrival and its wait: work no other CTA waits for, such as issuing copies into
// this CTA's own shared memory.
template <typename Work = NoWork>
__device__ __forceinline__ bool grid_sync_to(unsigned long long *cnt, unsigned long long target, uint32_t *status,
                                             int *s_flag, const PendingCopies *pc = nullptr, Work work = Work())
{
    __syncthreads();
    if (threadIdx.x == 0) red_release_add_u64(cnt, 1ull);   // release: the CTA's writes before the CTA barrier
    work();
    if (threadIdx.x == 0) {
        int ok = 1;
        if ((long long)(ld_acquire_u64(cnt) - target) < 0) {
            const unsigned long long t0 = globaltimer_ns();
            while ((long long)(ld_acquire_u64(cnt) - target) < 0) {
                if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
                    set_status(status, ST_TIMEOUT);
                    ok = 0;
                    if (pc) {
                        for (int k = 0; k < pc->ntiles; ++k)
                            if (pc->tile_par[k] >= 0) mbar_wait(&pc->tiles[k], (uint32_t)pc->tile_par[k]);
                        if (*pc->many_par >= 0)
                            for (int k = 0; k < pc->nmany; ++k) mbar_wait(&pc->many[k], (uint32_t)*pc->many_par);
                    }
                    break;
                }
                __nanosleep(64);   // fewer polls on the counter's line while the arrivals land
            }
        }
        *s_flag = ok;                      // the acquiring load above orders what follows
    }
    __syncthreads();
    return *s_flag != 0;
}

}  // namespace pi
