// Device helpers shared by the library's kernels: PTX wrappers for mbarriers, TMA, tcgen05
// and the bounded waits. Included by the .cu files only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lora_internal.h"

namespace lora {
namespace dev {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- cluster
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// All threads of every CTA in the cluster (also a CTA-wide barrier).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Shared::cluster address of the same shared variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes, uint32_t pred) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t"
        "@q mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar), "r"(bytes), "r"(pred)
        : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Arrive on a barrier given by its shared::cluster address (this CTA's or the peer's).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
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
    return ok != 0;
}
// Warp-wide form of wait_bounded for the converged producer and MMA warps: every lane
// tests the phase (one instruction for the warp); only if it is not complete yet does lane 0
// fall back to the bounded loop. Returns the same value in every lane.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status,
                                          uint64_t limit_ns);

// Waits for the phase with the given parity to complete. Gives up (returns false) when
// another role has aborted or when `limit_ns` of wall time pass; in the latter case it
// records the timeout in the status word and raises the CTA's abort flag.
static __device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status, uint64_t limit_ns, bool honour_abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (honour_abort && *abort_flag) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, 1);
            *abort_flag = 1;
            return false;
        }
    }
}

__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status,
                                          uint64_t limit_ns) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = wait_bounded(bar, parity, abort_flag, status, limit_ns, true);
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// ---------------------------------------------------------------- TMA
// 2-D tiled load into this CTA's shared memory, completing bytes on `bar` (a barrier of
// this CTA; with CG = 2 it may be the even CTA's barrier, as a shared::cluster address).
// Issued by the lanes with pred != 0 (one lane of a converged warp).
template <int CG>
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c_inner,
                                            int c_outer, uint32_t pred) {
    if (CG == 1) {
        asm volatile(
            "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\t"
            "@q cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%3, %4}], [%2];\n\t}" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c_inner), "r"(c_outer), "r"(pred)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\t"
            "@q cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
            " [%0], [%1, {%3, %4}], [%2];\n\t}" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c_inner), "r"(c_outer), "r"(pred)
            : "memory");
    }
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// Tensor maps written to global memory by the host: make the tensormap proxy see them.
__device__ __forceinline__ void tensormap_acquire(const CUtensorMap* map) {
    asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(
                     reinterpret_cast<uint64_t>(map))
                 : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// With CG = 2 one warp of each CTA of the pair executes these together.
template <int CG>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    if (CG == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                     "r"(ncols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    } else {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                     "r"(ncols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
}
template <int CG>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    if (CG == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate. Issued by the lane with
// pred != 0 of a converged warp: the MMA stream keeps the tensor pipe busy only when the
// issuing warp is converged (a lone diverged lane issues MMAs far more slowly).
template <int CG>
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate, uint32_t pred) {
    if (CG == 1)
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "setp.ne.b32 q, %5, 0;\n\t"
            "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(pred)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "setp.ne.b32 q, %5, 0;\n\t"
            "@q tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(pred)
            : "memory");
}
// Arrive once on `bar` (CG = 1: this CTA's; CG = 2: the barrier at that offset in both CTAs
// of the pair) when every tcgen05 op the issuing lane issued so far has completed.
template <int CG>
__device__ __forceinline__ void mma_commit(uint32_t bar, uint32_t pred) {
    if (CG == 1)
        asm volatile(
            "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %1, 0;\n\t"
            "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar),
            "r"(pred)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t"
            "@q tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
            " [%0], %1;\n\t}" ::"r"(bar), "h"((uint16_t)3), "r"(pred)
            : "memory");
}
// Same, arriving only on this CTA's barrier.
template <int CG>
__device__ __forceinline__ void mma_commit_local(uint32_t bar, uint32_t pred) {
    if (CG == 1)
        asm volatile(
            "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %1, 0;\n\t"
            "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar),
            "r"(pred)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %1, 0;\n\t"
            "@q tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar),
            "r"(pred)
            : "memory");
}
// 32 lanes x 32 bits x 16 columns: thread i of the warp gets 16 consecutive columns of lane
// (taddr.lane + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32"
        " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with a swizzle as wide
// as its rows: BK = 64 -> 128-byte rows and 128-byte swizzle (layout 2), BK = 32 ->
// 64-byte rows and 64-byte swizzle (layout 4). Groups of 8 rows are 8 x row bytes apart
// (stride byte offset); the leading byte offset is unused for these layouts; version 1.
// The tile base must be aligned to the swizzle pattern (1024 bytes here).
template <int BK>
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
    static_assert(BK == 64 || BK == 32, "K per stage must be 32 or 64");
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)((8 * BK * 2) >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)(BK == 64 ? 2 : 4) << 61;
    return d;
}
// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, shape M x N.
__device__ __forceinline__ uint32_t instr_desc_bf16(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Adapter id of row t among the merged segments (binary search over offsets).
__device__ __forceinline__ int row_adapter(const int32_t* off, const int32_t* ids, int n, int t) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return ids[lo];
}

// ---------------------------------------------------------------- programmatic dependent launch
// Lets the next kernel of the stream (launched with programmatic stream serialization) start
// while this one finishes; a no-op when none is.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Waits until the kernels this one depends on have completed and their writes are visible; returns
// at once when this kernel was launched without a programmatic dependency.
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------- cross-CTA flags
__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Generic-proxy global writes / reads ordered against the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void epilogue_bar_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kEpilogueThreads) : "memory");
}
// The same named barrier of the four epilogue warps, also ANDing a predicate over them.
__device__ __forceinline__ int epilogue_bar_and(int v) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, %2, q;\n\tselp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(v), "n"(kEpilogueThreads)
        : "memory");
    return r;
}
// Waits until *counter >= value (bounded like wait_bounded).
static __device__ __noinline__ bool wait_count(const int* counter, int value, volatile int* abort_flag, int* status,
                                        uint64_t limit_ns) {
    if (ld_acquire(counter) >= value) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        __nanosleep(64);
        if (ld_acquire(counter) >= value) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, 1);
            *abort_flag = 1;
            return false;
        }
    }
}
// Waits until *flag == value (bounded like wait_bounded).
static __device__ __noinline__ bool wait_flag(const int* flag, int value, volatile int* abort_flag, int* status,
                                       uint64_t limit_ns) {
    if (ld_acquire(flag) == value) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        __nanosleep(64);
        if (ld_acquire(flag) == value) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, 1);
            *abort_flag = 1;
            return false;
        }
    }
}

}  // namespace dev
}  // namespace lora
