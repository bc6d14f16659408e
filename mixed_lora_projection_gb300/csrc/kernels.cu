// sm_103a kernels of the shared-base, per-request LoRA projection.
//
// One persistent, warp-specialised tile GEMM serves both passes of the method ("Two 27B
// models on a single RTX 5090", section 4: the adapter's two thin matrices run beside
// the changed matrix and their output is added), as two kinds of work unit of one launch:
//
//   shrink unit:  U[t, 0:r]   = bf16( s_a * X[t,:] A_a^T )  for the rows of one adapter tile;
//                 rows of the tile that name no adapter get U = 0.
//   fused unit:   acc[t, n]   = X[t,:] W[n,:]^T           (K = d_in)
//                 acc[t, n]  += U[t,:] B_a[n,:]^T         (K = r, adapter tiles only, same
//                                                          TMEM accumulator)
//                 Y[t, n]     = bf16(acc[t, n])
//
// Shrink units come first in the unit order. A fused unit of an adapter tile waits, before
// its expand k-blocks, for a ready flag that the tile's shrink unit publishes (release /
// acquire at GPU scope, plus async-proxy fences because U is written with plain stores and
// read by TMA). A CTA only ever waits for units earlier in the order, which every other
// CTA reaches without waiting, so the dependency cannot cycle.
//
// Per CTA (one per SM, persistent over the work units):
//   warp 0      TMA loads (cp.async.bulk.tensor, swizzle as wide as the K-step) of the A
//               tile (128 rows) and the B tile per stage into a ring;
//   warp 1      owns 512 TMEM columns (two 128x256 fp32 accumulators); issues tcgen05.mma
//               kind::f16 and commits each stage back to the producer and each finished
//               accumulator to the epilogue;
//               both warps run their loops converged and let lane 0 issue (predicated): a
//               lone diverged lane cannot feed the tensor pipe back to back;
//   warps 2..5  epilogue: tcgen05.ld the accumulator (warp w reads TMEM lanes 32*(w%4)..),
//               round to bf16 and store the tile's rows with 16-byte stores.
// Two accumulators let the epilogue of one tile overlap the mainloop of the next.
//
// CTA group 2 (CG = 2): a cluster of two CTAs on an SM pair computes a 256-row unit (two
// row tiles that share the B tile) with tcgen05.mma.cta_group::2 (M = 256). Each CTA loads
// its own 128 A rows and one half of the B tile's rows; the even CTA issues the MMAs, which
// read the peer's half of B from the peer's shared memory, and each CTA's TMEM receives its
// own 128 rows. Each SM thus lands 32 KB per 64-wide K-step instead of 48 KB, which is what
// bounds the single-CTA form (the rate at which an SM's shared memory can be filled).
// Barriers: the even CTA's full barrier counts both CTAs' bytes; its MMA commits release
// both CTAs' stages and accumulators (multicast); both epilogues release the even CTA's
// accumulator barrier.
//
// Every mbarrier wait is bounded by a wall-clock limit; a wait that runs out sets bit 0
// of the status word and a CTA-wide abort flag, and all roles leave their loops, wait
// (bounded) for their own copies and MMAs in flight, free TMEM and return.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

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
__device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
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
// Waits until *flag == epoch (bounded like wait_bounded).
__device__ __noinline__ bool wait_flag(const int* flag, int epoch, volatile int* abort_flag, int* status,
                                       uint64_t limit_ns) {
    if (ld_acquire(flag) == epoch) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        __nanosleep(64);
        if (ld_acquire(flag) == epoch) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, 1);
            *abort_flag = 1;
            return false;
        }
    }
}

// One work unit, as every role decodes it.
struct Unit {
    Tile tile;
    int shrink;      // 1: shrink unit (U rows), 0: fused unit (Y block)
    int tile_index;  // ready-flag slot
    int n0;          // first output column
    int n;           // MMA N of this unit
    int nk;          // k-blocks
};

// The work list of a launch, in global memory or in the kernel parameters.
struct WorkList {
    const Tile* fused;
    const Tile* shrink;
    const int32_t* seg_off;
    const int32_t* seg_id;
    const float* scales;
    const CUtensorMap* tm_a;
    const CUtensorMap* tm_b;
};

__device__ __forceinline__ WorkList resolve_work_list(const GemmParams& p) {
    WorkList wl;
    if (p.inline_wl) {
        // the offset is stored, not derived from n_fused: a launch of the shrink units alone
        // runs with n_fused = 0 over the same list
        wl.fused = p.inline_tiles;
        wl.shrink = p.inline_tiles + p.inline_shrink_off;
        wl.seg_off = p.inline_seg;
        wl.seg_id = p.inline_seg + p.n_seg + 1;
        wl.scales = p.inline_scales;
        wl.tm_b = p.inline_maps;
        wl.tm_a = p.inline_maps + kInlineAdapters;
    } else {
        wl.fused = p.fused_tiles;
        wl.shrink = p.shrink_tiles;
        wl.seg_off = p.seg_off;
        wl.seg_id = p.seg_id;
        wl.scales = p.scales;
        wl.tm_b = p.tm_b;
        wl.tm_a = p.tm_a;
    }
    return wl;
}

__device__ __forceinline__ Unit decode_unit(const GemmParams& p, const WorkList& wl, int u, int rank) {
    Unit r;
    const int cs = p.cluster_size;
    if (u < p.n_shrink) {
        r.tile = wl.shrink[u * cs + rank];
        r.shrink = 1;
        r.tile_index = r.tile.fused_index;
        r.n0 = 0;
        r.n = p.shrink_n;
        r.nk = p.k_main_blocks;
    } else {
        const int v = u - p.n_shrink;
        int ti, nt;
        if (p.m_fastest == 2) {
            // column-tile groups of raster_group: all row tiles of a group, then the next group
            const int per = p.n_fused * p.raster_group;
            const int g = v / per, rr = v % per;
            const int gw = min(p.raster_group, p.n_ntiles - g * p.raster_group);
            ti = rr / gw;
            nt = g * p.raster_group + rr % gw;
        } else {
            ti = p.m_fastest ? (v % p.n_fused) : (v / p.n_ntiles);
            nt = p.m_fastest ? (v / p.n_fused) : (v % p.n_ntiles);
        }
        r.tile = wl.fused[ti * cs + rank];
        r.shrink = 0;
        r.tile_index = r.tile.fused_index;
        r.n0 = nt * p.tile_n;
        r.n = p.tile_n;
        r.nk = p.k_main_blocks + (r.tile.adapter ? p.k_lora_blocks : 0);
    }
    return r;
}

template <int BK, int CG, int QW>
__global__ void __launch_bounds__(QW ? kThreadsW4 : kThreads, 1)
    lora_gemm_kernel(const __grid_constant__ GemmParams p) {
    static_assert(!QW || BK == 64, "the 4-bit base uses 64-wide K-steps (32 packed bytes per row)");
    constexpr uint32_t kStageA = kTileM * BK * 2;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // carve: rings (1024-aligned), then barriers, then the TMEM slot and the abort flag
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const int stages = p.stages;
    const int b_rows = (p.tile_n > p.shrink_n ? p.tile_n : p.shrink_n) / CG;  // this CTA's B rows
    const uint32_t b_stage_bytes = (uint32_t)b_rows * BK * 2;
    uint8_t* a_ring = base;
    uint8_t* b_ring = a_ring + (size_t)stages * kStageA;
    // 4-bit base: staging rings of the packed tile (32 bytes per row) and its scales
    const int q_rows = QW ? p.tile_n / CG : 0;
    const uint32_t q_stage_bytes = (uint32_t)q_rows * (BK / 2);
    const uint32_t s_stage_bytes = ((uint32_t)q_rows * 2 + 127u) & ~127u;
    uint8_t* q_ring = b_ring + (size_t)stages * b_stage_bytes;
    uint8_t* s_ring = q_ring + (size_t)stages * q_stage_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_ring + (size_t)stages * s_stage_bytes);
    uint64_t* full = bars;
    uint64_t* empty = full + stages;
    uint64_t* pfull = empty + stages;
    uint64_t* tfull = pfull + stages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = CG > 1 ? (int)cluster_ctarank() : 0;
    const bool leader = rank == 0;                 // issues the MMAs of the pair
    const int group = (int)blockIdx.x / CG;        // cluster index
    const int n_groups = (int)gridDim.x / CG;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            // the producer's arrive, plus one arrive per converter warp of each CTA of the group
            mbar_init(smem_addr(&full[s]), 1 + (QW ? CG * (kConvertThreads / 32) : 0));
            mbar_init(smem_addr(&empty[s]), 1);
            mbar_init(smem_addr(&pfull[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_addr(&tfull[a]), 1);
            mbar_init(smem_addr(&tempty[a]), CG * kEpilogueThreads);  // both CTAs' epilogues
        }
        mbar_init(smem_addr(drain), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc<CG>(smem_addr(tmem_slot), 2 * kAccCols);
    tc_fence_before();
    if (CG > 1) cluster_sync();  // barrier inits visible to the peer before any remote arrive
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int n_units = p.n_shrink + p.n_fused * p.n_ntiles;
    const uint64_t limit = p.wait_limit_ns;
    const WorkList wl = resolve_work_list(p);

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // The whole warp runs the loop (converged); lane 0 issues.
        const uint32_t issuer = lane == 0 ? 1u : 0u;
        if (!p.debug_stall) {
            if (lane == 0) {
                tma_prefetch_desc(&p.tm_x);
                if (p.n_fused) {
                    tma_prefetch_desc(QW ? &p.tm_wq : &p.tm_w);
                    if (QW) tma_prefetch_desc(&p.tm_ws);
                    tma_prefetch_desc(&p.tm_u);
                }
            }
            __syncwarp();
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            int acquired_a = -1, acquired_b = -1;  // adapters whose global tensor maps were acquired
            bool ok = true;
            for (int u = group; u < n_units && ok; u += n_groups) {
                const Unit w = decode_unit(p, wl, u, rank);
                const int ad = w.tile.adapter;
                const CUtensorMap* bmain = &p.tm_w;
                if (w.shrink) {
                    bmain = &wl.tm_a[ad - 1];
                    if (acquired_a != ad) {
                        if (!p.inline_wl) tensormap_acquire(bmain);
                        acquired_a = ad;
                    }
                } else if (ad && acquired_b != ad) {
                    if (!p.inline_wl) tensormap_acquire(&wl.tm_b[ad - 1]);
                    acquired_b = ad;
                }
                const int half = w.n / CG;                       // B rows this CTA loads
                // bytes the (even CTA's) full barrier receives per stage, from the whole group
                const uint32_t tx = CG * (kStageA + (uint32_t)half * BK * 2);
                // 4-bit base: TMA brings only A to the full barrier; the B tile of a base step
                // comes from the converter warps, its packed form lands on pfull
                const bool w4_unit = QW && !w.shrink;
                const uint32_t tx_w4 = CG * kStageA;
                const uint32_t ptx = (uint32_t)half * (BK / 2) + (uint32_t)half * 2;
                for (int kb = 0; kb < w.nk; ++kb) {
                    if (kb == p.k_main_blocks && p.flags) {
                        // the expand reads U rows written by this tile's shrink unit
                        int fok = 1;
                        if (lane == 0) fok = wait_flag(&p.flags[w.tile_index], p.epoch, abort_flag, p.status, limit);
                        if (!__shfl_sync(0xffffffffu, fok, 0)) {
                            ok = false;
                            break;
                        }
                        fence_proxy_async_global();
                    }
                    if (!wait_warp(smem_addr(&empty[stage]), phase ^ 1, abort_flag, p.status, limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb_local = smem_addr(&full[stage]);
                    const bool main = kb < p.k_main_blocks;
                    const bool w4_step = w4_unit && main;
                    mbar_arrive_expect_tx(fb_local, w4_step ? tx_w4 : tx, leader ? issuer : 0u);
                    const uint32_t fb = CG > 1 ? map_to_rank(fb_local, 0) : fb_local;
                    const uint32_t sa = smem_addr(a_ring + (size_t)stage * kStageA);
                    const uint32_t sb = smem_addr(b_ring + (size_t)stage * b_stage_bytes);
                    const int k = main ? kb * BK : (kb - p.k_main_blocks) * BK;
                    tma_load_2d<CG>(sa, main ? &p.tm_x : &p.tm_u, fb, k, w.tile.row0, issuer);
                    if (w4_step) {
                        // packed rows and this K-step's scales, into this CTA's staging ring
                        const uint32_t pb = smem_addr(&pfull[stage]);
                        mbar_arrive_expect_tx(pb, ptx, issuer);
                        tma_load_2d<1>(smem_addr(q_ring + (size_t)stage * q_stage_bytes), &p.tm_wq, pb, kb * (BK / 2),
                                       w.n0 + rank * half, issuer);
                        tma_load_2d<1>(smem_addr(s_ring + (size_t)stage * s_stage_bytes), &p.tm_ws, pb,
                                       w.n0 + rank * half, (kb * BK) / kW4Group, issuer);
                    } else {
                        tma_load_2d<CG>(sb, main ? bmain : &wl.tm_b[ad - 1], fb, k, w.n0 + rank * half, issuer);
                    }
                    ++issued;
                    if (++stage == stages) { stage = 0; phase ^= 1; }
                }
            }
            if (lane == 0) {
                if (!ok && leader) {
                    // wait (bounded, ignoring the abort flag) for the copies still in flight
                    long long first = issued > stages ? issued - stages : 0;
                    for (long long j = first; j < issued; ++j)
                        wait_bounded(smem_addr(&full[j % stages]), (uint32_t)((j / stages) & 1), abort_flag,
                                     p.status, limit, false);
                }
                if (CG > 1) {
                    // the pair's MMAs have released every stage of this CTA: no copy into it and
                    // no remote arrive on its barriers is still pending when it exits
                    long long first = issued > stages ? issued - stages : 0;
                    for (long long j = first; j < issued; ++j)
                        wait_bounded(smem_addr(&empty[j % stages]), (uint32_t)((j / stages) & 1), abort_flag,
                                     p.status, limit, false);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (even CTA)
        // The whole warp runs the loop (converged); lane 0 issues the MMAs and commits.
        const uint32_t issuer = lane == 0 ? 1u : 0u;
        if (leader) {
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int u = group; u < n_units && ok; u += n_groups, ++it) {
                const Unit w = decode_unit(p, wl, u, rank);
                const uint32_t idesc = instr_desc_bf16(kTileM * CG, w.n);
                const int acc = it & 1;
                if (!wait_warp(smem_addr(&tempty[acc]), ((it >> 1) & 1) ^ 1, abort_flag, p.status, limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * kAccCols);
                for (int kb = 0; kb < w.nk; ++kb) {
                    if (!wait_warp(smem_addr(&full[stage]), phase, abort_flag, p.status, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = smem_desc<BK>(smem_addr(a_ring + (size_t)stage * kStageA));
                    const uint64_t bd = smem_desc<BK>(smem_addr(b_ring + (size_t)stage * b_stage_bytes));
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        // advance 16 bf16 = 32 bytes along K inside the swizzled rows
                        mma_bf16<CG>(d, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), idesc,
                                     (kb > 0 || k > 0) ? 1u : 0u, issuer);
                    }
                    mma_commit<CG>(smem_addr(&empty[stage]), issuer);
                    if (++stage == stages) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                mma_commit<CG>(smem_addr(&tfull[acc]), issuer);
            }
            // every MMA this warp issued has completed before TMEM is released
            mma_commit_local<CG>(smem_addr(drain), issuer);
            if (lane == 0) wait_bounded(smem_addr(drain), 0, abort_flag, p.status, limit, false);
        }
    } else if (QW && warp >= 6) {
        // ------------------------------------------------------------ 4-bit converter (warps 6..9)
        // Base K-steps of fused units: packed int4 rows + scales (staging ring) -> bf16 B tile in
        // the 128-byte-swizzled layout the MMA reads. W[n,k] = q * s, q = signed nibble (low
        // nibble = even k); (128 + (q ^ 8) - 136) is q exactly, then one RNE multiply by s.
        // Other K-steps (expand, shrink) load B by TMA; the converters only count themselves in.
        const int ct = threadIdx.x - 6 * 32;
        const uint32_t full_target_rank = 0;
        const __nv_bfloat162 magic = __floats2bfloat162_rn(136.0f, 136.0f);
        int stage = 0;
        uint32_t phase = 0, pbits = 0;
        bool ok = true;
        for (int u = group; u < n_units && ok; u += n_groups) {
            const Unit w = decode_unit(p, wl, u, rank);
            const bool w4_unit = !w.shrink;
            const int rows = w.n / CG;
            for (int kb = 0; kb < w.nk; ++kb) {
                if (!wait_warp(smem_addr(&empty[stage]), phase ^ 1, abort_flag, p.status, limit)) {
                    ok = false;
                    break;
                }
                if (w4_unit && kb < p.k_main_blocks) {
                    if (!wait_warp(smem_addr(&pfull[stage]), (pbits >> stage) & 1u, abort_flag, p.status, limit)) {
                        ok = false;
                        break;
                    }
                    pbits ^= 1u << stage;
                    const uint8_t* qs = q_ring + (size_t)stage * q_stage_bytes;
                    const __nv_bfloat16* ss = reinterpret_cast<const __nv_bfloat16*>(s_ring + (size_t)stage * s_stage_bytes);
                    uint8_t* bs = b_ring + (size_t)stage * b_stage_bytes;
                    for (int r = ct; r < rows; r += kConvertThreads) {
                        const uint4 q0 = *reinterpret_cast<const uint4*>(qs + (size_t)r * 32);
                        const uint4 q1 = *reinterpret_cast<const uint4*>(qs + (size_t)r * 32 + 16);
                        const __nv_bfloat162 s2 = __bfloat162bfloat162(ss[r]);
                        const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const uint32_t wv = words[c] ^ 0x88888888u;  // nibbles to offset binary q + 8
                            uint32_t o[4];
#pragma unroll
                            for (int pp = 0; pp < 4; ++pp) {
                                const uint32_t v = ((wv >> (8 * pp)) & 0xFu) | (((wv >> (8 * pp + 4)) & 0xFu) << 16) |
                                                   0x43004300u;  // bf16 pair 128 + (q + 8)
                                __nv_bfloat162 t = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&v), magic);
                                t = __hmul2(t, s2);
                                o[pp] = *reinterpret_cast<const uint32_t*>(&t);
                            }
                            *reinterpret_cast<uint4*>(bs + (size_t)r * 128 + (((uint32_t)c ^ ((uint32_t)r & 7u)) << 4)) =
                                make_uint4(o[0], o[1], o[2], o[3]);
                        }
                    }
                    // generic stores -> visible to the tensor core (async proxy) before the arrive
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                __syncwarp();
                if (lane == 0) {
                    const uint32_t fb_local = smem_addr(&full[stage]);
                    if (CG > 1)
                        mbar_arrive_cluster(map_to_rank(fb_local, full_target_rank));
                    else
                        mbar_arrive(fb_local);
                }
                if (++stage == stages) { stage = 0; phase ^= 1; }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 2..5)
        const int q = warp & 3;                      // TMEM lane quadrant this warp may read
        const int r_local = q * 32 + lane;           // tile row held by this thread
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        int it = 0;
        for (int u = group; u < n_units; u += n_groups, ++it) {
            const Unit w = decode_unit(p, wl, u, rank);
            const int acc = it & 1;
            int ok = 1;
            if (lane == 0)
                ok = wait_bounded(smem_addr(&tfull[acc]), (it >> 1) & 1, abort_flag, p.status, limit, true);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const int row = w.tile.row0 + r_local;
            const bool row_ok = r_local < w.tile.nrows;
            float scale = 1.0f;
            __nv_bfloat16* out;
            int n_out;
            if (w.shrink) {
                const int a = row_ok ? row_adapter(wl.seg_off, wl.seg_id, p.n_seg, row) : 0;
                scale = (a == w.tile.adapter) ? wl.scales[w.tile.adapter - 1] : 0.0f;
                out = reinterpret_cast<__nv_bfloat16*>(p.u) + (size_t)row * p.rank;
                n_out = p.rank;
            } else {
                out = reinterpret_cast<__nv_bfloat16*>(p.y) + (size_t)row * p.d_out + w.n0;
                n_out = p.d_out - w.n0;
            }
            const uint32_t taddr = tmem_base + (uint32_t)(acc * kAccCols) + lane_off;
            for (int c = 0; c < w.n; c += 32) {
                uint32_t v[32];
                const bool two = c + 16 < w.n;  // w.n is a multiple of 16
                tmem_ld16(taddr + (uint32_t)c, v);
                if (two) tmem_ld16(taddr + (uint32_t)c + 16, v + 16);
                tmem_ld_wait();
                if (row_ok) {
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        if ((h < 2 || two) && c + 8 * h < n_out) {
                            uint4 o;
                            o.x = pack_bf16x2(__uint_as_float(v[8 * h + 0]) * scale, __uint_as_float(v[8 * h + 1]) * scale);
                            o.y = pack_bf16x2(__uint_as_float(v[8 * h + 2]) * scale, __uint_as_float(v[8 * h + 3]) * scale);
                            o.z = pack_bf16x2(__uint_as_float(v[8 * h + 4]) * scale, __uint_as_float(v[8 * h + 5]) * scale);
                            o.w = pack_bf16x2(__uint_as_float(v[8 * h + 6]) * scale, __uint_as_float(v[8 * h + 7]) * scale);
                            *reinterpret_cast<uint4*>(out + c + 8 * h) = o;
                        }
                    }
                }
            }
            tc_fence_before();
            if (CG > 1)
                mbar_arrive_cluster(map_to_rank(smem_addr(&tempty[acc]), 0));  // the even CTA's barrier
            else
                mbar_arrive(smem_addr(&tempty[acc]));
            if (w.shrink && p.flags && w.tile_index >= 0) {
                // publish this tile's U rows to the fused units that wait for them
                fence_proxy_async_global();
                epilogue_bar_sync();
                if (warp == 2 && lane == 0) {
                    __threadfence();
                    st_release(&p.flags[w.tile_index], p.epoch);
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    if (CG > 1) cluster_sync();  // neither CTA of the pair touches the other's memory after this
    else __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, 2 * kAccCols);
    }
}

}  // namespace dev

size_t gemm_smem_bytes(int b_tile_rows, int stages, int bk, int w4_rows) {
    const size_t w4 = w4_rows ? (size_t)w4_rows * (bk / 2) + (((size_t)w4_rows * 2 + 127) & ~(size_t)127) : 0;
    return 1024 + (size_t)stages * ((size_t)kTileM * bk * 2 + (size_t)b_tile_rows * bk * 2 + w4) +
           8 * (3 * (size_t)stages + 5) + 16;
}

template <int BK, int CG, int QW>
static cudaError_t set_smem_attr() {
    return cudaFuncSetAttribute(dev::lora_gemm_kernel<BK, CG, QW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemLimit);
}

cudaError_t gemm_prepare_device() {
    cudaError_t e;
    if ((e = set_smem_attr<64, 1, 0>()) != cudaSuccess) return e;
    if ((e = set_smem_attr<64, 2, 0>()) != cudaSuccess) return e;
    if ((e = set_smem_attr<32, 1, 0>()) != cudaSuccess) return e;
    if ((e = set_smem_attr<32, 2, 0>()) != cudaSuccess) return e;
    if ((e = set_smem_attr<64, 1, 1>()) != cudaSuccess) return e;
    return set_smem_attr<64, 2, 1>();
}

static void launch_config(const GemmParams& p, int grid, cudaStream_t stream, cudaLaunchConfig_t* cfg,
                          cudaLaunchAttribute* attr) {
    const int b_rows = (p.tile_n > p.shrink_n ? p.tile_n : p.shrink_n) / p.cluster_size;
    memset(cfg, 0, sizeof(*cfg));
    cfg->gridDim = dim3(grid, 1, 1);
    cfg->blockDim = dim3(p.w4 ? kThreadsW4 : kThreads, 1, 1);
    cfg->dynamicSmemBytes = gemm_smem_bytes(b_rows, p.stages, p.bk, p.w4 ? p.tile_n / p.cluster_size : 0);
    cfg->stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.cluster_size;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg->attrs = attr;
    cfg->numAttrs = 1;
}

template <typename F>
static cudaError_t dispatch(const GemmParams& p, F&& f) {
    if (p.w4) {
        if (p.bk == 64 && p.cluster_size == 1) return f(dev::lora_gemm_kernel<64, 1, 1>);
        if (p.bk == 64 && p.cluster_size == 2) return f(dev::lora_gemm_kernel<64, 2, 1>);
        return cudaErrorInvalidValue;
    }
    if (p.bk == 64 && p.cluster_size == 1) return f(dev::lora_gemm_kernel<64, 1, 0>);
    if (p.bk == 64 && p.cluster_size == 2) return f(dev::lora_gemm_kernel<64, 2, 0>);
    if (p.bk == 32 && p.cluster_size == 1) return f(dev::lora_gemm_kernel<32, 1, 0>);
    if (p.bk == 32 && p.cluster_size == 2) return f(dev::lora_gemm_kernel<32, 2, 0>);
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm(const GemmParams& p, int grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    launch_config(p, grid, stream, &cfg, attr);
    return dispatch(p, [&](auto kernel) { return cudaLaunchKernelEx(&cfg, kernel, p); });
}

int gemm_max_clusters(const GemmParams& p) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    launch_config(p, p.cluster_size, nullptr, &cfg, attr);
    int n = 0;
    cudaError_t e = dispatch(p, [&](auto kernel) { return cudaOccupancyMaxActiveClusters(&n, kernel, &cfg); });
    if (e != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace lora
