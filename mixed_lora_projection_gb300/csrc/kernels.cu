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
// CTA reaches without waiting, so the dependency cannot cycle, given that the grid's CTAs
// are resident together (such launches are cooperative launches). The last CTA to finish
// clears the flags, so a launch depends on no value left by an earlier one (CUDA graphs
// replay it unchanged).
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
// Two unit forms wider than one MMA (SM pairs, 224 threads, each an instantiation of its own, so
// that neither changes the code of the others): each 16-wide K step takes a second MMA over the B
// stage rows past the first MMA's, issued by warp 6 beside warp 1's first (one warp waits ~80
// cycles between MMAs whatever their width), into the accumulator columns after the first MMA's;
// one accumulator of up to 512 columns, so a unit's epilogue no longer overlaps the next unit's
// MMAs.
//   token-column units (FORM 1, p.yt): for batches of at most 512 rows on one adapter, a unit
//     computes a block of Y^T: 256 output features (W rows as the A operand, 128 per CTA) for
//     every token row of the batch (X rows as the B operand, half of them per CTA), so W is read
//     once and no row tile is padded; the epilogue maps accumulator columns back to token rows
//     through a per-warp shared-memory buffer;
//   wide row tiles (FORM 2, tile_n of 272 to 512 columns): 256-row units as on SM pairs, with
//     more output columns per unit, so that a projection's units fill whole waves of SM pairs
//     (2,048 rows of a 5,120-column projection on 76 SM pairs: 144 units of 288 columns, two
//     waves, instead of 160 of 256, three); the epilogue maps accumulator columns back to output
//     columns in the order of the pair's B stage rows.
// The sums keep their order whatever the unit's shape, so the bits equal those of 256-column
// row tiles.
//
// Every mbarrier wait is bounded by a wall-clock limit; a wait that runs out sets bit 0
// of the status word and a CTA-wide abort flag, and all roles leave their loops, wait
// (bounded) for their own copies and MMAs in flight, free TMEM and return.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "dev_common.cuh"
#include "lora_internal.h"

namespace lora {
namespace dev {
// One work unit, as every role decodes it.
struct Unit {
    Tile tile;
    int shrink;      // 1: shrink unit (U rows), 0: fused unit (Y block)
    int tile_index;  // ready-flag slot
    int n0;          // first output column
    int n;           // MMA N of this unit
    int nk;          // k-blocks (base K-steps of this unit, then the expand's)
    int kb0;         // first base K-step
    int kmain;       // base K-steps of this unit
    int part;        // K part when the launch splits K (0 .. k_split - 1), else 0
    int slot;        // K parts: this block's counter pair
    int pchunk;      // K parts: float4 column chunk of the block's first column in `partials`
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

template <bool YT>
__device__ __forceinline__ Unit decode_unit(const GemmParams& p, const WorkList& wl, int u, int rank) {
    Unit r;
    const int cs = p.cluster_size;
    // with K split into S parts every block (shrink or fused) is S consecutive units, one per
    // part of the base K-steps (k_chunk each, the last one the rest); the expand's K-steps go with
    // the last part
    const int S = p.k_split > 1 ? p.k_split : 1;
    const bool split = S > 1;
    const int v0 = u / S;
    r.part = u - v0 * S;
    r.kb0 = r.part * p.k_chunk;
    r.kmain = r.part == S - 1 ? p.k_main_blocks - r.kb0 : p.k_chunk;
    const int srt = p.shrink_ntiles > 1 ? p.shrink_ntiles : 1;   // rank tiles per shrink group
    if (v0 < p.n_shrink * srt) {
        const int g = v0 / srt;
        r.tile = wl.shrink[g * cs + rank];
        r.shrink = 1;
        r.tile_index = r.tile.fused_index;
        r.n0 = (v0 - g * srt) * p.shrink_n;
        r.n = p.shrink_n;
        r.nk = r.kmain;
        r.slot = p.shrink_slot0 + g * cs + rank;
        r.pchunk = p.u_chunk0;
    } else if (YT) {
        // token-column unit: 256 output features (128 per CTA) for every token row
        const int v = v0 - p.n_shrink;
        r.tile = wl.fused[rank];
        r.tile.adapter = p.yt_adapter;
        r.shrink = 0;
        r.tile_index = 0;
        r.n0 = v * kTileM * cs;
        r.n = 2 * p.yt_h;
        r.nk = r.kmain + (p.yt_adapter ? p.k_lora_blocks : 0);
        r.slot = 0;
        r.pchunk = 0;
    } else {
        const int v = v0 - p.n_shrink;
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
        r.nk = r.kmain + ((r.tile.adapter && r.part == S - 1) ? p.k_lora_blocks : 0);
        r.slot = r.tile.split_index * p.n_ntiles + nt;
        r.pchunk = r.n0 >> 2;
    }
    return r;
}

// Row of the pair's B stages (the even CTA's `rows` rows, then the odd CTA's) that accumulator
// column c of a two-MMA unit multiplies: the first MMA's columns [0, 2 h) hold stage rows [0, h)
// of the even CTA, then of the odd CTA; the second MMA's columns hold stage rows [h, rows) of the
// even CTA, then of the odd CTA. It is the token row of a token-column unit and the output
// column (from the unit's first) of a wide row tile.
__device__ __forceinline__ int pair_b_row(int c, int h, int rows) {
    if (c < 2 * h) return c < h ? c : rows + c - h;
    const int cc = c - 2 * h, h1 = rows - h;
    return cc < h1 ? h + cc : rows + h + cc - h1;
}

// Epilogue of a token-column unit: this thread's TMEM lane is output feature f and each
// accumulator column a token row. Each 32-column chunk goes through the warp's 2 KB buffer
// ([32 tokens][32 features] bf16, written one token column per thread) and leaves as 16-byte
// stores: thread l writes 8 features of token row (l + 32 i) / 4, so a warp's store covers 8
// token rows of 64 bytes.
__device__ __forceinline__ void yt_store(const GemmParams& p, uint32_t taddr, int f0, int lane, uint8_t* stage) {
    const int h = p.yt_h, rows = p.yt_rows, n = 2 * p.yt_rows, T = p.yt_tokens;
    __nv_bfloat16* sb = reinterpret_cast<__nv_bfloat16*>(stage);
    for (int c = 0; c < n; c += 32) {
        uint32_t v[32];
        const bool two = c + 16 < n;  // n is a multiple of 16
        tmem_ld16(taddr + (uint32_t)c, v);
        if (two) tmem_ld16(taddr + (uint32_t)c + 16, v + 16);
        tmem_ld_wait();
        __syncwarp();                 // the buffer's previous chunk has been read by every lane
#pragma unroll
        for (int t = 0; t < 32; ++t) sb[t * 32 + lane] = __float2bfloat16_rn(__uint_as_float(v[t]));
        __syncwarp();
        const int m = two ? 32 : 16;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = lane + 32 * i;      // 16-byte piece k: token column k / 4, features 8 (k % 4) ..
            const int tc = k >> 2, seg = k & 3;
            const int tok = pair_b_row(c + tc, h, rows);
            const int f = f0 + 8 * seg;
            if (tc < m && tok < T && f < p.d_out) {
                const uint4 val = *reinterpret_cast<const uint4*>(stage + (size_t)k * 16);
                *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.y) + (size_t)tok * p.d_out + f) = val;
            }
        }
    }
}

// FORM: kFormRows (row tiles), kFormTokenColumns, kFormWideRows (see the file header).
template <int BK, int CG, int FORM>
__global__ void __launch_bounds__(FORM != kFormRows ? kThreadsWide : kThreads, 1)
    lora_gemm_kernel(const __grid_constant__ GemmParams p) {
    constexpr bool YT = FORM == kFormTokenColumns;   // token-column units
    constexpr bool WIDE = FORM != kFormRows;         // two MMAs per K16 step, two MMA warps
    static_assert(!WIDE || (CG == 2 && BK == 64), "two-MMA units run on SM pairs with 64-wide K-steps");
    // A stage: the tile's rows of X (or U) for this K-step; a batch of one short tile loads
    // only its rows (a_rows < 128), and the MMA's remaining A rows read unrelated shared memory
    // whose output rows are never stored
    const uint32_t kStageA = (uint32_t)(p.a_rows ? p.a_rows : kTileM) * BK * 2;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // carve: rings (1024-aligned), then barriers, then the TMEM slot and the abort flag
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const int stages = p.stages;
    // this CTA's B rows per stage: output-tile rows of W, rows of A_a, or token rows
    const int b_rows = YT ? max(p.yt_rows, p.shrink_n / CG) : (p.tile_n > p.shrink_n ? p.tile_n : p.shrink_n) / CG;
    const uint32_t b_stage_bytes = (uint32_t)b_rows * BK * 2;
    // units wider than one accumulator take all of TMEM: one accumulator at a time
    const int n_acc = (WIDE && (YT ? 2 * p.yt_rows : p.tile_n) > kAccCols) ? 1 : 2;
    uint8_t* a_ring = base;
    uint8_t* b_ring = a_ring + (size_t)stages * kStageA;
    // token-column units: the epilogue warps' transposing buffers (2 KB each) follow the rings
    uint8_t* yt_stage = b_ring + (size_t)stages * b_stage_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(yt_stage + (YT ? kYtStageBytes : 0));
    uint64_t* full = bars;
    uint64_t* empty = full + stages;
    uint64_t* tfull = empty + stages;
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

    // two-MMA units: two MMA warps (1 and 6) commit every stage, accumulator and drain
    constexpr uint32_t kIssuers = WIDE ? 2 : 1;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), kIssuers);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_addr(&tfull[a]), kIssuers);
            mbar_init(smem_addr(&tempty[a]), CG * kEpilogueThreads);  // both CTAs' epilogues
        }
        mbar_init(smem_addr(drain), kIssuers);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc<CG>(smem_addr(tmem_slot), 2 * kAccCols);
    tc_fence_before();
    if (CG > 1) cluster_sync();  // barrier inits visible to the peer before any remote arrive
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int n_units = (p.n_shrink * (p.shrink_ntiles > 1 ? p.shrink_ntiles : 1) + p.n_fused * p.n_ntiles) *
                        (p.k_split > 1 ? p.k_split : 1);
    const uint64_t limit = p.wait_limit_ns;
    const WorkList wl = resolve_work_list(p);
    // the next call's kernel may start on the SMs this one leaves, and stream its first W tiles
    if (p.pdl && threadIdx.x == 0) griddep_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // The whole warp runs the loop (converged); lane 0 issues.
        const uint32_t issuer = lane == 0 ? 1u : 0u;
        if (!p.debug_stall) {
            if (lane == 0) {
                tma_prefetch_desc(&p.tm_x);
                if (p.n_fused) {
                    tma_prefetch_desc(&p.tm_w);
                    tma_prefetch_desc(&p.tm_u);
                    if (YT) tma_prefetch_desc(&p.tm_xt);
                }
            }
            __syncwarp();
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            int acquired_a = -1, acquired_b = -1;  // adapters whose global tensor maps were acquired
            bool ok = true;
            // Launched ahead of the previous kernel's end: the W tiles of the first unit's first
            // ring stages (W is not written by that kernel) are requested before the wait, into
            // stages that are free at the start; their X rows follow the wait.
            int pre = 0;
            if (p.pdl) {
                if (group < n_units) {
                    const Unit w0 = decode_unit<YT>(p, wl, group, rank);
                    if (!w0.shrink) {
                        // W is the B operand, or the A operand of a token-column unit
                        const int half0 = w0.n / CG;
                        const uint32_t tx0 = YT ? CG * (kStageA + (uint32_t)p.yt_rows * BK * 2)
                                                  : CG * (kStageA + (uint32_t)half0 * BK * 2);
                        pre = w0.kmain < stages ? w0.kmain : stages;
                        for (int kb = 0; kb < pre; ++kb) {
                            const uint32_t fb_local = smem_addr(&full[kb]);
                            mbar_arrive_expect_tx(fb_local, tx0, leader ? issuer : 0u);
                            const uint32_t fb = CG > 1 ? map_to_rank(fb_local, 0) : fb_local;
                            if (YT)
                                tma_load_2d<CG>(smem_addr(a_ring + (size_t)kb * kStageA), &p.tm_w, fb,
                                                (w0.kb0 + kb) * BK, w0.n0 + rank * kTileM, issuer);
                            else
                                tma_load_2d<CG>(smem_addr(b_ring + (size_t)kb * b_stage_bytes), &p.tm_w, fb,
                                                (w0.kb0 + kb) * BK, w0.n0 + rank * half0, issuer);
                        }
                    }
                }
                griddep_wait();
            }
            for (int u = group; u < n_units && ok; u += n_groups) {
                const Unit w = decode_unit<YT>(p, wl, u, rank);
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
                const bool yt_unit = YT && !w.shrink;
                const int half = w.n / CG;                       // B rows this CTA loads
                // bytes the (even CTA's) full barrier receives per stage, from the whole group
                const uint32_t tx = yt_unit ? CG * (kStageA + (uint32_t)p.yt_rows * BK * 2)
                                            : CG * (kStageA + (uint32_t)half * BK * 2);
                for (int kb = 0; kb < w.nk; ++kb) {
                    if (kb == w.kmain && p.flags) {
                        // the expand reads U rows written by this tile's shrink unit (a token-column
                        // unit: by every tile's)
                        int fok = 1;
                        if (lane == 0) {
                            if (yt_unit) {
                                for (int i = 0; i < p.n_flags && fok; ++i)
                                    fok = wait_flag(&p.flags[i], 1, abort_flag, p.status, limit);
                            } else {
                                fok = wait_flag(&p.flags[w.tile_index], 1, abort_flag, p.status, limit);
                            }
                        }
                        if (!__shfl_sync(0xffffffffu, fok, 0)) {
                            ok = false;
                            break;
                        }
                        fence_proxy_async_global();
                    }
                    // a stage whose W tile went out before the dependency wait: armed and free
                    const bool prefetched = issued < pre;
                    if (!prefetched && !wait_warp(smem_addr(&empty[stage]), phase ^ 1, abort_flag, p.status, limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb_local = smem_addr(&full[stage]);
                    const bool main = kb < w.kmain;
                    if (!prefetched) mbar_arrive_expect_tx(fb_local, tx, leader ? issuer : 0u);
                    const uint32_t fb = CG > 1 ? map_to_rank(fb_local, 0) : fb_local;
                    const uint32_t sa = smem_addr(a_ring + (size_t)stage * kStageA);
                    const uint32_t sb = smem_addr(b_ring + (size_t)stage * b_stage_bytes);
                    const int k = main ? (w.kb0 + kb) * BK : (kb - w.kmain) * BK;
                    if (yt_unit) {
                        // A: this CTA's 128 output features of W (B_a); B: its token rows of X (U)
                        if (!prefetched)
                            tma_load_2d<CG>(sa, main ? &p.tm_w : &wl.tm_b[ad - 1], fb, k, w.n0 + rank * kTileM,
                                            issuer);
                        tma_load_2d<CG>(sb, main ? &p.tm_xt : &p.tm_u, fb, k, rank * p.yt_rows, issuer);
                    } else {
                        tma_load_2d<CG>(sa, main ? &p.tm_x : &p.tm_u, fb, k, main ? w.tile.row0 : w.tile.u_row,
                                        issuer);
                        if (!prefetched)
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
    } else if (warp == 1 || (WIDE && warp == 6)) {
        // ------------------------------------------------------------ MMA issuer (even CTA)
        // The whole warp runs the loop (converged); lane 0 issues the MMAs and commits. In the
        // two-MMA instantiations warp 6 issues each K16 step's second MMA (the B stage rows past the
        // first MMA's) beside warp 1's first: one warp waits ~80 cycles between MMAs whatever their
        // width, two warps keep the tensor pipe fed with both. Both commit every stage and
        // accumulator (the barriers count two arrivals).
        const uint32_t issuer = lane == 0 ? 1u : 0u;
        const bool second = WIDE && warp == 6;
        if (p.pdl) griddep_wait();
        if (leader) {
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int u = group; u < n_units && ok; u += n_groups, ++it) {
                const Unit w = decode_unit<YT>(p, wl, u, rank);
                // two-MMA units: the first MMA takes B stage rows [0, r1) of each CTA (N = n1), a
                // second, when n2 > 0, the rest (N = n2) into the accumulator columns after the
                // first's: token-column units past yt_h token rows per CTA, row tiles past 256 columns
                int n1 = w.n, n2 = 0, r1 = 0;
                if (WIDE && !w.shrink) {
                    if (YT) {
                        n2 = 2 * (p.yt_rows - p.yt_h);
                        r1 = p.yt_h;
                    } else if (w.n > kAccCols) {
                        n1 = kAccCols;
                        n2 = w.n - kAccCols;
                        r1 = kAccCols / CG;
                    }
                }
                const uint32_t idesc = instr_desc_bf16(kTileM * CG, n1);
                const bool mma2 = n2 > 0;
                const uint32_t idesc2 = instr_desc_bf16(kTileM * CG, mma2 ? n2 : 16);
                const uint64_t b_off2 = (uint64_t)((r1 * BK * 2) >> 4);
                const int acc = it % n_acc;
                if (!wait_warp(smem_addr(&tempty[acc]), ((it / n_acc) & 1) ^ 1, abort_flag, p.status, limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * kAccCols);
                // With mma_group 2 the stages are taken two at a time: a shared-memory read by
                // this warp (the barrier wait) does not complete before the MMAs it issued
                // earlier have, so each wait drains the tensor pipe; one wait per two K-steps
                // halves those drains.
                for (int kb = 0; kb < w.nk;) {
                    const int ns = (p.mma_group > 1 && kb + 1 < w.nk) ? 2 : 1;
                    int st1 = stage + 1;
                    uint32_t ph1 = phase;
                    if (st1 == stages) { st1 = 0; ph1 ^= 1; }
                    if (!wait_warp(smem_addr(&full[stage]), phase, abort_flag, p.status, limit) ||
                        (ns == 2 && !wait_warp(smem_addr(&full[st1]), ph1, abort_flag, p.status, limit))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int j = 0; j < ns; ++j) {
                        const int st = j ? st1 : stage;
                        const uint64_t ad = smem_desc<BK>(smem_addr(a_ring + (size_t)st * kStageA));
                        const uint64_t bd = smem_desc<BK>(smem_addr(b_ring + (size_t)st * b_stage_bytes));
                        if (!second) {
#pragma unroll
                            for (int k = 0; k < BK / 16; ++k) {
                                // advance 16 bf16 = 32 bytes along K inside the swizzled rows
                                mma_bf16<CG>(d, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), idesc,
                                             (kb + j > 0 || k > 0) ? 1u : 0u, issuer);
                            }
                        } else if (mma2) {
#pragma unroll
                            for (int k = 0; k < BK / 16; ++k) {
                                // the stage rows past the first r1 (whole 1024-byte swizzle atoms)
                                mma_bf16<CG>(d + (uint32_t)n1, ad + (uint64_t)(2 * k),
                                             bd + b_off2 + (uint64_t)(2 * k), idesc2,
                                             (kb + j > 0 || k > 0) ? 1u : 0u, issuer);
                            }
                        }
                        mma_commit<CG>(smem_addr(&empty[st]), issuer);
                    }
                    if (ns == 2) {
                        stage = st1 + 1;
                        phase = ph1;
                        if (stage == stages) { stage = 0; phase ^= 1; }
                    } else {
                        stage = st1;
                        phase = ph1;
                    }
                    kb += ns;
                }
                if (!ok) break;
                mma_commit<CG>(smem_addr(&tfull[acc]), issuer);
            }
            // every MMA this warp issued has completed before TMEM is released
            mma_commit_local<CG>(smem_addr(drain), issuer);
            if (lane == 0) wait_bounded(smem_addr(drain), 0, abort_flag, p.status, limit, false);
        }
    } else if (warp <= 5) {
        // ------------------------------------------------------------ epilogue (warps 2..5)
        const int q = warp & 3;                      // TMEM lane quadrant this warp may read
        const int r_local = q * 32 + lane;           // tile row held by this thread
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        // with K halves the four epilogue warps meet at named barriers in every unit: they first
        // agree on going on, so that none waits at a barrier for a warp that has left
        const bool split_launch = p.k_split > 1;
        const int n_parts = split_launch ? p.k_split : 1;
        volatile int* ticket = abort_flag + 1;       // this unit's K-part role, shared by the warps
        if (p.pdl) griddep_wait();                   // global reads and writes follow the previous kernel
        int it = 0;
        for (int u = group; u < n_units; u += n_groups, ++it) {
            const Unit w = decode_unit<YT>(p, wl, u, rank);
            const int acc = it % n_acc;
            int ok = 1;
            if (lane == 0)
                ok = wait_bounded(smem_addr(&tfull[acc]), (it / n_acc) & 1, abort_flag, p.status, limit, true);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (split_launch) ok = epilogue_bar_and(ok);
            if (!ok) break;
            tc_fence_after();
            // K parts: every part but the last to arrive stores its fp32 sums in its own slot; the
            // last waits until all of them are stored and adds the S sums in part order (P0 + P1,
            // then + P2, + P3), its own from registers: the same sum whichever part arrives last
            const bool split = split_launch && w.tile.nrows > 0;
            bool first = false;                      // this part stores its sums (not the last)
            int* ctr = nullptr;
            if (split) {
                ctr = p.split_ctr + 2 * (size_t)w.slot;
                if (warp == 2 && lane == 0) {
                    const int old = atomicAdd(ctr, 1);
                    int wok = 1;
                    if (old == n_parts - 1) wok = wait_count(ctr + 1, n_parts - 1, abort_flag, p.status, limit);
                    *ticket = (old < n_parts - 1 ? 1 : 0) | (wok ? 0 : 2);
                }
                epilogue_bar_sync();
                const int tk = *ticket;
                if (tk & 2) break;                   // the wait ran out: the CTA is aborting
                first = (tk & 1) != 0;
            }
            const uint32_t taddr = tmem_base + (uint32_t)(acc * kAccCols) + lane_off;
            if (YT && !w.shrink) {
                yt_store(p, taddr, w.n0 + rank * kTileM + q * 32, lane, yt_stage + (size_t)q * 2048);
            } else {
                const int row = w.tile.row0 + r_local;
                const bool row_ok = r_local < w.tile.nrows;
                float scale = 1.0f;
                __nv_bfloat16* out;
                int n_out;
                if (w.shrink) {
                    const int a = row_ok ? row_adapter(wl.seg_off, wl.seg_id, p.n_seg, row) : 0;
                    scale = (a == w.tile.adapter) ? wl.scales[w.tile.adapter - 1] : 0.0f;
                    out = reinterpret_cast<__nv_bfloat16*>(p.u) + (size_t)row * p.rank + w.n0;
                    n_out = p.rank - w.n0;
                } else {
                    out = reinterpret_cast<__nv_bfloat16*>(p.y) + (size_t)row * p.d_out + w.n0;
                    n_out = p.d_out - w.n0;
                }
                // partial sums of this row: part q's float4 chunk j (columns n0 + 4j ..) at
                // part_base[(q * part_chunks + j) * part_rows]
                const size_t part_stride = (size_t)p.part_chunks * p.part_rows;    // one part's slot
                float4* part = split ? p.partials + (size_t)w.pchunk * p.part_rows + row : nullptr;
                const bool wide_tile = FORM == kFormWideRows && !w.shrink && w.n > kAccCols;
                for (int c = 0; c < w.n; c += 32) {
                    uint32_t v[32];
                    const bool two = c + 16 < w.n;  // w.n is a multiple of 16
                    tmem_ld16(taddr + (uint32_t)c, v);
                    if (two) tmem_ld16(taddr + (uint32_t)c + 16, v + 16);
                    tmem_ld_wait();
                    if (row_ok && split) {
                        if (first) {
                            float4* pc = part + (size_t)w.part * part_stride + (size_t)(c >> 2) * p.part_rows;
#pragma unroll
                            for (int h = 0; h < 8; ++h)
                                if ((h < 4 || two) && c + 4 * h < n_out)
                                    __stcg(pc + (size_t)h * p.part_rows,
                                           make_float4(__uint_as_float(v[4 * h]), __uint_as_float(v[4 * h + 1]),
                                                       __uint_as_float(v[4 * h + 2]), __uint_as_float(v[4 * h + 3])));
                        } else {
                            // the sum in part order; each other part's eight loads of the chunk are in
                            // flight at once (addresses past the block's last column are clamped to it;
                            // those sums are never stored)
                            const int last = (n_out - 1) >> 2;
                            float acc[32];
                            for (int q = 0; q < n_parts; ++q) {
                                float t[32];
                                if (q == w.part) {
#pragma unroll
                                    for (int i = 0; i < 32; ++i) t[i] = __uint_as_float(v[i]);
                                } else {
                                    const float4* pq = part + (size_t)q * part_stride;
                                    float4 o[8];
#pragma unroll
                                    for (int h = 0; h < 8; ++h)
                                        o[h] = __ldcg(pq + (size_t)min((c >> 2) + h, last) * p.part_rows);
#pragma unroll
                                    for (int h = 0; h < 8; ++h) {
                                        t[4 * h] = o[h].x;
                                        t[4 * h + 1] = o[h].y;
                                        t[4 * h + 2] = o[h].z;
                                        t[4 * h + 3] = o[h].w;
                                    }
                                }
#pragma unroll
                                for (int i = 0; i < 32; ++i) acc[i] = q == 0 ? t[i] : acc[i] + t[i];
                            }
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(acc[i]);
                        }
                    }
                    if (row_ok && !first) {
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            // a wide row tile's accumulator columns follow its B stage rows
                            // (boundaries at multiples of 8 columns)
                            const int col = wide_tile ? pair_b_row(c + 8 * h, kAccCols / CG, w.n / CG) : c + 8 * h;
                            if ((h < 2 || two) && col < n_out) {
                                uint4 o;
                                o.x = pack_bf16x2(__uint_as_float(v[8 * h + 0]) * scale,
                                                  __uint_as_float(v[8 * h + 1]) * scale);
                                o.y = pack_bf16x2(__uint_as_float(v[8 * h + 2]) * scale,
                                                  __uint_as_float(v[8 * h + 3]) * scale);
                                o.z = pack_bf16x2(__uint_as_float(v[8 * h + 4]) * scale,
                                                  __uint_as_float(v[8 * h + 5]) * scale);
                                o.w = pack_bf16x2(__uint_as_float(v[8 * h + 6]) * scale,
                                                  __uint_as_float(v[8 * h + 7]) * scale);
                                *reinterpret_cast<uint4*>(out + col) = o;
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            if (CG > 1)
                mbar_arrive_cluster(map_to_rank(smem_addr(&tempty[acc]), 0));  // the even CTA's barrier
            else
                mbar_arrive(smem_addr(&tempty[acc]));
            if (first) {
                // every thread's partial sums are stored before the last part may read them
                __threadfence();
                epilogue_bar_sync();
                if (warp == 2 && lane == 0) {
                    __threadfence();
                    atomicAdd(ctr + 1, 1);
                }
            }
            if (w.shrink && p.flags && w.tile_index >= 0 && !first) {
                // publish this tile's U rows to the fused units that wait for them (with K
                // parts, the last part, which stored them)
                fence_proxy_async_global();
                epilogue_bar_sync();
                if (warp == 2 && lane == 0) {
                    if (p.debug_publish_delay_ns) {
                        // tests only: hold the flag back so that an expand that did not wait reads stale U
                        const uint64_t t0 = global_timer_ns();
                        while (global_timer_ns() - t0 < p.debug_publish_delay_ns) __nanosleep(1000);
                    }
                    __threadfence();
                    st_release(&p.flags[w.tile_index], 1);
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
    if (p.flags || p.split_ctr) {
        // The last CTA of the launch to get here clears the ready flags, the K-half counters and
        // the exit counter: every CTA counts itself in only after all of its flag and counter
        // reads, so none is still waiting, and the next launch on the stream (a replay of a
        // captured graph included) starts from zero.
        int last = 0;
        if (threadIdx.x == 0) {
            __threadfence();
            last = atomicAdd(p.done_count, 1) == (int)gridDim.x - 1;
        }
        last = __syncthreads_or(last);
        if (last) {
            __threadfence();
            if (p.flags)
                for (int i = threadIdx.x; i < p.n_flags; i += blockDim.x) p.flags[i] = 0;
            if (p.split_ctr)
                for (int i = threadIdx.x; i < 2 * p.n_split_slots; i += blockDim.x) p.split_ctr[i] = 0;
            if (threadIdx.x == 0) *p.done_count = 0;
        }
    }
}

// Plain 4-bit layout -> kernel layout, one 32-bit word (8 input features) per step:
// feature 8c+i sits in plain nibble i (two's complement); the kernel layout puts feature
// 8c+2j in nibble j and 8c+2j+1 in nibble j+4, offset binary (q + 8 = nibble ^ 8).
__global__ void w4_repack_kernel(const uint32_t* src, uint32_t* dst, long long n_words) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_words;
         i += (long long)gridDim.x * blockDim.x) {
        const uint32_t w = src[i];
        uint32_t o = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            o |= ((w >> (8 * j)) & 0xFu) << (4 * j);
            o |= ((w >> (8 * j + 4)) & 0xFu) << (4 * j + 16);
        }
        dst[i] = o ^ 0x88888888u;
    }
}

}  // namespace dev

cudaError_t w4_repack(const void* src, void* dst, long long n_words, int grid, cudaStream_t stream) {
    if (n_words <= 0) return cudaSuccess;
    // src may equal dst: each thread reads its word before writing it, no other thread touches it
    dev::w4_repack_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint32_t*>(src), static_cast<uint32_t*>(dst),
                                                    n_words);
    return cudaGetLastError();
}

size_t gemm_smem_bytes(int b_tile_rows, int stages, int bk, int a_rows, int yt) {
    return 1024 + (size_t)stages * ((size_t)a_rows * bk * 2 + (size_t)b_tile_rows * bk * 2) +
           (yt ? (size_t)kYtStageBytes : 0) + 8 * (2 * (size_t)stages + 5) + 16;
}

template <int BK, int CG, int FORM = kFormRows>
static cudaError_t set_smem_attr() {
    return cudaFuncSetAttribute(dev::lora_gemm_kernel<BK, CG, FORM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemLimit);
}

cudaError_t gemm_prepare_device() {
    cudaError_t e;
    if ((e = set_smem_attr<64, 1>()) != cudaSuccess) return e;
    if ((e = set_smem_attr<64, 2>()) != cudaSuccess) return e;
    if ((e = set_smem_attr<64, 2, kFormTokenColumns>()) != cudaSuccess) return e;
    if ((e = set_smem_attr<64, 2, kFormWideRows>()) != cudaSuccess) return e;
    if ((e = set_smem_attr<32, 1>()) != cudaSuccess) return e;
    return set_smem_attr<32, 2>();
}

// Cooperative launches can be switched off for a profiler (LORA_LINEAR_NONCOOPERATIVE=1 in the
// environment): Nsight Compute rejects the cooperative grid that fits without its
// instrumentation ("LaunchFailed"), and it runs one kernel at a time, so the grid is
// co-resident anyway.
static bool cooperative_launches() {
    static const bool on = [] {
        const char* v = getenv("LORA_LINEAR_NONCOOPERATIVE");
        return !(v && v[0] == '1');
    }();
    return on;
}

// Launches of a two-MMA instantiation: token-column units and row tiles wider than 256 columns.
bool gemm_wide(const GemmParams& p) {
    return p.yt || p.tile_n > kAccCols;
}

int gemm_b_rows(const GemmParams& p) {
    if (p.yt) return p.yt_rows > p.shrink_n / p.cluster_size ? p.yt_rows : p.shrink_n / p.cluster_size;
    return (p.tile_n > p.shrink_n ? p.tile_n : p.shrink_n) / p.cluster_size;
}

static void launch_config(const GemmParams& p, int grid, cudaStream_t stream, cudaLaunchConfig_t* cfg,
                          cudaLaunchAttribute* attr /* [3] */) {
    const int b_rows = gemm_b_rows(p);
    *cfg = cudaLaunchConfig_t{};
    cfg->gridDim = dim3(grid, 1, 1);
    cfg->blockDim = dim3(gemm_wide(p) ? kThreadsWide : kThreads, 1, 1);
    cfg->dynamicSmemBytes = gemm_smem_bytes(b_rows, p.stages, p.bk, p.a_rows ? p.a_rows : kTileM, p.yt);
    cfg->stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.cluster_size;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg->attrs = attr;
    cfg->numAttrs = 1;
    if (p.flags && cooperative_launches()) {
        // fused units wait for ready flags set by shrink units on other CTAs of the grid: a
        // cooperative launch starts only when every CTA can be resident at once, so a CTA never
        // waits on one that another kernel keeps from starting
        attr[1].id = cudaLaunchAttributeCooperative;
        attr[1].val.cooperative = 1;
        cfg->numAttrs = 2;
    } else if (p.pdl) {
        // may start while the previous kernel of the stream finishes (it waits for it before
        // touching anything but W)
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg->numAttrs = 2;
    }
}

template <typename F>
static cudaError_t dispatch(const GemmParams& p, F&& f) {
    const bool pair64 = p.bk == 64 && p.cluster_size == 2;
    if (p.yt) return pair64 ? f(dev::lora_gemm_kernel<64, 2, kFormTokenColumns>) : cudaErrorInvalidValue;
    if (p.tile_n > kAccCols) return pair64 ? f(dev::lora_gemm_kernel<64, 2, kFormWideRows>) : cudaErrorInvalidValue;
    if (p.bk == 64 && p.cluster_size == 1) return f(dev::lora_gemm_kernel<64, 1, kFormRows>);
    if (pair64) return f(dev::lora_gemm_kernel<64, 2, kFormRows>);
    if (p.bk == 32 && p.cluster_size == 1) return f(dev::lora_gemm_kernel<32, 1, kFormRows>);
    if (p.bk == 32 && p.cluster_size == 2) return f(dev::lora_gemm_kernel<32, 2, kFormRows>);
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm(const GemmParams& p, int grid, cudaStream_t stream) {
    // rank tiles only in a launch of shrink units alone, without ready flags or K parts
    if (p.shrink_ntiles > 1 && (p.n_fused || p.flags || p.k_split > 1 || p.shrink_n < 16 || (p.shrink_n & 15)))
        return cudaErrorInvalidValue;
    // wide row tiles: whole K per unit, a multiple of 16 columns, at most two 256-column MMAs
    if (!p.yt && p.tile_n > kAccCols &&
        (p.k_split > 1 || p.tile_n > kMaxWideTileN || (p.tile_n & 15) || (p.a_rows && p.a_rows != kTileM)))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[3];
    launch_config(p, grid, stream, &cfg, attr);
    return dispatch(p, [&](auto kernel) { return cudaLaunchKernelEx(&cfg, kernel, p); });
}

int gemm_max_clusters(const GemmParams& p) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[3];
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
