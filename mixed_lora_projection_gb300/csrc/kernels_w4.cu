// sm_103a kernel of the projection with a 4-bit base weight (W4A16 base, bf16 adapter).
//
// The 4-bit base has to be expanded to bf16 before the tensor core can use it. Doing that
// into shared memory puts a second full-width tile through the shared-memory port on every
// K-step, beside the TMA fills and the MMA's operand reads, and that port then sets the
// pace. Here the dequantised weights go to tensor memory instead: the tile is transposed,
//
//   D[n, t] = sum_k W[n, k] X[t, k]  (+ sum_j B_a[n, j] U[t, j] for adapter tokens)
//
// with the unit's 128 output features n on the MMA's M side (TMEM lanes) and its tokens t
// on N (up to 256: two planner tiles). tcgen05.mma kind::f16 reads A (the weights) from
// tensor memory, written with tcgen05.st by the converter warps, and B (the X rows) from
// shared memory, filled by TMA. The adapter's expand (B_a tile as A, U rows as B) runs
// from shared memory into the same accumulator; U comes from the shrink pass, launched
// before this kernel on the same stream.
//
// Per CTA (one per SM, persistent over the units, in the order W4Params::tokens_fastest
// selects: feature tiles or token groups fastest):
//   warp 0      TMA: X tiles (base K-steps), U and B_a tiles (expand K-steps);
//   warp 1      TMEM owner (512 columns: one 128 x 256 fp32 accumulator and one 32-column
//               stage of dequantised A per ring stage), issues the MMAs: one wait per two
//               ring stages, four MMAs per feature tile and one commit per K-step; with two
//               feature tiles per unit it issues the first tile's and warp 15 the second's
//               (one warp waits ~80 cycles between MMAs whatever their width, and these MMAs
//               are narrow: two warps keep the tensor pipe fed with both tiles);
//   warps 2..5  epilogue: warp w reads lanes 32 (w % 4) .. (one output feature per thread),
//               stages each whole 32-token chunk of Y in shared memory ([token][feature])
//               and writes it with one TMA store (a tile's ragged last chunk from registers);
//   warps 6..13 converters: warp w dequantises whole K-steps (6..9 the even ring stages,
//               10..13 the odd ones) for the 32 features of lane quadrant w % 4, packed
//               ring -> TMEM, and counts itself in on the stage's full barrier;
//   warp 14     TMA of the packed base and its scales (4 K-steps per box) into their ring;
//   warp 15     with two feature tiles per unit: the second tile's MMAs (see warp 1); with three
//               token tiles in a group: the third tile's MMAs (its rows the B operand, its
//               accumulator at columns 256 ..).
// Instantiations: FT (feature tiles per unit), SPLIT (K parts), TAIL (a third token tile); the
// code of each option stays out of the others' instantiations, where it cost registers and time.
// Every wait is bounded as in the bf16 kernel (status word, abort flag, orderly exit).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "dev_common.cuh"
#include "lora_internal.h"
#include "lora_w4.h"

namespace lora {
namespace dev {

namespace {

constexpr uint32_t kXStageMaxBytes = (256 + kW4TailRows) * 128;   // B operand: up to 256 + 96 token rows x 64 bf16
constexpr uint32_t kQStageBytes = 128 * kW4PackBytes;   // packed rows of 4 K-steps
constexpr uint32_t kSStageBytes = 2 * 128 * 2;          // two scale groups of 128 features
constexpr uint32_t kAccCols4 = 256;               // accumulator columns (tokens)
constexpr uint32_t kYChunkRows = 32;              // tokens per Y chunk (one tcgen05.ld of 32 columns)
constexpr uint32_t kYStageBytes = kYChunkRows * 128 * 2;   // [32 tokens][128 features] bf16

// Y chunk from shared memory to global memory through a tensor map, in this thread's bulk
// async-group; rows and features past the tensor's extent are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int c_inner, int c_outer) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c_inner), "r"(c_outer)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// all of this thread's bulk stores have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// all of this thread's bulk stores are complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// generic-proxy shared-memory writes made visible to the async proxy (the TMA store that follows)
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 (bf16 in, fp32 accumulate), issued by the lane
// with pred != 0 of a converged warp.
__device__ __forceinline__ void mma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate, uint32_t pred) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.ne.b32 q, %5, 0;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(pred)
        : "memory");
}

// 32 lanes x 32 bits x 16 columns from registers: thread i writes lane (taddr.lane + i).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0],"
        " {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Unit order: feature tiles fastest (each token group's X stays in L2 while the packed base
// streams past it), or token groups fastest (each packed feature tile is read once per wave
// while every group's X stays in L2: for a base too large to stay in L2 beside the output).
__device__ __forceinline__ int w4_group_of(const W4Params& p, int u) {
    return p.tokens_fastest ? u % p.n_groups : u / p.n_ntiles;
}
__device__ __forceinline__ int w4_ntile_of(const W4Params& p, int u) {
    return p.tokens_fastest ? u / p.n_groups : u % p.n_ntiles;
}

struct W4Unit {
    W4Group g;
    int n0;          // first output feature
    int n;           // MMA N of the base K-steps (tokens, multiple of 16)
    int n2;          // N of the second MMA (the third token tile's rows), 0 without one
    int kb0, kend;   // base K-steps [kb0, kend) of this unit
    int part;        // K part (0 .. k_split - 1), 0 without parts
    int block;       // (token group, feature tile) block: its split counters
    bool expand;     // runs the expand's K-steps (the last part)
};

template <int FT, bool SPLIT, bool TAIL>
__device__ __forceinline__ W4Unit w4_unit(const W4Params& p, const W4Group* groups, int u) {
    W4Unit r;
    const int S = SPLIT ? p.k_split : 1;
    const int v = u / S;
    r.part = u - v * S;
    r.block = v;
    r.kb0 = r.part * p.k_chunk;
    r.kend = r.part == S - 1 ? p.k_main_blocks : r.kb0 + p.k_chunk;
    r.expand = r.part == S - 1;
    const int gi = w4_group_of(p, v);
    r.g = groups[gi];
    r.n0 = w4_ntile_of(p, v) * kW4TileM * FT;
    // token tile h at accumulator columns 128 h: a third tile makes the first MMA cover both
    // of the first two tiles whole
    const bool third = TAIL && r.g.nrows[2] > 0;
    r.n = third              ? 256
          : r.g.nrows[1] > 0 ? 128 + ((r.g.nrows[1] + 15) & ~15)
                             : ((r.g.nrows[0] + 15) & ~15);
    r.n2 = third ? ((r.g.nrows[2] + 15) & ~15) : 0;
    return r;
}

// 64-bit counter reaches `value` (acquire), bounded like every other wait.
static __device__ __noinline__ bool wait_count64(const unsigned long long* counter, unsigned long long value,
                                                 volatile int* abort_flag, int* status, uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    while (true) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(counter) : "memory");
        if (v >= value) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, 1);
            *abort_flag = 1;
            return false;
        }
        __nanosleep(256);
    }
}

}  // namespace

// FT feature tiles of 128 per unit. FT = 2 serves batches of one token tile of at most 128 rows
// with no adapter rows (decode steps): the unit's two tiles share each K-step's X stage, barrier
// round trips and ring slots, which halves the K-steps an SM runs in sequence. Tensor memory
// then holds two 128-column accumulators (tile f at column 128 f) and A stages of 64 columns.
template <int FT, bool SPLIT, bool TAIL>
__global__ void __launch_bounds__(kW4Threads, 1) lora_w4_kernel(const __grid_constant__ W4Params p) {
    static_assert(!TAIL || FT == 1, "a third token tile only with one feature tile per unit");
    static_assert(FT == 1 || FT == 2, "one or two feature tiles per unit");
    constexpr uint32_t kQStage = FT * kQStageBytes;    // packed rows of the unit's feature tiles
    constexpr uint32_t kSStage = FT * kSStageBytes;    // their scales (two groups of 128 inputs)
    constexpr uint32_t kAStageCols = 32 * FT;          // TMEM columns of one A stage
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const int stages = p.stages, pstages = p.pstages;
    // ring stage s: base K-step -> X rows (B operand, up to 256 rows) in smem and the
    // dequantised weights (A operand) in TMEM columns 256 + 32 s; expand K-step -> U rows
    // (B operand) in the first 16 KB and the B_a tile (A operand) in the second 16 KB
    const uint32_t x_stage = (uint32_t)p.x_stage_bytes;
    uint8_t* x_ring = base;
    uint8_t* y_stage = x_ring + (size_t)stages * x_stage;   // 2 x 8 KB: Y chunks on their way out
    uint8_t* q_ring = y_stage + kYStageBytes * 2;
    uint8_t* s_ring = q_ring + (size_t)pstages * kQStage;
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_ring + (size_t)pstages * kSStage);
    uint64_t* full = bars;                          // TMA bytes + one arrive per converter quadrant
    uint64_t* empty = full + stages;                // MMA done with the stage (smem and TMEM)
    uint64_t* pfull = empty + stages;               // packed rows + scales landed
    uint64_t* pempty = pfull + pstages;             // converters done with them
    uint64_t* tfull = pempty + pstages;             // accumulator complete
    uint64_t* tempty = tfull + 1;                   // accumulator drained by the epilogue
    uint64_t* drain = tempty + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* ticket = abort_flag + 1;          // K parts: the unit's role, shared by the epilogue warps

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // MMA warps (one per feature tile of a unit, or two with a third token tile): each commits
    // every stage, accumulator and drain
    constexpr bool mma2 = FT == 2 || TAIL;
    constexpr uint32_t kIssuers = mma2 ? 2u : 1u;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(smem_addr(&full[s]), 1 + kW4ConvertWarps / 2);
            mbar_init(smem_addr(&empty[s]), kIssuers);
        }
        for (int s = 0; s < pstages; ++s) {
            mbar_init(smem_addr(&pfull[s]), 1);
            mbar_init(smem_addr(&pempty[s]), kW4ConvertWarps);
        }
        mbar_init(smem_addr(tfull), kIssuers);
        mbar_init(smem_addr(tempty), kEpilogueThreads);
        mbar_init(smem_addr(drain), kIssuers);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc<1>(smem_addr(tmem_slot), 2 * kAccCols4);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // A stages after the accumulators: columns 256 + 32 FT s, or 384 + 32 s past a third token tile
    const uint32_t tmem_a = tmem_base + (TAIL ? 3u * 128u : kAccCols4);

    const int n_units = p.n_groups * p.n_ntiles * (SPLIT ? p.k_split : 1);
    const uint64_t limit = p.wait_limit_ns;
    const W4Group* groups = p.inline_wl ? p.inline_groups : p.groups;
    const CUtensorMap* bmaps = p.inline_wl ? p.inline_bmaps : p.tm_b;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA: X, U, B_a
        const uint32_t issuer = lane == 0 ? 1u : 0u;
        if (!p.debug_stall) {
            if (lane == 0) {
                tma_prefetch_desc(&p.tm_x);
                tma_prefetch_desc(&p.tm_u);
            }
            __syncwarp();
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            int acquired = -1;
            bool ok = true;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                const W4Unit w = w4_unit<FT, SPLIT, TAIL>(p, groups, u);
                const int ntile = (TAIL && w.g.nrows[2] > 0) ? 3 : w.g.nrows[1] > 0 ? 2 : 1;
                // tiles 0 and 1: 128-row boxes; a third tile: its own box of tail_rows rows
                const uint32_t x_bytes = (ntile < 3 ? (uint32_t)ntile : 2u) * 16384u +
                                         (ntile == 3 ? (uint32_t)p.tail_rows * 128u : 0u);
                for (int kb = w.kb0; kb < w.kend; ++kb) {
                    if (!wait_warp(smem_addr(&empty[stage]), phase ^ 1, abort_flag, p.status, limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_addr(&full[stage]);
                    mbar_arrive_expect_tx(fb, x_bytes, issuer);
                    const uint32_t xs = smem_addr(x_ring + (size_t)stage * x_stage);
                    for (int h = 0; h < ntile; ++h)
                        tma_load_2d<1>(xs + (uint32_t)h * 16384u, h < 2 ? &p.tm_x : &p.tm_x3, fb, kb * 64,
                                       w.g.row0[h], issuer);
                    ++issued;
                    if (++stage == stages) { stage = 0; phase ^= 1; }
                }
                for (int h = 0; h < (TAIL ? 3 : 2) && ok && w.expand; ++h) {
                    const int a = w.g.adapter[h];
                    if (w.g.nrows[h] == 0 || a == 0) continue;
                    const CUtensorMap* bm = &bmaps[a - 1];
                    if (!p.inline_wl && acquired != a) {
                        tensormap_acquire(bm);
                        acquired = a;
                    }
                    for (int kr = 0; kr < p.k_lora_blocks; ++kr) {
                        if (!wait_warp(smem_addr(&empty[stage]), phase ^ 1, abort_flag, p.status, limit)) {
                            ok = false;
                            break;
                        }
                        const uint32_t fb = smem_addr(&full[stage]);
                        mbar_arrive_expect_tx(fb, 32768u, issuer);
                        const uint32_t xs = smem_addr(x_ring + (size_t)stage * x_stage);
                        tma_load_2d<1>(xs, &p.tm_u, fb, kr * 64, w.g.row0[h], issuer);
                        tma_load_2d<1>(xs + 16384u, bm, fb, kr * 64, w.n0, issuer);
                        ++issued;
                        if (++stage == stages) { stage = 0; phase ^= 1; }
                    }
                }
            }
            if (lane == 0 && !ok) {
                // wait (bounded, ignoring the abort flag) for the copies still in flight
                long long first = issued > stages ? issued - stages : 0;
                for (long long j = first; j < issued; ++j)
                    wait_bounded(smem_addr(&full[j % stages]), (uint32_t)((j / stages) & 1), abort_flag, p.status,
                                 limit, false);
            }
        }
    } else if (warp == 14) {
        // ------------------------------------------------------------ TMA: packed base + scales
        const uint32_t issuer = lane == 0 ? 1u : 0u;
        if (!p.debug_stall) {
            if (lane == 0) {
                tma_prefetch_desc(&p.tm_wq);
                tma_prefetch_desc(&p.tm_ws);
            }
            __syncwarp();
            int ps = 0;
            uint32_t pph = 0;
            long long issued = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                const W4Unit w = w4_unit<FT, SPLIT, TAIL>(p, groups, u);
                const int n0 = w.n0;
                // packed boxes of 4 K-steps; part boundaries are multiples of 4 K-steps
                for (int pb = w.kb0 >> 2; pb < ((w.kend + 3) >> 2); ++pb) {
                    if (!wait_warp(smem_addr(&pempty[ps]), pph ^ 1, abort_flag, p.status, limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t pbar = smem_addr(&pfull[ps]);
                    mbar_arrive_expect_tx(pbar, kQStage + kSStage, issuer);
                    tma_load_2d<1>(smem_addr(q_ring + (size_t)ps * kQStage), &p.tm_wq, pbar, pb * kW4PackBytes,
                                   n0, issuer);
                    tma_load_2d<1>(smem_addr(s_ring + (size_t)ps * kSStage), &p.tm_ws, pbar, n0, 2 * pb, issuer);
                    ++issued;
                    if (++ps == pstages) { ps = 0; pph ^= 1; }
                }
            }
            if (lane == 0 && !ok) {
                long long first = issued > pstages ? issued - pstages : 0;
                for (long long j = first; j < issued; ++j)
                    wait_bounded(smem_addr(&pfull[j % pstages]), (uint32_t)((j / pstages) & 1), abort_flag, p.status,
                                 limit, false);
            }
        }
    } else if (warp == 1 || (mma2 && warp == 15)) {
        // ------------------------------------------------------------ MMA issuers
        // Warp 1 issues feature tile 0's MMAs (and the expand's), warp 15 tile 1's, or with
        // three token tiles warp 1 the first two tiles' MMA and warp 15 the third's; both walk
        // every stage and commit it.
        const uint32_t issuer = lane == 0 ? 1u : 0u;
        const int my_tile = (mma2 && warp == 15) ? 1 : 0;
        int stage = 0;
        uint32_t phase = 0;
        int it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++it) {
            const W4Unit w = w4_unit<FT, SPLIT, TAIL>(p, groups, u);
            if (!wait_warp(smem_addr(tempty), (it & 1) ^ 1, abort_flag, p.status, limit)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // Stages are taken two at a time: a shared-memory read by this warp (the barrier
            // wait) does not complete before the MMAs it issued earlier have, so each wait
            // costs a drain of the tensor pipe; eight MMAs per wait hide it where four do not.
            const uint32_t idesc = instr_desc_bf16(kW4TileM, w.n);
            const uint32_t idesc2 = instr_desc_bf16(kW4TileM, w.n2 ? w.n2 : 16);
            // a part's K-steps are even in number (k_chunk % 4 == 0, k_main_blocks even: d_in % 128 == 0)
            for (int kb = w.kb0; kb < w.kend; kb += 2) {
                int st1 = stage + 1;
                uint32_t ph1 = phase;
                if (st1 == stages) { st1 = 0; ph1 ^= 1; }
                if (!wait_warp(smem_addr(&full[stage]), phase, abort_flag, p.status, limit) ||
                    !wait_warp(smem_addr(&full[st1]), ph1, abort_flag, p.status, limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int st = j ? st1 : stage;
                    const uint64_t bd = smem_desc<64>(smem_addr(x_ring + (size_t)st * x_stage));
                    if (FT == 2) {
                        const int f = my_tile;
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_tmem_a(tmem_base + (uint32_t)(128 * f),
                                       tmem_a + kAStageCols * st + (uint32_t)(32 * f + 8 * k), bd + (uint64_t)(2 * k),
                                       idesc, (kb > w.kb0 || j > 0 || k > 0) ? 1u : 0u, issuer);
                    } else if (!TAIL || my_tile == 0) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_tmem_a(tmem_base, tmem_a + kAStageCols * st + (uint32_t)(8 * k), bd + (uint64_t)(2 * k),
                                       idesc, (kb > w.kb0 || j > 0 || k > 0) ? 1u : 0u, issuer);
                    } else if (w.n2) {
                        // the third token tile: its rows follow the first two 16 KB boxes; its
                        // accumulator columns follow theirs
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_tmem_a(tmem_base + 256u, tmem_a + kAStageCols * st + (uint32_t)(8 * k),
                                       bd + (uint64_t)((32768 >> 4) + 2 * k), idesc2,
                                       (kb > w.kb0 || j > 0 || k > 0) ? 1u : 0u, issuer);
                    }
                    mma_commit<1>(smem_addr(&empty[st]), issuer);
                }
                stage = st1 + 1;
                phase = ph1;
                if (stage == stages) { stage = 0; phase ^= 1; }
            }
            const uint32_t idesc_e = instr_desc_bf16(kW4TileM, 128);
            for (int h = 0; h < (TAIL ? 3 : 2) && ok && w.expand; ++h) {
                if (w.g.nrows[h] == 0 || w.g.adapter[h] == 0) continue;
                for (int kr = 0; kr < p.k_lora_blocks; kr += 2) {
                    const int ns = kr + 1 < p.k_lora_blocks ? 2 : 1;
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
                        const uint32_t xs = smem_addr(x_ring + (size_t)st * x_stage);
                        const uint64_t ad = smem_desc<64>(xs + 16384u);
                        const uint64_t bd = smem_desc<64>(xs);
                        if (my_tile == 0) {
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                mma_bf16<1>(tmem_base + (uint32_t)(128 * h), ad + (uint64_t)(2 * k),
                                            bd + (uint64_t)(2 * k), idesc_e, 1u, issuer);
                        }
                        mma_commit<1>(smem_addr(&empty[st]), issuer);
                    }
                    if (ns == 2) {
                        stage = st1 + 1;
                        phase = ph1;
                    } else {
                        stage = st1;
                        phase = ph1;
                        continue;
                    }
                    if (stage == stages) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) break;
            mma_commit<1>(smem_addr(tfull), issuer);
        }
        // every MMA this warp issued has completed before TMEM is released
        mma_commit_local<1>(smem_addr(drain), issuer);
        if (lane == 0) wait_bounded(smem_addr(drain), 0, abort_flag, p.status, limit, false);
    } else if (warp >= 6 && warp <= 13) {
        // ------------------------------------------------------------ converters (warps 6..13)
        // Kernel layout of the packed base (lora_linear_w4_repack): 32-bit word c of a row's
        // K-step holds inputs 8c..8c+7 as offset-binary nibbles (q + 8), input 8c+2j in nibble
        // j and 8c+2j+1 in nibble j+4. ((word >> 4j) & 0x000F000F) | 0x43004300 is then the
        // bf16 pair (128 + q + 8) of inputs (8c+2j, 8c+2j+1), exact; minus 136 is q exactly,
        // and one round-to-nearest-even multiply gives q * s. The pair is one TMEM column.
        // Warp w serves the ring stages of parity (w - 6) / 4 for the 32 features of lane
        // quadrant w % 4: a whole base K-step (64 inputs, 32 columns) per stage, and on
        // expand K-steps only its arrive on the stage's full barrier.
        const int q = warp & 3;                       // lane quadrant: features 32q .. 32q+31
        const int par = (warp - 6) >> 2;              // ring-stage parity this warp serves
        const int nl = 32 * q + lane;                 // feature within the unit
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        const __nv_bfloat162 magic = __floats2bfloat162_rn(136.0f, 136.0f);
        int ps = 0, stage = 0;
        uint32_t pph = 0, phase = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            const W4Unit w = w4_unit<FT, SPLIT, TAIL>(p, groups, u);
            for (int kb = w.kb0; kb < w.kend; ++kb) {
                if ((kb & 3) == 0 &&
                    !wait_warp(smem_addr(&pfull[ps]), pph, abort_flag, p.status, limit)) {
                    ok = false;
                    break;
                }
                if ((stage & 1) == par) {
                    bool got = true;
#pragma unroll
                    for (int f = 0; f < FT && got; ++f) {
                        // the packed box rows are 128 bytes, 128-byte swizzled: 16-byte chunk c of
                        // row r sits at chunk c ^ (r % 8); feature tile f's rows start at 128 f
                        const int r = 128 * f + nl;
                        const uint8_t* row = q_ring + (size_t)ps * kQStage + (size_t)r * kW4PackBytes;
                        const uint32_t c0 = (uint32_t)(2 * (kb & 3)) ^ (uint32_t)(r & 7);
                        const uint32_t c1 = (uint32_t)(2 * (kb & 3) + 1) ^ (uint32_t)(r & 7);
                        const uint4 q0 = *reinterpret_cast<const uint4*>(row + (c0 << 4));
                        const uint4 q1 = *reinterpret_cast<const uint4*>(row + (c1 << 4));
                        const __nv_bfloat16* ss =
                            reinterpret_cast<const __nv_bfloat16*>(s_ring + (size_t)ps * kSStage);
                        const __nv_bfloat162 s2 =
                            __bfloat162bfloat162(ss[((kb & 3) >> 1) * (kW4TileM * FT) + r]);
                        const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                        uint32_t o[32];
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const uint32_t v = ((words[c] >> (4 * j)) & 0x000F000Fu) | 0x43004300u;
                                __nv_bfloat162 t = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&v), magic);
                                t = __hmul2(t, s2);
                                o[4 * c + j] = *reinterpret_cast<const uint32_t*>(&t);
                            }
                        }
                        if (f == 0) {
                            if (!wait_warp(smem_addr(&empty[stage]), phase ^ 1, abort_flag, p.status, limit)) {
                                got = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        const uint32_t ta = tmem_a + lane_off + kAStageCols * (uint32_t)stage + (uint32_t)(32 * f);
                        tmem_st16(ta, o);
                        tmem_st16(ta + 16u, o + 16);
                    }
                    if (!got) {
                        ok = false;
                        break;
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_addr(&full[stage]));
                }
                if ((kb & 3) == 3 || kb == w.kend - 1) {
                    // this packed slot is read (by this warp's K-steps in it): hand it back
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_addr(&pempty[ps]));
                    if (++ps == pstages) { ps = 0; pph ^= 1; }
                }
                if (++stage == stages) { stage = 0; phase ^= 1; }
            }
            // expand K-steps: no weights to convert, only this quadrant's arrive
            for (int h = 0; h < (TAIL ? 3 : 2) && ok && w.expand; ++h) {
                if (w.g.nrows[h] == 0 || w.g.adapter[h] == 0) continue;
                for (int kr = 0; kr < p.k_lora_blocks; ++kr) {
                    if ((stage & 1) == par) {
                        if (!wait_warp(smem_addr(&empty[stage]), phase ^ 1, abort_flag, p.status, limit)) {
                            ok = false;
                            break;
                        }
                        if (lane == 0) mbar_arrive(smem_addr(&full[stage]));
                        __syncwarp();
                    }
                    if (++stage == stages) { stage = 0; phase ^= 1; }
                }
            }
        }
    } else if (warp >= 2 && warp <= 5) {
        // ------------------------------------------------------------ epilogue (warps 2..5)
        const int q = warp & 3;
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        // Whole 32-token chunks go out through shared memory and TMA stores (two 8 KB buffers;
        // thread = feature, so each warp writes 64 contiguous bytes per token row), so the
        // accumulator is released once it has been read rather than after ~256 strided global
        // stores per thread; the ragged last chunk of a tile is stored from registers.
        __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(p.y);
        const bool issuer = warp == 2 && lane == 0;
        int chunk = 0;
        int it = 0;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++it) {
            const W4Unit w = w4_unit<FT, SPLIT, TAIL>(p, groups, u);
            int ok = 1;
            if (lane == 0) ok = wait_bounded(smem_addr(tfull), it & 1, abort_flag, p.status, limit, true);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            ok = epilogue_bar_and(ok);   // the four warps leave together (they share barriers)
            if (!ok) break;
            tc_fence_after();
            // K parts: every part but the last to arrive stores its fp32 sums; the last waits until
            // all of them are stored and adds the k_split sums in part order, its own from registers
            const int S = SPLIT ? p.k_split : 1;
            bool store_part = false;
            unsigned long long* ctr = nullptr;
            if (SPLIT) {
                ctr = p.split_ctr + 2 * (size_t)w.block;
                if (issuer) {
                    const unsigned long long old = atomicAdd(ctr, 1ull);
                    const unsigned long long s64 = (unsigned long long)S;
                    int role = old % s64 == s64 - 1 ? 0 : 1;
                    if (role == 0 && !wait_count64(ctr + 1, (old / s64 + 1) * (s64 - 1), abort_flag, p.status, limit))
                        role = 2;
                    *ticket = role;
                }
                epilogue_bar_sync();
                const int role = *ticket;
                if (role == 2) break;    // the wait ran out: the CTA is aborting
                store_part = role == 1;
            }
            // FT = 1: token tile h (up to three) at accumulator columns 128 h; FT = 2 (one token tile): feature
            // tile f at accumulator columns 128 f. The accumulator is released right after the
            // unit's last tensor-memory load, before that chunk's stores.
            const int last_hf = FT == 1 ? ((TAIL && w.g.nrows[2] > 0) ? 2 : w.g.nrows[1] > 0 ? 1 : 0) : 1;
            for (int hf = 0; hf < (TAIL ? 3 : 2); ++hf) {
                const int h = FT == 1 ? hf : 0;
                const int n_tile = w.n0 + (FT == 1 ? 0 : kW4TileM * hf);
                const int n = n_tile + 32 * q + lane;
                const bool n_ok = n < p.d_out;
                const int rows = (FT == 1 || hf < FT) ? w.g.nrows[h] : 0;
                for (int c = 0; c < rows; c += 32) {
                    uint32_t v[32];
                    const uint32_t taddr = tmem_base + lane_off + (uint32_t)(128 * hf + c);
                    tmem_ld16(taddr, v);
                    tmem_ld16(taddr + 16u, v + 16);
                    tmem_ld_wait();
                    if (hf == last_hf && c + 32 >= rows) {
                        tc_fence_before();
                        mbar_arrive(smem_addr(tempty));
                    }
                    const int m = rows - c < 32 ? rows - c : 32;
                    if (SPLIT) {
                        // partial sums of part q: row t, feature n at partials[(q * part_rows + t) * d_out + n]
                        const size_t t0 = (size_t)(w.g.row0[h] + c);
                        if (store_part) {
                            if (n_ok) {
                                float* pp = p.partials + ((size_t)w.part * p.part_rows + t0) * p.d_out + n;
#pragma unroll
                                for (int t = 0; t < 32; ++t)
                                    if (t < m) __stcg(pp + (size_t)t * p.d_out, __uint_as_float(v[t]));
                            }
                            continue;
                        }
                        // the sum in part order, eight tokens at a time; rows past m and features past
                        // d_out read row t0 / feature 0 of a slot (in range; those sums are never stored)
                        const float* pbase = p.partials + t0 * p.d_out + (n_ok ? n : 0);
#pragma unroll
                        for (int g8 = 0; g8 < 32; g8 += 8) {
                            float acc[8];
#pragma unroll
                            for (int qq = 0; qq < kMaxKSplit; ++qq) {
                                if (qq >= S) break;
                                float tv[8];
                                if (qq == w.part) {
#pragma unroll
                                    for (int t = 0; t < 8; ++t) tv[t] = __uint_as_float(v[g8 + t]);
                                } else {
                                    const float* pq = pbase + (size_t)qq * p.part_rows * p.d_out;
#pragma unroll
                                    for (int t = 0; t < 8; ++t)
                                        tv[t] = __ldcg(pq + (size_t)(g8 + t < m ? g8 + t : 0) * p.d_out);
                                }
#pragma unroll
                                for (int t = 0; t < 8; ++t) acc[t] = qq == 0 ? tv[t] : acc[t] + tv[t];
                            }
#pragma unroll
                            for (int t = 0; t < 8; ++t) v[g8 + t] = __float_as_uint(acc[t]);
                        }
                    }
                    if (m == 32) {
                        uint8_t* buf = y_stage + (size_t)(chunk & 1) * kYStageBytes;
                        __nv_bfloat16* sb = reinterpret_cast<__nv_bfloat16*>(buf) + 32 * q + lane;
#pragma unroll
                        for (int t = 0; t < 32; ++t) sb[t * 128] = __float2bfloat16_rn(__uint_as_float(v[t]));
                        fence_proxy_async_smem();
                        // the store issued from this buffer two chunks ago has read it before the
                        // barrier of the previous chunk; the one from the other buffer before this one
                        if (issuer) bulk_wait_read_all();
                        epilogue_bar_sync();
                        if (issuer) {
                            tma_store_2d(&p.tm_y, smem_addr(buf), n_tile, w.g.row0[h] + c);
                            bulk_commit_group();
                        }
                        ++chunk;
                    } else if (n_ok) {
                        __nv_bfloat16* col = y + (size_t)(w.g.row0[h] + c) * p.d_out + n;
#pragma unroll
                        for (int t = 0; t < 32; ++t)
                            if (t < m) col[(size_t)t * p.d_out] = __float2bfloat16_rn(__uint_as_float(v[t]));
                    }
                }
            }
            if (store_part) {
                // every thread's partial sums are stored before the last part may read them
                __threadfence();
                epilogue_bar_sync();
                if (issuer) {
                    __threadfence();
                    atomicAdd(ctr + 1, 1ull);
                }
            }
        }
        if (issuer) bulk_wait_all();
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<1>(tmem_base, 2 * kAccCols4);
    }
}

}  // namespace dev

size_t w4_smem_bytes(int stages, int pstages, int x_stage_bytes, int ft) {
    return 1024 + (size_t)stages * (size_t)x_stage_bytes + 2 * (size_t)dev::kYStageBytes +
           (size_t)pstages * (size_t)ft * (dev::kQStageBytes + dev::kSStageBytes) +
           8 * (2 * (size_t)stages + 2 * (size_t)pstages + 3) + 16;
}

template <int FT, bool SPLIT, bool TAIL>
static cudaError_t w4_smem_attr() {
    return cudaFuncSetAttribute(dev::lora_w4_kernel<FT, SPLIT, TAIL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemLimit);
}

cudaError_t w4_prepare_device() {
    cudaError_t e;
    if ((e = w4_smem_attr<1, false, false>()) != cudaSuccess || (e = w4_smem_attr<1, true, false>()) != cudaSuccess ||
        (e = w4_smem_attr<1, false, true>()) != cudaSuccess || (e = w4_smem_attr<2, false, false>()) != cudaSuccess)
        return e;
    return w4_smem_attr<2, true, false>();
}

// Cooperative launches can be switched off for a profiler (LORA_LINEAR_NONCOOPERATIVE=1), as for
// the bf16 kernel: Nsight Compute runs one kernel at a time, so the grid is co-resident anyway.
static bool w4_cooperative_launches() {
    static const bool on = [] {
        const char* v = getenv("LORA_LINEAR_NONCOOPERATIVE");
        return !(v && v[0] == '1');
    }();
    return on;
}

cudaError_t launch_w4(const W4Params& p, int grid, cudaStream_t stream) {
    // the TMEM A stages (32 FT columns each) sit after the 256 accumulator columns; the
    // converters' warp sets take alternate stages; an X stage holds the unit's token tiles (and,
    // with FT = 1, the expand's U and B_a boxes of 16 KB each)
    const int ft = p.feature_tiles;
    if ((ft != 1 && ft != 2) || w4_smem_bytes(p.stages, p.pstages, p.x_stage_bytes, ft) > (size_t)kSmemLimit ||
        p.stages < 2 || p.stages * 32 * ft > (p.tail_rows ? 128 : 256) || (p.stages & 1) || p.pstages < 2 ||
        (p.x_stage_bytes & 1023) ||
        p.x_stage_bytes < 16384 || p.x_stage_bytes > (int)dev::kXStageMaxBytes || (ft == 2 && p.n_ntiles * 256 < p.d_out))
        return cudaErrorInvalidValue;
    // a third token tile (FT = 1): its X box of at most kW4TailRows rows after the first two
    if (p.tail_rows && (ft != 1 || p.k_split > 1 || p.tail_rows > kW4TailRows || (p.tail_rows & 15) ||
                        p.x_stage_bytes < 32768 + p.tail_rows * 128))
        return cudaErrorInvalidValue;
    // K parts: every part a whole number of packed boxes (4 K-steps), the last one keeping at least one
    if (p.k_split > 1 && (p.k_chunk < 4 || (p.k_chunk & 3) || (p.k_split - 1) * p.k_chunk >= p.k_main_blocks ||
                          !p.partials || !p.split_ctr || p.part_rows < 1))
        return cudaErrorInvalidValue;
    const size_t smem = w4_smem_bytes(p.stages, p.pstages, p.x_stage_bytes, ft);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kW4Threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (p.k_split > 1 && w4_cooperative_launches()) {
        // the last part of a block waits for the block's other parts on other CTAs: a cooperative
        // launch starts only when its whole grid can be resident
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    const bool split = p.k_split > 1;
    if (ft == 2)
        return split ? cudaLaunchKernelEx(&cfg, dev::lora_w4_kernel<2, true, false>, p)
                     : cudaLaunchKernelEx(&cfg, dev::lora_w4_kernel<2, false, false>, p);
    if (p.tail_rows) return cudaLaunchKernelEx(&cfg, dev::lora_w4_kernel<1, false, true>, p);
    return split ? cudaLaunchKernelEx(&cfg, dev::lora_w4_kernel<1, true, false>, p)
                 : cudaLaunchKernelEx(&cfg, dev::lora_w4_kernel<1, false, false>, p);
}

}  // namespace lora
