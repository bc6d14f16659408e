// Internal declarations shared by the library's translation units (not installed).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

namespace lora {

constexpr int kTileM = 128;          // rows per tile = tcgen05 M (cta_group::1)
constexpr int kTileK = 64;           // default K per pipeline stage: one 128-byte swizzle row of bf16
constexpr int kMaxTileN = 256;       // widest output tile = one TMEM accumulator (256 fp32 columns)
constexpr int kMaxWideTileN = 512;   // widest row tile of the two-MMA instantiation (one 512-column accumulator)
constexpr int kAccCols = 256;        // TMEM columns per accumulator; two accumulators per CTA
constexpr int kStageBytesA = kTileM * kTileK * 2;      // 16 KB at K = 64
constexpr int kMaxStages = 16;
constexpr int kSmemLimit = 232448;                     // opt-in dynamic shared memory per CTA (227 KB)
constexpr int kThreads = 192;        // warp 0 TMA, warp 1 MMA + TMEM owner, warps 2..5 epilogue
constexpr int kThreadsWide = 224;    // two-MMA units: warp 6 issues the second MMA of each K16 step
// Unit forms of the bf16 kernel, one instantiation each: row tiles (up to 256 output columns),
// token-column units (blocks of Y^T), wide row tiles (272 to 512 output columns, SM pairs)
constexpr int kFormRows = 0, kFormTokenColumns = 1, kFormWideRows = 2;
constexpr int kYtStageBytes = 4 * 32 * 32 * 2;  // token-column epilogue: 32 tokens x 32 features bf16 per warp
constexpr int kEpilogueThreads = 128;
constexpr int kW4Group = 128;        // input features per scale of a 4-bit base
// Work lists this small travel inside the kernel parameters (no upload copy per call).
constexpr int kInlineTiles = 64;     // fused + shrink tiles (cluster groups included)
constexpr int kInlineSegs = 48;      // merged segments
constexpr int kInlineAdapters = 4;   // adapters named in the call
constexpr int kMaxKSplit = 4;        // most parts a block's K is split into

struct Tile {                        // one planner tile, as uploaded to the device
    int32_t row0, nrows, adapter;    // adapter: compact slot (1-based), 0 = none
    int32_t fused_index;             // ready-flag slot: index of these rows among the fused tiles
                                     // (-1 on a shrink tile that only pads a cluster group)
    int32_t u_row;                   // first U row the expand reads (fused tiles): row0, or a
                                     // block of U that is always zero for a base tile that shares
                                     // an SM pair (and so the pair's expand) with an adapter tile
    int32_t split_index;             // fused tiles: this tile's own index among the fused tiles
                                     // (its K-half counters; unlike fused_index, never a partner's)
};

// Parameters of one launch of the tile GEMM. Passed by value as a __grid_constant__.
// Work units: [0, n_shrink) are shrink units (U rows of adapter tiles, N = shrink_n), then
// n_fused x n_ntiles fused units (128 x tile_n blocks of Y: base K-loop over d_in, then,
// for adapter tiles, the expand K-loop over the rank into the same accumulator). With
// cluster_size 2 a unit is a group of two row tiles (tiles 2g and 2g+1 of the arrays, one
// per CTA of the cluster) that share the same B operand tile; each CTA loads half of that
// tile's rows and the pair runs M = 256 MMAs. Groups are padded with tiles of nrows 0.
// When `flags` is set, a fused unit's expand waits until flags[tile] == 1, which the shrink
// unit of that tile publishes after its U rows are stored (single-launch mode).
// With k_split == S > 1 every unit (shrink or fused) is split into S units over S parts of the
// base K-steps (the expand goes with the last part): every part but the last to finish stores its
// fp32 partial sums; the last adds the S sums in part order (so the sum does not depend on which
// part finishes last) and stores Y (or U, and publishes its flag).
struct GemmParams {
    // inline work list (used when inline_wl != 0): adapter tensor maps (B_a at [0, 4), A_a
    // at [4, 8)), tiles (fused then shrink), merged segments (offsets then ids), scales
    CUtensorMap inline_maps[2 * kInlineAdapters];
    Tile inline_tiles[kInlineTiles];
    int32_t inline_seg[2 * kInlineSegs + 1];
    float inline_scales[kInlineAdapters];
    int inline_wl;
    int inline_shrink_off;           // index of the first shrink tile in inline_tiles
    CUtensorMap tm_x;                // X [T, d_in], box 64 x 128
    CUtensorMap tm_w;                // W [d_out, d_in], box 64 x tile_n
    CUtensorMap tm_u;                // U [u_rows, rank], box 64 x 128
    const CUtensorMap* tm_b;         // device array per compact adapter: B_a [d_out, rank], box 64 x tile_n
    const CUtensorMap* tm_a;         // device array per compact adapter: A_a [rank, d_in], box 64 x shrink_n
    const Tile* shrink_tiles;        // device [n_shrink]
    const Tile* fused_tiles;         // device [n_fused]
    const int32_t* seg_off;          // merged segments (device), compact ids
    const int32_t* seg_id;
    const float* scales;             // per compact adapter (device)
    void* y;                         // Y [T, d_out] bf16
    void* u;                         // U [u_rows, rank] bf16
    int* flags;                      // per fused tile: 1 once its U rows are stored; nullptr = no
                                     // in-kernel dependency. Zero at launch, cleared at exit.
    int* done_count;                 // CTAs that finished the launch (the last one clears flags)
    int n_flags;                     // flags [0, n_flags) in use
    int* status;                     // device status word: bit 0 = a bounded wait ran out
    unsigned long long wait_limit_ns;
    int n_seg;
    int n_shrink;                    // shrink groups (tiles = cluster_size x groups)
    int n_fused;                     // fused row groups
    int n_ntiles;                    // output-column tiles of the fused units
    int tile_n;                      // fused output-tile width (multiple of 16, <= 256; on SM pairs with
                                     // whole K per unit up to 512: wide row tiles, whose 16-wide K
                                     // steps take a second MMA over the B rows past 128 per CTA)
    int shrink_n;                    // shrink output-tile width = rank rounded up to 16
    int stages;
    int m_fastest;                   // 1: row tiles first, 0: column tiles first, 2: column-tile groups
    int raster_group;                // column tiles per group when m_fastest == 2
    int k_main_blocks;               // ceil(d_in / 64)
    int k_lora_blocks;               // ceil(rank / 64)
    int d_out;
    int rank;
    int cluster_size;                // CTA group of the MMA: 1, or 2 (an SM pair, M = 256)
    int bk;                          // K per pipeline stage: 64 (128-byte swizzle) or 32 (64-byte swizzle)
    int mma_group;                   // stages the MMA warp waits for at once (1 or 2)
    int a_rows;                      // rows of one A box (tm_x, tm_u): 0 or 128, or fewer (a multiple
                                     // of 16) for a batch of one tile on single CTAs
    int debug_stall;
    unsigned long long debug_publish_delay_ns;   // tests: shrink units publish their flag this late
    // K parts (k_split == 2 or 4; 0 or 1 = whole K per unit)
    int k_split;
    int k_chunk;                     // base K-steps of every part but the last (which takes the rest)
    float4* partials;                // fp32 partial sums: part q's float4 chunk c (output columns
                                     // 4c .. 4c+3) of row t at [(q * part_chunks + c) * part_rows + t]
    int part_rows;                   // row stride of `partials` (>= T)
    int part_chunks;                 // float4 chunks per part: Y's columns, then U's
    int* split_ctr;                  // per (fused tile, column tile): {halves arrived, partials stored};
                                     // zero at launch, cleared at exit by the last CTA
    int n_split_slots;               // counter pairs in use: fused tiles x column tiles, then the
                                     // shrink tiles (padding included) from shrink_slot0
    int shrink_slot0;
    int u_chunk0;                    // float4 chunk of U's column 0 in `partials` (after Y's chunks)
    // Programmatic dependent launch: the launch may start before the previous kernel of the stream
    // ends; only the W tiles of its first unit's first ring stages are loaded before it waits for
    // that kernel, and it lets the next kernel start early in turn
    int pdl;
    // Token-column units (yt = 1, SM pairs, K-steps of 64): every fused unit computes a block of
    // Y^T, 256 output features (the MMA's M: 128 per CTA of the pair) for every token row of the
    // batch (the MMA's N), so a W tile is read once for all rows and no row tile is padded. CTA r
    // of the pair holds token rows [r * yt_rows, (r + 1) * yt_rows) of each stage. The first MMA
    // of a 16-wide K-step takes rows [0, yt_h) of both CTAs' stages (N = 2 yt_h) into accumulator
    // columns [0, 2 yt_h); when yt_rows > yt_h a second takes rows [yt_h, yt_rows) (N = 2 (yt_rows
    // - yt_h)) into the columns after them. The launch runs n_ntiles such units (n_fused = 1).
    // Every token row names the same adapter, yt_adapter (0: none, no expand); the expand reads U
    // through tm_u, whose box is then yt_rows rows.
    // Shrink units over rank tiles (a launch of shrink units alone, without ready flags or K
    // parts): every shrink group runs shrink_ntiles units of shrink_n rank columns each.
    int shrink_ntiles;               // 0 or 1: one unit over the whole rank
    int yt;
    int yt_tokens;                   // T: token rows stored
    int yt_rows;                     // token rows per CTA per stage (a multiple of 8, <= 256)
    int yt_h;                        // token rows per CTA of the first MMA (a multiple of 8, <= 128)
    int yt_adapter;
    CUtensorMap tm_xt;               // X [T, d_in], box 64 x yt_rows (token-column units)
};

// Token rows per CTA and per CTA of the first MMA of a token-column launch for T rows
// (T <= 2 * kMaxYtRows): an SM pair holds 2 * rows token rows; past 128 rows per CTA the first
// MMA takes 128 of them (N = 256) and a second the rest.
constexpr int kMaxYtRows = 256;
inline void yt_split(int T, int* rows, int* h) {
    int tb = (T + 1) / 2;
    tb = (tb + 7) / 8 * 8;
    *rows = tb;
    *h = tb < 128 ? tb : 128;
}

// The plan of one call: merged segments and tiles, ids remapped to compact adapter slots.
struct Plan {
    std::vector<int32_t> seg_off, seg_id;    // merged runs (compact ids)
    std::vector<Tile> fused, shrink;
    std::vector<int> used_adapters;          // compact slot -> caller's adapter index (0-based)
};

// planner.cpp
int plan_segments(const int32_t* seg_offsets, const int32_t* seg_ids, int n_seg, int T,
                  int n_adapters, Plan* plan);

// kernels.cu
size_t gemm_smem_bytes(int b_tile_rows, int stages, int bk, int a_rows = kTileM, int yt = 0);
cudaError_t gemm_prepare_device();           // sets the opt-in smem limit on the current device
cudaError_t launch_gemm(const GemmParams& p, int grid, cudaStream_t stream);
int gemm_max_clusters(const GemmParams& p);  // co-resident clusters of this launch shape
int gemm_b_rows(const GemmParams& p);        // B rows of one CTA's pipeline stage
bool gemm_wide(const GemmParams& p);         // the launch runs the two-MMA instantiation
cudaError_t w4_repack(const void* src, void* dst, long long n_words, int grid, cudaStream_t stream);

}  // namespace lora
