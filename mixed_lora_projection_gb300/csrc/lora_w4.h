// Internal declarations of the 4-bit-base kernel (kernels_w4.cu) and its host side (not
// installed). Kept apart from lora_internal.h so that the bf16 kernel's sources do not change
// when only this kernel's parameters do.
#pragma once

#include "lora_internal.h"

namespace lora {

// 4-bit base kernel (transposed tile: output features on the MMA's M side, tokens on N).
// A token group is one or two consecutive planner tiles (each <= 128 rows and one adapter);
// its X rows form the B operand of up to 256 columns. A batch of exactly three tiles whose last
// one has at most kW4TailRows rows is one group of three: the third tile's rows (its own X box)
// are the B operand of a second MMA per 16-wide K step, so each weight tile is dequantised once
// for the whole batch. Units = groups x output tiles of 128 features, in the order
// W4Params::tokens_fastest selects.
constexpr int kW4TileM = 128;         // output features per unit (TMEM lanes)
constexpr int kW4Threads = 512;       // warp 0 TMA (X, U, B_a), 1 MMA, 2..5 epilogue,
                                      // 6..13 dequantise into TMEM, 14 TMA of the packed base,
                                      // 15 the second MMA of a K16 step: the second feature
                                      // tile's (two feature tiles per unit) or the third token
                                      // tile's (three token tiles per group)
constexpr int kW4TailRows = 96;       // most rows of the third token tile of a group
constexpr int kW4ConvertWarps = 8;
constexpr int kW4AStages = 8;         // most ring stages (TMEM A stages of 32 columns each)
constexpr int kW4InlineGroups = 48;
constexpr int kW4PackBytes = 128;     // packed bytes per row per TMA box (4 K-steps of 64)

struct W4Group {
    int32_t row0[3], nrows[3], adapter[3];  // a tile is absent when its nrows is 0
};

struct W4Params {
    CUtensorMap inline_bmaps[kInlineAdapters];  // B_a [d_out, rank], box 64 x 128 (inline work list)
    W4Group inline_groups[kW4InlineGroups];
    int inline_wl;
    CUtensorMap tm_x;                // X [T, d_in] bf16, box 64 x 128, 128-byte swizzle
    CUtensorMap tm_x3;               // X, box 64 x tail_rows: the third token tile of a group
    CUtensorMap tm_u;                // U [u_rows, rank] bf16, box 64 x 128, 128-byte swizzle
    CUtensorMap tm_wq;               // packed base [d_out, d_in/2] u8 (kernel layout), box 128 x 128, swizzled
    CUtensorMap tm_ws;               // scales [d_in/128, d_out] bf16, box 128 x 2
    CUtensorMap tm_y;                // Y [T, d_out] bf16, box 128 x 32, no swizzle (whole 32-row chunks)
    const CUtensorMap* tm_b;         // device array per compact adapter (when not inline)
    const W4Group* groups;           // device array (when not inline)
    void* y;                         // Y [T, d_out] bf16
    int* status;
    unsigned long long wait_limit_ns;
    int n_groups;
    int n_ntiles;                    // ceil(d_out / 128)
    int k_main_blocks;               // ceil(d_in / 64)
    int k_lora_blocks;               // ceil(rank / 64)
    int k_pack_blocks;               // ceil(k_main_blocks / 4)
    int d_out;
    int stages;                      // X / U ring
    int pstages;                     // packed ring
    int x_stage_bytes;               // bytes per X / U ring stage (a multiple of 1024)
    int tokens_fastest;              // unit order: 1 = token groups fastest, 0 = feature tiles fastest
    int feature_tiles;               // 128-feature tiles per unit: 1, or 2 for one token tile of at
                                     // most 128 rows with no adapter rows (tm_wq / tm_ws boxes 128 x FT)
    int tail_rows;                   // FT = 1: rows of the third token tile's X box (a multiple of 16,
                                     // <= kW4TailRows) when the call's group has three tiles, else 0
    // K parts (k_split > 1): every (token group, feature tile) block runs as k_split units over
    // parts of the base K-steps (k_chunk each, a multiple of 4; the last part takes the rest and
    // the expand); every part but the last to finish stores its fp32 sums in `partials`, the last
    // adds the k_split sums in part order and stores Y. Counters only grow (64-bit): the k-th
    // launch's arrivals at a block are k_split k .. k_split k + k_split - 1.
    int k_split;
    int k_chunk;
    float* partials;                 // part q, row t, feature n at [(q * part_rows + t) * d_out + n]
    int part_rows;
    unsigned long long* split_ctr;   // per block: {parts arrived, partial sums stored}
    int debug_stall;
};

// kernels_w4.cu
size_t w4_smem_bytes(int stages, int pstages, int x_stage_bytes, int ft);
cudaError_t w4_prepare_device();
cudaError_t launch_w4(const W4Params& p, int grid, cudaStream_t stream);

}  // namespace lora
