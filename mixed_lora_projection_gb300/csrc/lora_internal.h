// Internal declarations shared by the library's translation units (not installed).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

namespace lora {

constexpr int kTileM = 128;          // rows per tile = tcgen05 M (cta_group::1)
constexpr int kTileK = 64;           // K per pipeline stage: one 128-byte swizzle row of bf16
constexpr int kMaxTileN = 256;       // widest output tile = one TMEM accumulator (256 fp32 columns)
constexpr int kAccCols = 256;        // TMEM columns per accumulator; two accumulators per CTA
constexpr int kStageBytesA = kTileM * kTileK * 2;      // 16 KB
constexpr int kMaxStages = 12;
constexpr int kSmemBudget = 232448 - 2048;             // opt-in dynamic smem minus slack
constexpr int kThreads = 192;        // warp 0 TMA, warp 1 MMA + TMEM owner, warps 2..5 epilogue
constexpr int kEpilogueThreads = 128;

enum Mode { kFused = 0, kShrink = 1 };

struct Tile {                        // one planner tile, as uploaded to the device
    int32_t row0, nrows, adapter, pad;
};

// Parameters of one launch of the tile GEMM. Passed by value as a __grid_constant__.
struct GemmParams {
    CUtensorMap tm_x;                // X [T, d_in], box 64 x 128
    CUtensorMap tm_w;                // W [d_out, d_in], box 64 x tile_n (fused only)
    CUtensorMap tm_u;                // U [u_rows, rank], box 64 x 128 (fused only)
    const CUtensorMap* tm_adapter;   // device array, per compact adapter: fused -> B_a, shrink -> A_a
    const Tile* tiles;               // device array [n_tiles]
    const int32_t* seg_off;          // merged segments (device), compact ids
    const int32_t* seg_id;
    const float* scales;             // per compact adapter (device)
    void* out;                       // Y [T, d_out] (fused) or U [u_rows, rank] (shrink), bf16
    int* status;                     // device status word: bit 0 = a bounded wait ran out
    unsigned long long wait_limit_ns;
    int n_seg;
    int n_tiles;                     // planner tiles in this launch
    int n_ntiles;                    // output-column tiles
    int tile_n;                      // output-tile width (multiple of 16, <= 256)
    int stages;
    int m_fastest;                   // 1: consecutive work units walk row tiles first
    int k_main_blocks;               // ceil(d_in / 64)
    int k_lora_blocks;               // ceil(rank / 64) (fused) or 0
    int ld_out;                      // row stride of out, elements
    int n_out;                       // valid output columns (d_out or rank)
    int debug_stall;
};

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
size_t gemm_smem_bytes(int tile_n, int stages);
cudaError_t gemm_prepare_device();           // sets the opt-in smem limit on the current device
cudaError_t launch_gemm(int mode, const GemmParams& p, int grid, cudaStream_t stream);

}  // namespace lora
