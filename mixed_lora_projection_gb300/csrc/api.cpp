// C-ABI of the shared-base, per-request LoRA projection: handle, argument checks,
// work-list upload and the two launches per call (shrink, then fused base+expand).
//
// Source: "Two 27B models on a single RTX 5090", sections 3-4 (W + B.A per changed
// matrix; the adapter's two thin matrices run only for the requests that name it, in
// the same batches as base requests).
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <unordered_map>
#include <vector>

#include "../../include/lora_linear.h"
#include "lora_internal.h"
#include "lora_w4.h"

using namespace lora;

namespace {

constexpr int kRing = 8;  // work-list slots in flight per handle

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct Slot {
    uint8_t* host = nullptr;   // pinned
    uint8_t* dev = nullptr;
    cudaEvent_t done = nullptr;
    bool pending = false;
};

struct TimingRec {
    cudaEvent_t ev[3];
    bool has_shrink;
};

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

int check_shape(int d_in, int d_out, int rank, int max_tokens, int max_segments) {
    if (d_in <= 0 || d_out <= 0 || (d_in % 8) || (d_out % 8)) return LORA_EINVAL;
    if (d_in > LORA_MAX_FEATURES || d_out > LORA_MAX_FEATURES) return LORA_EINVAL;
    if (rank < 8 || rank > LORA_MAX_RANK || (rank % 8)) return LORA_EINVAL;
    if (max_tokens < 1 || max_segments < 1 || max_tokens > LORA_MAX_TOKENS || max_segments > LORA_MAX_SEGMENTS)
        return LORA_EINVAL;
    return LORA_OK;
}

}  // namespace

struct lora_linear {
    int device = 0, d_in = 0, d_out = 0, rank = 0, max_tokens = 0, max_segments = 0;
    int num_sms = 0;
    void* u_ws = nullptr;       // bf16 [u_rows, rank]: shrink output, read by the fused pass
    int u_rows = 0;
    int* status = nullptr;      // device status word
    int* flags = nullptr;       // per fused tile: U rows ready (1) in the running launch; then the
                                // launch's exit counter. All zero between launches.
    int* status_host = nullptr; // pinned copy for forward_host
    Slot slots[kRing];
    size_t slot_bytes = 0;
    int next_slot = 0;
    int max_fused = 0;
    EncodeTiledFn encode = nullptr;
    // options
    int force_tile_n = 0, raster = 0, debug_stall = 0, timing = 0, two_launch = 0, cluster = 0;
    unsigned long long debug_publish_delay_ns = 0;
    int raster_group = 4, tile_k = 0, allow_inline = 1, mma_group = 0;  // 0: 2 for SM pairs, else 1
    int max_ctas = 0;           // LORA_OPT_MAX_CTAS: at most this many CTAs per launch (0 = one per SM)
    int pdl = 0;                // LORA_OPT_PDL: launches without ready flags may start early
    int yt_mode = 0;            // LORA_OPT_TOKEN_COLUMNS: 0 = auto, 1 = never, 2 = whenever a batch allows
    int wide_mode = 0;          // LORA_OPT_WIDE_TILES: 0 = auto, 1 = never
    // 4-bit base K parts: chosen once per handle like k_split
    int w4_k_split = 1;         // 1..4: every 4-bit block runs as that many units over parts of K
    int w4_k_split_opt = 0;     // LORA_OPT_W4_K_SPLIT: 0 = the handle's own choice
    float* w4_partials = nullptr;                 // [part][max_tokens][d_out] fp32
    int w4_partial_parts = 0;
    unsigned long long* w4_split_ctr = nullptr;   // per block {arrived, stored}, only ever growing
    size_t w4_split_blocks = 0;
    int max_clusters_cache[2][kMaxYtRows / 8 + 1] = {};  // co-resident clusters by (size, B rows per CTA)
    // K halves: chosen once per handle (every call on it sums each output the same way)
    int k_split = 1;            // 1, 2 or 4: every block runs as that many units over parts of K
    int k_split_opt = 0;        // LORA_OPT_K_SPLIT: 0 = the handle's own choice, 1, 2 or 4 = forced
    float4* partials = nullptr; // fp32 partial sums: per K part, the float4 chunks of Y's and U's
                                // columns x max_tokens rows
    int partial_parts = 0;      // K parts `partials` has room for
    int* split_ctr = nullptr;   // per (fused tile, column tile): halves arrived, partials stored
    size_t split_slots = 0;     // counter pairs allocated
    std::unordered_map<uint64_t, uint32_t> shape_cache;   // plan signature -> (cs << 16) | tile_n
    unsigned long long wait_limit_ns = 4000000000ull;
    std::vector<TimingRec> trec;
    std::vector<cudaEvent_t> ev_pool;
    long long launches = 0;
    // staging for forward_host: device copies of X and Y, copy streams, chunk events
    void* x_stage = nullptr;
    void* y_stage = nullptr;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t ev_in[16] = {}, ev_done[16] = {};
};

namespace {

struct DeviceGuard {
    int prev = -1;
    bool changed = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) {
            changed = cudaSetDevice(dev) == cudaSuccess;
        }
    }
    ~DeviceGuard() {
        if (changed) cudaSetDevice(prev);
    }
};

void free_handle(lora_linear* h) {
    if (!h) return;
    for (Slot& s : h->slots) {
        if (s.host) cudaFreeHost(s.host);
        if (s.dev) cudaFree(s.dev);
        if (s.done) cudaEventDestroy(s.done);
    }
    for (TimingRec& r : h->trec)
        for (cudaEvent_t e : r.ev) h->ev_pool.push_back(e);
    for (cudaEvent_t e : h->ev_pool) cudaEventDestroy(e);
    if (h->u_ws) cudaFree(h->u_ws);
    if (h->partials) cudaFree(h->partials);
    if (h->split_ctr) cudaFree(h->split_ctr);
    if (h->w4_partials) cudaFree(h->w4_partials);
    if (h->w4_split_ctr) cudaFree(h->w4_split_ctr);
    if (h->status) cudaFree(h->status);
    if (h->flags) cudaFree(h->flags);
    if (h->status_host) cudaFreeHost(h->status_host);
    if (h->x_stage) cudaFree(h->x_stage);
    if (h->y_stage) cudaFree(h->y_stage);
    if (h->s_in) cudaStreamDestroy(h->s_in);
    if (h->s_out) cudaStreamDestroy(h->s_out);
    for (int i = 0; i < 16; ++i) {
        if (h->ev_in[i]) cudaEventDestroy(h->ev_in[i]);
        if (h->ev_done[i]) cudaEventDestroy(h->ev_done[i]);
    }
    delete h;
}

cudaEvent_t take_event(lora_linear* h) {
    if (!h->ev_pool.empty()) {
        cudaEvent_t e = h->ev_pool.back();
        h->ev_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

CUresult encode_2d(lora_linear* h, CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                   uint32_t box_inner, uint32_t box_outer) {
    // the swizzle is as wide as the box rows: 64 bf16 -> 128 bytes, 32 bf16 -> 64 bytes
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return h->encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     box_inner == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Deepest ring that fits the opt-in shared memory, for `b_rows` B rows per CTA.
int stages_for(int b_rows, int bk, int a_rows = kTileM, int yt = 0) {
    int s = kMaxStages;
    while (s > 2 && gemm_smem_bytes(b_rows, s, bk, a_rows, yt) > (size_t)kSmemLimit) --s;
    return s;
}

// 2-D map of bytes whose 128-byte box rows are 128-byte swizzled (the 4-bit base's packed
// rows, read 16 bytes per thread without bank conflicts).
CUresult encode_u8_sw128(lora_linear* h, CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                         uint32_t box_outer) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner};
    cuuint32_t box[2] = {128, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return h->encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Token groups of the 4-bit base kernel: consecutive planner tiles in pairs.
std::vector<W4Group> make_w4_groups(const std::vector<Tile>& fused, bool allow_three = true) {
    std::vector<W4Group> g;
    // a batch of exactly three tiles whose last has at most kW4TailRows rows (a 300-row decision
    // beside chat rows) is one group: each weight tile is dequantised once for all of it (not on
    // handles that split the 4-bit K-steps)
    const size_t per = (allow_three && fused.size() == 3 && fused[2].nrows <= kW4TailRows) ? 3 : 2;
    for (size_t i = 0; i < fused.size(); i += per) {
        W4Group w;
        memset(&w, 0, sizeof(w));
        for (size_t k = 0; k < per && i + k < fused.size(); ++k) {
            w.row0[k] = fused[i + k].row0;
            w.nrows[k] = fused[i + k].nrows;
            w.adapter[k] = fused[i + k].adapter;
        }
        g.push_back(w);
    }
    return g;
}

// 2-D map without swizzle (the 4-bit base's packed rows and scales).
CUresult encode_plain_2d(lora_linear* h, CUtensorMap* m, CUtensorMapDataType dtype, int elem_bytes,
                         const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * (uint64_t)elem_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return h->encode(m, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// SMs a launch of this handle may use: all of them, or LORA_OPT_MAX_CTAS of them (so that
// calls on other streams can run beside it on the rest).
int usable_sms(const lora_linear* h) {
    return h->max_ctas > 0 ? std::min(h->num_sms, h->max_ctas) : h->num_sms;
}

// Output-tile width: the per-SM critical path is (waves x (tile_n + fixed cost)); narrow
// tiles only where the row count is small enough that the pass streams W from memory.
int choose_tile_n(const lora_linear* h, int n_fused, int n_groups, int slots, int k_split = 1) {
    if (h->force_tile_n) return h->force_tile_n;
    const bool small_batch = (long long)n_fused * kTileM <= 384;
    long long best_cost = -1;
    int best = kMaxTileN;
    for (int tn = kMaxTileN; tn >= 16; tn -= 16) {
        if (!small_batch && tn < 128) break;
        // with K halves every output block is two units of half the K-steps
        long long units = (long long)n_groups * ceil_div(h->d_out, tn) * k_split;
        long long waves = (units + slots - 1) / slots;
        long long cost = waves * (tn + 16);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = tn;
        }
    }
    return best;
}

// Rasterisation: consecutive work units run at the same time on different SMs (a
// "wave"). Walking output-column tiles fastest re-reads all of W every wave; walking row
// tiles fastest re-reads all of X. Pick the order whose per-wave DRAM bytes are smaller,
// counting an operand as L2-resident across waves when it fits in ~96 MB of the 129 MB L2.
int choose_m_fastest(const lora_linear* h, int n_tiles, int n_ntiles, int tile_n, int rows_per_unit,
                     int slots) {
    if (h->raster == 1) return 1;
    if (h->raster == 2) return 0;
    if (h->raster == 3) return 2;
    const double l2_budget = 96e6;
    const long long units = (long long)n_tiles * n_ntiles;
    const long long g = std::min<long long>(units, slots);
    const double xb = (double)rows_per_unit * h->d_in * 2, wb = (double)tile_n * h->d_in * 2;
    const double total_x = (double)n_tiles * xb, total_w = (double)n_ntiles * wb;
    const double rows_n = ceil_div(g, n_ntiles), cols_n = (double)std::min<long long>(g, n_ntiles);
    const double rows_m = (double)std::min<long long>(g, n_tiles), cols_m = ceil_div(g, n_tiles);
    const double cost_n = rows_n * xb + (total_w > l2_budget ? cols_n * wb : 0.0);
    const double cost_m = cols_m * wb + (total_x > l2_budget ? rows_m * xb : 0.0);
    if (cost_m < cost_n) return 1;
    // Column tiles fastest: when W is larger than ~40 MB, walking it in two halves (groups of
    // half the column tiles, all row tiles of a group before the next) reads X twice but keeps
    // each half of W in L2 across its waves. Measured under the power limit, where DRAM traffic
    // costs clock: 16k and 32k prefills +1.5-2% over whole rows of column tiles.
    if (total_w > 40e6 && n_ntiles >= 4) return 2;
    return 0;
}

// Launch shape of one call: cluster size, tile widths, pipeline depth, rasterisation.
struct Shape {
    int cs = 1, tile_n = 0, shrink_n = 0, n_ntiles = 0, stages = 0, m_fastest = 0, bk = 64, raster_group = 1;
    int a_rows = kTileM;   // rows of one A box: the tile's rows when the batch is one short tile
    int yt = 0, yt_rows = 0, yt_h = 0;   // token-column units (SM pairs, 256 features x every token row)
    std::vector<Tile> fused_groups, shrink_groups;  // cs tiles per group
};

// Groups of `cs` consecutive tiles that share the B tile of their MMAs. Shrink tiles pair
// when they name the same adapter (their B operand is A_a). Fused tiles pair when they name
// the same adapter or when one of them names none: the pair then runs the adapter's expand,
// and the base tile's half reads its U operand from `zero_row`, a block of U that is always
// zero, so its rows gain exact zeros. A tile without a partner is padded with a copy of
// itself that has no rows. A padding shrink tile gets flag slot -1 (it publishes nothing); a
// padding or base fused tile takes its partner's slot (it waits for the same U rows).
void make_groups(const std::vector<Tile>& tiles, int cs, bool shrink, int zero_row, std::vector<Tile>* out) {
    out->clear();
    for (size_t i = 0; i < tiles.size();) {
        if (cs == 1) {
            out->push_back(tiles[i]);
            ++i;
            continue;
        }
        const bool has_next = i + 1 < tiles.size();
        const int a0 = tiles[i].adapter, a1 = has_next ? tiles[i + 1].adapter : -1;
        if (has_next && (a0 == a1 || (!shrink && (a0 == 0 || a1 == 0)))) {
            Tile t0 = tiles[i], t1 = tiles[i + 1];
            if (a0 != a1) {
                Tile& base = a0 == 0 ? t0 : t1;
                const Tile& other = a0 == 0 ? t1 : t0;
                base.adapter = other.adapter;
                base.fused_index = other.fused_index;
                base.u_row = zero_row;
            }
            out->push_back(t0);
            out->push_back(t1);
            i += 2;
        } else {
            Tile pad = tiles[i];
            pad.nrows = 0;
            if (shrink) pad.fused_index = -1;
            out->push_back(tiles[i]);
            out->push_back(pad);
            i += 1;
        }
    }
}

int max_clusters(lora_linear* h, const GemmParams& p) {
    const int b_rows = gemm_b_rows(p);
    int& c = h->max_clusters_cache[p.cluster_size - 1][b_rows / 8];
    if (c == 0) c = gemm_max_clusters(p);
    return c;
}

// Per-SM cycles of one 64-wide K-step of an N-column unit, measured on GB300: a single CTA
// is bound by how fast its shared memory fills (A + B tile, ~61 bytes per clock); an SM pair
// lands only half of B per SM and its cost falls less than proportionally with N (the A tile
// and the per-step barrier round trips stay): fitted to 16k-prefill units of 256, 224 and 192
// columns, which cost 1 : 0.954 : 0.862 per unit.
//
// Wide row tiles (SM pairs, 288 to 320 columns) add a second MMA per 16-wide K step over the
// columns past 256, which costs ~50-90 cycles whatever its width (the tensor pipe's floor per
// instruction), and hold all of TMEM in one accumulator: measured per unit against a 256-column
// unit on 2,048-row projections, 1.31x (down, 17,408 -> 5,120) to 1.51x (o, 6,144 -> 5,120) for
// 12-25% more columns. They pay where they take a wave off a projection whose 256-column units
// leave the last wave of SM pairs at most half full (down at 2,048 rows: 160 units of 256 columns
// on 76 SM pairs, 3 waves, the last 17% full; 149 of 288, 2 waves: 271 -> 237 us; at 1,024 rows
// o and down 0.71x and 0.75x of the narrow tiles chosen before; o at 2,176 rows 0.92x), and are
// weighed only there: with the last wave 68% full (o, 3,456 rows) the model would expect 1% from
// them, o's measured 1.51x loses it. kWideKstepFactor is the per-K-step cost against a 256-column
// unit that reproduces the measured choices. Relative to the unit, the second MMA and the exposed
// epilogue cost more the shorter its K: on projections of 80 K-steps (d_in 5,120) wide units took
// 1.37-1.49x (qkv at 336 columns 177 against 172 us at 224; gate_up at 288-512 columns 490-555
// against 431 us at 256), so they are weighed only from kMinWideKSteps K-steps on.
constexpr double kWideKstepFactor = 1.32;
constexpr int kMinAutoWideTileN = 288, kMaxAutoWideTileN = 320, kMinWideKSteps = 96;

double kstep_cycles(int cs, int n) {
    if (cs > 1 && n > kMaxTileN) return kWideKstepFactor * kstep_cycles(2, kMaxTileN);
    if (cs > 1) return 300.0 + 1.58 * n;
    const double mma = 4.0 * std::max(n / 2.0, 48.0) + 130.0;
    const double fill = (kTileM + (double)n) * kTileK * 2.0 / 61.0;
    return std::max(fill, mma);
}

// Makespan (per-SM cycles) of the persistent round-robin schedule of one launch shape.
double makespan(const lora_linear* h, const std::vector<Tile>& fused_groups, const std::vector<Tile>& shrink_groups,
                int cs, int tile_n, int shrink_n, int slots, int k_split = 1) {
    const int k_main = ceil_div(h->d_in, kTileK), k_lora = ceil_div(h->rank, kTileK);
    const int n_ntiles = ceil_div(h->d_out, tile_n);
    const int nsg = (int)shrink_groups.size() / cs, nfg = (int)fused_groups.size() / cs;
    const double ks = kstep_cycles(cs, tile_n);
    const double c_shrink = k_main * kstep_cycles(cs, shrink_n);
    const double c_lora = k_lora * ks;
    // K parts: S units per block over k_chunk K-steps each (the last one the rest); with parts,
    // each unit pays about two K-steps more for the fp32 partial sums stored and read back
    const int S = k_split > 1 ? k_split : 1;
    const int k_chunk = ceil_div(k_main, S), extra = S > 1 ? 2 : 0;
    std::vector<double> load(slots, 0.0);
    long long u = 0;
    const double sk = c_shrink / k_main;
    for (int g = 0; g < nsg; ++g)
        for (int q = 0; q < S; ++q) {
            const int k = q == S - 1 ? k_main - (S - 1) * k_chunk : k_chunk;
            load[u++ % slots] += (k + extra) * sk;
        }
    // fused units in the kernel's order do not change the per-slot sums by much; use row-major
    for (int g = 0; g < nfg; ++g) {
        const double lora = fused_groups[(size_t)g * cs].adapter ? c_lora : 0.0;
        for (int t = 0; t < n_ntiles; ++t)
            for (int q = 0; q < S; ++q) {
                const int k = q == S - 1 ? k_main - (S - 1) * k_chunk : k_chunk;
                load[u++ % slots] += (k + extra) * ks + (q == S - 1 ? lora : 0.0);
            }
    }
    return *std::max_element(load.begin(), load.end());
}

// Per-SM cycles of one 64-wide K-step of a token-column unit whose pair holds 2 * rows token
// rows, its epilogue included, fitted to gate_up (5,120 -> 34,816) and qkv (5,120 -> 12,288)
// batches of 200 to 512 rows without adapter rows timed on GB300: one MMA per 16-wide step up to
// 128 rows per CTA (~940 cycles at 100 rows), a second one (from a second warp) and a single
// accumulator, whose epilogue no longer overlaps the next unit, past it (~1,150 cycles at 152
// rows, ~1,700 at 256). Units with an expand took ~8% more per K-step (the shrink units beside
// them and the wait for their flags). These units stream W from memory, so they run well above
// their MMA time.
double yt_kstep_cycles(int rows, bool adapter) {
    const double c = rows <= kTileM ? 850.0 + 0.9 * rows : 340.0 + 5.3 * rows;
    return adapter ? 1.08 * c : c;
}

// The row-tile model (kstep_cycles) is fitted to the tensor-bound shapes of large batches; on
// the batches token-column units serve (W streamed from memory) row tiles took 1.05-1.67x its
// makespan (gate_up and qkv, 200 to 512 rows). Token-column units are chosen when their makespan
// is below the row-tile makespan times this factor (the factor that lost least time over those
// 24 timed batches), and only up to kMaxYtAutoRows rows: past that the row tiles are four nearly
// full 128-row tiles on SM pairs and token-column units hold all of TMEM (gate_up at 512 rows:
// 134 against 115 us without adapter rows).
constexpr double kRowTileSmallBatchFactor = 1.40;
constexpr int kMaxYtAutoRows = 448;

// Token-column units serve a batch of at most 2 * kMaxYtRows rows whose tiles all name one
// adapter (or none), on SM pairs with 64-wide K-steps and whole K per unit; options that fix
// another shape rule them out.
bool yt_allowed(const lora_linear* h, const Plan& plan) {
    if (h->yt_mode == 1 || h->k_split > 1 || plan.fused.empty()) return false;
    if ((h->tile_k && h->tile_k != kTileK) || h->cluster == 1 || usable_sms(h) < 2) return false;
    if (h->force_tile_n && h->force_tile_n != kMaxTileN) return false;
    if (plan.seg_off.back() > 2 * kMaxYtRows) return false;
    for (const Tile& t : plan.fused)
        if (t.adapter != plan.fused[0].adapter) return false;
    return true;
}

// Makespan (per-SM cycles) of a token-column launch: the shrink groups (SM pairs), then one unit
// per 256 output features over every token row, round-robin over the SM pairs.
double yt_makespan(const lora_linear* h, const Plan& plan, int slots) {
    int rows = 0, hh = 0;
    yt_split(plan.seg_off.back(), &rows, &hh);
    const int k_main = ceil_div(h->d_in, kTileK), k_lora = ceil_div(h->rank, kTileK);
    const int shrink_n = ceil_div(h->rank, 16) * 16;
    std::vector<Tile> sg;
    make_groups(plan.shrink, 2, true, h->u_rows - kTileM, &sg);
    std::vector<double> load(slots, 0.0);
    long long u = 0;
    for (size_t g = 0; g < sg.size() / 2; ++g) load[u++ % slots] += k_main * kstep_cycles(2, shrink_n);
    const bool ad = plan.fused[0].adapter != 0;
    const double unit = (k_main + (ad ? k_lora : 0)) * yt_kstep_cycles(rows, ad);
    for (int t = 0; t < ceil_div(h->d_out, 2 * kTileM); ++t) load[u++ % slots] += unit;
    return *std::max_element(load.begin(), load.end());
}

// The launch shape (SM pair or single CTA, output-tile width) the makespan model expects to
// finish a plan soonest with K in `k_split` parts; cs / tn nonzero fix that choice; `wide` lets SM
// pairs weigh wide row tiles. Returns the expected makespan.
double search_shape(const lora_linear* h, const Plan& plan, int cs, int tn, int k_split, int* out_cs, int* out_tn,
                    bool wide = false) {
    const int nf = (int)plan.fused.size();
    const int shrink_n = ceil_div(h->rank, 16) * 16;
    const bool small_batch = (long long)nf * kTileM <= 384;
    if (small_batch && !cs) cs = 1;
    double best = -1;
    int best_cs = cs ? cs : 1, best_tn = tn ? tn : kMaxTileN;
    for (int c = 1; c <= 2; ++c) {
        if (cs && c != cs) continue;
        if (c == 2 && nf < 2) continue;
        std::vector<Tile> fg, sg;
        make_groups(plan.fused, c, false, h->u_rows - kTileM, &fg);
        make_groups(plan.shrink, c, true, h->u_rows - kTileM, &sg);
        const int slots = usable_sms(h) / c;
        if (small_batch) {
            const int t = tn ? tn : choose_tile_n(h, nf, (int)fg.size() / c, slots, k_split);
            const double m = makespan(h, fg, sg, c, t, shrink_n, slots, k_split);
            if (best < 0 || m < best) { best = m; best_cs = c; best_tn = t; }
            continue;
        }
        if (tn) {
            const double m = makespan(h, fg, sg, c, tn, shrink_n, slots, k_split);
            if (best < 0 || m < best * 0.999) { best = m; best_cs = c; best_tn = tn; }
            continue;
        }
        // Candidate widths in the order a tie goes to: 256 columns, then the wide tiles, then the
        // narrower ones. Wide tiles are weighed on SM pairs where 256-column units leave the last
        // wave at most half full (their gains were measured there: 2,048 rows of o and down 17%,
        // 1,024 rows 8%, 2,176 rows of o 43%).
        const long long u256 = (long long)(fg.size() / c) * ceil_div(h->d_out, kMaxTileN) + (long long)(sg.size() / c);
        const double last = (double)(u256 % slots) / slots;
        std::vector<int> widths{kMaxTileN};
        if (c == 2 && wide && last > 0.0 && last <= 0.5)
            for (int t = kMinAutoWideTileN; t <= kMaxAutoWideTileN; t += 16) widths.push_back(t);
        for (int t = kMaxTileN - 16; t >= 128; t -= 16) widths.push_back(t);
        for (const int t : widths) {
            const double m = makespan(h, fg, sg, c, t, shrink_n, slots, k_split);
            if (best < 0 || m < best * 0.999) { best = m; best_cs = c; best_tn = t; }
        }
    }
    *out_cs = best_cs;
    *out_tn = best_tn;
    return best;
}

Shape choose_shape(lora_linear* h, const Plan& plan, bool bf16 = true) {
    Shape sh;
    const int nf = (int)plan.fused.size();
    sh.shrink_n = ceil_div(h->rank, 16) * 16;
    sh.bk = h->tile_k ? h->tile_k : 64;
    const bool small_batch = (long long)nf * kTileM <= 384;
    int cs = h->cluster, tn = h->force_tile_n;
    // wide row tiles (past 256 columns) run on SM pairs of the bf16 kernel with whole K per unit
    if (tn > kMaxTileN) {
        if (!bf16 || cs == 1 || h->k_split > 1 || (h->tile_k && h->tile_k != kTileK)) tn = kMaxTileN;
        else cs = 2;
    }
    // K halves: whole 256-column blocks (narrower ones gained nothing where halves were measured)
    if (h->k_split > 1 && !small_batch && !tn) tn = kMaxTileN;
    const bool yt_ok = bf16 && yt_allowed(h, plan);
    int yt = 0;
    if (!cs || !tn || yt_ok) {
        const int cs0 = cs, tn0 = tn;
        if (small_batch && !cs) cs = 1;
        // plan signature: tile count and each tile's adapter / row count, then the options that
        // fix or restrict the choice, each mixed in on its own
        uint64_t key = 1469598103934665603ull ^ (uint64_t)nf;
        for (const Tile& t : plan.fused) key = (key ^ (uint64_t)(t.adapter * 131 + t.nrows)) * 1099511628211ull;
        for (const int v : {cs, tn, h->k_split, yt_ok ? 1 + h->yt_mode : 0, h->wide_mode, h->tile_k, h->max_ctas,
                            bf16 ? 1 : 0})
            key = (key ^ (uint64_t)(uint32_t)v) * 1099511628211ull;
        auto it = h->shape_cache.find(key);
        if (it != h->shape_cache.end()) {
            yt = (int)(it->second >> 31);
            cs = (int)((it->second >> 16) & 0x7FFF);
            tn = (int)(it->second & 0xFFFF);
        } else {
            double m = 0.0;
            // wide row tiles: bf16 base, whole K of at least kMinWideKSteps 64-wide K-steps
            const bool wide = bf16 && h->wide_mode != 1 && h->k_split <= 1 && (!h->tile_k || h->tile_k == kTileK) &&
                              ceil_div(h->d_in, kTileK) >= kMinWideKSteps;
            if (!cs || !tn) m = search_shape(h, plan, cs, tn, h->k_split, &cs, &tn, wide);
            if (yt_ok) {
                // token-column units when asked for, or, for batches of more than one row tile,
                // when the calibrated models expect them to finish sooner
                const int slots = usable_sms(h) / 2;
                if (h->yt_mode == 2 || (!cs0 && !tn0 && nf >= 2 && plan.seg_off.back() <= kMaxYtAutoRows &&
                                        yt_makespan(h, plan, slots) < kRowTileSmallBatchFactor * m))
                    yt = 1;
            }
            if (yt) {
                cs = 2;
                tn = kMaxTileN;
            }
            if (h->shape_cache.size() > 256) h->shape_cache.clear();
            h->shape_cache[key] = ((uint32_t)yt << 31) | ((uint32_t)cs << 16) | (uint32_t)tn;
        }
    }
    sh.cs = cs;
    make_groups(plan.fused, sh.cs, false, h->u_rows - kTileM, &sh.fused_groups);
    make_groups(plan.shrink, sh.cs, true, h->u_rows - kTileM, &sh.shrink_groups);
    const int nfg = (int)sh.fused_groups.size() / sh.cs;
    const int slots = usable_sms(h) / sh.cs;
    sh.tile_n = tn;
    sh.n_ntiles = ceil_div(h->d_out, sh.tile_n);
    // a batch of one tile of fewer than 128 rows (a decode step) on single CTAs loads only its
    // rows of X (and U): smaller A stages, a deeper ring for the W stream
    if (sh.cs == 1 && plan.fused.size() == 1) sh.a_rows = std::max(16, ceil_div(plan.fused[0].nrows, 16) * 16);
    if (plan.shrink.empty()) sh.shrink_n = 0;   // no shrink units: the B ring holds output tiles only
    sh.stages = stages_for(std::max(sh.tile_n, sh.shrink_n) / sh.cs, sh.bk, sh.a_rows);
    sh.m_fastest = choose_m_fastest(h, nfg, sh.n_ntiles, sh.tile_n, kTileM * sh.cs, slots);
    sh.raster_group = h->raster == 3 ? h->raster_group : ceil_div(sh.n_ntiles, 2);
    if (yt) {
        // one unit per 256 output features; a stage holds 128 W rows and this CTA's token rows
        sh.yt = 1;
        yt_split(plan.seg_off.back(), &sh.yt_rows, &sh.yt_h);
        sh.bk = kTileK;
        sh.a_rows = kTileM;
        sh.n_ntiles = ceil_div(h->d_out, 2 * kTileM);
        sh.stages = stages_for(std::max(sh.yt_rows, sh.shrink_n / 2), sh.bk, kTileM, 1);
        sh.m_fastest = 0;
    }
    return sh;
}

// Fused row groups of a launch shape: token-column units span every token row in one group.
int fused_row_groups(const Shape& sh) {
    return sh.yt ? 1 : (int)(sh.fused_groups.size() / sh.cs);
}

// K parts for a handle, decided once from its shape and max_tokens, so that every call on the
// handle sums each output the same way (a row's bits never depend on the batch it is in). The
// handle splits K in halves when it serves small batches (the single-CTA path: at most three
// 128-row tiles) of a projection with long K (at least 96 K-steps of 64, d_in >= 6,144) and the
// launch-shape model expects them to finish at least 7% sooner. Each SM then streams half of K
// over twice as many column blocks. Measured on 48-row batches: the o projection (6,144 ->
// 5,120) 1.3x and the down projection (17,408 -> 5,120) 2x faster with halves, qkv (5,120 ->
// 12,288) no faster; quarters were no faster than halves (o 30.0 against 25.2 us, down 47.4
// against 47.7 us: the last part reads three sets of partial sums), so the handle chooses them
// only when asked (LORA_OPT_K_SPLIT = 4). Past the small-batch path the round trip of the fp32
// partial sums through L2 cancels what the parts gain in the last wave (2,048 rows, halves: o
// +4%, down -4%, qkv -12%), so whole K stays.
int choose_k_split(lora_linear* h) {
    if (h->k_split_opt) {
        // as many parts as asked for, as long as every part keeps at least one K-step
        const int k64 = ceil_div(h->d_in, kTileK);
        int s = h->k_split_opt;
        while (s > 1 && (s - 1) * ceil_div(k64, s) >= k64) s /= 2;
        return s;
    }
    if (ceil_div(h->d_in, kTileK) < 96) return 1;
    const int32_t off[2] = {0, h->max_tokens}, ids[1] = {0};
    Plan plan;
    if (plan_segments(off, ids, 1, h->max_tokens, -1, &plan) != LORA_OK) return 1;
    if ((long long)plan.fused.size() * kTileM > 384) return 1;
    int cs = 0, tn = 0;
    const double whole = search_shape(h, plan, 0, 0, 1, &cs, &tn);
    const double halves = search_shape(h, plan, 0, 0, 2, &cs, &tn);
    return halves < 0.93 * whole ? 2 : 1;
}

// Device buffers of the K parts (fp32 partial sums per part and the per-block counters),
// allocated when the handle first splits K, and grown when it splits into more parts.
int ensure_split_buffers(lora_linear* h) {
    if (h->k_split < 2 || h->partial_parts >= h->k_split) return LORA_OK;
    // float4 chunks of Y's columns, then of U's, per part; counter pairs: (fused tile, column
    // tile), then shrink tiles (SM-pair padding included)
    const size_t chunks = (size_t)ceil_div(h->d_out, 4) + (size_t)ceil_div(h->rank, 4);
    const size_t slots = (size_t)std::min(h->max_fused, h->max_tokens) * ceil_div(h->d_out, 16) + 2 * (size_t)h->max_fused;
    if (h->partials) cudaFree(h->partials);
    h->partials = nullptr;
    h->partial_parts = 0;
    if (cudaMalloc((void**)&h->partials, (size_t)h->k_split * chunks * (size_t)h->max_tokens * sizeof(float4)) !=
        cudaSuccess) {
        cudaGetLastError();
        h->partials = nullptr;
        return LORA_ENOMEM;
    }
    h->partial_parts = h->k_split;
    if (!h->split_ctr) {
        if (cudaMalloc((void**)&h->split_ctr, 2 * slots * sizeof(int)) != cudaSuccess) {
            cudaGetLastError();
            h->split_ctr = nullptr;
            return LORA_ENOMEM;
        }
        if (cudaMemset(h->split_ctr, 0, 2 * slots * sizeof(int)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
            return LORA_ECUDA;
        h->split_slots = slots;
    }
    return LORA_OK;
}

// K parts of the 4-bit base for a handle, decided once from its shape and max_tokens (a row's
// bits never depend on the batch). Decode-sized handles (at most 128 rows: one token tile) of
// narrow projections leave most SMs without a unit of one 128-feature tile (o and down on 5,120
// outputs: 40 units for 152 SMs); they split the base K-steps into as many parts (at most 4,
// each at least 8 K-steps, a multiple of 4) as still fit one wave of units.
int choose_w4_k_split(const lora_linear* h) {
    const int k64 = ceil_div(h->d_in, kTileK);
    auto fits = [&](int s) {
        const int chunk = ceil_div(ceil_div(k64, s), 4) * 4;
        return s == 1 || (chunk >= 8 && (s - 1) * chunk < k64);
    };
    if (h->w4_k_split_opt) {
        int s = h->w4_k_split_opt;
        while (s > 1 && !fits(s)) --s;
        return s;
    }
    if (h->max_tokens > kTileM) return 1;
    const int units = ceil_div(h->d_out, kW4TileM);
    int best = 1;
    for (int s = 2; s <= 4; ++s)
        if (units * s <= usable_sms(h) && fits(s)) best = s;
    return best;
}

// The 4-bit K parts' device buffers: fp32 partial sums per part, and the block counters (zeroed
// whenever they are (re)allocated or the parts change).
int ensure_w4_split_buffers(lora_linear* h) {
    if (h->w4_k_split < 2) return LORA_OK;
    const size_t blocks = (size_t)h->max_fused * ceil_div(h->d_out, kW4TileM);
    if (h->w4_partial_parts < h->w4_k_split) {
        if (h->w4_partials) cudaFree(h->w4_partials);
        h->w4_partials = nullptr;
        h->w4_partial_parts = 0;
        if (cudaMalloc((void**)&h->w4_partials,
                       (size_t)h->w4_k_split * h->max_tokens * h->d_out * sizeof(float)) != cudaSuccess) {
            cudaGetLastError();
            h->w4_partials = nullptr;
            return LORA_ENOMEM;
        }
        h->w4_partial_parts = h->w4_k_split;
    }
    if (!h->w4_split_ctr) {
        if (cudaMalloc((void**)&h->w4_split_ctr, 2 * blocks * sizeof(unsigned long long)) != cudaSuccess) {
            cudaGetLastError();
            h->w4_split_ctr = nullptr;
            return LORA_ENOMEM;
        }
        h->w4_split_blocks = blocks;
    }
    if (cudaMemset(h->w4_split_ctr, 0, 2 * h->w4_split_blocks * sizeof(unsigned long long)) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
        return LORA_ECUDA;
    return LORA_OK;
}

// Launch shape of the 4-bit kernel for a call's token groups (host logic only).
struct W4Shape {
    int feature_tiles = 1, n_ntiles = 0, tokens_fastest = 0, x_stage_bytes = 0, stages = 4, pstages = 2;
    int tail_rows = 0;   // rows of the third token tile's X box (a group of three tiles), else 0
};

W4Shape w4_shape(const lora_linear* h, const std::vector<W4Group>& groups, int T) {
    W4Shape w;
    const int n = (int)groups.size();
    // a batch of one token tile of at most 128 rows and no adapter rows (a decode step) runs two
    // feature tiles per unit when that still gives most SMs a unit (gate_up: 136 units); narrower
    // projections keep one tile per unit, twice as many units (qkv 96, o and down 40)
    const bool one_tile =
        n == 1 && groups[0].nrows[1] == 0 && groups[0].nrows[0] <= kTileM && groups[0].adapter[0] == 0;
    w.feature_tiles = (one_tile && 4 * ceil_div(h->d_out, 2 * kW4TileM) >= 3 * usable_sms(h)) ? 2 : 1;
    w.n_ntiles = ceil_div(h->d_out, kW4TileM * w.feature_tiles);
    // unit order: token groups fastest when the packed base is too large to stay in L2 beside
    // the output stream while the batch's X fits there (the mixed batch on gate_up: 89 MB
    // packed, 42 MB of X), else feature tiles fastest; LORA_OPT_RASTER 1 / 2 force it
    const double packed_bytes = (double)h->d_out * h->d_in / 2, x_bytes = (double)T * h->d_in * 2;
    w.tokens_fastest = h->raster == 1   ? 1
                       : h->raster == 2 ? 0
                                        : (n > 1 && packed_bytes > 32e6 && x_bytes <= 64e6) ? 1 : 0;
    // X stages: two token tiles (and the expand's U + B_a boxes), or one tile when FT = 2, or
    // two tiles and a third tile's rows; the packed ring takes the rest of shared memory
    w.x_stage_bytes = w.feature_tiles == 2 ? kTileM * 128 : 2 * kTileM * 128;
    if (n == 1 && groups[0].nrows[2] > 0) {
        w.tail_rows = ceil_div(groups[0].nrows[2], 16) * 16;
        w.x_stage_bytes += w.tail_rows * 128;
    }
    while (w.pstages < 8 &&
           w4_smem_bytes(w.stages, w.pstages + 1, w.x_stage_bytes, w.feature_tiles) <= (size_t)kSmemLimit)
        ++w.pstages;
    return w;
}

Slot* acquire_slot(lora_linear* h) {
    Slot* s = &h->slots[h->next_slot];
    h->next_slot = (h->next_slot + 1) % kRing;
    if (s->pending) {
        if (cudaEventSynchronize(s->done) != cudaSuccess) return nullptr;
        s->pending = false;
    }
    return s;
}

}  // namespace

extern "C" {

const char* lora_linear_error_string(int code) {
    switch (code) {
        case LORA_OK: return "ok";
        case LORA_EINVAL: return "invalid argument";
        case LORA_ENOMEM: return "out of memory";
        case LORA_ECUDA: return "CUDA call failed";
        case LORA_ETIMEOUT: return "a kernel's bounded wait ran out";
        case LORA_EUNSUPPORTED: return "unsupported by this library";
        case LORA_ENODEV: return "no usable sm_103 device";
        default: return "unknown error";
    }
}

}  // extern "C"

static int validate_impl(int d_in, int d_out, int rank, int max_tokens, int max_segments, const void* x, int T,
                         const int32_t* seg_offsets, const int32_t* seg_adapter_ids, int n_seg, const void* W,
                         size_t w_bytes, const void* const* A, const void* const* B, const float* scale,
                         int n_adapters, const void* y) {
    int rc = check_shape(d_in, d_out, rank, max_tokens, max_segments);
    if (rc != LORA_OK) return rc;
    if (T < 0 || T > max_tokens || n_seg < 0 || n_seg > max_segments || n_adapters < 0)
        return LORA_EINVAL;
    if (T == 0) {
        if (n_seg == 0) return LORA_OK;
        if (!seg_offsets || !seg_adapter_ids) return LORA_EINVAL;
        for (int i = 0; i <= n_seg; ++i)
            if (seg_offsets[i] != 0) return LORA_EINVAL;
        for (int i = 0; i < n_seg; ++i)
            if (seg_adapter_ids[i] < 0 || seg_adapter_ids[i] > n_adapters) return LORA_EINVAL;
        return LORA_OK;
    }
    if (n_seg < 1 || !seg_offsets || !seg_adapter_ids) return LORA_EINVAL;
    if (!x || !y || !W || !aligned16(x) || !aligned16(y) || !aligned16(W)) return LORA_EINVAL;
    if (seg_offsets[0] != 0 || seg_offsets[n_seg] != T) return LORA_EINVAL;
    const size_t xb = (size_t)T * d_in * 2, yb = (size_t)T * d_out * 2, wb = w_bytes;
    const size_t ab = (size_t)rank * d_in * 2, bb = (size_t)d_out * rank * 2;
    if (overlaps(y, yb, x, xb) || overlaps(y, yb, W, wb)) return LORA_EINVAL;
    for (int i = 0; i < n_seg; ++i) {
        if (seg_offsets[i + 1] < seg_offsets[i]) return LORA_EINVAL;
        int a = seg_adapter_ids[i];
        if (a < 0 || a > n_adapters) return LORA_EINVAL;
        if (a == 0 || seg_offsets[i + 1] == seg_offsets[i]) continue;
        if (!A || !B || !scale) return LORA_EINVAL;
        const void* pa = A[a - 1];
        const void* pb = B[a - 1];
        if (!pa || !pb || !aligned16(pa) || !aligned16(pb)) return LORA_EINVAL;
        if (!std::isfinite(scale[a - 1])) return LORA_EINVAL;
        if (overlaps(y, yb, pa, ab) || overlaps(y, yb, pb, bb)) return LORA_EINVAL;
    }
    return LORA_OK;
}

extern "C" {

int lora_linear_validate(int d_in, int d_out, int rank, int max_tokens, int max_segments,
                         const void* x, int T, const int32_t* seg_offsets,
                         const int32_t* seg_adapter_ids, int n_seg, const void* W,
                         const void* const* A, const void* const* B, const float* scale,
                         int n_adapters, const void* y) {
    return validate_impl(d_in, d_out, rank, max_tokens, max_segments, x, T, seg_offsets, seg_adapter_ids, n_seg, W,
                         (size_t)d_out * d_in * 2, A, B, scale, n_adapters, y);
}

int lora_linear_create(lora_linear** out, int d_in, int d_out, int rank, int max_tokens,
                       int max_segments, int device) {
    if (!out) return LORA_EINVAL;
    *out = nullptr;
    int rc = check_shape(d_in, d_out, rank, max_tokens, max_segments);
    if (rc != LORA_OK) return rc;
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || device < 0 || device >= count) {
        cudaGetLastError();
        return LORA_ENODEV;
    }
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return LORA_ECUDA;
    if (prop.major != 10 || prop.minor != 3) return LORA_ENODEV;

    DeviceGuard guard(device);
    lora_linear* h = new lora_linear();
    h->device = device;
    h->d_in = d_in;
    h->d_out = d_out;
    h->rank = rank;
    h->max_tokens = max_tokens;
    h->max_segments = max_segments;
    h->num_sms = prop.multiProcessorCount;

    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
        free_handle(h);
        return LORA_ECUDA;
    }
    h->encode = reinterpret_cast<EncodeTiledFn>(fn);
    if (gemm_prepare_device() != cudaSuccess || w4_prepare_device() != cudaSuccess) {
        free_handle(h);
        return LORA_ECUDA;
    }

    h->u_rows = ceil_div(max_tokens, kTileM) * kTileM + kTileM;
    h->max_fused = ceil_div(max_tokens, kTileM) + max_segments + 1;
    h->k_split = choose_k_split(h);
    h->slot_bytes = align_up(2 * (size_t)max_segments * sizeof(CUtensorMap), 128) +
                    4 * (size_t)h->max_fused * sizeof(Tile) +
                    align_up(4 * (2 * (size_t)max_segments + 1), 16) +
                    align_up(4 * (size_t)max_segments, 16) + 256 +
                    // 4-bit base kernel: B_a maps of its own box and the token groups
                    align_up((size_t)max_segments * sizeof(CUtensorMap), 128) +
                    (size_t)(h->max_fused / 2 + 1) * sizeof(W4Group) + 256;
    if (cudaMalloc(&h->u_ws, (size_t)h->u_rows * rank * 2) != cudaSuccess ||
        cudaMalloc((void**)&h->status, sizeof(int)) != cudaSuccess ||
        cudaMalloc((void**)&h->flags, sizeof(int) * ((size_t)h->max_fused + 1)) != cudaSuccess ||
        cudaHostAlloc((void**)&h->status_host, sizeof(int), cudaHostAllocDefault) != cudaSuccess) {
        cudaGetLastError();
        free_handle(h);
        return LORA_ENOMEM;
    }
    for (Slot& s : h->slots) {
        if (cudaHostAlloc((void**)&s.host, h->slot_bytes, cudaHostAllocDefault) != cudaSuccess ||
            cudaMalloc((void**)&s.dev, h->slot_bytes) != cudaSuccess) {
            cudaGetLastError();
            free_handle(h);
            return LORA_ENOMEM;
        }
        if (cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming) != cudaSuccess) {
            free_handle(h);
            return LORA_ECUDA;
        }
    }
    rc = ensure_split_buffers(h);
    if (rc == LORA_OK) {
        h->w4_k_split = choose_w4_k_split(h);
        rc = ensure_w4_split_buffers(h);
    }
    if (rc != LORA_OK) {
        free_handle(h);
        return rc;
    }
    if (cudaMemset(h->status, 0, sizeof(int)) != cudaSuccess ||
        cudaMemset(h->flags, 0, sizeof(int) * ((size_t)h->max_fused + 1)) != cudaSuccess ||
        cudaMemset(h->u_ws, 0, (size_t)h->u_rows * rank * 2) != cudaSuccess) {
        free_handle(h);
        return LORA_ECUDA;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) {
        free_handle(h);
        return LORA_ECUDA;
    }
    *out = h;
    return LORA_OK;
}

int lora_linear_destroy(lora_linear* h) {
    if (!h) return LORA_OK;
    DeviceGuard guard(h->device);
    cudaDeviceSynchronize();
    free_handle(h);
    return LORA_OK;
}

int lora_linear_set_option(lora_linear* h, int option, long long value) {
    if (!h) return LORA_EINVAL;
    switch (option) {
        case LORA_OPT_TILE_N:
            if (value != 0 && (value < 16 || value > kMaxWideTileN || value % 16)) return LORA_EINVAL;
            h->force_tile_n = (int)value;
            return LORA_OK;
        case LORA_OPT_WAIT_LIMIT_US:
            if (value < 1000 || value > 60000000) return LORA_EINVAL;
            h->wait_limit_ns = (unsigned long long)value * 1000ull;
            return LORA_OK;
        case LORA_OPT_DEBUG_STALL:
            h->debug_stall = value ? 1 : 0;
            return LORA_OK;
        case LORA_OPT_DEBUG_PUBLISH_DELAY_US:
            if (value < 0 || value > 1000000) return LORA_EINVAL;
            h->debug_publish_delay_ns = (unsigned long long)value * 1000ull;
            return LORA_OK;
        case LORA_OPT_TIMING: {
            DeviceGuard guard(h->device);
            for (TimingRec& r : h->trec)
                for (cudaEvent_t e : r.ev) h->ev_pool.push_back(e);
            h->trec.clear();
            h->timing = value ? 1 : 0;
            return LORA_OK;
        }
        case LORA_OPT_RASTER:
            if (value < 0 || value > 3) return LORA_EINVAL;
            h->raster = (int)value;
            return LORA_OK;
        case LORA_OPT_RASTER_GROUP:
            if (value < 1 || value > 4096) return LORA_EINVAL;
            h->raster_group = (int)value;
            return LORA_OK;
        case LORA_OPT_MMA_GROUP:
            if (value < 0 || value > 2) return LORA_EINVAL;
            h->mma_group = (int)value;
            return LORA_OK;
        case LORA_OPT_INLINE_WORK_LIST:
            h->allow_inline = value ? 1 : 0;
            return LORA_OK;
        case LORA_OPT_TILE_K:
            if (value != 0 && value != 32 && value != 64) return LORA_EINVAL;
            h->tile_k = (int)value;
            return LORA_OK;
        case LORA_OPT_TWO_LAUNCH:
            h->two_launch = value ? 1 : 0;
            return LORA_OK;
        case LORA_OPT_CLUSTER:
            if (value < 0 || value > 2) return LORA_EINVAL;
            h->cluster = (int)value;
            return LORA_OK;
        case LORA_OPT_PDL:
            if (value < 0 || value > 1) return LORA_EINVAL;
            h->pdl = (int)value;
            return LORA_OK;
        case LORA_OPT_TOKEN_COLUMNS:
            if (value < 0 || value > 2) return LORA_EINVAL;
            h->yt_mode = (int)value;
            return LORA_OK;
        case LORA_OPT_WIDE_TILES:
            if (value < 0 || value > 1) return LORA_EINVAL;
            h->wide_mode = (int)value;
            return LORA_OK;
        case LORA_OPT_W4_K_SPLIT: {
            if (value < 0 || value > 4) return LORA_EINVAL;
            DeviceGuard guard(h->device);
            if (cudaDeviceSynchronize() != cudaSuccess) return LORA_ECUDA;
            const int prev_opt = h->w4_k_split_opt, prev = h->w4_k_split;
            h->w4_k_split_opt = (int)value;
            h->w4_k_split = choose_w4_k_split(h);
            const int rc = ensure_w4_split_buffers(h);
            if (rc != LORA_OK) {
                h->w4_k_split_opt = prev_opt;
                h->w4_k_split = prev;
            }
            return rc;
        }
        case LORA_OPT_MAX_CTAS:
            if (value < 0 || value > (1 << 20) || (value > 0 && value < 2)) return LORA_EINVAL;
            h->max_ctas = (int)value;
            h->shape_cache.clear();
            return LORA_OK;
        case LORA_OPT_K_SPLIT: {
            if (value != 0 && value != 1 && value != 2 && value != 4) return LORA_EINVAL;
            DeviceGuard guard(h->device);
            const int prev_opt = h->k_split_opt, prev = h->k_split;
            h->k_split_opt = (int)value;
            h->k_split = choose_k_split(h);
            const int rc = ensure_split_buffers(h);
            if (rc != LORA_OK) {
                h->k_split_opt = prev_opt;
                h->k_split = prev;
            }
            return rc;
        }
        default:
            return LORA_EINVAL;
    }
}

int lora_linear_timing(lora_linear* h, int kind, double* total_ms, long long* launches,
                       long long* all_launches) {
    if (!h || kind < 0 || kind > 1) return LORA_EINVAL;
    DeviceGuard guard(h->device);
    double sum = 0;
    long long n = 0;
    for (TimingRec& r : h->trec) {
        if (kind == 0 && !r.has_shrink) continue;
        if (cudaEventSynchronize(r.ev[2]) != cudaSuccess) return LORA_ECUDA;
        float ms = 0;
        cudaEvent_t a = kind == 0 ? r.ev[0] : r.ev[1];
        cudaEvent_t b = kind == 0 ? r.ev[1] : r.ev[2];
        if (cudaEventElapsedTime(&ms, a, b) != cudaSuccess) return LORA_ECUDA;
        sum += ms;
        ++n;
    }
    if (total_ms) *total_ms = sum;
    if (launches) *launches = n;
    if (all_launches) *all_launches = h->launches;
    return LORA_OK;
}

int lora_linear_status(lora_linear* h, int reset) {
    if (!h) return LORA_EINVAL;
    DeviceGuard guard(h->device);
    if (cudaDeviceSynchronize() != cudaSuccess) return LORA_ECUDA;
    int v = 0;
    if (cudaMemcpy(&v, h->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return LORA_ECUDA;
    if (reset && cudaMemset(h->status, 0, sizeof(int)) != cudaSuccess) return LORA_ECUDA;
    // a launch that gave up part-way may leave the 4-bit K-part counters between launches' counts
    if (reset && v && h->w4_split_ctr &&
        cudaMemset(h->w4_split_ctr, 0, 2 * h->w4_split_blocks * sizeof(unsigned long long)) != cudaSuccess)
        return LORA_ECUDA;
    if (reset && cudaDeviceSynchronize() != cudaSuccess) return LORA_ECUDA;
    return v ? LORA_ETIMEOUT : LORA_OK;
}

int lora_linear_describe(lora_linear* h, int T, const int32_t* seg_offsets,
                         const int32_t* seg_adapter_ids, int n_seg, int* tile_n, int* n_tiles,
                         int* n_units, int* grid, int* stages, int* has_shrink, int* unit_order) {
    if (!h) return LORA_EINVAL;
    Plan plan;
    int rc = plan_segments(seg_offsets, seg_adapter_ids, n_seg, T, -1, &plan);
    if (rc != LORA_OK) return rc;
    const int nf = (int)plan.fused.size();
    int units = 0, tn = 0, st = 0, g = 0, order = 0;
    if (nf) {
        Shape sh = choose_shape(h, plan);
        order = sh.yt ? 3 : sh.m_fastest;
        units = (fused_row_groups(sh) * sh.n_ntiles + (int)(sh.shrink_groups.size() / sh.cs)) * h->k_split;
        tn = sh.tile_n;
        st = sh.stages;
        int slots = usable_sms(h);
        if (sh.cs > 1) {
            GemmParams q;
            memset(&q, 0, sizeof(q));
            q.tile_n = sh.tile_n;
            q.shrink_n = sh.shrink_n;
            q.stages = sh.stages;
            q.cluster_size = sh.cs;
            q.bk = sh.bk;
            q.yt = sh.yt;
            q.yt_rows = sh.yt_rows;
            q.yt_h = sh.yt_h;
            DeviceGuard guard(h->device);
            slots = std::min(max_clusters(h, q), usable_sms(h) / sh.cs);
        }
        g = std::min(units, slots) * sh.cs;
    }
    if (tile_n) *tile_n = tn;
    if (n_tiles) *n_tiles = nf;
    if (n_units) *n_units = units;
    if (grid) *grid = g;
    if (stages) *stages = st;
    if (has_shrink) *has_shrink = plan.shrink.empty() ? 0 : 1;
    if (unit_order) *unit_order = order;
    return LORA_OK;
}

}  // extern "C"

namespace {
// The projection on `stream`. The call's work list is uploaded on `upload`: the same stream,
// or (host-buffer path) a copy stream that then also copies the call's X rows from `x_src`
// and records `ready`, on which `stream` waits before the launch. Keeping the small work-list
// copy on the copy stream, ahead of the X rows, stops it from queueing behind the next
// chunk's X copy.
int forward_impl(lora_linear* h, const void* x, int T, const int32_t* seg_offsets,
                 const int32_t* seg_adapter_ids, int n_seg, const void* W, const void* const* A,
                 const void* const* B, const float* scale, int n_adapters, void* y, cudaStream_t stream,
                 cudaStream_t upload, const void* x_src, cudaEvent_t ready, const void* Wq = nullptr,
                 const void* Ws = nullptr) {
    if (!h) return LORA_EINVAL;
    int rc = validate_impl(h->d_in, h->d_out, h->rank, h->max_tokens, h->max_segments, x, T, seg_offsets,
                           seg_adapter_ids, n_seg, Wq ? Wq : W,
                           Wq ? (size_t)h->d_out * h->d_in / 2 : (size_t)h->d_out * h->d_in * 2, A, B, scale,
                           n_adapters, y);
    if (rc != LORA_OK) return rc;
    if (T == 0) return LORA_OK;
    Plan plan;
    rc = plan_segments(seg_offsets, seg_adapter_ids, n_seg, T, n_adapters, &plan);
    if (rc != LORA_OK) return rc;
    if ((int)plan.fused.size() > h->max_fused) return LORA_EINVAL;

    // caller's adapter index -> compact slot (1-based) for the device work list
    const int n_used = (int)plan.used_adapters.size();
    std::vector<int> compact(n_adapters + 1, 0);
    for (int k = 0; k < n_used; ++k) compact[plan.used_adapters[k] + 1] = k + 1;
    for (Tile& t : plan.fused) t.adapter = compact[t.adapter];
    for (Tile& t : plan.shrink) t.adapter = compact[t.adapter];
    for (int32_t& a : plan.seg_id) a = compact[a];

    for (size_t i = 0; i < plan.fused.size(); ++i) plan.fused[i].fused_index = plan.fused[i].split_index = (int32_t)i;

    DeviceGuard guard(h->device);
    const bool w4 = Wq != nullptr;
    Shape sh = choose_shape(h, plan, !w4);
    // 4-bit base: the shrink pass runs on the bf16 kernel (64-wide K-steps), then the 4-bit
    // kernel runs the base and expand passes over token groups
    int shrink_rank_tiles = 1;
    if (w4) {
        // the 4-bit kernel reads X and U through the same maps with 128-row boxes
        sh.bk = 64;
        sh.a_rows = kTileM;
        // its shrink is a launch of its own: spread over rank tiles (multiples of 32 columns) so
        // that a few shrink groups still find most SMs (48 + 300 rows: 3 groups x 4 tiles of 64);
        // each U column is the same whole-K sum
        const int groups = (int)(sh.shrink_groups.size() / sh.cs);
        if (groups > 0 && h->k_split <= 1) {
            const int room = std::max(1, usable_sms(h) / sh.cs / groups);
            const int width = std::max(32, ceil_div(ceil_div(h->rank, std::min(room, 8)), 32) * 32);
            if (width < sh.shrink_n) {
                shrink_rank_tiles = ceil_div(h->rank, width);
                sh.shrink_n = width;
            }
        }
        sh.stages = stages_for(std::max(sh.tile_n, sh.shrink_n) / sh.cs, sh.bk);
    }
    const std::vector<W4Group> w4_groups =
        w4 ? make_w4_groups(plan.fused, h->w4_k_split <= 1) : std::vector<W4Group>();
    const int n_w4g = (int)w4_groups.size();
    const W4Shape w4s = w4 ? w4_shape(h, w4_groups, T) : W4Shape();
    const bool w4_inline = n_used <= kInlineAdapters && n_w4g <= kW4InlineGroups;
    const int cs = sh.cs, tile_n = sh.tile_n, shrink_n = sh.shrink_n, bk = sh.bk;
    // token-column units: one row group spanning every token row
    const int nfg = sh.yt ? 1 : (int)sh.fused_groups.size() / cs, nsg = (int)sh.shrink_groups.size() / cs;
    const int nft = (int)sh.fused_groups.size(), nst = (int)sh.shrink_groups.size();
    const int n_m = (int)plan.seg_id.size();
    const int nf = (int)plan.fused.size();

    GemmParams p;
    memset(&p, 0, sizeof(p));
    W4Params q;
    memset(&q, 0, sizeof(q));
    const bool inline_wl = h->allow_inline && nft + nst <= kInlineTiles && n_m <= kInlineSegs &&
                           n_used <= kInlineAdapters && (!w4 || w4_inline);
    // Under stream capture only calls whose whole work list travels in the kernel parameters
    // are recorded: an uploaded list would be read from a ring slot that later calls reuse.
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &capture) != cudaSuccess) return LORA_ECUDA;
    const bool capturing = capture != cudaStreamCaptureStatusNone;
    if (capturing && (!inline_wl || x_src)) return LORA_EUNSUPPORTED;
    const bool timing = h->timing && !capturing;   // timing events are read back eagerly
    Slot* slot = nullptr;
    if (inline_wl) {
        // small work list: it travels in the kernel parameters, no upload
        for (int k = 0; k < n_used; ++k) {
            int a = plan.used_adapters[k];
            if (encode_2d(h, &p.inline_maps[k], B[a], h->rank, h->d_out, bk, tile_n / cs) != CUDA_SUCCESS)
                return LORA_ECUDA;
            if (encode_2d(h, &p.inline_maps[kInlineAdapters + k], A[a], h->d_in, h->rank, bk, shrink_n / cs) !=
                CUDA_SUCCESS)
                return LORA_ECUDA;
            p.inline_scales[k] = scale[a];
        }
        memcpy(p.inline_tiles, sh.fused_groups.data(), (size_t)nft * sizeof(Tile));
        memcpy(p.inline_tiles + nft, sh.shrink_groups.data(), (size_t)nst * sizeof(Tile));
        memcpy(p.inline_seg, plan.seg_off.data(), 4 * (size_t)(n_m + 1));
        memcpy(p.inline_seg + n_m + 1, plan.seg_id.data(), 4 * (size_t)n_m);
        p.inline_wl = 1;
        p.inline_shrink_off = nft;
        if (w4) {
            for (int k = 0; k < n_used; ++k)
                if (encode_2d(h, &q.inline_bmaps[k], B[plan.used_adapters[k]], h->rank, h->d_out, 64, kW4TileM) !=
                    CUDA_SUCCESS)
                    return LORA_ECUDA;
            memcpy(q.inline_groups, w4_groups.data(), (size_t)n_w4g * sizeof(W4Group));
            q.inline_wl = 1;
        }
        if (x_src &&
            cudaMemcpyAsync(const_cast<void*>(x), x_src, (size_t)T * h->d_in * 2, cudaMemcpyHostToDevice, upload) !=
                cudaSuccess)
            return LORA_ECUDA;
        if (upload != stream &&
            (cudaEventRecord(ready, upload) != cudaSuccess || cudaStreamWaitEvent(stream, ready, 0) != cudaSuccess))
            return LORA_ECUDA;
    } else {
        slot = acquire_slot(h);
        if (!slot) return LORA_ECUDA;
        // work list: [B_a maps][A_a maps][fused groups][shrink groups][seg_off][seg_id][scales]
        size_t off_bmaps = 0;
        size_t off_amaps = off_bmaps + (size_t)n_used * sizeof(CUtensorMap);
        size_t off_fused = align_up(off_amaps + (size_t)n_used * sizeof(CUtensorMap), 128);
        size_t off_shrink = off_fused + (size_t)nft * sizeof(Tile);
        size_t off_segoff = align_up(off_shrink + (size_t)nst * sizeof(Tile), 16);
        size_t off_segid = off_segoff + 4 * (size_t)(n_m + 1);
        size_t off_scale = align_up(off_segid + 4 * (size_t)n_m, 16);
        size_t used_bytes = off_scale + 4 * (size_t)n_used;
        // 4-bit base kernel: its B_a maps and token groups follow
        const size_t off_w4maps = align_up(used_bytes, 128);
        const size_t off_w4groups = off_w4maps + (size_t)n_used * sizeof(CUtensorMap);
        if (w4) used_bytes = off_w4groups + (size_t)n_w4g * sizeof(W4Group);
        if (used_bytes > h->slot_bytes) return LORA_EINVAL;

        uint8_t* hb = slot->host;
        CUtensorMap* bmaps = reinterpret_cast<CUtensorMap*>(hb + off_bmaps);
        CUtensorMap* amaps = reinterpret_cast<CUtensorMap*>(hb + off_amaps);
        for (int k = 0; k < n_used; ++k) {
            int a = plan.used_adapters[k];
            if (encode_2d(h, &bmaps[k], B[a], h->rank, h->d_out, bk, tile_n / cs) != CUDA_SUCCESS) return LORA_ECUDA;
            if (encode_2d(h, &amaps[k], A[a], h->d_in, h->rank, bk, shrink_n / cs) != CUDA_SUCCESS) return LORA_ECUDA;
        }
        memcpy(hb + off_fused, sh.fused_groups.data(), (size_t)nft * sizeof(Tile));
        memcpy(hb + off_shrink, sh.shrink_groups.data(), (size_t)nst * sizeof(Tile));
        memcpy(hb + off_segoff, plan.seg_off.data(), 4 * (size_t)(n_m + 1));
        memcpy(hb + off_segid, plan.seg_id.data(), 4 * (size_t)n_m);
        float* sc = reinterpret_cast<float*>(hb + off_scale);
        for (int k = 0; k < n_used; ++k) sc[k] = scale[plan.used_adapters[k]];
        if (w4) {
            CUtensorMap* w4maps = reinterpret_cast<CUtensorMap*>(hb + off_w4maps);
            for (int k = 0; k < n_used; ++k)
                if (encode_2d(h, &w4maps[k], B[plan.used_adapters[k]], h->rank, h->d_out, 64, kW4TileM) !=
                    CUDA_SUCCESS)
                    return LORA_ECUDA;
            memcpy(hb + off_w4groups, w4_groups.data(), (size_t)n_w4g * sizeof(W4Group));
            q.tm_b = reinterpret_cast<const CUtensorMap*>(slot->dev + off_w4maps);
            q.groups = reinterpret_cast<const W4Group*>(slot->dev + off_w4groups);
        }
        if (cudaMemcpyAsync(slot->dev, hb, used_bytes, cudaMemcpyHostToDevice, upload) != cudaSuccess)
            return LORA_ECUDA;
        if (x_src &&
            cudaMemcpyAsync(const_cast<void*>(x), x_src, (size_t)T * h->d_in * 2, cudaMemcpyHostToDevice, upload) !=
                cudaSuccess)
            return LORA_ECUDA;
        if (upload != stream &&
            (cudaEventRecord(ready, upload) != cudaSuccess || cudaStreamWaitEvent(stream, ready, 0) != cudaSuccess))
            return LORA_ECUDA;

        p.tm_b = reinterpret_cast<const CUtensorMap*>(slot->dev + off_bmaps);
        p.tm_a = reinterpret_cast<const CUtensorMap*>(slot->dev + off_amaps);
        p.shrink_tiles = reinterpret_cast<const Tile*>(slot->dev + off_shrink);
        p.fused_tiles = reinterpret_cast<const Tile*>(slot->dev + off_fused);
        p.seg_off = reinterpret_cast<const int32_t*>(slot->dev + off_segoff);
        p.seg_id = reinterpret_cast<const int32_t*>(slot->dev + off_segid);
        p.scales = reinterpret_cast<const float*>(slot->dev + off_scale);
    }
    if (encode_2d(h, &p.tm_x, x, h->d_in, T, bk, (uint32_t)sh.a_rows) != CUDA_SUCCESS) return LORA_ECUDA;
    if (w4) {
        q.tm_x = p.tm_x;
        q.feature_tiles = w4s.feature_tiles;
        q.tail_rows = w4s.tail_rows;
        if (w4s.tail_rows &&
            encode_2d(h, &q.tm_x3, x, h->d_in, T, 64, (uint32_t)w4s.tail_rows) != CUDA_SUCCESS)
            return LORA_ECUDA;
        const uint32_t q_box = (uint32_t)(kW4TileM * q.feature_tiles);
        if (encode_u8_sw128(h, &q.tm_wq, Wq, (uint64_t)h->d_in / 2, h->d_out, q_box) != CUDA_SUCCESS ||
            encode_plain_2d(h, &q.tm_ws, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Ws, h->d_out,
                            (uint64_t)h->d_in / kW4Group, q_box, 2) != CUDA_SUCCESS)
            return LORA_ECUDA;
    } else if (encode_2d(h, &p.tm_w, W, h->d_in, h->d_out, bk, tile_n / cs) != CUDA_SUCCESS) {
        return LORA_ECUDA;
    }
    // the expand reads U as the A operand (a_rows-row boxes), or as the B operand of token-column
    // units (yt_rows-row boxes)
    if (encode_2d(h, &p.tm_u, h->u_ws, h->rank, h->u_rows, bk, (uint32_t)(sh.yt ? sh.yt_rows : sh.a_rows)) !=
        CUDA_SUCCESS)
        return LORA_ECUDA;
    if (sh.yt) {
        if (encode_2d(h, &p.tm_xt, x, h->d_in, T, bk, (uint32_t)sh.yt_rows) != CUDA_SUCCESS) return LORA_ECUDA;
        p.yt = 1;
        p.yt_tokens = T;
        p.yt_rows = sh.yt_rows;
        p.yt_h = sh.yt_h;
        p.yt_adapter = plan.fused[0].adapter;
    }
    p.y = y;
    p.u = h->u_ws;
    p.status = h->status;
    p.wait_limit_ns = h->wait_limit_ns;
    p.n_seg = n_m;
    p.n_shrink = nsg;
    p.n_fused = nfg;
    p.n_ntiles = sh.n_ntiles;
    p.tile_n = tile_n;
    p.shrink_n = shrink_n;
    p.stages = sh.stages;
    p.m_fastest = sh.m_fastest;
    p.raster_group = sh.raster_group;
    p.k_main_blocks = ceil_div(h->d_in, bk);
    p.k_lora_blocks = ceil_div(h->rank, bk);
    p.bk = bk;
    // the MMA warp takes two stages per wait on SM pairs and on batches of one tile (decode
    // steps: 48-row batches of qkv, o and down measured 7-8% faster); one elsewhere
    p.mma_group = h->mma_group ? h->mma_group : ((cs > 1 || nf == 1) ? 2 : 1);
    p.a_rows = sh.a_rows;
    p.d_out = h->d_out;
    p.rank = h->rank;
    p.cluster_size = cs;
    p.debug_stall = h->debug_stall;
    p.debug_publish_delay_ns = h->debug_publish_delay_ns;
    // K halves (bf16 base): every fused output block runs as two units; the split point is set
    // in 64-wide K-steps, so that it does not move with the K-step width of the stages
    // K parts (bf16 base): every block runs as k_split units; the part boundaries are set in
    // 64-wide K-steps, so that they do not move with the K-step width of the stages
    const int k_split = (!w4 && h->k_split > 1) ? h->k_split : 1;
    if (k_split > 1) {
        if (!h->partials || h->partial_parts < k_split || (size_t)nf * sh.n_ntiles + nst > h->split_slots ||
            T > h->max_tokens)
            return LORA_ENOMEM;
        p.k_split = k_split;
        p.k_chunk = ceil_div(ceil_div(h->d_in, 64), k_split) * 64 / bk;
        if (p.k_chunk < 1 || (k_split - 1) * p.k_chunk >= p.k_main_blocks) return LORA_EINVAL;
        p.partials = h->partials;
        p.part_rows = h->max_tokens;
        p.part_chunks = ceil_div(h->d_out, 4) + ceil_div(h->rank, 4);
        p.split_ctr = h->split_ctr;
        p.shrink_slot0 = nf * sh.n_ntiles;
        p.n_split_slots = nf * sh.n_ntiles + nst;
        p.u_chunk0 = ceil_div(h->d_out, 4);
        p.done_count = h->flags + h->max_fused;
    }
    const int slots = cs > 1 ? std::min(max_clusters(h, p), usable_sms(h) / cs) : usable_sms(h);
    if (slots < 1) return LORA_ECUDA;
    // every tile the kernel will decode names a valid adapter slot and flag slot: the kernel
    // indexes tensor maps and flags with them, so a malformed list must never reach it
    for (const Tile& t : sh.fused_groups)
        if (t.adapter < 0 || t.adapter > n_used || t.fused_index < 0 || t.fused_index >= nf ||
            t.split_index < 0 || t.split_index >= nf ||
            t.row0 < 0 || t.nrows < 0 || t.row0 + t.nrows > T ||
            (t.adapter && t.u_row != t.row0 && t.u_row != h->u_rows - kTileM))
            return LORA_EINVAL;
    for (const Tile& t : sh.shrink_groups)
        if (t.adapter < 1 || t.adapter > n_used || t.fused_index < -1 || t.fused_index >= nf || t.row0 < 0 ||
            t.nrows < 0 || t.row0 + t.nrows > T)
            return LORA_EINVAL;

    TimingRec rec{};
    if (timing) {
        for (int i = 0; i < 3; ++i) {
            rec.ev[i] = take_event(h);
            if (!rec.ev[i]) return LORA_ECUDA;
        }
        cudaEventRecord(rec.ev[0], stream);
    }
    const int fused_units = nfg * sh.n_ntiles * k_split;
    const int shrink_units = nsg * k_split;
    if (w4) {
        // shrink (bf16 kernel), then base + expand on the 4-bit kernel, ordered by the stream
        if (nsg > 0) {
            GemmParams sp = p;
            sp.n_fused = 0;
            sp.shrink_ntiles = shrink_rank_tiles;
            if (launch_gemm(sp, std::min(nsg * shrink_rank_tiles, slots) * cs, stream) != cudaSuccess) return LORA_ECUDA;
            ++h->launches;
            rec.has_shrink = true;
        }
        if (timing) cudaEventRecord(rec.ev[1], stream);
        for (const W4Group& g : w4_groups)
            for (int k = 0; k < 3; ++k)
                if (g.adapter[k] < 0 || g.adapter[k] > n_used || g.nrows[k] < 0 || g.row0[k] < 0 ||
                    g.row0[k] + g.nrows[k] > T || g.nrows[k] > kTileM || (k == 0 && g.nrows[0] == 0) ||
                    (k == 2 && g.nrows[2] > 0 && (g.nrows[1] == 0 || g.nrows[2] > w4s.tail_rows)))
                    return LORA_EINVAL;
        q.tm_u = p.tm_u;
        q.y = y;
        q.status = h->status;
        q.wait_limit_ns = h->wait_limit_ns;
        q.n_groups = n_w4g;
        q.n_ntiles = w4s.n_ntiles;
        q.tokens_fastest = w4s.tokens_fastest;
        q.k_main_blocks = ceil_div(h->d_in, 64);
        q.k_lora_blocks = ceil_div(h->rank, 64);
        q.k_pack_blocks = ceil_div(q.k_main_blocks, 4);
        q.d_out = h->d_out;
        q.x_stage_bytes = w4s.x_stage_bytes;
        if (h->w4_k_split > 1) {
            if (!h->w4_partials || h->w4_partial_parts < h->w4_k_split || !h->w4_split_ctr ||
                (size_t)n_w4g * w4s.n_ntiles > h->w4_split_blocks || T > h->max_tokens)
                return LORA_ENOMEM;
            q.k_split = h->w4_k_split;
            q.k_chunk = ceil_div(ceil_div(ceil_div(h->d_in, 64), h->w4_k_split), 4) * 4;
            q.partials = h->w4_partials;
            q.part_rows = h->max_tokens;
            q.split_ctr = h->w4_split_ctr;
        }
        q.stages = w4s.stages;
        q.pstages = w4s.pstages;
        // whole 32-row chunks of Y leave through TMA stores (Y 16-byte aligned, d_out % 8 == 0:
        // both checked before any launch)
        if (encode_plain_2d(h, &q.tm_y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, y, h->d_out, T, kW4TileM, 32) !=
            CUDA_SUCCESS)
            return LORA_ECUDA;
        q.debug_stall = h->debug_stall;
        const int units = q.n_groups * q.n_ntiles * (q.k_split > 1 ? q.k_split : 1);
        if (launch_w4(q, std::min(units, usable_sms(h)), stream) != cudaSuccess) return LORA_ECUDA;
        ++h->launches;
    } else if (h->two_launch && nsg > 0) {
        // shrink, then fused base+expand ordered by the stream
        GemmParams s = p;
        s.n_fused = 0;
        if (launch_gemm(s, std::min(shrink_units, slots) * cs, stream) != cudaSuccess) return LORA_ECUDA;
        ++h->launches;
        rec.has_shrink = true;
        if (timing) cudaEventRecord(rec.ev[1], stream);
        GemmParams f = p;
        f.n_shrink = 0;
        if (launch_gemm(f, std::min(fused_units, slots) * cs, stream) != cudaSuccess) return LORA_ECUDA;
        ++h->launches;
    } else {
        // one launch: shrink units first, fused units wait on the per-tile ready flags
        if (timing) cudaEventRecord(rec.ev[1], stream);
        if (nsg > 0) {
            p.flags = h->flags;
            p.done_count = h->flags + h->max_fused;
            p.n_flags = nf;
        }
        // a launch with ready flags is cooperative and starts on its own; others may start early
        p.pdl = (h->pdl && !p.flags) ? 1 : 0;
        if (launch_gemm(p, std::min(shrink_units + fused_units, slots) * cs, stream) != cudaSuccess) return LORA_ECUDA;
        ++h->launches;
    }
    if (timing) {
        cudaEventRecord(rec.ev[2], stream);
        h->trec.push_back(rec);
    }
    if (slot) {
        if (cudaEventRecord(slot->done, stream) != cudaSuccess) return LORA_ECUDA;
        slot->pending = true;
    }
    return LORA_OK;
}
}  // namespace

extern "C" {

int lora_linear_forward(lora_linear* h, const void* x, int T, const int32_t* seg_offsets,
                        const int32_t* seg_adapter_ids, int n_seg, const void* W,
                        const void* const* A, const void* const* B, const float* scale,
                        int n_adapters, void* y, void* stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    return forward_impl(h, x, T, seg_offsets, seg_adapter_ids, n_seg, W, A, B, scale, n_adapters, y, stream,
                        stream, nullptr, nullptr);
}

int lora_linear_w4_repack(const void* src, void* dst, long long n_bytes, void* stream) {
    if (n_bytes < 0 || (n_bytes % 4) != 0) return LORA_EINVAL;
    if (n_bytes == 0) return LORA_OK;
    if (!src || !dst || (reinterpret_cast<uintptr_t>(src) & 3) || (reinterpret_cast<uintptr_t>(dst) & 3))
        return LORA_EINVAL;
    // partial overlap would let one thread read a word another has already rewritten
    if (src != dst && overlaps(dst, (size_t)n_bytes, src, (size_t)n_bytes)) return LORA_EINVAL;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return LORA_ECUDA;
    const long long n_words = n_bytes / 4;
    const long long want = (n_words + 255) / 256;
    const int grid = (int)std::min<long long>(want, (long long)sms * 8);
    return w4_repack(src, dst, n_words, grid, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? LORA_OK
                                                                                                   : LORA_ECUDA;
}

int lora_linear_forward_w4(lora_linear* h, const void* x, int T, const int32_t* seg_offsets,
                           const int32_t* seg_adapter_ids, int n_seg, const void* Wq, const void* Ws,
                           const void* const* A, const void* const* B, const float* scale, int n_adapters,
                           void* y, void* stream_) {
    if (!h) return LORA_EINVAL;
    if (h->d_in % kW4Group) return LORA_EINVAL;
    if (T > 0) {
        if (!Wq || !Ws || !aligned16(Wq) || !aligned16(Ws)) return LORA_EINVAL;
        const size_t yb = (size_t)T * h->d_out * 2;
        if (overlaps(y, yb, Wq, (size_t)h->d_out * h->d_in / 2) ||
            overlaps(y, yb, Ws, (size_t)(h->d_in / kW4Group) * h->d_out * 2))
            return LORA_EINVAL;
    }
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    return forward_impl(h, x, T, seg_offsets, seg_adapter_ids, n_seg, nullptr, A, B, scale, n_adapters, y, stream,
                        stream, nullptr, nullptr, Wq, Ws);
}

}  // extern "C"

// Row boundaries of the host-buffer path's chunks: {0, T} below 2,048 rows; else chunks of up to
// max(1024, T / 8) rows (multiples of 128) between ramps that halve down to max(256, T / 32) rows
// at both ends.
static std::vector<int> host_chunk_bounds(int T) {
    std::vector<int> b(1, 0);
    if (T < 2048) {
        b.push_back(T);
        return b;
    }
    // chunk sizes in whole 128-row tiles: a ramp of small chunks (small, 2 small, ... up to half
    // the middle chunks' size, at most four), the middle split evenly, the ramp mirrored; only
    // the last chunk takes the rows past the last whole tile
    const int tiles = T / kTileM;
    const int big = std::max(8, tiles / 8), small = std::max(2, tiles / 32);
    std::vector<int> ramp;
    for (int v = small; v <= big / 2 && (int)ramp.size() < 4; v *= 2) ramp.push_back(v);
    int ramp_tiles = 0;
    for (int v : ramp) ramp_tiles += 2 * v;
    if (ramp_tiles >= tiles) {
        ramp.clear();
        ramp_tiles = 0;
    }
    const int mid = tiles - ramp_tiles, n_mid = std::max(1, ceil_div(mid, big));
    std::vector<int> sizes(ramp);
    for (int i = 0; i < n_mid; ++i) sizes.push_back(mid / n_mid + (i < mid % n_mid ? 1 : 0));
    for (int i = (int)ramp.size() - 1; i >= 0; --i) sizes.push_back(ramp[i]);
    for (int v : sizes) b.push_back(b.back() + v * kTileM);
    b.back() = T;
    return b;
}

static int forward_host_impl(lora_linear* h, const void* x_host, int T, const int32_t* seg_offsets,
                             const int32_t* seg_adapter_ids, int n_seg, const void* W, const void* Wq,
                             const void* Ws, const void* const* A, const void* const* B, const float* scale,
                             int n_adapters, void* y_host, void* stream_) {
    if (!h) return LORA_EINVAL;
    if (T < 0 || T > h->max_tokens) return LORA_EINVAL;
    if (T > 0 && (!x_host || !y_host)) return LORA_EINVAL;
    // the call's segments are checked once, up front (the chunks only re-slice them); each
    // chunk's device-side arguments are checked by lora_linear_forward
    if (n_seg > h->max_segments) return LORA_EINVAL;
    {
        Plan whole;
        int prc = plan_segments(seg_offsets, seg_adapter_ids, n_seg, T, n_adapters, &whole);
        if (prc != LORA_OK) return prc;
    }
    int rc = LORA_OK;
    DeviceGuard guard(h->device);
    if (!h->x_stage) {
        if (cudaMalloc(&h->x_stage, (size_t)h->max_tokens * h->d_in * 2) != cudaSuccess ||
            cudaMalloc(&h->y_stage, (size_t)h->max_tokens * h->d_out * 2) != cudaSuccess) {
            cudaGetLastError();
            if (h->x_stage) cudaFree(h->x_stage);
            h->x_stage = nullptr;
            h->y_stage = nullptr;
            return LORA_ENOMEM;
        }
    }
    if (!h->s_in) {
        if (cudaStreamCreateWithFlags(&h->s_in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&h->s_out, cudaStreamNonBlocking) != cudaSuccess)
            return LORA_ECUDA;
        for (int i = 0; i < 16; ++i)
            if (cudaEventCreateWithFlags(&h->ev_in[i], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&h->ev_done[i], cudaEventDisableTiming) != cudaSuccess)
                return LORA_ECUDA;
    }
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    // Row chunks: copy-in of chunk c+1 and copy-out of chunk c-1 overlap the kernel of chunk c
    // (rows are independent, so each chunk is a call of its own on its rows). The host link is
    // the bound, and only the first chunk's copy-in and the last chunk's kernel and copy-out
    // overlap nothing, so the chunks ramp up from and back down to small ones.
    std::vector<int> bounds = host_chunk_bounds(T);
    const uint8_t* xh = static_cast<const uint8_t*>(x_host);
    uint8_t* yh = static_cast<uint8_t*>(y_host);
    uint8_t* xd = static_cast<uint8_t*>(h->x_stage);
    uint8_t* yd = static_cast<uint8_t*>(h->y_stage);
    const size_t xrow = (size_t)h->d_in * 2, yrow = (size_t)h->d_out * 2;
    std::vector<int32_t> off, ids;
    // one chunk: nothing to overlap, so copy-in, kernel and copy-out stay on the caller's stream
    // (no cross-stream events on the path of a short call)
    const bool single = bounds.size() == 2;
    cudaStream_t s_in = single ? stream : h->s_in, s_out = single ? stream : h->s_out;
    // an error after the first chunk was issued waits for the copies already queued, so that
    // none of them touches the caller's host buffers after this call has returned
    const auto fail = [&](int code) {
        cudaStreamSynchronize(stream);
        if (!single) {
            cudaStreamSynchronize(s_in);
            cudaStreamSynchronize(s_out);
        }
        cudaGetLastError();
        return code;
    };
    for (int c = 0; c + 1 < (int)bounds.size(); ++c) {
        const int a = bounds[c], b = bounds[c + 1];
        const int n = b - a;
        // the segments restricted to rows [a, b), offsets made relative to a
        off.assign(1, 0);
        ids.clear();
        for (int i = 0; i < n_seg; ++i) {
            int lo = std::max(seg_offsets[i], a), hi = std::min(seg_offsets[i + 1], b);
            if (hi <= lo) continue;
            off.push_back(hi - a);
            ids.push_back(seg_adapter_ids[i]);
        }
        if (ids.empty() && n > 0) return fail(LORA_EINVAL);
        const int e = c % 16;
        // work list (on s_in, planned and uploaded by forward_impl), then X rows, both
        // ordered before the event the kernel waits on
        rc = forward_impl(h, xd + (size_t)a * xrow, n, off.data(), ids.data(), (int)ids.size(), W, A, B, scale,
                          n_adapters, yd + (size_t)a * yrow, stream, s_in, xh + (size_t)a * xrow, h->ev_in[e],
                          Wq, Ws);
        if (rc != LORA_OK) return fail(rc);
        if (n > 0) {
            if (!single && (cudaEventRecord(h->ev_done[e], stream) != cudaSuccess ||
                            cudaStreamWaitEvent(s_out, h->ev_done[e], 0) != cudaSuccess))
                return fail(LORA_ECUDA);
            if (cudaMemcpyAsync(yh + (size_t)a * yrow, yd + (size_t)a * yrow, (size_t)n * yrow, cudaMemcpyDeviceToHost,
                                s_out) != cudaSuccess)
                return fail(LORA_ECUDA);
        }
    }
    // the status word travels back with the last rows of Y (on the copy-out stream, after the
    // last kernel), so the call ends with waits only and no further round trip
    if (!single && (cudaEventRecord(h->ev_done[15], stream) != cudaSuccess ||
                    cudaStreamWaitEvent(s_out, h->ev_done[15], 0) != cudaSuccess))
        return fail(LORA_ECUDA);
    if (cudaMemcpyAsync(h->status_host, h->status, sizeof(int), cudaMemcpyDeviceToHost, s_out) != cudaSuccess)
        return fail(LORA_ECUDA);
    if (cudaStreamSynchronize(stream) != cudaSuccess || (!single && cudaStreamSynchronize(s_out) != cudaSuccess))
        return LORA_ECUDA;
    return *h->status_host ? LORA_ETIMEOUT : LORA_OK;
}


extern "C" {

int lora_linear_forward_host(lora_linear* h, const void* x_host, int T, const int32_t* seg_offsets,
                             const int32_t* seg_adapter_ids, int n_seg, const void* W,
                             const void* const* A, const void* const* B, const float* scale,
                             int n_adapters, void* y_host, void* stream) {
    return forward_host_impl(h, x_host, T, seg_offsets, seg_adapter_ids, n_seg, W, nullptr, nullptr, A, B, scale,
                             n_adapters, y_host, stream);
}

int lora_linear_forward_host_w4(lora_linear* h, const void* x_host, int T, const int32_t* seg_offsets,
                                const int32_t* seg_adapter_ids, int n_seg, const void* Wq, const void* Ws,
                                const void* const* A, const void* const* B, const float* scale, int n_adapters,
                                void* y_host, void* stream) {
    if (!h) return LORA_EINVAL;
    if (h->d_in % kW4Group) return LORA_EINVAL;
    if (T > 0 && (!Wq || !Ws || !aligned16(Wq) || !aligned16(Ws))) return LORA_EINVAL;
    return forward_host_impl(h, x_host, T, seg_offsets, seg_adapter_ids, n_seg, nullptr, Wq, Ws, A, B, scale,
                             n_adapters, y_host, stream);
}

}  // extern "C"

extern "C" {

int lora_linear_shape(int d_in, int d_out, int rank, int num_sms, int T, const int32_t* seg_offsets,
                      const int32_t* seg_adapter_ids, int n_seg, int w4, int* cluster, int* tile_n, int* bk,
                      int* stages, int* unit_order, int* fused_units, int* shrink_units) {
    int* outs[] = {cluster, tile_n, bk, stages, unit_order, fused_units, shrink_units};
    for (int* o : outs)
        if (o) *o = 0;
    if (num_sms < 2 || T < 0 || (w4 && d_in % kW4Group)) return LORA_EINVAL;
    int rc = check_shape(d_in, d_out, rank, std::max(T, 1), std::max(n_seg, 1));
    if (rc != LORA_OK) return rc;
    Plan plan;
    rc = plan_segments(seg_offsets, seg_adapter_ids, n_seg, T, -1, &plan);
    if (rc != LORA_OK || plan.fused.empty()) return rc;
    // a handle on the host alone: the shape model reads only its sizes and options
    lora_linear h;
    h.d_in = d_in;
    h.d_out = d_out;
    h.rank = rank;
    h.max_tokens = std::max(T, 1);
    h.num_sms = num_sms;
    h.u_rows = ceil_div(h.max_tokens, kTileM) * kTileM + kTileM;
    if (!w4) h.k_split = choose_k_split(&h);   // a handle of max_tokens = T
    else h.w4_k_split = choose_w4_k_split(&h);
    for (size_t i = 0; i < plan.fused.size(); ++i) plan.fused[i].fused_index = plan.fused[i].split_index = (int32_t)i;
    const Shape sh = choose_shape(&h, plan, !w4);
    if (w4) {
        // the 4-bit kernel over token groups; the shrink runs as the bf16 kernel's shrink units
        const std::vector<W4Group> groups = make_w4_groups(plan.fused, h.w4_k_split <= 1);
        const W4Shape ws = w4_shape(&h, groups, T);
        if (cluster) *cluster = 1;
        if (tile_n) *tile_n = kW4TileM * ws.feature_tiles;
        if (bk) *bk = 64;
        if (stages) *stages = ws.stages;
        if (unit_order) *unit_order = ws.tokens_fastest;
        if (fused_units) *fused_units = (int)groups.size() * ws.n_ntiles * h.w4_k_split;
        if (shrink_units) *shrink_units = (int)(sh.shrink_groups.size() / sh.cs);
        return LORA_OK;
    }
    if (cluster) *cluster = sh.cs;
    if (tile_n) *tile_n = sh.tile_n;
    if (bk) *bk = sh.bk;
    if (stages) *stages = sh.stages;
    if (unit_order) *unit_order = sh.yt ? 3 : sh.m_fastest;   // 0, 1, 2, 3 as documented
    if (fused_units) *fused_units = fused_row_groups(sh) * sh.n_ntiles * h.k_split;
    if (shrink_units) *shrink_units = (int)(sh.shrink_groups.size() / sh.cs) * h.k_split;
    return LORA_OK;
}

int lora_linear_k_split(int d_in, int d_out, int rank, int max_tokens, int num_sms, int* k_split) {
    if (!k_split) return LORA_EINVAL;
    *k_split = 0;
    if (num_sms < 2) return LORA_EINVAL;
    int rc = check_shape(d_in, d_out, rank, max_tokens, 1);
    if (rc != LORA_OK) return rc;
    lora_linear h;
    h.d_in = d_in;
    h.d_out = d_out;
    h.rank = rank;
    h.max_tokens = max_tokens;
    h.num_sms = num_sms;
    h.u_rows = ceil_div(max_tokens, kTileM) * kTileM + kTileM;
    *k_split = choose_k_split(&h);
    return LORA_OK;
}

int lora_linear_host_chunks(int T, int32_t* bounds, int* n) {
    if (T < 0 || !bounds || !n) return LORA_EINVAL;
    const std::vector<int> b = host_chunk_bounds(T);
    if ((int)b.size() - 1 > LORA_MAX_HOST_CHUNKS) return LORA_EINVAL;   // never: the schedule's bound
    for (size_t i = 0; i < b.size(); ++i) bounds[i] = b[i];
    *n = (int)b.size() - 1;
    return LORA_OK;
}

}  // extern "C"
