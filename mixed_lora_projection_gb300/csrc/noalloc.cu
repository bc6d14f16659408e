// lora_linear_forward_noalloc: the projection for callers that cannot allocate memory.
//
// Some callers cannot call cudaMalloc: a serving engine that reserved its device pools at
// start-up (a raw allocation then fails or fragments them), latency-critical code where
// cudaMalloc's device-wide synchronisation would stall other streams, and plugins whose
// host forbids allocations after start-up. This entry point needs no handle: its scratch
// (the shrink output U, the device work list and a status word) is one file-scope
// __device__ array of fixed size, resident on every GPU that loads the library. It runs
// the same kernels as lora_linear_forward and allocates nothing, on the device or the
// host: the plan and the work list are built in fixed-size arrays on the stack, and a
// small work list travels in the kernel parameters instead of being copied.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "../../include/lora_linear.h"
#include "lora_internal.h"

namespace {

using lora::GemmParams;
using lora::Tile;

constexpr int kMaxTokens = LORA_NOALLOC_MAX_TOKENS;
constexpr int kMaxSegs = LORA_NOALLOC_MAX_SEGMENTS;
constexpr int kURows = kMaxTokens + lora::kTileM;           // a tile's TMA read runs up to 127 rows past T
constexpr size_t kUBytes = (size_t)kURows * LORA_MAX_RANK * 2;
constexpr int kMaxTiles = kMaxTokens / lora::kTileM + kMaxSegs + 1;
// work list: [B_a maps][A_a maps][fused tiles][shrink tiles][seg_off][seg_id][scales]
constexpr size_t kOffBMaps = 0;
constexpr size_t kOffAMaps = kOffBMaps + (size_t)kMaxSegs * sizeof(CUtensorMap);
constexpr size_t kOffFused = kOffAMaps + (size_t)kMaxSegs * sizeof(CUtensorMap);
constexpr size_t kOffShrink = kOffFused + (size_t)kMaxTiles * sizeof(Tile);
constexpr size_t kOffSegOff = kOffShrink + (size_t)kMaxTiles * sizeof(Tile);
constexpr size_t kOffSegId = kOffSegOff + 4 * (size_t)(kMaxSegs + 4);
constexpr size_t kOffScale = kOffSegId + 4 * (size_t)(kMaxSegs + 4);
constexpr size_t kWorkBytes = kOffScale + 4 * (size_t)(kMaxSegs + 4);
constexpr size_t kOffStatus = kUBytes + ((kWorkBytes + 255) / 256) * 256;
constexpr size_t kScratchBytes = LORA_NOALLOC_SCRATCH_BYTES;
static_assert(kOffStatus + 256 <= kScratchBytes, "scratch layout exceeds LORA_NOALLOC_SCRATCH_BYTES");

// Layout of the scratch array: [U: kURows x 256 bf16][work list][status word].
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kMaxDevices = 64;
struct DeviceSetup {
    bool ready = false;
    unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch on this device
    int num_sms = 0;
};
DeviceSetup g_setup[kMaxDevices];
EncodeTiledFn g_encode = nullptr;
std::mutex g_setup_mutex;

// Once per device, with that device current: the scratch array's device address (host
// code only has a host-side stand-in for the symbol), the SM count and the kernels'
// shared-memory opt-in.
int setup_device(int dev, DeviceSetup** out) {
    if (dev < 0 || dev >= kMaxDevices) return LORA_ENODEV;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    DeviceSetup& s = g_setup[dev];
    if (!s.ready) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return LORA_ENODEV;
        if (prop.major != 10 || prop.minor != 3) return LORA_ENODEV;
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                return LORA_ECUDA;
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return LORA_ECUDA;
        if (lora::gemm_prepare_device() != cudaSuccess) return LORA_ECUDA;
        s.scratch = static_cast<unsigned char*>(ptr);
        s.num_sms = prop.multiProcessorCount;
        s.ready = true;
    }
    *out = &s;
    return LORA_OK;
}

CUresult encode(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
                uint32_t box_outer) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

inline int cdiv(long long a, long long b) { return (int)((a + b - 1) / b); }

// The planner's tiling in fixed-size arrays (same rule as lora_linear_plan): merged runs,
// greedy 128-row tiles that never hold two different adapters, adapter tiles ordered by id.
struct FixedPlan {
    int n_m = 0, n_fused = 0, n_shrink = 0, n_used = 0;
    int32_t seg_off[kMaxSegs + 1];
    int32_t seg_id[kMaxSegs];
    Tile fused[kMaxTiles];
    Tile shrink[kMaxTiles];
    int used[kMaxSegs];  // compact slot -> caller's adapter index (0-based), ascending
};

void plan_fixed(const int32_t* off, const int32_t* ids, int n_seg, FixedPlan* p) {
    for (int i = 0; i < n_seg; ++i) {
        int lo = off[i], hi = off[i + 1], a = ids[i];
        if (hi == lo) continue;
        if (p->n_m && p->seg_id[p->n_m - 1] == a) {
            p->seg_off[p->n_m] = hi;
        } else {
            if (!p->n_m) p->seg_off[0] = lo;
            p->seg_id[p->n_m] = a;
            p->seg_off[++p->n_m] = hi;
        }
    }
    Tile cur{0, 0, 0, 0, 0};
    for (int r = 0; r < p->n_m; ++r) {
        int pos = p->seg_off[r], hi = p->seg_off[r + 1], a = p->seg_id[r];
        while (pos < hi) {
            if (cur.nrows == lora::kTileM || (a != 0 && cur.adapter != 0 && a != cur.adapter)) {
                p->fused[p->n_fused++] = cur;
                cur = Tile{pos, 0, 0, 0, pos};
            }
            int take = hi - pos < lora::kTileM - cur.nrows ? hi - pos : lora::kTileM - cur.nrows;
            cur.nrows += take;
            pos += take;
            if (a != 0) cur.adapter = a;
        }
    }
    if (cur.nrows) p->fused[p->n_fused++] = cur;
    for (int i = 0; i < p->n_fused; ++i)  // stable insertion by adapter id
        if (p->fused[i].adapter) {
            int j = p->n_shrink++;
            while (j > 0 && p->shrink[j - 1].adapter > p->fused[i].adapter) {
                p->shrink[j] = p->shrink[j - 1];
                --j;
            }
            p->shrink[j] = p->fused[i];
            p->shrink[j].fused_index = i;
        }
    for (int i = 0; i < p->n_shrink; ++i)
        if (!p->n_used || p->used[p->n_used - 1] != p->shrink[i].adapter - 1) p->used[p->n_used++] = p->shrink[i].adapter - 1;
}

int compact_of(const FixedPlan& p, int id) {
    if (id == 0) return 0;
    for (int k = 0; k < p.n_used; ++k)
        if (p.used[k] == id - 1) return k + 1;
    return 0;
}

}  // namespace

extern "C" int lora_linear_forward_noalloc(const void* x, int T, const int32_t* seg_offsets,
                                           const int32_t* seg_adapter_ids, int n_seg, int d_in, int d_out,
                                           int rank, const void* W, const void* const* A,
                                           const void* const* B, const float* scale, int n_adapters,
                                           void* y, void* stream_) {
    int rc = lora_linear_validate(d_in, d_out, rank, kMaxTokens, kMaxSegs, x, T, seg_offsets, seg_adapter_ids,
                                  n_seg, W, A, B, scale, n_adapters, y);
    if (rc != LORA_OK) return rc;
    if (T == 0) return LORA_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ECUDA;
    DeviceSetup* ds = nullptr;
    rc = setup_device(dev, &ds);
    if (rc != LORA_OK) return rc;

    FixedPlan plan;
    plan_fixed(seg_offsets, seg_adapter_ids, n_seg, &plan);
    for (int i = 0; i < plan.n_fused; ++i) plan.fused[i].adapter = compact_of(plan, plan.fused[i].adapter);
    for (int i = 0; i < plan.n_shrink; ++i) plan.shrink[i].adapter = compact_of(plan, plan.shrink[i].adapter);
    for (int i = 0; i < plan.n_m; ++i) plan.seg_id[i] = compact_of(plan, plan.seg_id[i]);

    const int tile_n = lora::kMaxTileN;
    const int shrink_n = cdiv(rank, 16) * 16;
    auto stages_for = [](int tn) {
        int s = lora::kMaxStages;
        while (s > 2 && lora::gemm_smem_bytes(tn, s, lora::kTileK) > (size_t)lora::kSmemLimit) --s;
        return s < 2 ? 2 : (s > lora::kMaxStages ? lora::kMaxStages : s);
    };

    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    // The work list below lives on this call's stack (or in the kernel parameters); a stream
    // capture would record work that reads it after the call has returned, so no work is
    // enqueued while the stream is capturing.
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &capture) != cudaSuccess) return LORA_ECUDA;
    if (capture != cudaStreamCaptureStatusNone) return LORA_EUNSUPPORTED;

    unsigned char* scratch = ds->scratch;
    unsigned char* wdev = scratch + kUBytes;
    int* status = reinterpret_cast<int*>(scratch + kOffStatus);
    GemmParams p;
    memset(&p, 0, sizeof(p));
    // Every tensor map is encoded before anything is enqueued, so a failed call leaves the
    // stream untouched. A work list within the kernel-parameter limits travels in the
    // parameters (no copy at all); a larger one is copied into the scratch array.
    const bool inline_wl = plan.n_fused + plan.n_shrink <= lora::kInlineTiles && plan.n_m <= lora::kInlineSegs &&
                           plan.n_used <= lora::kInlineAdapters;
    alignas(128) unsigned char work[kWorkBytes];
    CUtensorMap* bmaps = inline_wl ? p.inline_maps : reinterpret_cast<CUtensorMap*>(work + kOffBMaps);
    CUtensorMap* amaps =
        inline_wl ? p.inline_maps + lora::kInlineAdapters : reinterpret_cast<CUtensorMap*>(work + kOffAMaps);
    for (int k = 0; k < plan.n_used; ++k) {
        int a = plan.used[k];
        if (encode(&bmaps[k], B[a], rank, d_out, lora::kTileK, tile_n) != CUDA_SUCCESS) return LORA_ECUDA;
        if (encode(&amaps[k], A[a], d_in, rank, lora::kTileK, shrink_n) != CUDA_SUCCESS) return LORA_ECUDA;
    }
    if (encode(&p.tm_x, x, d_in, T, lora::kTileK, lora::kTileM) != CUDA_SUCCESS) return LORA_ECUDA;
    if (encode(&p.tm_w, W, d_in, d_out, lora::kTileK, tile_n) != CUDA_SUCCESS) return LORA_ECUDA;
    if (encode(&p.tm_u, scratch, rank, kURows, lora::kTileK, lora::kTileM) != CUDA_SUCCESS) return LORA_ECUDA;
    if (inline_wl) {
        memcpy(p.inline_tiles, plan.fused, sizeof(Tile) * plan.n_fused);
        memcpy(p.inline_tiles + plan.n_fused, plan.shrink, sizeof(Tile) * plan.n_shrink);
        memcpy(p.inline_seg, plan.seg_off, 4 * (size_t)(plan.n_m + 1));
        memcpy(p.inline_seg + plan.n_m + 1, plan.seg_id, 4 * (size_t)plan.n_m);
        for (int k = 0; k < plan.n_used; ++k) p.inline_scales[k] = scale[plan.used[k]];
        p.inline_wl = 1;
        p.inline_shrink_off = plan.n_fused;
    } else {
        memcpy(work + kOffFused, plan.fused, sizeof(Tile) * plan.n_fused);
        memcpy(work + kOffShrink, plan.shrink, sizeof(Tile) * plan.n_shrink);
        memcpy(work + kOffSegOff, plan.seg_off, 4 * (size_t)(plan.n_m + 1));
        memcpy(work + kOffSegId, plan.seg_id, 4 * (size_t)plan.n_m);
        float* sc = reinterpret_cast<float*>(work + kOffScale);
        for (int k = 0; k < plan.n_used; ++k) sc[k] = scale[plan.used[k]];
        p.tm_b = reinterpret_cast<const CUtensorMap*>(wdev + kOffBMaps);
        p.tm_a = reinterpret_cast<const CUtensorMap*>(wdev + kOffAMaps);
        p.shrink_tiles = reinterpret_cast<const Tile*>(wdev + kOffShrink);
        p.fused_tiles = reinterpret_cast<const Tile*>(wdev + kOffFused);
        p.seg_off = reinterpret_cast<const int32_t*>(wdev + kOffSegOff);
        p.seg_id = reinterpret_cast<const int32_t*>(wdev + kOffSegId);
        p.scales = reinterpret_cast<const float*>(wdev + kOffScale);
        // cudaMemcpyAsync from pageable memory returns once the source has been read, so the
        // stack buffer may go away with this call
        if (cudaMemcpyAsync(wdev, work, kWorkBytes, cudaMemcpyHostToDevice, stream) != cudaSuccess) return LORA_ECUDA;
    }
    if (cudaMemsetAsync(status, 0, sizeof(int), stream) != cudaSuccess) return LORA_ECUDA;

    p.y = y;
    p.u = scratch;
    p.status = status;
    p.wait_limit_ns = 4000000000ull;
    p.n_seg = plan.n_m;
    p.n_fused = plan.n_fused;
    p.n_ntiles = cdiv(d_out, tile_n);
    p.tile_n = tile_n;
    p.shrink_n = shrink_n;
    p.stages = stages_for(tile_n > shrink_n ? tile_n : shrink_n);
    // keep the smaller operand L2-resident: walk row tiles first when X is smaller than W
    p.m_fastest = ((long long)plan.n_fused * lora::kTileM < (long long)d_out) ? 1 : 0;
    p.k_main_blocks = cdiv(d_in, lora::kTileK);
    p.k_lora_blocks = cdiv(rank, lora::kTileK);
    p.d_out = d_out;
    p.rank = rank;
    p.cluster_size = 1;
    p.raster_group = 1;
    p.bk = lora::kTileK;
    p.mma_group = 1;  // single CTAs: one stage per wait
    // two launches ordered by the stream: the shrink units, then the fused units
    if (plan.n_shrink > 0) {
        GemmParams s = p;
        s.n_shrink = plan.n_shrink;
        s.n_fused = 0;
        int grid = plan.n_shrink < ds->num_sms ? plan.n_shrink : ds->num_sms;
        if (lora::launch_gemm(s, grid, stream) != cudaSuccess) return LORA_ECUDA;
    }
    long long units = (long long)plan.n_fused * p.n_ntiles;
    int grid = units < ds->num_sms ? (int)units : ds->num_sms;
    if (lora::launch_gemm(p, grid, stream) != cudaSuccess) return LORA_ECUDA;
    return LORA_OK;
}
