// Token-segment planner: request segments -> tiles of the fused pass and of the shrink.
//
// Source: "Two 27B models on a single RTX 5090", section 4 -- requests that name the
// adapter and requests that do not run in the same batches, and the adapter applies only
// to the former. The planner turns the batch's segments into 128-row tiles so that one
// tile never mixes two different adapters, while base rows fill the tiles of their
// neighbours instead of forcing ragged tiles.
#include <algorithm>

#include "../../include/lora_linear.h"
#include "lora_internal.h"

namespace lora {

int plan_segments(const int32_t* seg_offsets, const int32_t* seg_ids, int n_seg, int T,
                  int n_adapters, Plan* plan) {
    plan->seg_off.clear();
    plan->seg_id.clear();
    plan->fused.clear();
    plan->shrink.clear();
    plan->used_adapters.clear();
    if (T < 0 || n_seg < 0) return LORA_EINVAL;
    if (n_seg == 0) return T == 0 ? LORA_OK : LORA_EINVAL;
    if (!seg_offsets || !seg_ids) return LORA_EINVAL;
    if (seg_offsets[0] != 0 || seg_offsets[n_seg] != T) return LORA_EINVAL;
    for (int i = 0; i < n_seg; ++i) {
        if (seg_offsets[i + 1] < seg_offsets[i]) return LORA_EINVAL;
        if (seg_ids[i] < 0 || (n_adapters >= 0 && seg_ids[i] > n_adapters)) return LORA_EINVAL;
    }
    // merged runs: drop empty segments, join neighbours with equal ids
    for (int i = 0; i < n_seg; ++i) {
        int lo = seg_offsets[i], hi = seg_offsets[i + 1], a = seg_ids[i];
        if (hi == lo) continue;
        if (!plan->seg_id.empty() && plan->seg_id.back() == a) {
            plan->seg_off.back() = hi;
        } else {
            if (plan->seg_id.empty()) plan->seg_off.push_back(lo);
            plan->seg_off.push_back(hi);
            plan->seg_id.push_back(a);
        }
    }
    if (plan->seg_id.empty()) {
        plan->seg_off.assign(1, 0);
        return LORA_OK;
    }
    // fused tiles: greedy walk; cut at kTileM rows or where a second nonzero id would enter
    Tile cur{0, 0, 0, 0, 0};
    for (size_t r = 0; r < plan->seg_id.size(); ++r) {
        int pos = plan->seg_off[r], hi = plan->seg_off[r + 1], a = plan->seg_id[r];
        while (pos < hi) {
            if (cur.nrows == kTileM || (a != 0 && cur.adapter != 0 && a != cur.adapter)) {
                plan->fused.push_back(cur);
                cur = Tile{pos, 0, 0, 0, pos};
            }
            int take = std::min(hi - pos, kTileM - cur.nrows);
            cur.nrows += take;
            pos += take;
            if (a != 0) cur.adapter = a;
        }
    }
    if (cur.nrows) plan->fused.push_back(cur);
    // shrink tiles: adapter tiles, stably ordered by adapter id
    for (size_t i = 0; i < plan->fused.size(); ++i)
        if (plan->fused[i].adapter) {
            Tile t = plan->fused[i];
            t.fused_index = (int32_t)i;
            plan->shrink.push_back(t);
        }
    std::stable_sort(plan->shrink.begin(), plan->shrink.end(),
                     [](const Tile& a, const Tile& b) { return a.adapter < b.adapter; });
    // compact adapter slots in order of id (used by the device work list)
    for (const Tile& t : plan->shrink)
        if (plan->used_adapters.empty() || plan->used_adapters.back() != t.adapter - 1)
            plan->used_adapters.push_back(t.adapter - 1);
    return LORA_OK;
}

}  // namespace lora

extern "C" int lora_linear_plan(const int32_t* seg_offsets, const int32_t* seg_adapter_ids,
                                int n_seg, int T, int32_t* fused_tiles, int* n_fused,
                                int32_t* shrink_tiles, int* n_shrink) {
    if (!n_fused || !n_shrink) return LORA_EINVAL;
    lora::Plan plan;
    int rc = lora::plan_segments(seg_offsets, seg_adapter_ids, n_seg, T, -1, &plan);
    if (rc != LORA_OK) return rc;
    if ((int)plan.fused.size() > *n_fused || (int)plan.shrink.size() > *n_shrink) return LORA_EINVAL;
    if ((!fused_tiles && !plan.fused.empty()) || (!shrink_tiles && !plan.shrink.empty())) return LORA_EINVAL;
    for (size_t i = 0; i < plan.fused.size(); ++i) {
        fused_tiles[3 * i + 0] = plan.fused[i].row0;
        fused_tiles[3 * i + 1] = plan.fused[i].nrows;
        fused_tiles[3 * i + 2] = plan.fused[i].adapter;
    }
    for (size_t i = 0; i < plan.shrink.size(); ++i) {
        shrink_tiles[3 * i + 0] = plan.shrink[i].row0;
        shrink_tiles[3 * i + 1] = plan.shrink[i].nrows;
        shrink_tiles[3 * i + 2] = plan.shrink[i].adapter;
    }
    *n_fused = (int)plan.fused.size();
    *n_shrink = (int)plan.shrink.size();
    return LORA_OK;
}
