// moe_runtime.cuh -- host side of expert residency: an LRU cache of expert
// slots in the device arena, filled from an expert source on a miss.
//
// Page spark_model/layers/moe_v41.rs (module doc: the ExpertLru gathers the
// picked experts' raw slices into its device-visible slots, misses read from
// the source) and page spark_model/layers/moe_v41/device_route.rs (module
// doc: the host reads the header, touches the picks in the cache, fetches the
// misses and uploads the cache's slot changes to the device table; fn
// slot_table_update). The cache owns n_slots arena slots; (layer, expert) ->
// slot, least recently used first out. The device slot table is kept equal to
// the cache's map: after a change the table rows that changed are uploaded
// (from pageable host memory, so the copy has taken the data when the call
// returns). Host code only; no kernel.
#pragma once
#include <cstdint>
#include <list>
#include <unordered_map>
#include <vector>

#include "../../include/moe.h"

namespace moe {

struct ExpertCache {
    int n_layers = 0, n_routed = 0, n_slots = 0;
    const char *arena_base = nullptr;
    uint64_t slot_bytes = 0;
    int32_t *table_dev = nullptr;  // [n_layers][n_routed] device slot table (NULL: host-only, for tests)
    moe_expert_fetch_fn fetch = nullptr;
    void *user = nullptr;
    std::vector<int32_t> table;    // host copy of the slot table
    std::vector<int64_t> owner;    // slot -> layer * n_routed + expert, -1 free
    std::list<int> lru;            // slots, most recently used at the front
    std::vector<std::list<int>::iterator> where;  // slot -> its place in lru
    uint64_t hits = 0, misses = 0, evictions = 0;

    int init(int layers, int routed, int slots, const moe_arena *arena, int32_t *tdev, moe_expert_fetch_fn f, void *u)
    {
        n_layers = layers;
        n_routed = routed;
        n_slots = slots;
        arena_base = static_cast<const char *>(arena->base);
        slot_bytes = arena->slot_bytes;
        table_dev = tdev;
        fetch = f;
        user = u;
        table.assign((size_t)layers * routed, -1);
        owner.assign(slots, -1);
        where.resize(slots);
        for (int s = slots - 1; s >= 0; --s) {  // free slots at the back: taken first
            lru.push_front(s);
            where[s] = lru.begin();
        }
        return MOE_OK;
    }

    void touch(int s)
    {
        lru.erase(where[s]);
        lru.push_front(s);
        where[s] = lru.begin();
    }
};

}  // namespace moe
