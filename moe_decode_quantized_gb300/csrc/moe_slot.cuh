// moe_slot.cuh -- the slot-table update (page
// spark_model/layers/moe_v41/device_route.rs, fn slot_table_update and
// struct Kernels slot_table_set): table[layer][expert] = slot for a batch of
// (layer, expert, slot) triples, one thread per triple. The triples of one
// launch land in parallel, so the caller dedupes them (last write wins).
#pragma once
#include "moe_common.cuh"

namespace moe {

__global__ void moe_slot_table_kernel(int32_t *table, int n_routed, const int32_t *triples, int n,
                                      uint32_t *status)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    pdl_wait();
    if (i >= n)
        return;
    const int l = triples[3 * i], e = triples[3 * i + 1], s = triples[3 * i + 2];
    if (l < 0 || l >= MOE_SLOT_TABLE_LAYERS || e < 0 || e >= n_routed) {
        if (status)
            atomicOr(status, (uint32_t)MOE_WS_TRIPLE);
        return;
    }
    table[(size_t)l * n_routed + e] = s;
}

}  // namespace moe
