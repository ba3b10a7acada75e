// Expert-parallel sharding on the host (xinfer docs "Options": each rank loads and offloads its own expert
// shard while NCCL combines the rank-local MoE results).  The partition is a plain contiguous split of the
// expert ids; the rank's layer is an ordinary layer whose map holds only its own experts, so its hot routes
// are exactly the routes to its shard and its cold list is the routes to the other ranks' shards.
#include <cstdint>

#include "../../include/moe.h"

extern "C" int moe_ep_local_map(int32_t E, int32_t world, int32_t rank, int32_t *expert_to_slot, int32_t *first,
                                int32_t *count) {
    if (E < 1 || world < 1 || world > E || rank < 0 || rank >= world || !expert_to_slot) return MOE_EINVAL;
    const int32_t base = E / world, extra = E % world;
    const int32_t n = base + (rank < extra ? 1 : 0);
    const int32_t f = rank * base + (rank < extra ? rank : extra);
    for (int32_t e = 0; e < E; ++e) expert_to_slot[e] = (e >= f && e < f + n) ? e - f : -1;
    if (first) *first = f;
    if (count) *count = n;
    return MOE_OK;
}
