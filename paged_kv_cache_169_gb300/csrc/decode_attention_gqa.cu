// Grouped-query decode attention: the instantiations with 2, 4 or 8 query heads per KV
// head ("大模型推理加速——KV Cache篇" §6.2: MQA/GQA share one K/V head among a group of
// query heads, so each K/V tile is read once for the whole group).  fp16 and FP8 pools.

#include "attention_kernel.cuh"

namespace kvp {
namespace {

template <int G>
int launch_g(const kv_pool* pool, const AttnArgs& a, const AttnPlan& plan, unsigned* counters,
             cudaStream_t stream) {
    const kv_pool_desc& d = pool->desc;
    if (d.dtype == KV_F16) {
        if (d.head_dim == 128) {
            // tensor cores when the pool has its swizzled tensor maps (head-pair stages when
            // the head count is even), else CUDA cores
            if (pool->tmaps && plan.pairs)
                return launch_typed<Cfg<128, __half, __half, G, true, 1, 0, false, true>>(pool, a, plan, counters, stream);
            if (pool->tmaps) return launch_typed<Cfg<128, __half, __half, G, true>>(pool, a, plan, counters, stream);
            return launch_typed<Cfg<128, __half, __half, G>>(pool, a, plan, counters, stream);
        }
        return launch_typed<Cfg<64, __half, __half, G>>(pool, a, plan, counters, stream);
    }
    if (d.dtype == KV_FP8_E4M3) {
        if (d.head_dim == 128) {
            // tensor cores when the pool has its swizzled tensor maps (K and V fragments
            // converted in registers from the E4M3 codes), else CUDA cores
            if (pool->tmaps && plan.pairs)           // head-pair stages
                return launch_typed<Cfg<128, uint8_t, __half, G, true, 1, 0, false, true>>(pool, a, plan, counters,
                                                                                            stream);
            if (pool->tmaps) return launch_typed<Cfg<128, uint8_t, __half, G, true>>(pool, a, plan, counters, stream);
            return launch_typed<Cfg<128, uint8_t, __half, G>>(pool, a, plan, counters, stream);
        }
        return launch_typed<Cfg<64, uint8_t, __half, G>>(pool, a, plan, counters, stream);
    }
    return KV_ERR_UNSUPPORTED;
}

}  // namespace

int launch_attention_grouped(int group, const kv_pool* pool, const AttnArgs& args, const AttnPlan& plan,
                             unsigned* counters, cudaStream_t stream) {
    switch (group) {
        case 2: return launch_g<2>(pool, args, plan, counters, stream);
        case 4: return launch_g<4>(pool, args, plan, counters, stream);
        case 8: return launch_g<8>(pool, args, plan, counters, stream);
        default: return KV_ERR_INVALID_ARG;
    }
}

}  // namespace kvp
