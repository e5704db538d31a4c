// paged_decode_attention host side: partition plan, workspace layout and launches of the
// kernel in attention_kernel.cuh (head groups of 1 here; larger groups in
// decode_attention_gqa.cu).

#include "attention_kernel.cuh"

namespace kvp {
namespace {

template <typename C>
int consumers_of() { return C::NC * C::CPS; }      // per SM

template <typename C>
int rings_of() { return C::NR * C::CPS; }

template <int G>
int consumers_for_g(const kv_pool* pool) {
    const kv_pool_desc& d = pool->desc;
    if constexpr (G > 1) {                         // grouped-query tensor-core configuration
        // head-pair stages (FP8): rings of two warps, each ring's items covering two K/V heads
        if (d.dtype == KV_FP8_E4M3 && d.head_dim == 128 && pool->tmaps && pair_stages(pool, false))
            return rings_of<Cfg<128, uint8_t, __half, G, true, 1, 0, false, true>>();
        if (d.dtype == KV_F16 && d.head_dim == 128 && pool->tmaps && pair_stages(pool, false))
            return rings_of<Cfg<128, __half, __half, G, true, 1, 0, false, true>>();
        if (d.dtype == KV_F16 && d.head_dim == 128 && pool->tmaps)
            return consumers_of<Cfg<128, __half, __half, G, true>>();
        if (d.dtype == KV_FP8_E4M3 && d.head_dim == 128 && pool->tmaps)
            return consumers_of<Cfg<128, uint8_t, __half, G, true>>();
    }
    if constexpr (G == 1) {                        // fp32 pools have no grouped path
        if (d.dtype == KV_F32) return d.head_dim == 128 ? consumers_of<Cfg<128, float, float>>()
                                                        : consumers_of<Cfg<64, float, float>>();
    }
    if (d.dtype == KV_F16) return d.head_dim == 128 ? consumers_of<Cfg<128, __half, __half, G>>()
                                                    : consumers_of<Cfg<64, __half, __half, G>>();
    return d.head_dim == 128 ? consumers_of<Cfg<128, uint8_t, __half, G>>()
                             : consumers_of<Cfg<64, uint8_t, __half, G>>();
}

}  // namespace

// Heads per work item of this pool's single-query decode (Cfg HP: 1, 2 or 4).  Pools whose
// (block, head) tiles are small pay for every copy, so one copy brings a block's tiles of
// several adjacent heads: FP8 pools with B = 8 take four (4 KiB copies), FP8 pools with
// B = 16 and fp16 pools with B = 8 two (head_dim 128; the head count a multiple of the
// group).  KVP_NO_HEAD_PAIRS (tuning builds only) turns it off.
int head_group(const kv_pool_desc& d, int group) {
#if defined(KVP_NO_HEAD_PAIRS)
    (void)d; (void)group;
    return 1;
#else
    if (group != 1 || d.head_dim != 128) return 1;
    if (d.dtype == KV_FP8_E4M3 && d.block_size == 8 && d.num_heads % 4 == 0) return 4;
    if (d.num_heads % 2 != 0) return 1;
    if (d.dtype == KV_FP8_E4M3 && (d.block_size == 8 || d.block_size == 16)) return 2;
    if (d.dtype == KV_F16 && d.block_size == 8) return 2;
    return 1;
#endif
}

bool pair_stages(const kv_pool* pool, bool prefix) {
#if defined(KVP_NO_PAIR_STAGES)
    (void)pool;
    (void)prefix;
    return false;                                  // tuning builds only
#else
    // Measured (GB300): shared-prefix launches +16 % (8 KiB instead of 4 KiB copies lift
    // the per-SM copy rate that bounds them), FP8 grouped-query +4 %; fp16 grouped-query
    // +1.5 % once two CTAs share each SM (1 % slower with one CTA of nine warps per SM).
    (void)prefix;
    if (!pool->tmaps || !pool->pmaps || pool->desc.num_heads % 2 != 0) return false;
    return true;
#endif
}

namespace {

// K/V heads covered by one work item of this launch shape: head groups of the single-query
// CUDA-core consumer, or the head pairs of the tensor-core consumer
int kv_heads_per_item(const kv_pool* pool, int group) {
    if (group > 1 && pool->tmaps && pool->desc.head_dim == 128 && pair_stages(pool, false)) return 2;
    return head_group(pool->desc, group);
}

int consumers_for(const kv_pool* pool, int group) {
    const int hp = head_group(pool->desc, group);
    if (hp == 4) return consumers_of<Cfg<128, uint8_t, __half, 1, false, 4, 8>>();
    if (hp == 2) {
        if (pool->desc.dtype == KV_F16) return consumers_of<Cfg<128, __half, __half, 1, false, 2, 8>>();
        return pool->desc.block_size == 8 ? consumers_of<Cfg<128, uint8_t, __half, 1, false, 2, 8>>()
                                          : consumers_of<Cfg<128, uint8_t, __half, 1, false, 2, 16>>();
    }
    switch (group) {
        case 2: return consumers_for_g<2>(pool);
        case 4: return consumers_for_g<4>(pool);
        case 8: return consumers_for_g<8>(pool);
        default: return consumers_for_g<1>(pool);
    }
}

constexpr size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

bool valid_group(const kv_pool_desc& d, int group) {
    if (group == 1) return true;
    return (group == 2 || group == 4 || group == 8) && d.dtype != KV_F32;
}

int plan_attention(const kv_pool* pool, int batch, int max_context, int partition_tokens,
                   AttnPlan* plan, int group, int window) {
    const kv_pool_desc& d = pool->desc;
    if (batch < 0 || max_context < 0 || window < 0 || batch > kMaxBatch * kMaxSub) return KV_ERR_INVALID_ARG;
    static_assert(kMaxBatch * kMaxSub == KV_MAX_DECODE_BATCH, "the documented batch limit");
    // a sliding window bounds the tokens read per sequence (window + up to 31 masked rows)
    const int span = (window > 0 && window + 32 < max_context) ? window + 32 : max_context;
    if (!valid_group(d, group)) return KV_ERR_INVALID_ARG;
    const int cap = 1 << 24;                       // block ids are fetched per chunk: no per-item cap
    constexpr int kAutoPartMax = 1024;             // library choice: 256 .. 1024 tokens per item
    constexpr int kAutoPartMin = 256;
    constexpr int kAutoPartAlt = 192;              // finer split of one-round launches (kernel's choice)
    const int nc = consumers_for(pool, group);
    int P;
    if (partition_tokens > 0) {
        if (partition_tokens % kPartAlign != 0 || partition_tokens > cap) return KV_ERR_INVALID_ARG;
        P = partition_tokens;
    } else if (partition_tokens == 0) {
        // work items are (sequence, KV head or head pair, partition), handed out dynamically
        const int64_t units = static_cast<int64_t>(batch > 0 ? batch : 1) * d.num_heads /
                              kv_heads_per_item(pool, group);
        const int64_t warps = static_cast<int64_t>(pool->num_sms) * nc;
        int64_t parts;
        if (group == 1) {
            // about 8 items per consumer warp, so the dynamic hand-out evens out the tail
            parts = (8 * warps + units - 1) / units;
        } else {
            // an item of a grouped launch also stages G query rows and writes (and merges)
            // G partial rows: fewer, longer items, about one round of them
            parts = warps / units;
        }
        if (parts < 1) parts = 1;
        int64_t p = (span + parts - 1) / parts;
        p = (p + kPartAlign - 1) / kPartAlign * kPartAlign;
        // every item also pays a claim, a query copy, a partial and its share of a merge:
        // below 256 tokens that costs more than the finer balance gains
        if (p < kAutoPartMin) p = kAutoPartMin;
        // the longest item bounds the tail when contexts are ragged (the host sees only
        // the longest context)
        if (p > kAutoPartMax) p = kAutoPartMax;
        P = static_cast<int>(p);
    } else {
        return KV_ERR_INVALID_ARG;
    }
    plan->partition = P;
    plan->fine_partition = P;
    plan->fine_from = batch;
    plan->alt_partition = P;
    if (partition_tokens == 0 && group == 1 && P == kAutoPartMin) {
        // a small launch (the 256-token floor was reached): the kernel may split finer, to
        // 192 tokens, when the lengths it reads still give at most one item per consumer
        // warp (measured: the 7B decode loop 0.72 -> 0.76 of the copy peak)
        plan->alt_partition = kAutoPartAlt;
    }
    if (partition_tokens == 0 && P >= 512) {
        // A launch of several rounds of work items ends with the last round: items claimed
        // last finish up to an item's time apart.  With long items (512 tokens and more)
        // the sequences handed out last, about one round of items' worth of tokens, take
        // half-size partitions (measured: ragged 256 sequences +1 % fp16, +4 % FP8; with
        // 256-token items it gained nothing and the doubled split count of long contexts
        // cost 3 %).
        const int hu = d.num_heads / kv_heads_per_item(pool, group);
        const int64_t warps = static_cast<int64_t>(pool->num_sms) * nc;
        const int64_t items = static_cast<int64_t>(batch) * hu * ((span + P - 1) / P);
        if (items >= 2 * warps) {
            const int64_t per_seq = static_cast<int64_t>(span) * hu;
            const int64_t n_fine = (warps * P + per_seq - 1) / per_seq;
            plan->fine_from = static_cast<int>(batch - (n_fine < batch ? n_fine : batch));
            plan->fine_partition = (P / 2 + kPartAlign - 1) / kPartAlign * kPartAlign;
        }
    }
    const int pmin = plan->fine_from < batch ? plan->fine_partition : plan->alt_partition;
    plan->max_parts = span <= pmin ? 1 : (span + pmin - 1) / pmin;
    // the kernel numbers a launch's work items with an int, and the workspace is sized in
    // size_t: refuse sizes that would overflow either (about 10^9 items per launch, far
    // beyond any pool a GPU holds)
    const int64_t launch_items = static_cast<int64_t>(batch < kMaxBatch ? batch : kMaxBatch) *
                                 d.num_heads * plan->max_parts;
    if (launch_items > (int64_t{1} << 30)) return KV_ERR_INVALID_ARG;
    plan->consumers = nc;
    plan->group = group;
    plan->window = window;
    plan->flags = 0;
    plan->pairs = group > 1 && kv_heads_per_item(pool, group) == 2;
    size_t ws = kCounterBytes;                      // work and exit counters
    if (plan->max_parts > 1) {
        const size_t n = static_cast<size_t>(batch) * d.num_heads * group * plan->max_parts;
        ws += plan->arrivals_bytes(batch, d.num_heads);
        ws += align256(n * 2 * sizeof(float));
        ws += align256(n * d.head_dim * sizeof(float));
    }
    plan->ws_bytes = ws;
    return KV_OK;
}

int plan_attention_prefix(const kv_pool* pool, int batch, int max_context, int partition_tokens,
                          AttnPlan* plan) {
    const kv_pool_desc& d = pool->desc;
    if (batch < 0 || max_context < 0 || batch > kMaxBatch * kMaxSub) return KV_ERR_INVALID_ARG;
    if (!pool->tmaps || d.head_dim != 128 || (d.dtype != KV_F16 && d.dtype != KV_FP8_E4M3))
        return KV_ERR_UNSUPPORTED;
    // A member's context splits at the end of its shared prefix into at most
    // ceil(max_context / P) + 1 partitions, which must fit one merge step.
    const int64_t pmin64 = ((static_cast<int64_t>(max_context) + kPfxMaxParts - 2) / (kPfxMaxParts - 1) +
                            kPartAlign - 1) / kPartAlign * kPartAlign;
    const int pmin = static_cast<int>(pmin64 < kPartAlign ? kPartAlign : pmin64);
    int P;
    if (partition_tokens > 0) {
        if (partition_tokens % kPartAlign != 0 || partition_tokens < pmin || partition_tokens > (1 << 24))
            return KV_ERR_INVALID_ARG;
        P = partition_tokens;
    } else if (partition_tokens == 0) {
        // library choice: short items, so a group's shared prefix (read once for all its
        // members) spreads over many SMs: about 8 partitions of the longest context, 64 to
        // 1024 tokens each.  With two rings of head pairs per SM, parallel sampling (8
        // members, 40 heads, 1030-1158 tokens) then fits one round of items: 160-token
        // partitions measured 0.349 of the copy peak, against 0.29-0.30 at 96 and 128
        // tokens (more items than rings) and 0.343 at 192.
        int64_t p = (static_cast<int64_t>(max_context) + 7) / 8;
        p = (p + kPartAlign - 1) / kPartAlign * kPartAlign;
        if (p < 64) p = 64;
        if (p > 1024) p = 1024;
        P = static_cast<int>(p < pmin ? pmin : p);
    } else {
        return KV_ERR_INVALID_ARG;
    }
    plan->partition = P;
    plan->fine_partition = P;
    plan->fine_from = batch;
    plan->alt_partition = P;
    plan->max_parts = max_context <= 0 ? 1 : (max_context + P - 1) / P + 1;
    const int64_t launch_items = static_cast<int64_t>(batch < kMaxBatch ? batch : kMaxBatch) *
                                 d.num_heads * plan->max_parts;
    if (launch_items > (int64_t{1} << 30)) return KV_ERR_INVALID_ARG;
    plan->pairs = pair_stages(pool, true);
    if (plan->pairs)
        plan->consumers = d.dtype == KV_F16 ? rings_of<Cfg<128, __half, __half, 8, true, 1, 0, true, true>>()
                                            : rings_of<Cfg<128, uint8_t, __half, 8, true, 1, 0, true, true>>();
    else
        plan->consumers = d.dtype == KV_F16 ? consumers_of<Cfg<128, __half, __half, 8, true, 1, 0, true>>()
                                            : consumers_of<Cfg<128, uint8_t, __half, 8, true, 1, 0, true>>();
    plan->group = 1;
    plan->window = 0;
    plan->flags = 0;
    plan->groups = nullptr;
    plan->n_groups = 0;
    size_t ws = kCounterBytes;
    if (plan->max_parts > 1) {
        const size_t n = static_cast<size_t>(batch) * d.num_heads * plan->max_parts;
        ws += plan->arrivals_bytes(batch, d.num_heads);
        ws += align256(n * 2 * sizeof(float));
        ws += align256(n * d.head_dim * sizeof(float));
    }
    plan->ws_bytes = ws;
    return KV_OK;
}

int launch_attention(const kv_pool* pool, int layer, const void* q, float* out,
                     const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                     int batch, int max_context, float scale, const AttnPlan& plan,
                     void* workspace, cudaStream_t stream) {
    return launch_attention_append(pool, layer, q, nullptr, nullptr, 0, out, block_tables, max_blocks,
                                   context_lens, batch, max_context, scale, plan, workspace, stream);
}

int launch_attention_append(const kv_pool* pool, int layer, const void* q, const void* k_new,
                            const void* v_new, int in_bytes, void* out, const int32_t* block_tables,
                            int max_blocks, const int32_t* context_lens, int batch, int max_context,
                            float scale, const AttnPlan& plan, void* workspace, cudaStream_t stream) {
    const kv_pool_desc& d = pool->desc;
    if (batch == 0) return KV_OK;
    const int group = plan.group;
    char* ws = static_cast<char*>(workspace);
    unsigned* counters = reinterpret_cast<unsigned*>(ws);
    const size_t arrivals_bytes = plan.arrivals_bytes(batch, d.num_heads);
    // the counters must be zero when the kernel starts; every launch leaves them zero when
    // it completes without a device error, so a caller that keeps the workspace for decode
    // calls may say so (KV_DECODE_WORKSPACE_ZEROED) and skip this clearing
    if (!(plan.flags & KV_DECODE_WORKSPACE_ZEROED) &&
        cudaMemsetAsync(counters, 0, kCounterBytes + arrivals_bytes, stream) != cudaSuccess)
        return KV_ERR_CUDA;

    AttnArgs a{};
    a.kpool = static_cast<char*>(pool->k_layers[layer]);
    a.vpool = static_cast<char*>(pool->v_layers[layer]);
    a.k_new = static_cast<const char*>(k_new);
    a.v_new = static_cast<const char*>(v_new);
    a.in_bytes = in_bytes;
    a.kscale = pool->k_scales ? pool->k_scales[layer] : nullptr;
    a.vscale = pool->v_scales ? pool->v_scales[layer] : nullptr;
    a.q = q;
    a.out = out;
    a.tables = block_tables;
    a.lens = context_lens;
    if (plan.max_parts > 1) {
        const size_t n = static_cast<size_t>(batch) * d.num_heads * group * plan.max_parts;
        a.arrivals = reinterpret_cast<unsigned*>(ws + kCounterBytes);
        a.grp_arrivals =
            reinterpret_cast<unsigned*>(ws + kCounterBytes + align256(static_cast<size_t>(batch) * d.num_heads * 4));
        a.n_grp = merge_groups(plan.max_parts);
        a.part_ml = reinterpret_cast<float*>(ws + kCounterBytes + arrivals_bytes);
        a.part_o = reinterpret_cast<float*>(ws + kCounterBytes + arrivals_bytes + align256(n * 2 * sizeof(float)));
    }
    a.err = pool->d_err;
    a.batch = batch;
    a.H = d.num_heads;
    a.B = d.block_size;
    a.max_blocks = max_blocks;
    const int64_t lim_tables = static_cast<int64_t>(max_blocks) * d.block_size;
    a.ctx_limit = static_cast<int>(lim_tables < max_context ? lim_tables : max_context);
    a.P = plan.partition;
    a.early_tables = (plan.flags & KV_DECODE_PDL) && (plan.flags & KV_DECODE_EARLY_TABLES) ? 1 : 0;
    a.out_f16 = (plan.flags & KV_DECODE_OUT_F16) ? 1 : 0;
    a.early_pool = a.early_tables && (plan.flags & KV_DECODE_EARLY_POOL) ? 1 : 0;
    a.P_fine = plan.fine_partition;
    a.P_alt = plan.alt_partition;
    a.s_fine = plan.fine_from;
    a.max_parts = plan.max_parts;
    a.num_blocks = d.num_blocks;
    a.qscale = scale * 1.4426950408889634f;        // log2(e): softmax evaluated with 2^x
    a.window = plan.window;
    if (pool->tmaps) {                             // the layer's swizzled tile maps
        const CUtensorMap* maps = plan.pairs ? pool->pmaps : pool->tmaps;
        a.kmap = maps[2 * layer];
        a.vmap = maps[2 * layer + 1];
    }
    a.fused = k_new != nullptr ? 1 : 0;

    if (plan.n_groups > 0) {                       // shared prompt prefixes
        if (!pool->tmaps || group != 1 || plan.window != 0) return KV_ERR_UNSUPPORTED;
        a.groups = plan.groups;
        a.n_groups = plan.n_groups;
        if (plan.pairs) {
            if (d.dtype == KV_F16)
                return launch_typed<Cfg<128, __half, __half, 8, true, 1, 0, true, true>>(pool, a, plan, counters,
                                                                                          stream);
            if (d.dtype == KV_FP8_E4M3)
                return launch_typed<Cfg<128, uint8_t, __half, 8, true, 1, 0, true, true>>(pool, a, plan, counters,
                                                                                           stream);
            return KV_ERR_UNSUPPORTED;
        }
        if (d.dtype == KV_F16)
            return launch_typed<Cfg<128, __half, __half, 8, true, 1, 0, true>>(pool, a, plan, counters, stream);
        if (d.dtype == KV_FP8_E4M3)
            return launch_typed<Cfg<128, uint8_t, __half, 8, true, 1, 0, true>>(pool, a, plan, counters, stream);
        return KV_ERR_UNSUPPORTED;
    }

    if (group != 1) return launch_attention_grouped(group, pool, a, plan, counters, stream);
    if (d.dtype == KV_F32) {
        if (d.head_dim == 128) return launch_typed<Cfg<128, float, float>>(pool, a, plan, counters, stream);
        return launch_typed<Cfg<64, float, float>>(pool, a, plan, counters, stream);
    }
    const int hp = head_group(d, 1);
    if (hp == 4)                                     // four heads per work item
        return launch_typed<Cfg<128, uint8_t, __half, 1, false, 4, 8>>(pool, a, plan, counters, stream);
    if (hp == 2) {                                   // two heads per work item
        if (d.dtype == KV_F16)
            return launch_typed<Cfg<128, __half, __half, 1, false, 2, 8>>(pool, a, plan, counters, stream);
        if (d.block_size == 8)
            return launch_typed<Cfg<128, uint8_t, __half, 1, false, 2, 8>>(pool, a, plan, counters, stream);
        return launch_typed<Cfg<128, uint8_t, __half, 1, false, 2, 16>>(pool, a, plan, counters, stream);
    }
    if (d.dtype == KV_F16) {
        if (d.head_dim == 128) return launch_typed<Cfg<128, __half, __half>>(pool, a, plan, counters, stream);
        return launch_typed<Cfg<64, __half, __half>>(pool, a, plan, counters, stream);
    }
    if (d.head_dim == 128) return launch_typed<Cfg<128, uint8_t, __half>>(pool, a, plan, counters, stream);
    return launch_typed<Cfg<64, uint8_t, __half>>(pool, a, plan, counters, stream);
}

}  // namespace kvp
