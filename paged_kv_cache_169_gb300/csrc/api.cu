// C ABI of kvpaged: argument validation and dispatch to the launchers.
// Declarations and the contract of every entry point are in include/kvpaged.h.

#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "kvp_internal.cuh"

namespace {

bool valid_desc(const kv_pool_desc* d) {
    if (!d) return false;
    if (d->num_layers < 1 || d->num_layers > 4096) return false;
    if (d->num_blocks < 1) return false;
    if (d->block_size != 8 && d->block_size != 16 && d->block_size != 32) return false;
    if (d->num_heads < 1 || d->num_heads > 256) return false;
    if (d->head_dim != 64 && d->head_dim != 128) return false;
    if (d->dtype != KV_F32 && d->dtype != KV_F16 && d->dtype != KV_FP8_E4M3) return false;
    // element offsets of a whole layer must fit the kernels' int64 arithmetic with room
    const long long elems = 1ll * d->num_blocks * d->num_heads * d->block_size * d->head_dim;
    return elems > 0 && elems < (1ll << 40);
}

void free_pool(kv_pool* p) {
    if (!p) return;
    std::free(p->tmaps_raw);
    std::free(p->k_layers);
    std::free(p->v_layers);
    std::free(p->k_scales);
    std::free(p->v_scales);
    delete p;
}

// Tensor maps of an fp16 or FP8, head_dim 128 pool for the grouped-query tensor-core path.
// fp16: each layer's K and V viewed as [rows][2][64] fp16 (rows = num_blocks*H*B, a row
// being one token of one head), box {64, 2, min(B, 16)}, 128-byte swizzle.  FP8: K and V
// viewed as [rows][128] bytes, box {128, min(B, 32)}, 128-byte swizzle (one token row is
// one swizzle line).  Leaves p->tmaps null if the driver's encoder is unavailable or
// refuses (the CUDA-core path then serves).
void make_tensor_maps(kv_pool* p) {
    const kv_pool_desc& d = p->desc;
    const bool fp8 = d.dtype == KV_FP8_E4M3;
    if (d.head_dim != 128 || (d.dtype != KV_F16 && !fp8)) return;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
        cudaGetLastError();
        return;
    }
    using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    Encode encode = reinterpret_cast<Encode>(fn);
    const int L = d.num_layers;
    void* raw = std::malloc(4 * L * sizeof(CUtensorMap) + 64);
    if (!raw) return;
    CUtensorMap* maps = reinterpret_cast<CUtensorMap*>((reinterpret_cast<uintptr_t>(raw) + 63) & ~uintptr_t(63));
    // a token row of one head (128 halves) seen as two 64-half halves: the copied tile of
    // up to 16 rows lands half-major ([2][rows][64]), so 8 consecutive tokens of one half
    // are 8 consecutive 128-byte lines and their swizzled 16-byte pieces hit distinct banks
    const cuuint64_t rows = static_cast<cuuint64_t>(d.num_blocks) * d.num_heads * d.block_size;
    const cuuint64_t dims[3] = {64, rows, 2};
    const cuuint64_t strides[2] = {256, 128};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(d.block_size < 16 ? d.block_size : 16), 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    const cuuint64_t dims8[2] = {128, rows};
    const cuuint64_t strides8[1] = {128};
    const cuuint32_t box8[2] = {128, static_cast<cuuint32_t>(d.block_size < 32 ? d.block_size : 32)};
    // head-pair stages: a whole block of two adjacent heads (2*B consecutive rows) per copy
    const bool pairs = fp8 || d.block_size <= 16;
    const cuuint32_t boxp[3] = {64, static_cast<cuuint32_t>(2 * d.block_size), 2};
    const cuuint32_t boxp8[2] = {128, static_cast<cuuint32_t>(2 * d.block_size)};
    for (int set = 0; set < (pairs ? 2 : 1); ++set) {
        for (int l = 0; l < L; ++l) {
            for (int kv = 0; kv < 2; ++kv) {
                void* base = kv == 0 ? p->k_layers[l] : p->v_layers[l];
                CUtensorMap* m = &maps[set * 2 * L + 2 * l + kv];
                const CUresult rc =
                    fp8 ? encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims8, strides8, set ? boxp8 : box8, estr,
                                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE)
                        : encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, strides, set ? boxp : box, estr,
                                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
                if (rc != CUDA_SUCCESS) {
                    if (set == 0) {
                        std::free(raw);
                        return;
                    }
                    p->tmaps = maps;                   // single-head maps only
                    p->tmaps_raw = raw;
                    return;
                }
            }
        }
    }
    p->tmaps = maps;
    p->pmaps = pairs ? maps + 2 * L : nullptr;
    p->tmaps_raw = raw;
}

}  // namespace

extern "C" {

const char* kv_status_str(int status) {
    switch (status) {
        case KV_OK: return "ok";
        case KV_ERR_INVALID_ARG: return "invalid argument";
        case KV_ERR_NO_BLOCKS: return "no free blocks";
        case KV_ERR_STATE: return "invalid allocator state";
        case KV_ERR_CUDA: return "CUDA runtime error";
        case KV_ERR_DEVICE: return "device-side error flag set";
        case KV_ERR_UNSUPPORTED: return "unsupported";
        default: return "unknown status";
    }
}

int kv_version(void) { return 101; }

int kv_pool_create(const kv_pool_desc* desc, void* const* k_layers, void* const* v_layers,
                   float* const* k_scales, float* const* v_scales, kv_pool** out) {
    if (!out) return KV_ERR_INVALID_ARG;
    *out = nullptr;
    if (!valid_desc(desc) || !k_layers || !v_layers) return KV_ERR_INVALID_ARG;
    const bool fp8 = desc->dtype == KV_FP8_E4M3;
    if (fp8 != (k_scales != nullptr) || fp8 != (v_scales != nullptr)) return KV_ERR_INVALID_ARG;
    const int L = desc->num_layers;
    for (int l = 0; l < L; ++l) {
        if (!k_layers[l] || !v_layers[l] || !kvp::aligned16(k_layers[l]) || !kvp::aligned16(v_layers[l]))
            return KV_ERR_INVALID_ARG;
        if (fp8 && (!k_scales[l] || !v_scales[l] || !kvp::aligned16(k_scales[l]) ||
                    !kvp::aligned16(v_scales[l])))
            return KV_ERR_INVALID_ARG;
    }
    kv_pool* p = new (std::nothrow) kv_pool{};
    if (!p) return KV_ERR_INVALID_ARG;
    p->desc = *desc;
    p->k_layers = static_cast<void**>(std::calloc(L, sizeof(void*)));
    p->v_layers = static_cast<void**>(std::calloc(L, sizeof(void*)));
    if (fp8) {
        p->k_scales = static_cast<float**>(std::calloc(L, sizeof(float*)));
        p->v_scales = static_cast<float**>(std::calloc(L, sizeof(float*)));
    }
    if (!p->k_layers || !p->v_layers || (fp8 && (!p->k_scales || !p->v_scales))) {
        free_pool(p);
        return KV_ERR_INVALID_ARG;
    }
    std::memcpy(p->k_layers, k_layers, L * sizeof(void*));
    std::memcpy(p->v_layers, v_layers, L * sizeof(void*));
    if (fp8) {
        std::memcpy(p->k_scales, k_scales, L * sizeof(float*));
        std::memcpy(p->v_scales, v_scales, L * sizeof(float*));
    }
    if (cudaGetDevice(&p->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess ||
        cudaMalloc(&p->d_err, sizeof(int)) != cudaSuccess) {
        free_pool(p);
        return KV_ERR_CUDA;
    }
    if (cudaMemset(p->d_err, 0, sizeof(int)) != cudaSuccess) {
        cudaFree(p->d_err);
        free_pool(p);
        return KV_ERR_CUDA;
    }
    make_tensor_maps(p);
    *out = p;
    return KV_OK;
}

int kv_pool_destroy(kv_pool* pool) {
    if (!pool) return KV_ERR_INVALID_ARG;
    int rc = cudaFree(pool->d_err) == cudaSuccess ? KV_OK : KV_ERR_CUDA;
    free_pool(pool);
    return rc;
}

int kv_pool_get_desc(const kv_pool* pool, kv_pool_desc* desc) {
    if (!pool || !desc) return KV_ERR_INVALID_ARG;
    *desc = pool->desc;
    return KV_OK;
}

int kv_pool_features(const kv_pool* pool, unsigned* flags) {
    if (!pool || !flags) return KV_ERR_INVALID_ARG;
    *flags = pool->tmaps ? KV_FEATURE_TENSOR_MAPS : 0u;
    return KV_OK;
}

int kv_selftest_wait_timeout(kv_pool* pool, uint64_t limit_ns, kv_stream_t stream) {
    if (!pool || limit_ns < 1 || limit_ns > 1000000000ull) return KV_ERR_INVALID_ARG;
    return kvp::launch_selftest_wait(pool, limit_ns, static_cast<cudaStream_t>(stream));
}

int kv_get_device_error(kv_pool* pool, kv_stream_t stream, int clear, int* code) {
    if (!pool || !code) return KV_ERR_INVALID_ARG;
    int h = 0;
    if (cudaMemcpyAsync(&h, pool->d_err, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return KV_ERR_CUDA;
    if (clear && cudaMemsetAsync(pool->d_err, 0, sizeof(int), stream) != cudaSuccess) return KV_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return KV_ERR_CUDA;
    *code = h;
    return h ? KV_ERR_DEVICE : KV_OK;
}

int kv_append(kv_pool* pool, int layer, const void* k, const void* v, kv_dtype in_dtype,
              const int64_t* slot_mapping, int num_tokens, kv_stream_t stream) {
    if (!pool || layer < 0 || layer >= pool->desc.num_layers || num_tokens < 0) return KV_ERR_INVALID_ARG;
    if (num_tokens == 0) return KV_OK;
    if (!k || !v || !slot_mapping || !kvp::aligned16(k) || !kvp::aligned16(v)) return KV_ERR_INVALID_ARG;
    const kv_dtype pd = pool->desc.dtype;
    if (pd == KV_FP8_E4M3) {
        if (in_dtype != KV_F16 && in_dtype != KV_F32) return KV_ERR_INVALID_ARG;
    } else if (in_dtype != pd) {
        return KV_ERR_INVALID_ARG;
    }
    return kvp::launch_append(pool, layer, k, v, in_dtype, slot_mapping, num_tokens, stream);
}

int kv_copy_blocks(kv_pool* pool, const int32_t* pairs, int num_pairs, int layer_begin,
                   int layer_end, kv_stream_t stream) {
    if (!pool || num_pairs < 0 || layer_begin < 0 || layer_end < layer_begin ||
        layer_end > pool->desc.num_layers)
        return KV_ERR_INVALID_ARG;
    if (num_pairs == 0 || layer_end == layer_begin) return KV_OK;
    if (!pairs || num_pairs > 65535) return KV_ERR_INVALID_ARG;
    return kvp::launch_copy_blocks(pool, pairs, num_pairs, layer_begin, layer_end, stream);
}

size_t paged_decode_workspace_size(const kv_pool* pool, int batch, int max_context,
                                   int partition_tokens) {
    if (!pool) return 0;
    kvp::AttnPlan plan;
    if (kvp::plan_attention(pool, batch, max_context, partition_tokens, &plan) != KV_OK) return 0;
    return plan.ws_bytes;
}

int paged_decode_attention(kv_pool* pool, int layer, const void* q, float* out,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, int batch, int max_context,
                           float scale, int partition_tokens, void* workspace,
                           size_t workspace_bytes, kv_stream_t stream) {
    if (!pool || layer < 0 || layer >= pool->desc.num_layers || batch < 0 || max_context < 0)
        return KV_ERR_INVALID_ARG;
    if (batch == 0) return KV_OK;
    if (!q || !out || !block_tables || !context_lens || !workspace || max_blocks_per_seq < 1)
        return KV_ERR_INVALID_ARG;
    if (!kvp::aligned16(q) || !kvp::aligned16(out) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return KV_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !(scale < 3.0e38f)) return KV_ERR_INVALID_ARG;
    kvp::AttnPlan plan;
    int rc = kvp::plan_attention(pool, batch, max_context, partition_tokens, &plan);
    if (rc != KV_OK) return rc;
    if (workspace_bytes < plan.ws_bytes) return KV_ERR_INVALID_ARG;
    return kvp::launch_attention(pool, layer, q, out, block_tables, max_blocks_per_seq, context_lens,
                                 batch, max_context, scale, plan, workspace, stream);
}

int paged_decode_attention_append(kv_pool* pool, int layer, const void* q, const void* k_new,
                                  const void* v_new, kv_dtype in_dtype, float* out,
                                  const int32_t* block_tables, int max_blocks_per_seq,
                                  const int32_t* context_lens, int batch, int max_context, float scale,
                                  int partition_tokens, void* workspace, size_t workspace_bytes,
                                  kv_stream_t stream) {
    if (!pool || layer < 0 || layer >= pool->desc.num_layers || batch < 0 || max_context < 0)
        return KV_ERR_INVALID_ARG;
    if (batch == 0) return KV_OK;
    if (!q || !k_new || !v_new || !out || !block_tables || !context_lens || !workspace ||
        max_blocks_per_seq < 1)
        return KV_ERR_INVALID_ARG;
    if (!kvp::aligned16(q) || !kvp::aligned16(out) || !kvp::aligned16(k_new) || !kvp::aligned16(v_new) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return KV_ERR_INVALID_ARG;
    const kv_dtype pd = pool->desc.dtype;
    if (pd == KV_FP8_E4M3) {
        if (in_dtype != KV_F16 && in_dtype != KV_F32) return KV_ERR_INVALID_ARG;
    } else if (in_dtype != pd) {
        return KV_ERR_INVALID_ARG;
    }
    if (!(scale > 0.f) || !(scale < 3.0e38f)) return KV_ERR_INVALID_ARG;
    kvp::AttnPlan plan;
    int rc = kvp::plan_attention(pool, batch, max_context, partition_tokens, &plan);
    if (rc != KV_OK) return rc;
    if (workspace_bytes < plan.ws_bytes) return KV_ERR_INVALID_ARG;
    return kvp::launch_attention_append(pool, layer, q, k_new, v_new, kvp::elem_bytes(in_dtype), out,
                                        block_tables, max_blocks_per_seq, context_lens, batch,
                                        max_context, scale, plan, workspace, stream);
}

size_t paged_decode_workspace_size_gqa(const kv_pool* pool, int batch, int num_q_heads, int max_context,
                                       int partition_tokens) {
    if (!pool || num_q_heads < 1 || num_q_heads % pool->desc.num_heads != 0) return 0;
    kvp::AttnPlan plan;
    if (kvp::plan_attention(pool, batch, max_context, partition_tokens, &plan,
                            num_q_heads / pool->desc.num_heads) != KV_OK)
        return 0;
    return plan.ws_bytes;
}

int paged_decode_attention_gqa(kv_pool* pool, int layer, const void* q, int num_q_heads,
                               const void* k_new, const void* v_new, kv_dtype in_dtype, float* out,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, int batch, int max_context, float scale,
                               int partition_tokens, void* workspace, size_t workspace_bytes,
                               kv_stream_t stream) {
    if (!pool || layer < 0 || layer >= pool->desc.num_layers || batch < 0 || max_context < 0)
        return KV_ERR_INVALID_ARG;
    if (num_q_heads < 1 || num_q_heads % pool->desc.num_heads != 0) return KV_ERR_INVALID_ARG;
    const int group = num_q_heads / pool->desc.num_heads;
    if (!kvp::valid_group(pool->desc, group)) return KV_ERR_INVALID_ARG;
    if (batch == 0) return KV_OK;
    if (!q || !out || !block_tables || !context_lens || !workspace || max_blocks_per_seq < 1)
        return KV_ERR_INVALID_ARG;
    if ((k_new == nullptr) != (v_new == nullptr)) return KV_ERR_INVALID_ARG;
    if (!kvp::aligned16(q) || !kvp::aligned16(out) || (k_new && (!kvp::aligned16(k_new) || !kvp::aligned16(v_new))) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return KV_ERR_INVALID_ARG;
    if (k_new) {
        const kv_dtype pd = pool->desc.dtype;
        if (pd == KV_FP8_E4M3) {
            if (in_dtype != KV_F16 && in_dtype != KV_F32) return KV_ERR_INVALID_ARG;
        } else if (in_dtype != pd) {
            return KV_ERR_INVALID_ARG;
        }
    }
    if (!(scale > 0.f) || !(scale < 3.0e38f)) return KV_ERR_INVALID_ARG;
    kvp::AttnPlan plan;
    int rc = kvp::plan_attention(pool, batch, max_context, partition_tokens, &plan, group);
    if (rc != KV_OK) return rc;
    if (workspace_bytes < plan.ws_bytes) return KV_ERR_INVALID_ARG;
    return kvp::launch_attention_append(pool, layer, q, k_new, v_new, k_new ? kvp::elem_bytes(in_dtype) : 0,
                                        out, block_tables, max_blocks_per_seq, context_lens, batch,
                                        max_context, scale, plan, workspace, stream);
}

size_t paged_decode_workspace_size_ex(const kv_pool* pool, const kv_decode_args* x) {
    if (!pool || !x) return 0;
    const int hq = x->num_q_heads ? x->num_q_heads : pool->desc.num_heads;
    if (hq < 1 || hq % pool->desc.num_heads != 0) return 0;
    kvp::AttnPlan plan;
    if (x->num_prefix_groups > 0) {
        if (hq != pool->desc.num_heads || x->window != 0 ||
            kvp::plan_attention_prefix(pool, x->batch, x->max_context, x->partition_tokens, &plan) != KV_OK)
            return 0;
        return plan.ws_bytes;
    }
    if (kvp::plan_attention(pool, x->batch, x->max_context, x->partition_tokens, &plan,
                            hq / pool->desc.num_heads, x->window) != KV_OK)
        return 0;
    return plan.ws_bytes;
}

int paged_decode_attention_ex(kv_pool* pool, const kv_decode_args* x) {
    if (!pool || !x) return KV_ERR_INVALID_ARG;
    if (x->layer < 0 || x->layer >= pool->desc.num_layers || x->batch < 0 || x->max_context < 0 ||
        x->window < 0)
        return KV_ERR_INVALID_ARG;
    const int hq = x->num_q_heads ? x->num_q_heads : pool->desc.num_heads;
    if (hq < 1 || hq % pool->desc.num_heads != 0) return KV_ERR_INVALID_ARG;
    const int group = hq / pool->desc.num_heads;
    if (!kvp::valid_group(pool->desc, group)) return KV_ERR_INVALID_ARG;
    if (x->batch == 0) return KV_OK;
    if (!x->q || !x->out || !x->block_tables || !x->context_lens || !x->workspace || x->max_blocks_per_seq < 1)
        return KV_ERR_INVALID_ARG;
    if ((x->k_new == nullptr) != (x->v_new == nullptr)) return KV_ERR_INVALID_ARG;
    if (!kvp::aligned16(x->q) || !kvp::aligned16(x->out) ||
        (x->k_new && (!kvp::aligned16(x->k_new) || !kvp::aligned16(x->v_new))) ||
        (reinterpret_cast<uintptr_t>(x->workspace) & 255u) != 0)
        return KV_ERR_INVALID_ARG;
    if (x->k_new) {
        const kv_dtype pd = pool->desc.dtype;
        if (pd == KV_FP8_E4M3) {
            if (x->in_dtype != KV_F16 && x->in_dtype != KV_F32) return KV_ERR_INVALID_ARG;
        } else if (x->in_dtype != pd) {
            return KV_ERR_INVALID_ARG;
        }
    }
    if (!(x->scale > 0.f) || !(x->scale < 3.0e38f)) return KV_ERR_INVALID_ARG;
    if (x->flags & ~(KV_DECODE_WORKSPACE_ZEROED | KV_DECODE_PDL | KV_DECODE_EARLY_TABLES | KV_DECODE_OUT_F16 |
                     KV_DECODE_EARLY_POOL))
        return KV_ERR_INVALID_ARG;
    if (x->num_prefix_groups < 0 || (x->num_prefix_groups > 0) != (x->prefix_groups != nullptr) ||
        x->num_prefix_groups > x->batch || (reinterpret_cast<uintptr_t>(x->prefix_groups) & 3u) != 0)
        return KV_ERR_INVALID_ARG;
    kvp::AttnPlan plan;
    int rc;
    if (x->num_prefix_groups > 0) {
        if (group != 1 || x->window != 0) return KV_ERR_UNSUPPORTED;
        rc = kvp::plan_attention_prefix(pool, x->batch, x->max_context, x->partition_tokens, &plan);
        plan.groups = x->prefix_groups;
        plan.n_groups = x->num_prefix_groups;
    } else {
        rc = kvp::plan_attention(pool, x->batch, x->max_context, x->partition_tokens, &plan, group, x->window);
    }
    if (rc != KV_OK) return rc;
    if (x->workspace_bytes < plan.ws_bytes) return KV_ERR_INVALID_ARG;
    plan.flags = x->flags;
    return kvp::launch_attention_append(pool, x->layer, x->q, x->k_new, x->v_new,
                                        x->k_new ? kvp::elem_bytes(x->in_dtype) : 0, x->out, x->block_tables,
                                        x->max_blocks_per_seq, x->context_lens, x->batch, x->max_context,
                                        x->scale, plan, x->workspace, x->stream);
}

int kv_decode_step(kv_alloc* alloc, kv_pool* pool, const int32_t* seqs, int n, int max_blocks,
                   int32_t* staging, int32_t* dev_meta, const void* inputs_h, void* inputs_d,
                   size_t inputs_bytes, void* out_h, size_t out_bytes, const kv_decode_args* args) {
    if (!alloc || !pool || !args || !seqs || n < 1 || max_blocks < 1 || !staging || !dev_meta)
        return KV_ERR_INVALID_ARG;
    if ((inputs_bytes && (!inputs_h || !inputs_d)) || (out_bytes && (!out_h || !args->out)))
        return KV_ERR_INVALID_ARG;
    const int64_t tab = static_cast<int64_t>(n) * max_blocks;
    if (args->batch != n || args->max_blocks_per_seq != max_blocks || args->block_tables != dev_meta ||
        args->context_lens != dev_meta + tab || !args->k_new || !args->v_new ||
        (args->flags & (KV_DECODE_EARLY_TABLES | KV_DECODE_EARLY_POOL)))
        return KV_ERR_INVALID_ARG;
    // every table must still fit max_blocks once this step's token is in it
    const int B = pool->desc.block_size;
    for (int i = 0; i < n; ++i) {
        int len = 0, nb = 0;
        const int rc = kv_alloc_seq_info(alloc, seqs[i], &len, &nb);
        if (rc != KV_OK) return rc;
        if ((static_cast<int64_t>(len) + 1 + B - 1) / B > max_blocks) return KV_ERR_INVALID_ARG;
    }
    int32_t* lens = staging + tab;
    int32_t* pairs = lens + n;
    // the slots themselves reach the kernel through the tables and lengths
    static thread_local std::vector<int64_t> slots;
    slots.resize(static_cast<size_t>(n));
    int n_cow = 0;
    int rc = kv_alloc_decode_step(alloc, seqs, n, slots.data(), pairs, &n_cow);
    if (rc != KV_OK) return rc;
    rc = kv_alloc_build_tables(alloc, seqs, n, staging, max_blocks, lens);
    if (rc != KV_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(args->stream);
    const size_t meta_bytes = sizeof(int32_t) * static_cast<size_t>(tab + 3 * static_cast<int64_t>(n));
    // inputs placed at the same offset after the staging buffer on both sides (at most 256
    // bytes of padding) travel with it in one copy: each copy has a fixed cost in the stream
    // (addresses compared as integers: the buffers are separate allocations)
    const uintptr_t ih = reinterpret_cast<uintptr_t>(inputs_h), sh = reinterpret_cast<uintptr_t>(staging);
    const uintptr_t id = reinterpret_cast<uintptr_t>(inputs_d), sd = reinterpret_cast<uintptr_t>(dev_meta);
    const bool one_copy = inputs_bytes && ih >= sh + meta_bytes && ih <= sh + meta_bytes + 256 &&
                          id >= sd && id - sd == ih - sh;
    const size_t first = one_copy ? static_cast<size_t>(ih - sh) + inputs_bytes : meta_bytes;
    if (cudaMemcpyAsync(dev_meta, staging, first, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return KV_ERR_CUDA;
    if (inputs_bytes && !one_copy &&
        cudaMemcpyAsync(inputs_d, inputs_h, inputs_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return KV_ERR_CUDA;
    if (n_cow > 0) {
        rc = kv_copy_blocks(pool, dev_meta + tab + n, n_cow, 0, pool->desc.num_layers, args->stream);
        if (rc != KV_OK) return rc;
    }
    rc = paged_decode_attention_ex(pool, args);
    if (rc != KV_OK) return rc;
    if (out_bytes && cudaMemcpyAsync(out_h, args->out, out_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return KV_ERR_CUDA;
    return n_cow;
}

size_t kv_swap_bytes(const kv_pool* pool, int num_blocks, int layer_begin, int layer_end) {
    if (!pool || num_blocks < 0 || layer_begin < 0 || layer_end < layer_begin ||
        layer_end > pool->desc.num_layers)
        return 0;
    return kvp::swap_bytes(pool, num_blocks, layer_begin, layer_end);
}

static int swap_common(kv_pool* pool, bool out, const int32_t* blocks, int num_blocks, int layer_begin,
                       int layer_end, void* host, kv_stream_t stream) {
    if (!pool || num_blocks < 0 || layer_begin < 0 || layer_end < layer_begin ||
        layer_end > pool->desc.num_layers || num_blocks > 65535)
        return KV_ERR_INVALID_ARG;
    if (num_blocks == 0 || layer_end == layer_begin) return KV_OK;
    if (!blocks || !host || !kvp::aligned16(host)) return KV_ERR_INVALID_ARG;
    return kvp::launch_swap(pool, out, blocks, num_blocks, layer_begin, layer_end, host, stream);
}

int kv_swap_out(kv_pool* pool, const int32_t* blocks, int num_blocks, int layer_begin, int layer_end,
                void* host_dst, kv_stream_t stream) {
    return swap_common(pool, true, blocks, num_blocks, layer_begin, layer_end, host_dst, stream);
}

int kv_swap_in(kv_pool* pool, const void* host_src, const int32_t* blocks, int num_blocks, int layer_begin,
               int layer_end, kv_stream_t stream) {
    return swap_common(pool, false, blocks, num_blocks, layer_begin, layer_end, const_cast<void*>(host_src),
                       stream);
}

}  // extern "C"
