// kv_append (slot-mapped cache write) and kv_copy_blocks (copy-on-write block copy).
//
// Append: "大模型推理加速——KV Cache篇" §3.1 writes the new token's K/V into the
// cache at its position before attention reads the cache; "KV Cache与PagedAttention"
// §3.3 (write_KV_to_block) writes into the sequence's current physical block.  The
// host turns (sequence, position) into a slot id = block * B + offset.
// FP8 append: "KV缓存机制解析" §8 stores history K/V in 8-bit floats with a scaling
// factor; the stored code is RNE-satfinite(x / scale[block]).
// Copy: "KV Cache与PagedAttention" §3.3 copy_block — the whole physical block.

#include "kvp_internal.cuh"

namespace kvp {
namespace {

// One CTA per token; threads stride over the token's H*D elements in 16-byte input
// vectors.  Pool offset of (block, head h, offset, j): ((block*H + h)*B + offset)*D + j.
template <typename TIn, typename TOut>
__global__ void __launch_bounds__(256) append_kernel(
    const TIn* __restrict__ k, const TIn* __restrict__ v, const int64_t* __restrict__ slots,
    TOut* __restrict__ kpool, TOut* __restrict__ vpool, const float* __restrict__ kscale,
    const float* __restrict__ vscale, int H, int D, int B, int64_t num_slots, int* err) {
    const int tok = blockIdx.x;
    const int64_t slot = slots[tok];
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (threadIdx.x == 0) atomicOr(err, KV_DEVERR_SLOT);
        return;
    }
    const int64_t blk = slot / B;
    const int off = static_cast<int>(slot % B);
    constexpr int VEC = 16 / sizeof(TIn);        // input elements per 16-byte vector
    const int n_vec = H * D / VEC;
    const TIn* ksrc = k + static_cast<int64_t>(tok) * H * D;
    const TIn* vsrc = v + static_cast<int64_t>(tok) * H * D;
    float ks = 1.f, vs = 1.f;
    if constexpr (sizeof(TOut) == 1) {
        ks = kscale[blk];
        vs = vscale[blk];
    }
    for (int i = threadIdx.x; i < n_vec; i += blockDim.x) {
        const int e = i * VEC;
        const int h = e / D, j = e % D;
        const int64_t dst = ((blk * H + h) * B + off) * static_cast<int64_t>(D) + j;
        const uint4 kin = *reinterpret_cast<const uint4*>(ksrc + e);
        const uint4 vin = *reinterpret_cast<const uint4*>(vsrc + e);
        if constexpr (sizeof(TOut) == sizeof(TIn)) {
            *reinterpret_cast<uint4*>(kpool + dst) = kin;
            *reinterpret_cast<uint4*>(vpool + dst) = vin;
        } else {
            // FP8 pool: quantise VEC elements with the block's scale.
            const TIn* kx = reinterpret_cast<const TIn*>(&kin);
            const TIn* vx = reinterpret_cast<const TIn*>(&vin);
            uint16_t kq[VEC / 2], vq[VEC / 2];
            #pragma unroll
            for (int u = 0; u < VEC / 2; ++u) {
                const float k0 = __fdiv_rn(static_cast<float>(kx[2 * u]), ks);
                const float k1 = __fdiv_rn(static_cast<float>(kx[2 * u + 1]), ks);
                const float v0 = __fdiv_rn(static_cast<float>(vx[2 * u]), vs);
                const float v1 = __fdiv_rn(static_cast<float>(vx[2 * u + 1]), vs);
                kq[u] = float2_to_e4m3x2(k0, k1);
                vq[u] = float2_to_e4m3x2(v0, v1);
            }
            if constexpr (VEC == 8) {
                *reinterpret_cast<uint2*>(kpool + dst) = *reinterpret_cast<uint2*>(kq);
                *reinterpret_cast<uint2*>(vpool + dst) = *reinterpret_cast<uint2*>(vq);
            } else {
                *reinterpret_cast<uint32_t*>(kpool + dst) = *reinterpret_cast<uint32_t*>(kq);
                *reinterpret_cast<uint32_t*>(vpool + dst) = *reinterpret_cast<uint32_t*>(vq);
            }
        }
    }
}

constexpr int kMaxCopyLayers = 64;
struct LayerPtrs {
    void* k[kMaxCopyLayers];
    void* v[kMaxCopyLayers];
    float* ks[kMaxCopyLayers];
    float* vs[kMaxCopyLayers];
};

// grid = (pairs, layers, 2 [K or V]).  Each CTA copies one block tensor of
// `block_bytes` (a multiple of 16) with 16-byte loads/stores; the FP8 scale goes along.
__global__ void __launch_bounds__(256) copy_blocks_kernel(
    const int32_t* __restrict__ pairs, LayerPtrs ptrs, int64_t block_bytes, int num_blocks, int* err) {
    const int pair = blockIdx.x, layer = blockIdx.y, which = blockIdx.z;
    const int src = pairs[2 * pair], dst = pairs[2 * pair + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && layer == 0 && which == 0) atomicOr(err, KV_DEVERR_BLOCK_ID);
        return;
    }
    char* base = static_cast<char*>(which == 0 ? ptrs.k[layer] : ptrs.v[layer]);
    const uint4* s = reinterpret_cast<const uint4*>(base + static_cast<int64_t>(src) * block_bytes);
    uint4* d = reinterpret_cast<uint4*>(base + static_cast<int64_t>(dst) * block_bytes);
    const int64_t n = block_bytes / 16;
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) d[i] = s[i];
    if (threadIdx.x == 0) {
        float* sc = which == 0 ? ptrs.ks[layer] : ptrs.vs[layer];
        if (sc) sc[dst] = sc[src];
    }
}

// Swap: grid = (blocks, layers, 2 [K or V]).  Each CTA moves one block tensor between the
// pool and its slot in a pinned host image (reached through its device mapping), 16 bytes
// per access.  Image layout: [block i][layer l][K, V][block_bytes], then the FP8 scales
// [block i][layer l][K, V] as float32.
template <bool OUT>
__global__ void __launch_bounds__(256) swap_kernel(const int32_t* __restrict__ blocks, LayerPtrs ptrs,
                                                   char* image, int64_t block_bytes, int nblocks_listed,
                                                   int nl, int num_blocks, int* err) {
    const int i = blockIdx.x, layer = blockIdx.y, which = blockIdx.z;
    const int b = blocks[i];
    if (b < 0 || b >= num_blocks) {
        if (threadIdx.x == 0 && layer == 0 && which == 0) atomicOr(err, KV_DEVERR_BLOCK_ID);
        return;
    }
    char* pool = static_cast<char*>(which == 0 ? ptrs.k[layer] : ptrs.v[layer]) + static_cast<int64_t>(b) * block_bytes;
    char* img = image + ((static_cast<int64_t>(i) * nl + layer) * 2 + which) * block_bytes;
    uint4* dst = reinterpret_cast<uint4*>(OUT ? img : pool);
    const uint4* src = reinterpret_cast<const uint4*>(OUT ? pool : img);
    const int64_t n = block_bytes / 16;
    for (int64_t k = threadIdx.x; k < n; k += blockDim.x) dst[k] = src[k];
    if (threadIdx.x == 0) {
        float* sc = which == 0 ? ptrs.ks[layer] : ptrs.vs[layer];
        if (sc) {
            float* img_sc = reinterpret_cast<float*>(image + static_cast<int64_t>(nblocks_listed) * nl * 2 * block_bytes) +
                            (static_cast<int64_t>(i) * nl + layer) * 2 + which;
            if (OUT) *img_sc = sc[b];
            else sc[b] = *img_sc;
        }
    }
}

}  // namespace

int launch_append(const kv_pool* pool, int layer, const void* k, const void* v, kv_dtype in_dtype,
                  const int64_t* slot_mapping, int num_tokens, cudaStream_t stream) {
    const kv_pool_desc& d = pool->desc;
    if (num_tokens == 0) return KV_OK;
    const dim3 grid(num_tokens), block(128);
    const int64_t num_slots = static_cast<int64_t>(d.num_blocks) * d.block_size;
    void* kp = pool->k_layers[layer];
    void* vp = pool->v_layers[layer];
    if (d.dtype == KV_F32) {
        append_kernel<float, float><<<grid, block, 0, stream>>>(
            static_cast<const float*>(k), static_cast<const float*>(v), slot_mapping,
            static_cast<float*>(kp), static_cast<float*>(vp), nullptr, nullptr, d.num_heads,
            d.head_dim, d.block_size, num_slots, pool->d_err);
    } else if (d.dtype == KV_F16) {
        append_kernel<__half, __half><<<grid, block, 0, stream>>>(
            static_cast<const __half*>(k), static_cast<const __half*>(v), slot_mapping,
            static_cast<__half*>(kp), static_cast<__half*>(vp), nullptr, nullptr, d.num_heads,
            d.head_dim, d.block_size, num_slots, pool->d_err);
    } else if (in_dtype == KV_F16) {
        append_kernel<__half, uint8_t><<<grid, block, 0, stream>>>(
            static_cast<const __half*>(k), static_cast<const __half*>(v), slot_mapping,
            static_cast<uint8_t*>(kp), static_cast<uint8_t*>(vp), pool->k_scales[layer],
            pool->v_scales[layer], d.num_heads, d.head_dim, d.block_size, num_slots, pool->d_err);
    } else {
        append_kernel<float, uint8_t><<<grid, block, 0, stream>>>(
            static_cast<const float*>(k), static_cast<const float*>(v), slot_mapping,
            static_cast<uint8_t*>(kp), static_cast<uint8_t*>(vp), pool->k_scales[layer],
            pool->v_scales[layer], d.num_heads, d.head_dim, d.block_size, num_slots, pool->d_err);
    }
    return cudaGetLastError() == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

int launch_copy_blocks(const kv_pool* pool, const int32_t* pairs, int num_pairs, int layer_begin,
                       int layer_end, cudaStream_t stream) {
    const kv_pool_desc& d = pool->desc;
    if (num_pairs == 0 || layer_end == layer_begin) return KV_OK;
    const int64_t block_bytes =
        static_cast<int64_t>(d.num_heads) * d.block_size * d.head_dim * elem_bytes(d.dtype);
    for (int l0 = layer_begin; l0 < layer_end; l0 += kMaxCopyLayers) {
        const int nl = (layer_end - l0) < kMaxCopyLayers ? (layer_end - l0) : kMaxCopyLayers;
        LayerPtrs p{};
        for (int i = 0; i < nl; ++i) {
            p.k[i] = pool->k_layers[l0 + i];
            p.v[i] = pool->v_layers[l0 + i];
            p.ks[i] = pool->k_scales ? pool->k_scales[l0 + i] : nullptr;
            p.vs[i] = pool->v_scales ? pool->v_scales[l0 + i] : nullptr;
        }
        copy_blocks_kernel<<<dim3(num_pairs, nl, 2), 256, 0, stream>>>(pairs, p, block_bytes,
                                                                        d.num_blocks, pool->d_err);
        if (cudaGetLastError() != cudaSuccess) return KV_ERR_CUDA;
    }
    return KV_OK;
}

}  // namespace kvp

namespace kvp {

size_t swap_bytes(const kv_pool* pool, int num_blocks, int layer_begin, int layer_end) {
    const kv_pool_desc& d = pool->desc;
    const int64_t block_bytes =
        static_cast<int64_t>(d.num_heads) * d.block_size * d.head_dim * elem_bytes(d.dtype);
    const int64_t nl = layer_end - layer_begin;
    int64_t n = static_cast<int64_t>(num_blocks) * nl * 2 * block_bytes;
    if (d.dtype == KV_FP8_E4M3) n += static_cast<int64_t>(num_blocks) * nl * 2 * sizeof(float);
    return static_cast<size_t>(n);
}

int launch_swap(const kv_pool* pool, bool out, const int32_t* blocks, int num_blocks, int layer_begin,
                int layer_end, void* host, cudaStream_t stream) {
    const kv_pool_desc& d = pool->desc;
    if (num_blocks == 0 || layer_end == layer_begin) return KV_OK;
    if (layer_end - layer_begin > kMaxCopyLayers) return KV_ERR_UNSUPPORTED;
    void* dev = nullptr;
    // the host image must be addressable by the device: pinned memory, or any host memory
    // where the GPU has coherent pageable-memory access
    if (cudaHostGetDevicePointer(&dev, host, 0) != cudaSuccess || !dev) {
        cudaGetLastError();
        return KV_ERR_INVALID_ARG;
    }
    const int64_t block_bytes =
        static_cast<int64_t>(d.num_heads) * d.block_size * d.head_dim * elem_bytes(d.dtype);
    const int nl = layer_end - layer_begin;
    LayerPtrs p{};
    for (int i = 0; i < nl; ++i) {
        p.k[i] = pool->k_layers[layer_begin + i];
        p.v[i] = pool->v_layers[layer_begin + i];
        p.ks[i] = pool->k_scales ? pool->k_scales[layer_begin + i] : nullptr;
        p.vs[i] = pool->v_scales ? pool->v_scales[layer_begin + i] : nullptr;
    }
    const dim3 grid(num_blocks, nl, 2);
    if (out)
        swap_kernel<true><<<grid, 256, 0, stream>>>(blocks, p, static_cast<char*>(dev), block_bytes, num_blocks,
                                                    nl, d.num_blocks, pool->d_err);
    else
        swap_kernel<false><<<grid, 256, 0, stream>>>(blocks, p, static_cast<char*>(dev), block_bytes, num_blocks,
                                                     nl, d.num_blocks, pool->d_err);
    return cudaGetLastError() == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

namespace {
// One warp waits on an mbarrier that nothing arrives at, through the same bounded wait the
// attention kernel uses: the wait gives up after limit_ns, sets KV_DEVERR_TIMEOUT and the
// kernel returns normally.
__global__ void selftest_wait_kernel(uint64_t limit_ns, int* err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    __syncwarp();
    mbar_wait_bounded(smem_u32(&bar), 0, err, limit_ns);
}
}  // namespace

int launch_selftest_wait(const kv_pool* pool, uint64_t limit_ns, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(limit_ns, pool->d_err);
    return cudaGetLastError() == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

}  // namespace kvp
