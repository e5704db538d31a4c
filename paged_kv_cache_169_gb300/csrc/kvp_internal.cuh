// Internal declarations shared by the kvpaged CUDA translation units.
#pragma once

#include <cuda.h>            // CUtensorMap (the encode entry point is fetched at run time)
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvpaged.h"

struct kv_pool {
    kv_pool_desc desc;
    int device;
    int num_sms;
    void** k_layers;     // host copies of the caller's per-layer device pointers
    void** v_layers;
    float** k_scales;    // FP8 pools only, else nullptr
    float** v_scales;
    int* d_err;          // device error bits (the library's only allocation)
    // fp16, head_dim 128 pools: per layer a K and a V tensor map of the pool viewed as
    // [rows = num_blocks*H*B][2][64] halves with a {64, 2, min(B,16)} box and 128-byte
    // swizzle (the grouped-query tensor-core path); nullptr when unavailable
    CUtensorMap* tmaps;  // [2 * num_layers], 64-byte aligned
    // the same views with boxes of 2*B rows (a block's tiles of two adjacent heads) for the
    // head-pair stages: fp16 pools with B <= 16 and FP8 pools; nullptr otherwise
    CUtensorMap* pmaps;  // [2 * num_layers]
    void* tmaps_raw;
};

namespace kvp {

inline int elem_bytes(kv_dtype t) { return t == KV_F32 ? 4 : (t == KV_F16 ? 2 : 1); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- launchers
int launch_append(const kv_pool* pool, int layer, const void* k, const void* v, kv_dtype in_dtype,
                  const int64_t* slot_mapping, int num_tokens, cudaStream_t stream);
int launch_copy_blocks(const kv_pool* pool, const int32_t* pairs, int num_pairs, int layer_begin,
                       int layer_end, cudaStream_t stream);
size_t swap_bytes(const kv_pool* pool, int num_blocks, int layer_begin, int layer_end);
int launch_swap(const kv_pool* pool, bool out, const int32_t* blocks, int num_blocks, int layer_begin,
                int layer_end, void* host, cudaStream_t stream);

// Split-context partials merge in one step up to this many partitions per (sequence,
// head); longer splits merge in two levels (groups of kMergeFan, then the groups).
constexpr int kMergeFan = 16;
inline int merge_groups(int max_parts) { return max_parts > kMergeFan ? (max_parts + kMergeFan - 1) / kMergeFan : 0; }

// Start of every decode workspace: kMaxSub work counters, then kMaxSub exit counters
// (u32 each); the arrival counters and the partials follow.
constexpr size_t kCounterBytes = 512;

struct AttnPlan {
    unsigned flags = 0;  // KV_DECODE_* of the call (kv_decode_args.flags)
    int partition;       // tokens per split-context partition
    int fine_partition;  // tokens per partition of the sequences from fine_from on
    int fine_from;       // first sequence with the finer partitions (batch: none)
    int alt_partition;   // < partition: the kernel takes it when that still fits one round of items
    int max_parts;       // ceil(max_context / smallest partition)
    int consumers;       // consumer warps per CTA
    int group;           // query heads per KV head
    int window;          // > 0: sliding window of the last `window` tokens
    bool pairs = false;  // tensor-core consumer with head-pair stages
    const int32_t* groups = nullptr;   // shared prompt prefixes: device [n_groups][3], or none
    int n_groups = 0;
    size_t ws_bytes;     // workspace bytes
    // zero-initialised counters after the kCounterBytes of work counters: the per-(sequence, head)
    // arrivals, then the per-partition-group arrivals
    size_t arrivals_bytes(int batch, int heads) const {
        if (max_parts <= 1) return 0;
        const size_t units = static_cast<size_t>(batch) * heads;
        return ((units * 4 + 255) & ~size_t(255)) + ((units * merge_groups(max_parts) * 4 + 255) & ~size_t(255));
    }
};
// group: query heads per KV head (1, or 2/4/8 for fp16 and FP8 pools)
bool valid_group(const kv_pool_desc& d, int group);
// whether a tensor-core launch on this pool (prefix: with shared prompt prefixes) uses
// head-pair stages
bool pair_stages(const kv_pool* pool, bool prefix);
// heads per work item of this pool's single-query decode (1, 2 or 4)
int head_group(const kv_pool_desc& d, int group);
int plan_attention(const kv_pool* pool, int batch, int max_context, int partition_tokens,
                   AttnPlan* plan, int group = 1, int window = 0);
// Plan of a call with shared prompt prefixes (one query per head, tensor-map pools only;
// KV_ERR_UNSUPPORTED otherwise).  The caller sets plan->groups and n_groups.
int plan_attention_prefix(const kv_pool* pool, int batch, int max_context, int partition_tokens,
                          AttnPlan* plan);
int launch_attention(const kv_pool* pool, int layer, const void* q, float* out,
                     const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                     int batch, int max_context, float scale, const AttnPlan& plan,
                     void* workspace, cudaStream_t stream);
// Same, with the fused append of each sequence's newest token (k_new/v_new [batch][H][D]).
int launch_attention_append(const kv_pool* pool, int layer, const void* q, const void* k_new,
                            const void* v_new, int in_bytes, void* out, const int32_t* block_tables,
                            int max_blocks, const int32_t* context_lens, int batch, int max_context,
                            float scale, const AttnPlan& plan, void* workspace, cudaStream_t stream);

// ---------------------------------------------------------------- device helpers
#ifdef __CUDACC__

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for completion of the phase with the given parity, for at most ~1 s.
// On time-out: set KV_DEVERR_TIMEOUT in *err and return false (no trap, no hang).
constexpr uint64_t kWaitLimitNs = 1000000000ull;
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, int* err,
                                                  uint64_t limit_ns = kWaitLimitNs) {
    #pragma unroll 1
    for (int i = 0; i < 256; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    #pragma unroll 1
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(err, KV_DEVERR_TIMEOUT);
            return false;
        }
    }
}

int launch_selftest_wait(const kv_pool* pool, uint64_t limit_ns, cudaStream_t stream);

// 1-D bulk copy global -> shared (the issuing CTA's own shared memory), completion
// counted in bytes on the mbarrier.  dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// 3-D tiled bulk tensor load global -> shared through a tensor map (param/const/global
// address), completion counted on the mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int x, int y, int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// Four 8x8 b16 matrices from shared memory (lane L gives row L%8 of matrix L/8).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}

// Two 16x16 byte matrices from shared memory, transposed (lanes 0-15 give the 16 row
// addresses of the first, lanes 16-31 of the second).  Lane 4g+t receives, of each
// matrix, the bytes of column g in rows 4t..4t+3 (r[0], r[2]) and of column g+8 in rows
// 4t..4t+3 (r[1], r[3]), in row order.
__device__ __forceinline__ void ldsm_b8_x2_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m16n16.x2.trans.shared.b8 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}

// D += A(16x16, fp16, row) * B(16x8, fp16, col) with fp32 accumulation.
// Transpose of an 8x8 b16 matrix held one row pair per lane (lane 4r + c: row r, cols 2c, 2c+1).
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t r;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
    return r;
}

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Arrival ticket with acquire-release semantics at GPU scope: the partials this warp wrote
// (ordered before the call by __syncwarp) are visible to whoever draws a later ticket, and
// the caller sees every partial released before its own ticket.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two E4M3 bytes (low byte = first element) -> two floats, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_half2_bits(uint16_t v) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
    return h2;
}

__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t v) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
    __half2 h = *reinterpret_cast<__half2*>(&h2);
    return __half22float2(h);
}

// Two floats -> two E4M3 bytes (low byte = a), round to nearest even, saturating.
__device__ __forceinline__ uint16_t float2_to_e4m3x2(float a, float b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return r;
}

#endif  // __CUDACC__

}  // namespace kvp
