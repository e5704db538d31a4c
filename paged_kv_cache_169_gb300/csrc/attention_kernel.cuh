// Decode-attention kernel template (shared by the MHA and grouped-query translation
// units).
//
// paged_decode_attention: one query token per (sequence, head) against that
// sequence's cached K/V, read through its block table.
//
// What is computed ("大模型推理加速——KV Cache篇" §3.1; "KV缓存机制解析" §5.1):
//   out[s,h] = softmax_t(scale * q[s,h] . K[s,t,h]) . V[s,t,h],  t < context_lens[s]
// with the cache stored in fixed-size physical blocks found through a block table
// ("KV Cache与PagedAttention" §2.1, §3.2).  The page's kernel sketch loads each
// block into shared memory and attends block by block; here the same idea is laid
// out for sm_103a:
//
// * Work items are (sequence, head, partition) triples (a head pair or quad for pools
//   with small tiles); a partition is at most P tokens (split-context, flash-decoding
//   style).  Items are handed out dynamically with one atomic counter, so ragged
//   batches balance.
// * Each CTA is persistent (one per SM): warps 0..NC-1 are consumers, warp NC is the
//   producer.  Producer lane w serves consumer w: it polls that consumer's ring without
//   blocking, and for every physical block of the next CT-token chunk issues one 1-D
//   bulk copy (cp.async.bulk, the TMA engine) of the contiguous (block, head) K tile
//   and one of the V tile into the ring stage, completing on the stage's mbarrier (the
//   tensor-core consumer's tiles come through swizzling tensor-map copies instead).
//   Block-table entries are fetched one chunk ahead, work items one item ahead.
// * A consumer warp owns NSW ring stages.  Its two half-warps read two token rows per
//   16-byte shared-memory load (lane: head_dim/16 dims of one row).  Each lane forms
//   partial dot products for its CT/2 tokens; a transpose-reduce over the 16 lanes of
//   a half leaves one token's score per lane.  Softmax runs in fp32 in the log2
//   domain with a running maximum that is only raised (and the state rescaled) when
//   some score exceeds it by more than 8; V is accumulated in fp32 with p_t broadcast
//   by shuffle, and the two halves are summed once per item.  ("KV Cache篇" §6.3:
//   tiles in on-chip SRAM, softmax state kept on chip.)
// * A sequence that fits one partition is normalised and written directly; longer
//   ones write (m, l, o) partials.  Each (sequence, head) counts its finished
//   partitions with an atomic ticket; the warp that finishes the last one merges them
//   (exact log-sum-exp merge) — no second kernel, and no warp ever waits for another.
//
// One query row per head is a matrix-vector product bound by HBM: it runs on the CUDA
// cores.  Grouped queries (G query heads per K/V head) make each K and V tile a small
// dense contraction: for fp16 and FP8 pools with head_dim 128 it runs on the tensor
// cores (consumer_mma below).

#pragma once

#include <math_constants.h>

#include "kvp_internal.cuh"

namespace kvp {

struct AttnArgs {
    CUtensorMap kmap;      // tensor-core path: the layer's K and V as swizzled tiles
    CUtensorMap vmap;
    char* kpool;           // written only by the fused append (the new token's slot)
    char* vpool;
    const float* kscale;
    const float* vscale;
    const void* q;
    void* out;             // [batch][H*G][D]: float, or __half when out_f16
    const int32_t* tables;
    const int32_t* lens;
    float* part_ml;        // [batch*H*max_parts][2]  (m in log2 units, l)
    float* part_o;         // [batch*H*max_parts][D]  unnormalised
    unsigned* counter;     // work items claimed so far (this launch)
    unsigned* exit_counter;  // producer warps that have finished (this launch)
    unsigned* arrivals;    // [batch*H] partitions (or partition groups) finished per (sequence, head)
    unsigned* grp_arrivals;  // [batch*H][n_grp] partitions finished per group of kMergeFan
    int n_grp;             // ceil(max_parts / kMergeFan) when max_parts > kMergeFan, else 0
    const char* k_new;     // fused append: [batch][H][D] new-token K (nullptr: no append)
    const char* v_new;
    int in_bytes;          // element size of k_new / v_new (2 or 4)
    int window;            // > 0: attend only to the last `window` tokens of each sequence
    int* err;
    int batch, H, B, max_blocks, ctx_limit, P, max_parts, num_blocks;
    int P_fine, s_fine;    // sequences s >= s_fine split into partitions of P_fine tokens (< P)
    int P_alt;             // < P: use P_alt instead when it still gives at most one item per consumer warp
    int early_tables;      // lens and tables may be read before griddepcontrol.wait (KV_DECODE_EARLY_TABLES)
    int early_pool;        // with early_tables: the first stages may be filled before it (KV_DECODE_EARLY_POOL)
    int out_f16;           // the result is stored as float16, rounded to nearest (KV_DECODE_OUT_F16)
    float qscale;          // scale * log2(e)
    // shared prompt prefixes (Cfg PFX): [n_groups][3] of (first sequence, members, shared
    // tokens), sequence indices of the whole call; s_base = this sub-launch's first sequence
    const int32_t* groups;
    int n_groups, s_base, fused;
};

// Launch the grouped-query instantiations (decode_attention_gqa.cu), group in {2, 4, 8}.
int launch_attention_grouped(int group, const kv_pool* pool, const AttnArgs& args, const AttnPlan& plan,
                             unsigned* counters, cudaStream_t stream);

namespace {

constexpr int kMaxBatch = 1024;    // sequences per launch (prefix table in shared memory)
constexpr int kMaxSub = 64;        // launches per call -> batch <= 65536
static_assert(2 * kMaxSub * sizeof(unsigned) <= kCounterBytes, "work + exit counters");
constexpr int kPartAlign = 32;     // partition sizes are multiples of this
#if defined(KVP_CLAIM_LEAD)
constexpr int kClaimLead = KVP_CLAIM_LEAD;   // tuning sweeps only
#else
constexpr int kClaimLead = 6;      // claim the next item this many fills before it is needed
#endif
constexpr unsigned FULL = 0xffffffffu;

enum : int { F_FIRST = 1, F_LAST = 2, F_TERM = 4, F_SINGLE = 8, F_PATCH = 16 };

struct __align__(16) Meta {
    int s, h, p, ntok;      // item (sequence, head, partition); valid tokens in the chunk
    int flags;
    int patch_row;          // F_PATCH: chunk row of the token appended by this call
    int patch_id, patch_off;   // F_PATCH: its physical block and offset inside the block
    int ids[4];             // physical block of each copy in the chunk (FP8: scale lookup)
    int lo;                 // sliding window: chunk rows below lo lie before the window
    int nq;                 // shared prefixes: query rows of the item (sequences s .. s+nq-1)
    int pad[2];
};

// Shared prompt prefixes: per sequence of a launch, the tokens it shares with its group
// (bits 0-23; 0: none) and, for the group's first sequence, the member count (bits 24-27).
constexpr int kPfxTokMask = (1 << 24) - 1;
// A sequence of a prefix group has at most this many partitions (shared part + private
// part); they merge in one step.
constexpr int kPfxMaxParts = 32;

constexpr int round_up(int a, int b) { return (a + b - 1) / b * b; }

// Launch shape per storage type: tokens per chunk (CT), consumer warps per SM (NC), ring
// stages per consumer (NSW).  Compile-time overrides exist only for tuning sweeps
// (KVP_F16_CT/NC/NSW, KVP_FP8_CT/NC/NSW).
template <int ESZ> struct Tune { static constexpr int CT = 32, NC = 0, NSW = 0; };   // 0: by stage size
#if !defined(KVP_F16_CT)
template <> struct Tune<2> { static constexpr int CT = 16, NC = 12, NSW = 0; };
#endif
#if !defined(KVP_FP8_CT)
template <> struct Tune<1> { static constexpr int CT = 32, NC = 12, NSW = 0; };
#endif
#if defined(KVP_F16_CT) && defined(KVP_F16_NC) && defined(KVP_F16_NSW)
template <> struct Tune<2> { static constexpr int CT = KVP_F16_CT, NC = KVP_F16_NC, NSW = KVP_F16_NSW; };
#endif
#if defined(KVP_FP8_CT) && defined(KVP_FP8_NC) && defined(KVP_FP8_NSW)
template <> struct Tune<1> { static constexpr int CT = KVP_FP8_CT, NC = KVP_FP8_NC, NSW = KVP_FP8_NSW; };
#endif
// CTAs per SM by launch shape (overrides: tuning sweeps)
#if !defined(KVP_F16_CPS)
#define KVP_F16_CPS 2              // fp16, one head per item
#endif
#if !defined(KVP_F16P_CPS)
#define KVP_F16P_CPS 2             // fp16, head pairs (B 8)
#endif
#if !defined(KVP_FP8_CPS)
#define KVP_FP8_CPS 2              // FP8, one head or head pairs per item
#endif
#if !defined(KVP_PR_CPS)
#define KVP_PR_CPS 2               // tensor-core head-pair stages, grouped queries
#endif
#if !defined(KVP_PFX_CPS)
#define KVP_PFX_CPS 2              // tensor-core head-pair stages, shared prefixes
#endif

// G_: query heads per KV head (grouped-query attention; 1 = one query per KV head).
// MMA_: grouped-query tensor-core consumer (head_dim 128, G >= 2).  Both pool types are fed
// by 128-byte-swizzled tensor-map copies: fp16 tiles as [2][rows][64] halves, FP8 tiles as
// [rows][128 codes], whose mma fragments are converted from the E4M3 codes in registers.
// HP_ = 2 (one query per KV head only): a work item covers two adjacent heads.  Their
// (block, head) tiles are adjacent in the pool, so one bulk copy brings both: half as many
// copies per byte, which is what limits pools with small tiles (FP8, and fp16 with B = 8).
// The two half-warps take one head each.  BR_ is then the block size (8 or 16), fixed at
// compile time because each copy holds whole blocks of both heads.
// PFX_ (tensor-core consumer, one query per head): shared prompt prefixes.  A work item is
// either (group, head, partition of the shared prefix), whose K/V tiles serve the query rows
// of up to G_ = 8 member sequences at once, or (sequence, head, partition of the tokens after
// the prefix) with one query row.
// PR_ (tensor-core consumer): head-pair stages.  One copy brings a block's tiles of two
// adjacent K/V heads (adjacent in the pool), and the stage is shared by two consumer warps,
// one head each: copies of 2B rows instead of B, half as many copies per byte (the copy
// rate per SM bounds small tiles).  Needs whole blocks per copy (B <= CT).
template <int D_, typename KV_, typename QT_, int G_ = 1, bool MMA_ = false, int HP_ = 1, int BR_ = 0,
          bool PFX_ = false, bool PR_ = false>
struct Cfg {
    static constexpr int D = D_;
    static constexpr int G = G_;
    static constexpr bool MMA = MMA_;
    static constexpr bool PFX = PFX_;
    static constexpr bool PR = PR_;
    static_assert(!PR || MMA, "head-pair stages: tensor-core consumer");
    static_assert(!PFX || (MMA && G == 8), "shared prefixes: tensor-core consumer with 8 query rows");
    // query rows of the output (and of q) per (sequence, KV head)
    static constexpr int GO = PFX ? 1 : G_;
    static constexpr int HP = HP_;
    static constexpr int BR = BR_;
    static constexpr int GE = G_ * HP_;                   // output rows per work item
    static constexpr int KVH = HP_ * (PR_ ? 2 : 1);       // K/V heads per work item (per copy)
    static_assert(!MMA || (sizeof(KV_) <= 2 && D_ == 128 && G_ >= 2), "tensor-core path: fp16 or FP8, d 128, G >= 2");
    static_assert(HP == 1 || ((HP == 2 || HP == 4) && G == 1 && !MMA && (BR == 8 || BR == 16)),
                  "head groups: one query per head");
    using KV = KV_;
    using QT = QT_;
    static constexpr int ESZ = sizeof(KV);
    static constexpr bool FP8 = (ESZ == 1);
    // G*CT/2 sums per lane bound the CUDA-core consumer; the tensor-core consumer takes 16
    // tokens per step (FP8: two steps per 32-token chunk, so a chunk moves as many bytes
    // as an fp16 one).  Head pairs: a chunk of CT tokens of two heads (fp16: 8, FP8: 16),
    // as many bytes as the single-head chunk.
    static constexpr int CT = MMA ? (ESZ == 1 ? 32 : 16)
                                  : HP == 4 ? 8 : HP == 2 ? 16 / ESZ : (G >= 4 ? 16 : Tune<ESZ>::CT);
    static_assert(HP == 1 || BR <= CT, "head pairs: whole blocks per copy");
    static constexpr int TPL = HP >= 2 ? CT : CT / 2;     // tokens per lane per chunk
    static constexpr int LPR = HP == 4 ? 8 : 16;          // lanes per token row
    static constexpr int DPL = D / LPR;                   // dims per lane
    static_assert(TPL <= LPR, "the transpose-reduce leaves one token per lane");
    static constexpr int CBMAX = CT >= 8 ? CT / 8 : 1;    // blocks per chunk at B = 8
    static constexpr int ROW = D * ESZ;                   // bytes of one token row of one head
    static constexpr int KV_BYTES = CT * ROW * KVH;       // bytes of K (or V) per chunk
    static constexpr int Q_BYTES = GE * D * sizeof(QT);   // the query rows of one item
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = KV_BYTES;
    static constexpr int Q_OFF = 2 * KV_BYTES;
    // the fp16 tensor-core path keeps its 1024-aligned stages to exactly K and V (8 KiB):
    // its query rows go to a region of their own, one slot per stage.  The FP8 tensor-core
    // path reads its query rows from global memory once per item.
    static constexpr bool SWZ_STAGE = MMA && !FP8;        // stages hold swizzled tensor-map tiles
    // FP8 tensor-core path: K and V tiles arrive 128-byte swizzled through the layer's 2-D
    // tensor maps, and the mma fragments are built straight from the E4M3 codes
    static constexpr bool SWZ_K = MMA && FP8;
    static constexpr int Q_STAGE = MMA ? 0 : Q_BYTES;
    // head-pair stages take their query rows from global memory (no per-stage slot)
    static constexpr int QR_BYTES = SWZ_STAGE && !PR ? Q_BYTES : 0;
    static constexpr int STAGE = round_up(Q_OFF + Q_STAGE, (SWZ_STAGE || SWZ_K) ? 1024 : 128);
    static constexpr int NC_AUTO = STAGE <= 9 * 1024 ? 8 : (STAGE <= 17 * 1024 ? 4 : 3);
    // CTAs resident per SM.  Two halve the granularity at which an SM passes from one
    // launch to the next under programmatic dependent launch and at which a launch's tail
    // frees SMs: each CTA gets half of the SM's 228 KiB (less the 1 KiB the system keeps
    // per CTA) and half of its consumer warps or rings.  Head quads (FP8, B 8) keep one:
    // half their stages would not double-buffer.
    static constexpr int CPS = (!MMA && G == 1 && HP == 1 && ESZ == 2) ? KVP_F16_CPS
                             : (!MMA && G == 1 && ESZ == 2) ? KVP_F16P_CPS
                             : (!MMA && G == 1 && ESZ == 1 && HP <= 2) ? KVP_FP8_CPS
                             : (PR && !PFX) ? KVP_PR_CPS
                             : (PR && PFX) ? KVP_PFX_CPS : 1;
    // more query heads per warp need more registers: fewer consumer warps
#if defined(KVP_MMA_NC)
    static constexpr int NC_MMA = KVP_MMA_NC;      // tuning sweeps only
#else
    static constexpr int NC_MMA = 7;               // 8 warps: the register cap stays at 255
#endif
#if defined(KVP_PR_RINGS)
    static constexpr int NR_PAIR = KVP_PR_RINGS;   // tuning sweeps only
#else
    // head-pair stages: 4 rings of 2 consumer warps per SM; shared-prefix launches, whose
    // items are few and short, take 2 rings per SM with deeper stages instead (up to 6
    // chunks of an item in flight, most of them fetched before the previous launch ends).
    // The SM's CTAs share them out.
    static constexpr int NR_PAIR = (PFX ? 2 : 4) / CPS;
#endif
    static constexpr int NC = PR ? 2 * NR_PAIR
                                 : MMA ? NC_MMA
                                       : G == 1 ? (Tune<ESZ>::NC ? Tune<ESZ>::NC : NC_AUTO) / CPS
                                                : (G == 2 ? 12 : (G == 4 ? 8 : 6));
    static constexpr int NR = PR ? NR_PAIR : NC;   // rings (one producer lane each)
    // stages that fit beside the prefix table and the barriers
    static constexpr int TABLES = (PFX ? 3 : 2) * kMaxBatch * 4;   // per-sequence launch tables
    // beside the stages: the tables and the reserve (alignment slack, barriers, zero line,
    // launch-wide values)
    static constexpr int RESERVE = 1024 + (MMA ? 2048 : 0);
    static constexpr int SMEM_BUDGET = CPS == 1 ? 227 * 1024 : 228 * 1024 / CPS - 1024;
    static constexpr int NSW_FIT =
        (SMEM_BUDGET - TABLES - RESERVE) /
        (NR * (STAGE + (int)sizeof(Meta) + QR_BYTES));
    // FP8 stages hold twice the tokens per byte; shared-prefix rings are few and deep
    static constexpr int NSW_CAP = (MMA && (FP8 || (PR && PFX))) ? 6 : 4;
    static constexpr int NSW = Tune<ESZ>::NSW && !MMA ? Tune<ESZ>::NSW : (NSW_FIT > NSW_CAP ? NSW_CAP : NSW_FIT);
    static_assert(NSW >= 2, "at least double buffering");
    static_assert(NR >= 1 && NC >= 1, "at least one ring per CTA");
    static constexpr int THREADS = (NC + 1) * 32;
    static constexpr int META_R = NR * NSW * STAGE;                   // one Meta per stage
    static constexpr int QR_OFF = META_R + NR * NSW * (int)sizeof(Meta);   // MMA: one q slot per stage
    static constexpr int BAR_OFF = round_up(QR_OFF + NR * NSW * QR_BYTES, 128);
    static constexpr int PREFIX_OFF = BAR_OFF + 2 * NR * NSW * 8;
    static constexpr int ZERO_OFF = PREFIX_OFF + TABLES;  // 128 zero bytes (FP8 mma: masked rows)
    static constexpr int MISC_OFF = ZERO_OFF + 128;             // launch-wide values (the partition size)
    static constexpr int ALIGN_SLACK = MMA ? 1024 : 0;           // to 1024-align the base
    static constexpr int SMEM = MISC_OFF + 16 + ALIGN_SLACK;
    static_assert(SMEM <= SMEM_BUDGET, "shared memory budget");
    static_assert(NC <= 32 && (CT == 8 || CT == 16 || CT == 32), "launch shape");
    static_assert(Q_OFF % 16 == 0 && META_R % 16 == 0 && QR_OFF % 16 == 0, "alignment");
};



__device__ __forceinline__ int nparts_of(int ctx, int P) { return ctx <= P ? 1 : (ctx + P - 1) / P; }

// Partition size of sequence s under the launch's partition size P: the sequences handed
// out last (s >= s_fine) take finer partitions, so the last round of work items is short
// and the launch ends evenly.
__device__ __forceinline__ int part_of(int P, const AttnArgs& a, int s) { return s >= a.s_fine ? a.P_fine : P; }

// Sliding window: the first attended token, and the first token actually read — rounded
// down to a whole copy unit (rpc rows) so every copy stays inside blocks the window still
// holds.  Rows in [first, start) are read but masked.
__device__ __forceinline__ int attend_start(int ctx, int window) {
    return (window > 0 && ctx > window) ? ctx - window : 0;
}
__device__ __forceinline__ int attend_first(int ctx, int window, int rpc) {
    return attend_start(ctx, window) / rpc * rpc;
}

__device__ __forceinline__ float warp_max(float v) {
    #pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
    #pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
    return v;
}
// over each group of W consecutive lanes (W = 16: half-warps, 8: quarter-warps)
template <int W>
__device__ __forceinline__ float group_max(float v) {
    #pragma unroll
    for (int o = W / 2; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
    return v;
}
template <int W>
__device__ __forceinline__ float group_sum(float v) {
    #pragma unroll
    for (int o = W / 2; o; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
    return v;
}

// d = a * b + c on two fp32 lanes at once (packed FFMA2, sm_100 family)
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// The lane's DPL consecutive elements of one token row, as DPL/2 float pairs.
template <typename C>
__device__ __forceinline__ void load_row(const char* row, int sub, float2 (&x)[C::DPL / 2]) {
    const char* p = row + sub * C::DPL * C::ESZ;
    if constexpr (C::ESZ == 4) {
        #pragma unroll
        for (int i = 0; i < C::DPL / 4; ++i) {
            const float4 v = reinterpret_cast<const float4*>(p)[i];
            x[2 * i] = make_float2(v.x, v.y);
            x[2 * i + 1] = make_float2(v.z, v.w);
        }
    } else if constexpr (C::ESZ == 2) {
        if constexpr (C::DPL == 8) {
            const uint4 v = *reinterpret_cast<const uint4*>(p);
            x[0] = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
            x[1] = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
            x[2] = __half22float2(*reinterpret_cast<const __half2*>(&v.z));
            x[3] = __half22float2(*reinterpret_cast<const __half2*>(&v.w));
        } else {
            const uint2 v = *reinterpret_cast<const uint2*>(p);
            x[0] = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
            x[1] = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
        }
    } else {
        if constexpr (C::DPL == 16) {                  // head quads: 16 codes per lane
            const uint4 v = *reinterpret_cast<const uint4*>(p);
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
            #pragma unroll
            for (int k = 0; k < 4; ++k) {
                x[2 * k] = e4m3x2_to_float2(static_cast<uint16_t>(w4[k] & 0xffffu));
                x[2 * k + 1] = e4m3x2_to_float2(static_cast<uint16_t>(w4[k] >> 16));
            }
        } else if constexpr (C::DPL == 8) {
            const uint2 v = *reinterpret_cast<const uint2*>(p);
            x[0] = e4m3x2_to_float2(static_cast<uint16_t>(v.x & 0xffffu));
            x[1] = e4m3x2_to_float2(static_cast<uint16_t>(v.x >> 16));
            x[2] = e4m3x2_to_float2(static_cast<uint16_t>(v.y & 0xffffu));
            x[3] = e4m3x2_to_float2(static_cast<uint16_t>(v.y >> 16));
        } else {
            const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
            x[0] = e4m3x2_to_float2(static_cast<uint16_t>(v & 0xffffu));
            x[1] = e4m3x2_to_float2(static_cast<uint16_t>(v >> 16));
        }
    }
}

// c.x += lo(a)·lo(b), c.y += hi(a)·hi(b): fp16 operands, fp32 accumulation.  The product
// of two fp16 values is exact in fp32, so this equals widening both operands first.
__device__ __forceinline__ float2 hfma2_f32(uint32_t a, uint32_t b, float2 c) {
    float2 d;
    asm("{\n\t.reg .f16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %4;\n\tfma.rn.f32.f16 %1, ah, bh, %5;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "r"(a), "r"(b), "f"(c.x), "f"(c.y));
    return d;
}

// The lane's DPL consecutive elements of one fp16 or FP8 token row as DPL/2 fp16 pairs
// (E4M3 -> fp16 is exact).
template <typename C>
__device__ __forceinline__ void load_row_h(const char* row, int sub, uint32_t (&x)[C::DPL / 2]) {
    const char* p = row + sub * C::DPL * C::ESZ;
    if constexpr (C::ESZ == 2) {
        if constexpr (C::DPL == 8) {
            const uint4 v = *reinterpret_cast<const uint4*>(p);
            x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
        } else {
            const uint2 v = *reinterpret_cast<const uint2*>(p);
            x[0] = v.x; x[1] = v.y;
        }
    } else {
        static_assert(C::ESZ == 1, "fp16 or FP8 rows");
        if constexpr (C::DPL == 16) {
            const uint4 v = *reinterpret_cast<const uint4*>(p);
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
            #pragma unroll
            for (int k = 0; k < 4; ++k) {
                x[2 * k] = e4m3x2_to_half2_bits(static_cast<uint16_t>(w4[k] & 0xffffu));
                x[2 * k + 1] = e4m3x2_to_half2_bits(static_cast<uint16_t>(w4[k] >> 16));
            }
        } else if constexpr (C::DPL == 8) {
            const uint2 v = *reinterpret_cast<const uint2*>(p);
            x[0] = e4m3x2_to_half2_bits(static_cast<uint16_t>(v.x & 0xffffu));
            x[1] = e4m3x2_to_half2_bits(static_cast<uint16_t>(v.x >> 16));
            x[2] = e4m3x2_to_half2_bits(static_cast<uint16_t>(v.y & 0xffffu));
            x[3] = e4m3x2_to_half2_bits(static_cast<uint16_t>(v.y >> 16));
        } else {
            const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
            x[0] = e4m3x2_to_half2_bits(static_cast<uint16_t>(v & 0xffffu));
            x[1] = e4m3x2_to_half2_bits(static_cast<uint16_t>(v >> 16));
        }
    }
}

template <typename C>
__device__ __forceinline__ void load_q(const char* qrow, int sub, float qs, float2 (&x)[C::DPL / 2]) {
    using QT = typename C::QT;
    const QT* p = reinterpret_cast<const QT*>(qrow) + sub * C::DPL;
    #pragma unroll
    for (int i = 0; i < C::DPL / 2; ++i)
        x[i] = make_float2(static_cast<float>(p[2 * i]) * qs, static_cast<float>(p[2 * i + 1]) * qs);
}

struct __align__(16) Item {
    int s, h, p, tok0, ntok, nchunks, single, valid, last;   // last: final partition
    int lo;                                                    // masked rows at the start
    int nq;                                                    // shared prefixes: query rows
};

// (s, h, p) of compact item index `it` (items ordered by sequence, head, partition).
template <int CT>
__device__ __forceinline__ Item decode_item(int it, int n_items, const int* s_ctx, const int* s_end,
                                            int batch, int H, int P_coarse, int s_fine, int P_fine, int window,
                                            int rpc) {
    Item r{};
    r.valid = it < n_items;
    if (!r.valid) return r;
    int lo = 0, hi = batch - 1;          // first s with s_end[s] > it
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (s_end[mid] > it) hi = mid; else lo = mid + 1;
    }
    const int s = lo;
    const int P = s >= s_fine ? P_fine : P_coarse;
    const int start = s ? s_end[s - 1] : 0;
    const int ctx = s_ctx[s];
    const int first = attend_first(ctx, window, rpc);
    const int np = nparts_of(ctx - first, P);
    const int rr = it - start;
    r.s = s;
    r.h = rr / np;
    r.p = rr - r.h * np;
    // the np partitions of a context split it evenly (each a multiple of kPartAlign tokens,
    // at most P): items of one sequence have about one size, which evens out the finish
    const int ps = np > 1 ? ((ctx - first + np - 1) / np + kPartAlign - 1) / kPartAlign * kPartAlign : P;
    r.tok0 = first + r.p * ps;
    r.ntok = min(ps, ctx - r.tok0);
    r.lo = r.p == 0 ? attend_start(ctx, window) - first : 0;
    r.nchunks = r.ntok > 0 ? (r.ntok + CT - 1) / CT : 1;
    r.single = np == 1;
    r.last = r.p == np - 1;
    r.nq = 1;
    return r;
}

// Shared prompt prefixes.  A prefix-group member's context is split in two: the shared
// prefix [0, S) and its own tokens [S, ctx), each evenly as decode_item splits a context.
// Its partitions are numbered shared first (0 .. ns-1), then its own (ns .. ns+no-1).
__device__ __forceinline__ int pfx_shared_parts(int S, int P) { return S > 0 ? nparts_of(S, P) : 0; }
__device__ __forceinline__ int pfx_own_parts(int ctx, int S, int P) {
    return (S > 0 && ctx <= S) ? 0 : nparts_of(ctx - S, P);
}
__device__ __forceinline__ int even_part(int len, int np, int P) {
    return np > 1 ? ((len + np - 1) / np + kPartAlign - 1) / kPartAlign * kPartAlign : P;
}

// Item `it` of a launch with prefix groups.  Items are ordered by sequence; a group's first
// sequence lists the group's shared items (head, shared partition: nq = member count query
// rows, sequences s .. s+nq-1) before its own items (head, own partition: one query row).
template <int CT>
__device__ __forceinline__ Item decode_item_pfx(int it, int n_items, const int* s_ctx, const int* s_end,
                                                const int* s_pfx, int batch, int H, int P) {
    Item r{};
    r.valid = it < n_items;
    if (!r.valid) return r;
    int lo = 0, hi = batch - 1;          // first s with s_end[s] > it
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (s_end[mid] > it) hi = mid; else lo = mid + 1;
    }
    const int s = lo;
    const int ctx = s_ctx[s];
    const int S = s_pfx[s] & kPfxTokMask, k = s_pfx[s] >> 24;
    const int ns = pfx_shared_parts(S, P);
    const int shared_items = k ? H * ns : 0;
    int rr = it - (s ? s_end[s - 1] : 0);
    r.s = s;
    if (rr < shared_items) {
        r.h = rr / ns;
        const int p = rr - r.h * ns;
        const int ps = even_part(S, ns, P);
        r.tok0 = p * ps;
        r.ntok = min(ps, S - r.tok0);
        r.p = p;
        r.nq = k;
    } else {
        rr -= shared_items;
        const int no = pfx_own_parts(ctx, S, P);
        r.h = rr / no;
        const int p = rr - r.h * no;
        const int ps = even_part(ctx - S, no, P);
        r.tok0 = S + p * ps;
        r.ntok = min(ps, ctx - r.tok0);
        r.p = ns + p;
        r.nq = 1;
        r.single = ns + no == 1;
        r.last = p == no - 1;
    }
    r.nchunks = r.ntok > 0 ? (r.ntok + CT - 1) / CT : 1;
    return r;
}

// Split-context merge of the np partials of one (sequence, head), by one warp:
// M = max m_p, L = sum l_p 2^(m_p - M), out = sum o_p 2^(m_p - M) / L.
// The partials were written by other SMs; they are read through L2 (ld.global.cg).
template <int D, int G, bool FINAL>
__device__ __forceinline__ void merge_rows(const AttnArgs& a, int64_t row, int first, int count, int stride,
                                           int lane) {
    // merges partials first, first+stride, ... (count of them) of G rows at once, 32/G
    // lanes per row (`row`: this lane group's (sequence, query head)), so every lane's
    // loads are independent and all rows' loads are in flight together (a merge sits on
    // the critical path).  A lane group with count 0 stores nothing.  FINAL writes the
    // normalised output; otherwise the merged, still unnormalised partial (with its m, l)
    // replaces partial `first`.
    constexpr int LPH = 32 / G;                     // lanes per row
    constexpr int DL = D / LPH;                     // dims per lane
    constexpr int VEC = DL % 4 == 0 ? 4 : 2;
    constexpr int UNR = G == 1 ? 4 : 2;
    const int q = lane % LPH;
    const bool act = count > 0;
    const int64_t base = row * a.max_parts + first;
    const float2* ml = reinterpret_cast<const float2*>(a.part_ml) + base;
    float mx = -CUDART_INF_F;
    for (int k = q; k < count; k += LPH) mx = fmaxf(mx, __ldcg(ml + static_cast<int64_t>(k) * stride).x);
    #pragma unroll
    for (int off = LPH / 2; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, off));
    float L = 0.f, acc[DL];
    #pragma unroll
    for (int i = 0; i < DL; ++i) acc[i] = 0.f;
    #pragma unroll UNR
    for (int k = 0; k < count; ++k) {
        const int64_t kr = static_cast<int64_t>(k) * stride;
        const float2 v = __ldcg(ml + kr);
        const float wgt = ex2_approx(v.x - mx);
        L = fmaf(v.y, wgt, L);
        const float* o = a.part_o + (base + kr) * D;
        #pragma unroll
        for (int i = 0; i < DL / VEC; ++i) {
            if constexpr (VEC == 4) {
                const float4 x = __ldcg(reinterpret_cast<const float4*>(o) + i * LPH + q);
                acc[4 * i] = fmaf(wgt, x.x, acc[4 * i]); acc[4 * i + 1] = fmaf(wgt, x.y, acc[4 * i + 1]);
                acc[4 * i + 2] = fmaf(wgt, x.z, acc[4 * i + 2]); acc[4 * i + 3] = fmaf(wgt, x.w, acc[4 * i + 3]);
            } else {
                const float2 x = __ldcg(reinterpret_cast<const float2*>(o) + i * LPH + q);
                acc[2 * i] = fmaf(wgt, x.x, acc[2 * i]); acc[2 * i + 1] = fmaf(wgt, x.y, acc[2 * i + 1]);
            }
        }
    }
    const float inv = FINAL ? 1.f / L : 1.f;
    if (FINAL && !act) return;
    if (FINAL && a.out_f16) {                          // rounded once, from the float32 result
        __half* oh = static_cast<__half*>(a.out) + row * D;
        #pragma unroll
        for (int i = 0; i < DL / VEC; ++i) {
            if constexpr (VEC == 4) {
                const __half2 lo = __floats2half2_rn(acc[4 * i] * inv, acc[4 * i + 1] * inv);
                const __half2 hi = __floats2half2_rn(acc[4 * i + 2] * inv, acc[4 * i + 3] * inv);
                uint2 w;
                w.x = *reinterpret_cast<const unsigned*>(&lo);
                w.y = *reinterpret_cast<const unsigned*>(&hi);
                reinterpret_cast<uint2*>(oh)[i * LPH + q] = w;
            } else {
                reinterpret_cast<__half2*>(oh)[i * LPH + q] = __floats2half2_rn(acc[2 * i] * inv, acc[2 * i + 1] * inv);
            }
        }
        return;
    }
    float* out = FINAL ? static_cast<float*>(a.out) + row * D : a.part_o + base * D;
    if (!FINAL) {
        __syncwarp();                                  // every lane has read partial `first`
        if (!act) return;
        if (q == 0) reinterpret_cast<float2*>(a.part_ml)[base] = make_float2(mx, L);
    }
    #pragma unroll
    for (int i = 0; i < DL / VEC; ++i) {
        if constexpr (VEC == 4) {
            reinterpret_cast<float4*>(out)[i * LPH + q] =
                make_float4(acc[4 * i] * inv, acc[4 * i + 1] * inv, acc[4 * i + 2] * inv, acc[4 * i + 3] * inv);
        } else {
            reinterpret_cast<float2*>(out)[i * LPH + q] = make_float2(acc[2 * i] * inv, acc[2 * i + 1] * inv);
        }
    }
}

// The G consecutive rows sh0 .. sh0+G-1 (the query heads of one K/V head).
template <int D, int G, bool FINAL>
__device__ __forceinline__ void merge_partials(const AttnArgs& a, int64_t sh0, int first, int count, int stride,
                                               int lane) {
    merge_rows<D, G, FINAL>(a, sh0 + lane / (32 / G), first, count, stride, lane);
}

// The final merge of one row (partials 0, stride, 2*stride, ... of it; count <= 32) with
// all 32 lanes (head_dim 128: a float4 of the row per lane).  Lane k loads partial k's
// (m, l) while the rows of the first eight partials are already in flight, so up to eight
// partials cost one L2 round trip (merge_rows' first pass over the maxima costs one more).
// The same operations in the same order as merge_rows with one row: the same bits.
template <int D>
__device__ __forceinline__ void merge_row_fast(const AttnArgs& a, int64_t row, int count, int stride, int lane) {
    static_assert(D == 128, "a float4 of the row per lane");
    const float2* ml = reinterpret_cast<const float2*>(a.part_ml) + row * a.max_parts;
    const float4* o = reinterpret_cast<const float4*>(a.part_o + row * a.max_parts * D) + lane;
    const float2 v = lane < count ? __ldcg(ml + static_cast<int64_t>(lane) * stride) : make_float2(-CUDART_INF_F, 0.f);
    // the weights and the denominator are summed in partition order, as merge_rows does,
    // so a row's result does not depend on which of the two merged it
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wk = 0.f, L = 0.f;
    #pragma unroll 1
    for (int k0 = 0; k0 < count; k0 += 8) {
        float4 x[8];
        #pragma unroll
        for (int k = 0; k < 8; ++k)
            x[k] = k0 + k < count ? __ldcg(o + static_cast<int64_t>(k0 + k) * stride * (D / 4))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
        if (k0 == 0) {
            const float mx = warp_max(v.x);
            wk = lane < count ? ex2_approx(v.x - mx) : 0.f;
        }
        #pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float w = __shfl_sync(FULL, wk, (k0 + k) & 31);
            const float lk = __shfl_sync(FULL, v.y, (k0 + k) & 31);
            if (k0 + k < count) L = fmaf(lk, w, L);
            acc.x = fmaf(w, x[k].x, acc.x);
            acc.y = fmaf(w, x[k].y, acc.y);
            acc.z = fmaf(w, x[k].z, acc.z);
            acc.w = fmaf(w, x[k].w, acc.w);
        }
    }
    const float inv = 1.f / L;
    if (a.out_f16) {                                   // rounded once, from the float32 result
        const __half2 lo = __floats2half2_rn(acc.x * inv, acc.y * inv);
        const __half2 hi = __floats2half2_rn(acc.z * inv, acc.w * inv);
        uint2 wv;
        wv.x = *reinterpret_cast<const unsigned*>(&lo);
        wv.y = *reinterpret_cast<const unsigned*>(&hi);
        reinterpret_cast<uint2*>(static_cast<__half*>(a.out) + row * D)[lane] = wv;
    } else {
        reinterpret_cast<float4*>(static_cast<float*>(a.out) + row * D)[lane] =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
}

// Partition p of (sequence, KV head) shk has written its partials: publish them and take
// a ticket.  Up to kMergeFan partitions merge in one step, by the warp that finishes last.
// Longer splits merge in two levels, which shortens the merge that ends the split: the
// last finisher of each group of kMergeFan partitions folds the group into the group's
// first slot, and the last group to fold merges the ceil(np / kMergeFan) groups.
// The ticket's atomic is issued at the end of the item and read one chunk later
// (ticket_resolve), so its round trip overlaps the next chunk instead of stalling the warp.
struct Ticket {
    unsigned prev;          // lane 0: the atomic's result (in flight until read)
    int64_t shk;
    int p, np;
    bool pending;
};

__device__ __forceinline__ void ticket_issue(const AttnArgs& a, Ticket& tk, int64_t shk, int p, int np, int lane) {
    __syncwarp();                                      // every lane's partial is written
    unsigned* ctr = np > kMergeFan ? a.grp_arrivals + shk * a.n_grp + p / kMergeFan : a.arrivals + shk;
    if (lane == 0) tk.prev = atom_add_acq_rel_gpu(ctr, 1u);
    tk.shk = shk;
    tk.p = p;
    tk.np = np;
    tk.pending = true;
}

template <int D, int G>
__device__ __forceinline__ void ticket_resolve(const AttnArgs& a, Ticket& tk, int lane) {
    if (!tk.pending) return;
    tk.pending = false;
    unsigned prev = __shfl_sync(FULL, tk.prev, 0);
    int count = tk.np, stride = 1;
    if (tk.np > kMergeFan) {
        const int grp = tk.p / kMergeFan;
        const int gsz = min(kMergeFan, tk.np - grp * kMergeFan);
        if (prev != static_cast<unsigned>(gsz - 1)) return;
        if (lane == 0) a.grp_arrivals[tk.shk * a.n_grp + grp] = 0;   // left zero for the next call
        __syncwarp();
        merge_partials<D, G, false>(a, tk.shk * G, grp * kMergeFan, gsz, 1, lane);
        __syncwarp();
        count = (tk.np + kMergeFan - 1) / kMergeFan;
        stride = kMergeFan;
        unsigned p2 = 0;
        if (lane == 0) p2 = atom_add_acq_rel_gpu(a.arrivals + tk.shk, 1u);
        prev = __shfl_sync(FULL, p2, 0);
    }
    if (prev != static_cast<unsigned>(count - 1)) return;
    if (lane == 0) a.arrivals[tk.shk] = 0;                             // left zero for the next call
    __syncwarp();
    if constexpr (D == 128 && G == 1) {
        if (count <= 32) {
            merge_row_fast<D>(a, tk.shk, count, stride, lane);
            return;
        }
    }
    merge_partials<D, G, true>(a, tk.shk * G, 0, count, stride, lane);
}

// Shared prefixes: an item writes a partial for each of its query rows (a shared item for
// every member of the group), so lane r takes the ticket of row r.  A member has at most
// kPfxMaxParts partitions, merged in one step.
struct PfxTicket {
    unsigned prev;          // the row's arrival count before this partition (in flight until read)
    int sq, np;             // the row's (sequence, head) and its number of partitions
    bool pending;
};

template <int D>
__device__ __forceinline__ void pfx_ticket_resolve(const AttnArgs& a, PfxTicket& tk, int lane) {
    const bool last = tk.pending && tk.prev == static_cast<unsigned>(tk.np - 1);
    tk.pending = false;
    const unsigned m = __ballot_sync(FULL, last);
    if (!m) return;
    if (last) a.arrivals[tk.sq] = 0;                                   // left zero for the next call
    __syncwarp();
    if (__popc(m) == 1) {                          // one row: all 32 lanes on it
        const int r = __ffs(m) - 1;
        merge_row_fast<D>(a, __shfl_sync(FULL, tk.sq, r), __shfl_sync(FULL, tk.np, r), 1, lane);
    } else {                                       // rows side by side, 4 lanes each (row r: lanes 4r..4r+3)
        const int r = lane >> 2;
        const int sq = __shfl_sync(FULL, tk.sq, r);
        const int np = __shfl_sync(FULL, tk.np, r);
        merge_rows<D, 8, true>(a, sq, 0, ((m >> r) & 1) ? np : 0, 1, lane);
    }
}

// Fused append: lane's D/32 elements of one new-token row (src, in_bytes per element)
// are converted to the pool type (FP8: RNE-satfinite(x / scale)) and written both into
// the consumer's stage row and into the pool slot, so the attention below sees exactly
// the bytes a separate kv_append would have stored.
template <typename C>
__device__ __forceinline__ void patch_row(const char* src, int in_bytes, char* srow, char* grow,
                                          float scale, int lane, int swz = 0) {
    constexpr int DW = C::D / 32;
    const int e0 = lane * DW;
    if constexpr (C::ESZ == 4) {
        static_assert(DW == 4 || DW == 2, "head_dim 64 or 128");
        if constexpr (DW == 4) {
            const float4 v = *reinterpret_cast<const float4*>(src + e0 * 4);
            *reinterpret_cast<float4*>(srow + e0 * 4) = v;
            *reinterpret_cast<float4*>(grow + e0 * 4) = v;
        } else {
            const float2 v = *reinterpret_cast<const float2*>(src + e0 * 4);
            *reinterpret_cast<float2*>(srow + e0 * 4) = v;
            *reinterpret_cast<float2*>(grow + e0 * 4) = v;
        }
    } else if constexpr (C::ESZ == 2) {
        if constexpr (DW == 4) {
            const uint2 v = *reinterpret_cast<const uint2*>(src + e0 * 2);
            *reinterpret_cast<uint2*>(srow + e0 * 2) = v;
            *reinterpret_cast<uint2*>(grow + e0 * 2) = v;
        } else {
            const uint32_t v = *reinterpret_cast<const uint32_t*>(src + e0 * 2);
            *reinterpret_cast<uint32_t*>(srow + e0 * 2) = v;
            *reinterpret_cast<uint32_t*>(grow + e0 * 2) = v;
        }
    } else {
        float x[DW];
        #pragma unroll
        for (int i = 0; i < DW; ++i)
            x[i] = in_bytes == 2 ? __half2float(reinterpret_cast<const __half*>(src)[e0 + i])
                                 : reinterpret_cast<const float*>(src)[e0 + i];
        uint16_t q[DW / 2];
        #pragma unroll
        for (int i = 0; i < DW / 2; ++i)
            q[i] = float2_to_e4m3x2(__fdiv_rn(x[2 * i], scale), __fdiv_rn(x[2 * i + 1], scale));
        if constexpr (DW == 4) {
            // swz != 0: the stage row is 128-byte swizzled (16-byte piece c at c ^ swz)
            const uint32_t v = static_cast<uint32_t>(q[0]) | (static_cast<uint32_t>(q[1]) << 16);
            *reinterpret_cast<uint32_t*>(srow + ((((e0 >> 4) ^ swz) << 4) | (e0 & 15))) = v;
            *reinterpret_cast<uint32_t*>(grow + e0) = v;
        } else {
            *reinterpret_cast<uint16_t*>(srow + e0) = q[0];
            *reinterpret_cast<uint16_t*>(grow + e0) = q[0];
        }
    }
}

// Byte offset inside a 128-byte-swizzled stage of element byte `off` of the logical
// [token][256 B] layout (tensor-map copies swap 16-byte chunks within each 128-byte row
// by the row's index mod 8).
__device__ __forceinline__ uint32_t swz128(uint32_t off) { return off ^ (((off >> 7) & 7u) << 4); }

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Grouped-query consumer on the tensor cores (fp16 or FP8 pools, head_dim 128, G query
// heads per K/V head).  Per 16-token step, with the tokens (and output dims) as the M side
// of mma.m16n8k16 and the query heads, padded to 8, as its N side:
//   S^T  = K Q^T      8 k-steps over the 128 dims; K fragments by ldmatrix (fp16) or
//                     converted from 16-byte reads of E4M3 codes (FP8)
//   softmax           per query column (the 8 lanes of equal lane%4), in the log2 domain
//   O^T += V^T P^T    P^T from the S accumulators by movmatrix.trans; V^T fragments by
//                     ldmatrix.trans (fp16) or the 8-bit transposing ldmatrix (FP8);
//                     8 output tiles of 16 dims
// fp32 accumulation and softmax, exact running max (FP8: one update per 32-token chunk).
template <typename C>
__device__ __forceinline__ void consumer_mma(const AttnArgs& a, char* smem, const int* s_ctx, int w, int lane,
                                             int P_eff) {
    constexpr int NSW = C::NSW, D = C::D, G = C::G, CT = C::CT;
    static_assert((CT == 16 || (C::FP8 && CT == 32)) && D == 128, "tensor-core consumer shape");
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    // head-pair stages: warps 2r and 2r+1 share ring r, taking the pair's heads 0 and 1
    const int wr = C::PR ? (w >> 1) : w;             // this warp's ring
    const int e = C::PR ? (w & 1) : 0;               // this warp's head of the item's pair
    // S^T = K Q^T and O^T += V^T P^T: the 16 tokens of a chunk (and 16 dims of an output
    // tile) are the mma's M side, the query heads (padded to 8) its N side, so no mma row
    // is padding.  Lane (g, t): token rows g and g+8, query columns 2t and 2t+1.
    const int g = lane >> 2, t = lane & 3;
    // byte x (0..255) of fp16 token row tok in a chunk: copies of rpc rows (8 or 16), each
    // laid out half-major [2][rpc][64 halves], 128-byte swizzled by the tensor-map copies
    // (rpc = min(B, 16)).  FP8 stages hold plain [rows][128 codes], also 128-byte swizzled:
    // 16-byte piece c of row r sits at piece c ^ (r % 8).
    // With head-pair stages a copy holds 2*rpc rows (head 0's rpc rows, then head 1's), so
    // this warp's token tok of a copy sits e*rpc rows further.
    const int rpc_ = a.B < CT ? a.B : CT;
    const int rs = rpc_ == 32 ? 5 : (rpc_ == 16 ? 4 : 3);
    const int cs = rs + (C::PR ? 1 : 0);             // log2 rows of one copy (per half for fp16)
    const int erow = C::PR ? (e << rs) : 0;
    auto tile_off = [rs, cs, erow](int tok, int x) -> uint32_t {
        const int rpc = 1 << rs;
        return swz128(static_cast<uint32_t>(((tok >> rs) << (cs + 8)) +
                                            ((((x >> 7) << cs) + erow + (tok & (rpc - 1))) << 7) + (x & 127)));
    };
    // FP8 stages: the stage row of this warp's token tok (rows % 8 are those of tok)
    auto row8 = [rs, erow](int tok) -> int {
        if constexpr (C::PR) return ((tok >> rs) << (rs + 1)) + erow + (tok & ((1 << rs) - 1));
        else return tok;
    };
    uint32_t qa[8][2];                 // B fragments of Q^T: query g, dims 16k+2t.. and 16k+8+2t..
    float ot[8][4];                    // O^T tile i: dims 16i+g / 16i+g+8, queries 2t / 2t+1
    float m2[2] = {-CUDART_INF_F, -CUDART_INF_F}, l2[2] = {0.f, 0.f};   // queries 2t, 2t+1
    #pragma unroll
    for (int i = 0; i < 8; ++i) { qa[i][0] = 0u; qa[i][1] = 0u; }
    #pragma unroll
    for (int i = 0; i < 8; ++i) { ot[i][0] = ot[i][1] = ot[i][2] = ot[i][3] = 0.f; }
    Ticket tk{};
    PfxTicket ptk{};
    const int* s_pfx = s_ctx + 2 * kMaxBatch;       // shared prefixes (PFX launches only)

    for (int j = 0;; ++j) {
        const int st = j % NSW;
        const uint32_t par = (j / NSW) & 1;
        const uint32_t fb = smem_u32(&bars[wr * NSW + st]);
        if (!mbar_wait_bounded(fb, par, a.err)) {
            mbar_wait_bounded(fb, par, a.err);      // let copies in flight land, then leave
            break;
        }
        char* stg = smem + (wr * NSW + st) * C::STAGE;
        const Meta* mp = reinterpret_cast<const Meta*>(smem + C::META_R + (wr * NSW + st) * sizeof(Meta));
        const int flags = mp->flags;
        if (flags & F_TERM) break;
        const int nt = mp->ntok, lo = mp->lo, ms = mp->s, mpart = mp->p;
        const int mh = C::PR ? 2 * mp->h + e : mp->h;   // this warp's K/V head
        // query rows of the item: G heads of one sequence, or (shared prefixes) one head of
        // the nq sequences ms .. ms+nq-1
        const int nq = C::PFX ? mp->nq : G;
        uint32_t kbase = smem_u32(stg + C::K_OFF), vbase = smem_u32(stg + C::V_OFF);
        if (flags & F_FIRST) {
            m2[0] = m2[1] = -CUDART_INF_F;
            l2[0] = l2[1] = 0.f;
            #pragma unroll
            for (int i = 0; i < 8; ++i) { ot[i][0] = ot[i][1] = ot[i][2] = ot[i][3] = 0.f; }
            // B fragments of the G query rows (fp16: staged with the item's first chunk;
            // FP8 and head-pair stages: read from global memory once per item)
            const bool real = g < nq && nt > 0;
            const int64_t qr = C::PFX ? static_cast<int64_t>(ms + (real ? g : 0)) * a.H + mh
                                      : (static_cast<int64_t>(ms) * a.H + mh) * G + (real ? g : 0);
            const uint32_t* qrow = (C::FP8 || C::PR)
                ? reinterpret_cast<const uint32_t*>(static_cast<const char*>(a.q) + qr * D * 2)
                : reinterpret_cast<const uint32_t*>(smem + C::QR_OFF + (wr * NSW + st) * C::QR_BYTES +
                                                    (real ? g : 0) * D * 2);
            #pragma unroll
            for (int k = 0; k < 8; ++k) {
                // FP8: k-index pairs (2t, 2t+1) and (2t+8, 2t+9) of k-step k = 4j + i stand
                // for dims 32t+16j+4i.. and 32t+16j+4i+2.. (the order the K fragments are
                // read in; a dot product is the same in any consistent order of its dims)
                if constexpr (C::FP8) {
                    const int h2 = 16 * t + 8 * (k >> 2) + 2 * (k & 3);   // uint32 = 2 dims
                    qa[k][0] = real ? qrow[h2] : 0u;
                    qa[k][1] = real ? qrow[h2 + 1] : 0u;
                    continue;
                }
                qa[k][0] = real ? qrow[8 * k + t] : 0u;
                qa[k][1] = real ? qrow[8 * k + 4 + t] : 0u;
            }
        }
        if (C::FP8 && (flags & F_PATCH)) {
            // the new token, quantised with its block's scale, into the stage row and the slot
            const int r = mp->patch_row;
            const int64_t sh = static_cast<int64_t>(ms) * a.H + mh;
            const int64_t grow = (static_cast<int64_t>(mp->patch_id) * a.H + mh) * a.B + mp->patch_off;
            // K and V rows sit 128-byte swizzled in the stage (16-byte piece c of row r at c ^ (r % 8))
            patch_row<C>(a.k_new + sh * D * a.in_bytes, a.in_bytes, stg + C::K_OFF + row8(r) * C::ROW,
                         a.kpool + grow * C::ROW, __ldg(a.kscale + mp->patch_id), lane, r & 7);
            patch_row<C>(a.v_new + sh * D * a.in_bytes, a.in_bytes, stg + C::V_OFF + row8(r) * C::ROW,
                         a.vpool + grow * C::ROW, __ldg(a.vscale + mp->patch_id), lane, r & 7);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
        } else if (flags & F_PATCH) {
            // the new token's row, into the swizzled stage and into the pool slot
            const int r = mp->patch_row;
            const int64_t sh = static_cast<int64_t>(ms) * a.H + mh;
            const int64_t grow = (static_cast<int64_t>(mp->patch_id) * a.H + mh) * a.B + mp->patch_off;
            const int e0 = lane * 4;
            const uint2 kv = *reinterpret_cast<const uint2*>(a.k_new + (sh * D + e0) * 2);
            const uint2 vv = *reinterpret_cast<const uint2*>(a.v_new + (sh * D + e0) * 2);
            const uint32_t so = tile_off(r, e0 * 2);
            *reinterpret_cast<uint2*>(stg + C::K_OFF + so) = kv;
            *reinterpret_cast<uint2*>(stg + C::V_OFF + so) = vv;
            *reinterpret_cast<uint2*>(a.kpool + grow * C::ROW + e0 * 2) = kv;
            *reinterpret_cast<uint2*>(a.vpool + grow * C::ROW + e0 * 2) = vv;
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
        }
        // 16-token steps (a 32-token FP8 chunk has two): every step's S mma first, one
        // softmax update over the whole chunk, then every step's P V mma.  A step with no
        // token in [lo, nt) is skipped.
        constexpr int NS = CT / 16;
        bool act[NS];
        bool any = false;
        #pragma unroll
        for (int u = 0; u < NS; ++u) {
            act[u] = 16 * u < nt && 16 * u + 16 > lo;
            any = any || act[u];
        }
        if (!C::FP8 && any && (nt < CT || lo > 0)) {
            // rows outside [lo, nt) may hold anything (unused slots): zero their V so
            // that p = 0 rows contribute exactly nothing to P V
            #pragma unroll 1
            for (int r = 0; r < CT; ++r)
                if ((r < lo || r >= nt) && lane < 16)
                    *reinterpret_cast<uint4*>(stg + C::V_OFF + tile_off(r, lane * 16)) = make_uint4(0, 0, 0, 0);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
        }
        if (any) {
            const int mi = lane >> 3, mr = lane & 7;
            float x[NS][4];
            float vsc[NS][2];                  // V scales of this lane's rows (FP8; else 1)
            #pragma unroll
            for (int u = 0; u < NS; ++u) {
                const int t16 = 16 * u;
                x[u][0] = x[u][1] = x[u][2] = x[u][3] = -CUDART_INF_F;
                vsc[u][0] = vsc[u][1] = 1.f;
                if (!act[u]) continue;
                // FP8: per-block scales of this lane's token rows (t16 + g and t16 + g + 8)
                float ks0 = 1.f, ks1 = 1.f;
                if constexpr (C::FP8) {
                    const int rpc = a.B < CT ? a.B : CT;
                    const int id0 = mp->ids[t16 / rpc], id1 = mp->ids[(t16 + 8) / rpc];
                    ks0 = __ldg(a.kscale + id0);
                    ks1 = __ldg(a.kscale + id1);
                    vsc[u][0] = __ldg(a.vscale + id0);
                    vsc[u][1] = __ldg(a.vscale + id1);
                }
                // S^T = K Q^T, the even and odd k-steps in two accumulators (shorter chains)
                float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
                // FP8: this lane's K rows t16 + g and t16 + g + 8 of the swizzled stage
                // (both have row % 8 == g): 16-byte pieces 2t and 2t+1 of each (dims
                // 32t..32t+31), piece c sitting at c ^ g.  A quarter-warp reads rows g and
                // g+1 (g even), whose pieces (2t+j)^g and (2t+j)^g^1 are 8 distinct ones:
                // no bank conflicts.
                uint4 kw[2][2];
                if constexpr (C::FP8) {
                    const char* kr0 = stg + C::K_OFF + row8(t16 + g) * C::ROW;
                    const char* kr1 = stg + C::K_OFF + row8(t16 + g + 8) * C::ROW;
                    #pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        kw[0][j] = *reinterpret_cast<const uint4*>(kr0 + (((2 * t + j) ^ g) << 4));
                        kw[1][j] = *reinterpret_cast<const uint4*>(kr1 + (((2 * t + j) ^ g) << 4));
                    }
                }
                #pragma unroll
                for (int k = 0; k < 8; ++k) {
                    uint32_t kf[4];
                    if constexpr (C::FP8) {
                        // A fragment straight from the E4M3 codes: the 4 codes of dims
                        // 32t+16j+4i.. of each row (k = 4j + i)
                        const uint32_t w0 = reinterpret_cast<const uint32_t*>(&kw[0][k >> 2])[k & 3];
                        const uint32_t w1 = reinterpret_cast<const uint32_t*>(&kw[1][k >> 2])[k & 3];
                        kf[0] = e4m3x2_to_half2_bits(static_cast<uint16_t>(w0 & 0xffffu));
                        kf[1] = e4m3x2_to_half2_bits(static_cast<uint16_t>(w1 & 0xffffu));
                        kf[2] = e4m3x2_to_half2_bits(static_cast<uint16_t>(w0 >> 16));
                        kf[3] = e4m3x2_to_half2_bits(static_cast<uint16_t>(w1 >> 16));
                    } else {
                        // A = K: (tok 0-7, dims 16k..) (tok 8-15, 16k..) (tok 0-7, +8..) (tok 8-15, +8..)
                        const int tok = t16 + (mi & 1) * 8 + mr, cp = 2 * k + (mi >> 1);
                        ldsm_x4(kbase + tile_off(tok, cp * 16), kf);
                    }
                    if (k & 1) mma_16816(sb, kf[0], kf[1], kf[2], kf[3], qa[k][0], qa[k][1]);
                    else mma_16816(sa, kf[0], kf[1], kf[2], kf[3], qa[k][0], qa[k][1]);
                }
                // log2-domain scores of tokens g (x0: query 2t, x1: 2t+1) and g+8 (x2, x3)
                const float qk0 = a.qscale * ks0, qk1 = a.qscale * ks1;   // K scales; 1 for fp16 pools
                const bool v0 = t16 + g >= lo && t16 + g < nt, v1 = t16 + g + 8 >= lo && t16 + g + 8 < nt;
                if (v0) { x[u][0] = (sa[0] + sb[0]) * qk0; x[u][1] = (sa[1] + sb[1]) * qk0; }
                if (v1) { x[u][2] = (sa[2] + sb[2]) * qk1; x[u][3] = (sa[3] + sb[3]) * qk1; }
            }
            // column maxima over the chunk's tokens: the 8 lanes of equal t hold them
            float mxa = -CUDART_INF_F, mxb = -CUDART_INF_F;
            #pragma unroll
            for (int u = 0; u < NS; ++u) {
                mxa = fmaxf(mxa, fmaxf(x[u][0], x[u][2]));
                mxb = fmaxf(mxb, fmaxf(x[u][1], x[u][3]));
            }
            #pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mxa = fmaxf(mxa, __shfl_xor_sync(FULL, mxa, off));
                mxb = fmaxf(mxb, __shfl_xor_sync(FULL, mxb, off));
            }
            const float ma = fmaxf(m2[0], mxa), mb = fmaxf(m2[1], mxb);
            const float ca = ex2_approx(m2[0] - ma), cb = ex2_approx(m2[1] - mb);
            l2[0] *= ca;
            l2[1] *= cb;
            m2[0] = ma;
            m2[1] = mb;
            #pragma unroll
            for (int i = 0; i < 8; ++i) { ot[i][0] *= ca; ot[i][2] *= ca; ot[i][1] *= cb; ot[i][3] *= cb; }
            #pragma unroll
            for (int u = 0; u < NS; ++u) {
                if (!act[u]) continue;
                const int t16 = 16 * u;
                const float p0 = ex2_approx(x[u][0] - ma), p1 = ex2_approx(x[u][1] - mb);
                const float p2 = ex2_approx(x[u][2] - ma), p3 = ex2_approx(x[u][3] - mb);
                l2[0] += p0 + p2;                    // this lane's tokens only; summed at the end
                l2[1] += p1 + p3;
                // P^T as the B operand: the 8x8 blocks (tokens x queries) this lane holds a
                // row pair of, transposed in registers (V scales folded in; 1 for fp16 pools)
                uint32_t pb0 = movmatrix_t(pack_half2(p0 * vsc[u][0], p1 * vsc[u][0]));
                uint32_t pb1 = movmatrix_t(pack_half2(p2 * vsc[u][1], p3 * vsc[u][1]));
                if constexpr (C::FP8) {
                    // the FP8 V fragments below pair tokens (4t, 4t+1) and (4t+2, 4t+3)
                    // as k pairs (2t, 2t+1) and (2t+8, 2t+9): fetch P^T in that order
                    // (tokens 4t.. sit with lane t' = 2t mod 4 of the first or second
                    // 8-token block)
                    const int s0 = 4 * g + ((2 * t) & 3), s1 = s0 + 1;
                    const uint32_t a0 = __shfl_sync(FULL, pb0, s0), b0 = __shfl_sync(FULL, pb1, s0);
                    const uint32_t a1 = __shfl_sync(FULL, pb0, s1), b1 = __shfl_sync(FULL, pb1, s1);
                    pb0 = t < 2 ? a0 : b0;
                    pb1 = t < 2 ? a1 : b1;
                }
                // O^T += V^T P^T, one 16-dim tile per mma
                if constexpr (C::FP8) {
                    // A = V^T from the E4M3 codes by a transposing byte ldmatrix: lanes 0-15
                    // address the 16 token rows of dim tile 2pp, lanes 16-31 those of tile
                    // 2pp+1 (16-byte piece of the swizzled row); lane (g, t) receives dims g
                    // and g+8 of tokens 4t..4t+3, converted exactly to the fp16 pairs of
                    // k pairs (2t, 2t+1) and (2t+8, 2t+9).  Rows outside [lo, nt) point at
                    // a zero line (their p is 0; their slots may hold anything).
                    const int vr = t16 + (lane & 15);
                    const bool vzero = (t16 + 16 > nt || t16 < lo) && (vr < lo || vr >= nt);
                    const uint32_t zaddr = smem_u32(smem + C::ZERO_OFF);
                    #pragma unroll
                    for (int pp = 0; pp < 4; ++pp) {
                        const int tile = 2 * pp + (lane >> 4);
                        const uint32_t addr = vzero ? zaddr : vbase + row8(vr) * C::ROW + ((tile ^ (vr & 7)) << 4);
                        uint32_t r[4];
                        ldsm_b8_x2_t(addr, r);
                        mma_16816(ot[2 * pp], e4m3x2_to_half2_bits(static_cast<uint16_t>(r[0] & 0xffffu)),
                                  e4m3x2_to_half2_bits(static_cast<uint16_t>(r[1] & 0xffffu)),
                                  e4m3x2_to_half2_bits(static_cast<uint16_t>(r[0] >> 16)),
                                  e4m3x2_to_half2_bits(static_cast<uint16_t>(r[1] >> 16)), pb0, pb1);
                        mma_16816(ot[2 * pp + 1], e4m3x2_to_half2_bits(static_cast<uint16_t>(r[2] & 0xffffu)),
                                  e4m3x2_to_half2_bits(static_cast<uint16_t>(r[3] & 0xffffu)),
                                  e4m3x2_to_half2_bits(static_cast<uint16_t>(r[2] >> 16)),
                                  e4m3x2_to_half2_bits(static_cast<uint16_t>(r[3] >> 16)), pb0, pb1);
                    }
                } else {
                    #pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        // A = V^T: (dims 16i.., tok 0-7) (dims 16i+8.., tok 0-7) (16i.., tok 8-15) (16i+8.., tok 8-15)
                        const int tok = t16 + (mi >> 1) * 8 + mr, cp = 2 * i + (mi & 1);
                        uint32_t vf[4];
                        ldsm_x4_t(vbase + tile_off(tok, cp * 16), vf);
                        mma_16816(ot[i], vf[0], vf[1], vf[2], vf[3], pb0, pb1);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars[C::NR * NSW + wr * NSW + st]));
        if constexpr (C::PFX) pfx_ticket_resolve<D>(a, ptk, lane);   // the previous item's tickets
        else ticket_resolve<D, G>(a, tk, lane);
        if (C::PFX && (flags & F_LAST)) {
            float la = l2[0], lb = l2[1];
            #pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                la += __shfl_xor_sync(FULL, la, off);
                lb += __shfl_xor_sync(FULL, lb, off);
            }
            // query row r = 2t + h2 belongs to sequence ms + r: its result directly when that
            // sequence has one partition, else its partial and (lane r) its ticket
            auto parts_of_row = [&](int r) {
                const int sm = ms + r, S = s_pfx[sm] & kPfxTokMask;
                return pfx_shared_parts(S, P_eff) + pfx_own_parts(s_ctx[sm], S, P_eff);
            };
            #pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int r = 2 * t + h2;
                if (r >= nq) continue;
                const int64_t sq = static_cast<int64_t>(ms + r) * a.H + mh;
                if (parts_of_row(r) == 1) {
                    const float inv = nt > 0 ? 1.f / (h2 ? lb : la) : 0.f;
                    if (a.out_f16) {
                        __half* dh = static_cast<__half*>(a.out) + sq * D;
                        #pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            dh[16 * i + g] = __float2half_rn(ot[i][h2] * inv);
                            dh[16 * i + 8 + g] = __float2half_rn(ot[i][2 + h2] * inv);
                        }
                    } else {
                        float* dst = static_cast<float*>(a.out) + sq * D;
                        #pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            dst[16 * i + g] = ot[i][h2] * inv;
                            dst[16 * i + 8 + g] = ot[i][2 + h2] * inv;
                        }
                    }
                } else {
                    const int64_t idx = sq * a.max_parts + mpart;
                    if (g == 0) {
                        a.part_ml[2 * idx] = m2[h2];
                        a.part_ml[2 * idx + 1] = h2 ? lb : la;
                    }
                    float* dst = a.part_o + idx * D;
                    #pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        dst[16 * i + g] = ot[i][h2];
                        dst[16 * i + 8 + g] = ot[i][2 + h2];
                    }
                }
            }
            __syncwarp();                               // every row's partial is written
            if (lane < nq) {
                const int np = parts_of_row(lane);
                if (np > 1) {
                    ptk.sq = (ms + lane) * a.H + mh;
                    ptk.np = np;
                    ptk.prev = atom_add_acq_rel_gpu(a.arrivals + ptk.sq, 1u);
                    ptk.pending = true;
                }
            }
        } else if (flags & F_LAST) {
            float la = l2[0], lb = l2[1];
            #pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                la += __shfl_xor_sync(FULL, la, off);
                lb += __shfl_xor_sync(FULL, lb, off);
            }
            const int64_t shk = static_cast<int64_t>(ms) * a.H + mh;
            #pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {              // query 2t + h2
                const int q = 2 * t + h2;
                if (q >= G) continue;
                const int64_t sq = shk * G + q;
                float inv = 1.f;
                float* dst;
                if (flags & F_SINGLE) {
                    inv = nt > 0 ? 1.f / (h2 ? lb : la) : 0.f;
                    if (a.out_f16) {
                        __half* dh = static_cast<__half*>(a.out) + sq * D;
                        #pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            dh[16 * i + g] = __float2half_rn(ot[i][h2] * inv);
                            dh[16 * i + 8 + g] = __float2half_rn(ot[i][2 + h2] * inv);
                        }
                        continue;
                    }
                    dst = static_cast<float*>(a.out) + sq * D;
                } else {
                    const int64_t idx = sq * a.max_parts + mpart;
                    if (g == 0) {
                        a.part_ml[2 * idx] = m2[h2];
                        a.part_ml[2 * idx + 1] = h2 ? lb : la;
                    }
                    dst = a.part_o + idx * D;
                }
                #pragma unroll
                for (int i = 0; i < 8; ++i) {
                    dst[16 * i + g] = ot[i][h2] * inv;
                    dst[16 * i + 8 + g] = ot[i][2 + h2] * inv;
                }
            }
            if (!(flags & F_SINGLE)) {
                const int ctx_s = s_ctx[ms];
                const int np = nparts_of(ctx_s - attend_first(ctx_s, a.window, a.B < CT ? a.B : CT), part_of(P_eff, a, ms));
                ticket_issue(a, tk, shk, mpart, np, lane);
            }
        }
    }
    if constexpr (C::PFX) pfx_ticket_resolve<D>(a, ptk, lane);
    else ticket_resolve<D, G>(a, tk, lane);
}

template <typename C>
__global__ void __launch_bounds__(C::THREADS, C::CPS) attention_partition_kernel(const __grid_constant__ AttnArgs a) {
    constexpr int NC = C::NC, NR = C::NR, NSW = C::NSW, D = C::D, CT = C::CT, TPL = C::TPL, DPL = C::DPL;
    constexpr int CBMAX = C::CBMAX;
    extern __shared__ __align__(128) char smem_raw[];
    // swizzled stages need a 1024-byte aligned base (the slack is part of C::SMEM)
    char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u) * (C::MMA ? 1 : 0);
    static_assert(!C::MMA || (C::STAGE % 1024 == 0 || !C::SWZ_STAGE), "swizzled stages 1024-aligned");
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);   // full[NR*NSW], empty[NR*NSW]
    int* s_ctx = reinterpret_cast<int*>(smem + C::PREFIX_OFF);
    int* s_end = s_ctx + kMaxBatch;
    int* s_pfx = s_ctx + 2 * kMaxBatch;         // shared prefixes (PFX launches only)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int HU = a.H / C::KVH;                // work units (single K/V heads or head groups) per sequence

    if (tid == 0) {
        // full barriers: the producer's arrival (with the copies' bytes); empty barriers: the
        // release by the stage's consumer warp (both warps of a head pair)
        for (int i = 0; i < 2 * NR * NSW; ++i) mbar_init(smem_u32(&bars[i]), i < NR * NSW ? 1 : NC / NR);
        fence_mbar_init();
    }
    if (tid < 32) reinterpret_cast<uint32_t*>(smem + C::ZERO_OFF)[tid] = 0u;   // read after the prologue's sync
    // Programmatic dependent launch: nothing above read global memory.  Wait for the
    // kernels this launch depends on (a no-op when it was launched without that
    // attribute), then let the next launch on the stream begin scheduling: its CTAs start
    // as this launch's CTAs exit and wait here in turn.  With early_tables the caller has
    // written context_lens and block_tables before the previous kernel began, so the
    // prologue and the first block ids are read first and every warp waits just before
    // its first other global access (producer: the first copies and claims; consumers:
    // their first stage).
    const bool early = a.early_tables != 0;
    if (!early) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    // ---- prologue: clamp lengths, items per sequence, inclusive prefix
    for (int s = tid; s < a.batch; s += C::THREADS) {
        int c = a.lens[s];
        if (c < 0 || c > a.ctx_limit) {
            if (blockIdx.x == 0) atomicOr(a.err, KV_DEVERR_CONTEXT);
            c = c < 0 ? 0 : a.ctx_limit;
        }
        s_ctx[s] = c;
        if constexpr (C::PFX) s_pfx[s] = 0;
        else s_end[s] = HU * nparts_of(c - attend_first(c, a.window, a.B < CT ? a.B : CT), part_of(a.P, a, s));
    }
    __syncthreads();
    if constexpr (C::PFX) {
        // This sub-launch's prefix groups: the shared token count of every member, and the
        // member count at the first member.  A group must list 2 to 8 sequences inside this
        // sub-launch, follow the previous group without overlap, share whole blocks, and
        // leave every member at least its newest token of its own when this call appends;
        // one that does not is attended without sharing and flagged.
        for (int gi = tid; gi < a.n_groups; gi += C::THREADS) {
            const int g0 = a.groups[3 * gi], k = a.groups[3 * gi + 1], S = a.groups[3 * gi + 2];
            const int first = g0 - a.s_base;
            if (first < 0 || first >= a.batch) continue;         // another sub-launch's group
            bool ok = k >= 2 && k <= 8 && first + k <= a.batch && S >= 0 && S % a.B == 0 && S <= kPfxTokMask;
            if (ok && gi > 0) ok = a.groups[3 * gi - 3] + a.groups[3 * gi - 2] <= g0;
            for (int m = 0; ok && m < k; ++m) ok = S + a.fused <= s_ctx[first + m];
            if (!ok) {
                if (blockIdx.x == 0) atomicOr(a.err, KV_DEVERR_PREFIX);
                continue;
            }
            if (S == 0) continue;
            for (int m = 0; m < k; ++m) s_pfx[first + m] = S | (m == 0 ? k << 24 : 0);
        }
        __syncthreads();
        for (int s = tid; s < a.batch; s += C::THREADS) {
            const int S = s_pfx[s] & kPfxTokMask, k = s_pfx[s] >> 24;
            s_end[s] = (k ? HU * pfx_shared_parts(S, a.P) : 0) + HU * pfx_own_parts(s_ctx[s], S, a.P);
        }
        __syncthreads();
    }
    int* s_misc = reinterpret_cast<int*>(smem + C::MISC_OFF);
    if (warp == 0) {
        // A launch whose items all fit in one round balances best with the smallest
        // partition that still gives every item a consumer warp: take P_alt when it does.
        int P_eff = a.P;
        if (a.P_alt < a.P) {
            int alt = 0;
            for (int s = lane; s < a.batch; s += 32) {
                const int c = s_ctx[s];
                alt += HU * nparts_of(c - attend_first(c, a.window, a.B < CT ? a.B : CT), a.P_alt);
            }
            alt = __reduce_add_sync(FULL, alt);
            if (alt <= static_cast<int>(gridDim.x) * NR) {
                P_eff = a.P_alt;
                for (int s = lane; s < a.batch; s += 32) {
                    const int c = s_ctx[s];
                    s_end[s] = HU * nparts_of(c - attend_first(c, a.window, a.B < CT ? a.B : CT), a.P_alt);
                }
                __syncwarp();
            }
        }
        if (lane == 0) s_misc[0] = P_eff;
        int carry = 0;
        for (int base = 0; base < a.batch; base += 32) {
            int v = base + lane < a.batch ? s_end[base + lane] : 0;
            #pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int n = __shfl_up_sync(FULL, v, o);
                if (lane >= o) v += n;
            }
            v += carry;
            if (base + lane < a.batch) s_end[base + lane] = v;
            carry = __shfl_sync(FULL, v, 31);
        }
    }
    __syncthreads();
    const int n_items = s_end[a.batch - 1];
    const int P_eff = s_misc[0];                // the launch's partition size

    auto full_bar = [&](int w, int st) { return smem_u32(&bars[w * NSW + st]); };
    auto empty_bar = [&](int w, int st) { return smem_u32(&bars[NR * NSW + w * NSW + st]); };
    auto stage_ptr = [&](int w, int st) { return smem + (w * NSW + st) * C::STAGE; };

    if (warp == NC) {
        // ================================================================ producer
        // Lane w feeds ring w (consumer w, or the head pair of consumers 2w, 2w+1); lanes
        // >= NR only take part in warp votes.
        const bool mine = lane < NR;
        const int w = mine ? lane : 0;
        const int rpc = a.B < CT ? a.B : CT;           // token rows per copy (whole block if B <= CT)
        // bytes per copy: rpc rows of each of the item's KVH heads (adjacent in the pool)
        const uint32_t tile = static_cast<uint32_t>(rpc) * C::ROW * C::KVH;
        // Items are claimed one at a time: the next one only while the current item's last
        // two chunks are filled (its atomic then has a chunk's time to return), so no lane
        // holds more than two items and the tail stays balanced when items are few.
        unsigned pending = 0;                          // claimed next item (atomic in flight)
        bool claimed = false;
        // the first item of every lane is fixed, so the first copies need no atomic round
        // trip; claimed items are numbered after them.  Lane-major order spreads a job with
        // fewer items than consumer warps evenly over the SMs.
        const unsigned first_claim = gridDim.x * NR;
        auto claim = [&]() { pending = atomicAdd(a.counter, 1u) + first_claim; claimed = true; };
        auto decode = [&](unsigned idx) {
            if constexpr (C::PFX)
                return decode_item_pfx<CT>(static_cast<int>(idx), n_items, s_ctx, s_end, s_pfx, a.batch, HU, P_eff);
            else
                return decode_item<CT>(static_cast<int>(idx), n_items, s_ctx, s_end, a.batch, HU, P_eff, a.s_fine,
                                       a.P_fine, a.window, rpc);
        };
        int ids[CBMAX];
        auto load_ids = [&](const Item& it, int chunk) {
            const int nt = it.valid ? min(CT, it.ntok - chunk * CT) : 0;
            const int ncp = nt > 0 ? (nt + rpc - 1) / rpc : 0;
            const int64_t row = static_cast<int64_t>(it.s) * a.max_blocks;
            const int t0 = it.tok0 + chunk * CT;
            #pragma unroll
            for (int j = 0; j < CBMAX; ++j) ids[j] = j < ncp ? a.tables[row + (t0 + j * rpc) / a.B] : 0;
        };
        Item cur{};
        int c = 0, fills = 0;
        bool alive = mine;
        if (mine) {
            cur = decode(lane * gridDim.x + blockIdx.x);
            load_ids(cur, 0);
        }
        // the query rows of cur, into stage st (they complete on that stage's barrier)
        auto copy_q = [&](int st) {
            const uint32_t qdst = C::QR_BYTES ? smem_u32(smem + C::QR_OFF + (w * NSW + st) * C::QR_BYTES)
                                              : smem_u32(stage_ptr(w, st)) + C::Q_OFF;
            if constexpr (C::PFX) {
                // one row per member sequence (rows of one head, H rows apart in q)
                constexpr uint32_t RB = C::D * sizeof(typename C::QT);
                for (int r = 0; r < cur.nq; ++r)
                    bulk_g2s(qdst + r * RB, static_cast<const char*>(a.q) + (static_cast<int64_t>(cur.s + r) * a.H + cur.h) * RB,
                             RB, full_bar(w, st));
            } else {
                const char* qsrc = static_cast<const char*>(a.q) + (static_cast<int64_t>(cur.s) * HU + cur.h) * C::Q_BYTES;
                bulk_g2s(qdst, qsrc, C::Q_BYTES, full_bar(w, st));
            }
        };
        // Fill stage st with chunk c of cur (or the end marker) and advance.  pre: before
        // griddepcontrol.wait (KV_DECODE_EARLY_POOL): K and V tiles only, the query copy
        // is left to q_stage and no item is claimed.
        int q_stage = -1;
        auto fill = [&](int st, bool pre) {
            char* stg = stage_ptr(w, st);
            Meta* meta = reinterpret_cast<Meta*>(smem + C::META_R + (w * NSW + st) * sizeof(Meta));
            const uint32_t fb = full_bar(w, st);
            if (!cur.valid) {
                meta->flags = F_TERM;
                mbar_arrive(fb);
                alive = false;
            } else {
                const int nt = min(CT, cur.ntok - c * CT);     // 0 only for an empty sequence
                const int nblk = nt > 0 ? (nt + rpc - 1) / rpc : 0;   // copies of this chunk
                const int row0 = (cur.tok0 + c * CT) % a.B;   // first row inside the block
                #pragma unroll
                for (int j = 0; j < CBMAX; ++j) {
                    if (j < nblk && (ids[j] < 0 || ids[j] >= a.num_blocks)) {
                        atomicOr(a.err, KV_DEVERR_BLOCK_ID);
                        ids[j] = 0;
                    }
                }
                const bool with_q = (c == 0) && nt > 0 && (C::Q_STAGE > 0 || C::QR_BYTES > 0);
                const uint32_t q_bytes = C::PFX ? cur.nq * C::D * sizeof(typename C::QT) : C::Q_BYTES;
                const uint32_t bytes = nblk * 2 * tile + (with_q ? q_bytes : 0);
                meta->s = cur.s;
                meta->h = cur.h;
                meta->p = cur.p;
                meta->ntok = nt;
                meta->lo = c == 0 ? cur.lo : 0;
                meta->nq = cur.nq;
                // fused append: the sequence's newest token is the last row of the
                // last chunk of its last partition
                const bool patch = a.k_new != nullptr && cur.last && c == cur.nchunks - 1 && nt > 0;
                meta->flags = (c == 0 ? F_FIRST : 0) | (c == cur.nchunks - 1 ? F_LAST : 0) |
                              (cur.single ? F_SINGLE : 0) | (patch ? F_PATCH : 0);
                if (patch) {
                    const int r = nt - 1, jr = r / rpc;
                    int pid = ids[0];
                    #pragma unroll
                    for (int j = 1; j < CBMAX; ++j) if (j == jr) pid = ids[j];
                    meta->patch_row = r;
                    meta->patch_id = pid;
                    meta->patch_off = row0 + r % rpc;
                }
                #pragma unroll
                for (int j = 0; j < CBMAX; ++j) meta->ids[j] = ids[j];
                if (bytes) mbar_arrive_expect_tx(fb, bytes);
                else mbar_arrive(fb);
                const uint32_t dst = smem_u32(stg);
                #pragma unroll
                for (int j = 0; j < CBMAX; ++j) {
                    if (j < nblk) {
                        const int64_t toff = ((static_cast<int64_t>(ids[j]) * a.H + cur.h * C::KVH) * a.B +
                                              row0) * C::ROW;
                        if constexpr (C::SWZ_STAGE) {
                            // rpc token rows of one head as [2][rows][64], 128-byte swizzled
                            const int row = static_cast<int>(toff / C::ROW);
                            tma_load_3d(dst + C::K_OFF + j * tile, &a.kmap, 0, row, 0, fb);
                            tma_load_3d(dst + C::V_OFF + j * tile, &a.vmap, 0, row, 0, fb);
                        } else if constexpr (C::SWZ_K) {
                            // rpc rows of 128 codes each, 128-byte swizzled
                            const int row = static_cast<int>(toff / C::ROW);
                            tma_load_2d(dst + C::K_OFF + j * tile, &a.kmap, 0, row, fb);
                            tma_load_2d(dst + C::V_OFF + j * tile, &a.vmap, 0, row, fb);
                        } else {
                            bulk_g2s(dst + C::K_OFF + j * tile, a.kpool + toff, tile, fb);
                            bulk_g2s(dst + C::V_OFF + j * tile, a.vpool + toff, tile, fb);
                        }
                    }
                }
                if (with_q) {
                    if (pre) q_stage = st;                // copied once the wait has returned
                    else copy_q(st);
                }
                if (pre) {                                // never the item's last chunk: no claim
                    ++c;
                    load_ids(cur, c);
                    return;
                }
                const int rem = cur.nchunks - 1 - c;      // chunks of cur still to fill
                if (rem <= kClaimLead && !claimed) claim();
                if (rem == 0) {
                    if (!claimed) claim();
                    cur = decode(pending);
                    claimed = false;
                    c = 0;
                    if (cur.valid && cur.nchunks - 1 <= kClaimLead) claim();
                } else {
                    ++c;
                }
                load_ids(cur, c);                  // used at this lane's next fill
            }
        };
        // KV_DECODE_EARLY_POOL: the previous kernel on the stream writes no pool row this
        // launch reads except each sequence's last two (context_len - 2: the token the
        // previous decode step appended; context_len - 1: this call's slot), so the first
        // stages of every lane's first item may be filled before the wait: up to NSW full
        // chunks lying wholly below those rows, never the item's last chunk (which would
        // need a claim).
        if (a.early_pool) {
            for (int k = 0; k < NSW; ++k) {
                if (mine && cur.valid && c < cur.nchunks - 1 && cur.tok0 + (c + 1) * CT <= s_ctx[cur.s] - 2) {
                    fill(fills % NSW, true);
                    ++fills;
                }
            }
        }
        if (early) asm volatile("griddepcontrol.wait;" ::: "memory");
        if (q_stage >= 0) copy_q(q_stage);
        if (mine && cur.valid && cur.nchunks - 1 - c <= kClaimLead) claim();
        bool failed = false;
        uint64_t idle_since = 0;
        while (__any_sync(FULL, alive) && !failed) {
            const int st = fills % NSW;
            bool ready = false;
            if (alive) ready = mbar_test_wait(empty_bar(w, st), ((fills / NSW) & 1) ^ 1);
            if (ready) {
                fill(st, false);
                ++fills;
            }
            // watchdog: no stage became free anywhere for about a second -> give up
            if (__any_sync(FULL, ready)) {
                idle_since = 0;
            } else {
                const uint64_t now = global_timer_ns();
                if (idle_since == 0) idle_since = now;
                else if (now - idle_since > kWaitLimitNs) {
                    if (lane == 0) atomicOr(a.err, KV_DEVERR_TIMEOUT);
                    failed = true;
                }
                __nanosleep(32);
            }
        }
        // Drain: every fill this lane issued has landed before the CTA may exit.
        if (mine) {
            for (int st = 0; st < NSW && st < fills; ++st) {
                const int last = fills - 1 - ((fills - 1 - st) % NSW);
                mbar_wait_bounded(full_bar(w, st), (last / NSW) & 1, a.err);
            }
        }
        // The last producer warp of the launch to finish (all claims made and read) leaves
        // the work and exit counters zero for the next call on this workspace.
        if (lane == 0) {
            __threadfence();
            if (atomicAdd(a.exit_counter, 1u) == gridDim.x - 1) {
                *reinterpret_cast<volatile unsigned*>(a.counter) = 0u;
                *reinterpret_cast<volatile unsigned*>(a.exit_counter) = 0u;
            }
        }
        return;
    }

    // ==================================================================== consumer
    if (early) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    if constexpr (C::MMA) {
        consumer_mma<C>(a, smem, s_ctx, warp, lane, P_eff);
        return;
    }
    constexpr int G = C::G, HP = C::HP, GE = C::GE, BR = C::BR, LPR = C::LPR;
    const int w = warp;
    // single heads: the half-warps take alternate tokens (half = which token of each row
    // pair); head groups: lane group e (16 lanes for pairs, 8 for quads) takes head e of
    // the item, every token of the chunk
    const int half = lane / LPR;
    const int sub = lane & (LPR - 1);           // which DPL-element slice of the row
    const int tok_l = HP >= 2 ? (lane & (TPL - 1)) : 2 * (lane & (TPL - 1)) + half;   // token whose score this lane holds
    const bool primary = (lane & (LPR - 1)) < TPL;       // one holder per token when TPL < LPR
    // stage byte offset of token row t (of the lane's head, from its K/V base): with head
    // pairs each copy holds BR rows of head 0, then BR rows of head 1
    auto tok_off = [](int t) -> int {
        if constexpr (HP >= 2) return (t / BR) * HP * BR * C::ROW + (t % BR) * C::ROW;
        else return t * C::ROW;
    };
    const int head_off = HP >= 2 ? half * BR * C::ROW : half * C::ROW;
    // fp16 and FP8 rows with fp16 queries: products of fp16 operands accumulated in fp32
    // (fma.f32.f16), no widening of the K/V elements; the query stays unscaled fp16 and
    // the score scale multiplies the reduced dot product.  fp32 pools: fp32 throughout.
    constexpr bool MX = C::ESZ <= 2 && sizeof(typename C::QT) == 2;
    uint32_t qh[G][DPL / 2];
    float2 q2[G][DPL / 2], acc[G][DPL / 2];
    float m[G], lsum[G];
    #pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = -CUDART_INF_F;
        lsum[g] = 0.f;
        #pragma unroll
        for (int i = 0; i < DPL / 2; ++i) {
            q2[g][i] = make_float2(0.f, 0.f);
            qh[g][i] = 0u;
            acc[g][i] = make_float2(0.f, 0.f);
        }
    }
    Ticket tk{};

    for (int j = 0;; ++j) {
        const int st = j % NSW;
        const uint32_t par = (j / NSW) & 1;
        const uint32_t fb = full_bar(w, st);
        if (!mbar_wait_bounded(fb, par, a.err)) {
            mbar_wait_bounded(fb, par, a.err);      // let copies in flight land, then leave
            break;
        }
        const char* stg = stage_ptr(w, st);
        const char* mst = smem + C::META_R + (w * NSW + st) * sizeof(Meta);
        struct { int s, h, p, ntok, flags; } meta;
        {
            const int4 m0 = *reinterpret_cast<const int4*>(mst);
            meta.s = m0.x; meta.h = m0.y; meta.p = m0.z; meta.ntok = m0.w;
            meta.flags = reinterpret_cast<const Meta*>(mst)->flags;
        }
        if (meta.flags & F_TERM) break;
        const int nt = meta.ntok;
        const int lo = reinterpret_cast<const Meta*>(mst)->lo;
        if (meta.flags & F_FIRST) {
            #pragma unroll
            for (int g = 0; g < G; ++g) {
                m[g] = -CUDART_INF_F;
                lsum[g] = 0.f;
                #pragma unroll
                for (int i = 0; i < DPL / 2; ++i) acc[g][i] = make_float2(0.f, 0.f);
                const char* qrow = stg + C::Q_OFF + (HP >= 2 ? half : g) * D * sizeof(typename C::QT);
                if constexpr (MX) {
                    if (nt > 0) {
                        const uint32_t* qp = reinterpret_cast<const uint32_t*>(qrow) + sub * (DPL / 2);
                        #pragma unroll
                        for (int i = 0; i < DPL / 2; ++i) qh[g][i] = qp[i];
                    }
                } else {
                    if (nt > 0) load_q<C>(qrow, sub, a.qscale, q2[g]);
                }
            }
        }
        if (meta.flags & F_PATCH) {
            // this warp owns the stage now: put the new token into its row and its slot
            const Meta* mp = reinterpret_cast<const Meta*>(mst);
            const int r = mp->patch_row;
            float ksc = 1.f, vsc = 1.f;
            if constexpr (C::FP8) {
                ksc = __ldg(a.kscale + mp->patch_id);
                vsc = __ldg(a.vscale + mp->patch_id);
            }
            char* srow = const_cast<char*>(stg);
            #pragma unroll
            for (int e = 0; e < HP; ++e) {          // every head of the item
                const int head = meta.h * HP + e;
                const int64_t sh = static_cast<int64_t>(meta.s) * a.H + head;
                const int64_t grow = (static_cast<int64_t>(mp->patch_id) * a.H + head) * a.B + mp->patch_off;
                const int so = tok_off(r) + (HP >= 2 ? e * BR * C::ROW : 0);
                patch_row<C>(a.k_new + sh * D * a.in_bytes, a.in_bytes, srow + C::K_OFF + so,
                             a.kpool + grow * C::ROW, ksc, lane);
                patch_row<C>(a.v_new + sh * D * a.in_bytes, a.in_bytes, srow + C::V_OFF + so,
                             a.vpool + grow * C::ROW, vsc, lane);
            }
            // the stage is refilled by the TMA engine later: order these generic writes first
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
        }
        if (nt > 0) {
            float ks = 1.f, vs = 1.f;
            if constexpr (C::FP8) {
                // per-block scales of this lane's token, loaded now and used after the dot
                // products; the producer validated the ids
                const int id = reinterpret_cast<const Meta*>(mst)->ids[tok_l / (a.B < CT ? a.B : CT)];
                ks = __ldg(a.kscale + id);
                vs = __ldg(a.vscale + id);
            }
            const char* K = stg + C::K_OFF + head_off;
            const char* V = stg + C::V_OFF + head_off;
            float part[G][TPL];
            #pragma unroll
            for (int i = 0; i < TPL; ++i) {          // token 2i + half (pairs: i); one K load serves G queries
                if constexpr (MX) {
                    uint32_t kx[DPL / 2];
                    load_row_h<C>(K + tok_off(HP >= 2 ? i : 2 * i), sub, kx);
                    #pragma unroll
                    for (int g = 0; g < G; ++g) {
                        float2 d2 = make_float2(0.f, 0.f);
                        #pragma unroll
                        for (int u = 0; u < DPL / 2; ++u) d2 = hfma2_f32(qh[g][u], kx[u], d2);
                        part[g][i] = d2.x + d2.y;
                    }
                } else {
                    float2 kx[DPL / 2];
                    load_row<C>(K + tok_off(HP >= 2 ? i : 2 * i), sub, kx);
                    #pragma unroll
                    for (int g = 0; g < G; ++g) {
                        float2 d2 = make_float2(0.f, 0.f);
                        #pragma unroll
                        for (int u = 0; u < DPL / 2; ++u) d2 = ffma2(q2[g][u], kx[u], d2);
                        part[g][i] = d2.x + d2.y;
                    }
                }
            }
            // log2-domain score scale of this lane's token (FP8: times its block's K scale)
            const float xs = MX ? (C::FP8 ? ks * a.qscale : a.qscale) : (C::FP8 ? ks : 1.f);
            float pv[G];
            #pragma unroll
            for (int g = 0; g < G; ++g) {
                // transpose-reduce over the 16 lanes of each half: lane ends with token tok_l
                #pragma unroll
                for (int off = TPL / 2; off >= 1; off >>= 1) {
                    const bool upper = (lane & off) != 0;
                    #pragma unroll
                    for (int i = 0; i < off; ++i) {
                        const float send = upper ? part[g][i] : part[g][i + off];
                        const float keep = upper ? part[g][i + off] : part[g][i];
                        part[g][i] = keep + __shfl_xor_sync(FULL, send, off);
                    }
                }
                float x = part[g][0];
                #pragma unroll
                for (int off = TPL; off < LPR; off <<= 1) x += __shfl_xor_sync(FULL, x, off);
                x *= xs;
                x = (tok_l < nt && tok_l >= lo) ? x : -CUDART_INF_F;
                if (__any_sync(FULL, x > m[g] + 8.f)) {   // raise the running max only when needed
                    const float m_new = fmaxf(m[g], HP >= 2 ? group_max<LPR>(x) : warp_max(x));
                    const float corr = ex2_approx(m[g] - m_new);
                    lsum[g] *= corr;
                    #pragma unroll
                    for (int i = 0; i < DPL / 2; ++i) { acc[g][i].x *= corr; acc[g][i].y *= corr; }
                    m[g] = m_new;
                }
                const float pr = ex2_approx(x - m[g]);
                if (primary) lsum[g] += pr;
                pv[g] = pr * vs;
            }
            // MX: p goes to the V products as fp16 (as the tensor-core consumer's P operand
            // does), packed once per lane and broadcast packed.  Measured against fp32 p with
            // widened V: 0.5 % faster on the 13B step, 2-4 % on FP8 pools.
            constexpr bool PH = MX;
            uint32_t pvh[G];
            #pragma unroll
            for (int g = 0; g < G; ++g) pvh[g] = PH ? pack_half2(pv[g], pv[g]) : 0u;
            #pragma unroll
            for (int i = 0; i < TPL; ++i) {          // token 2i + half (pairs: i), its p from lane i (+16)
                const int ti = HP >= 2 ? i : 2 * i + half;
                if constexpr (PH) {
                    uint32_t ph[G];
                    #pragma unroll
                    for (int g = 0; g < G; ++g) ph[g] = __shfl_sync(FULL, pvh[g], i + (lane & ~(LPR - 1)));
                    if ((nt == CT && lo == 0) || (ti < nt && ti >= lo)) {
                        uint32_t vx[DPL / 2];
                        load_row_h<C>(V + tok_off(HP >= 2 ? i : 2 * i), sub, vx);
                        #pragma unroll
                        for (int g = 0; g < G; ++g) {
                            #pragma unroll
                            for (int u = 0; u < DPL / 2; ++u) acc[g][u] = hfma2_f32(ph[g], vx[u], acc[g][u]);
                        }
                    }
                } else {
                    float pt[G];
                    #pragma unroll
                    for (int g = 0; g < G; ++g) pt[g] = __shfl_sync(FULL, pv[g], i + (lane & ~(LPR - 1)));
                    if ((nt == CT && lo == 0) || (ti < nt && ti >= lo)) {
                        float2 vx[DPL / 2];
                        load_row<C>(V + tok_off(HP >= 2 ? i : 2 * i), sub, vx);
                        #pragma unroll
                        for (int g = 0; g < G; ++g) {
                            const float2 p2 = make_float2(pt[g], pt[g]);
                            #pragma unroll
                            for (int u = 0; u < DPL / 2; ++u) acc[g][u] = ffma2(p2, vx[u], acc[g][u]);
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(w, st));
        ticket_resolve<D, GE>(a, tk, lane);           // the previous item's ticket
        if (meta.flags & F_LAST) {
            const int64_t shk = static_cast<int64_t>(meta.s) * HU + meta.h;   // (sequence, work unit)
            #pragma unroll
            for (int g = 0; g < G; ++g) {
                const float l = HP >= 2 ? group_sum<LPR>(lsum[g]) : warp_sum(lsum[g]);
                float2 o[DPL / 2];
                #pragma unroll
                for (int i = 0; i < DPL / 2; ++i) {
                    if constexpr (HP >= 2) {
                        o[i] = acc[g][i];              // each lane group holds its own head
                    } else {                           // the two halves saw different tokens
                        o[i].x = acc[g][i].x + __shfl_xor_sync(FULL, acc[g][i].x, 16);
                        o[i].y = acc[g][i].y + __shfl_xor_sync(FULL, acc[g][i].y, 16);
                    }
                }
                const int64_t sq = shk * GE + (HP >= 2 ? half : g);   // (sequence, query head)
                if (meta.flags & F_SINGLE) {
                    if (HP >= 2 || half == 0) {
                        const float inv = nt > 0 ? 1.f / l : 0.f;   // empty sequence -> zeros
                        if (a.out_f16) {
                            __half2* dst = reinterpret_cast<__half2*>(static_cast<__half*>(a.out) + sq * D + sub * DPL);
                            #pragma unroll
                            for (int i = 0; i < DPL / 2; ++i)
                                dst[i] = __floats2half2_rn(nt > 0 ? o[i].x * inv : 0.f, nt > 0 ? o[i].y * inv : 0.f);
                        } else {
                            float2* dst = reinterpret_cast<float2*>(static_cast<float*>(a.out) + sq * D + sub * DPL);
                            #pragma unroll
                            for (int i = 0; i < DPL / 2; ++i)
                                dst[i] = nt > 0 ? make_float2(o[i].x * inv, o[i].y * inv) : make_float2(0.f, 0.f);
                        }
                    }
                } else {
                    const int64_t idx = sq * a.max_parts + meta.p;
                    if (HP >= 2 ? sub == 0 : lane == 0) {
                        a.part_ml[2 * idx] = m[g];
                        a.part_ml[2 * idx + 1] = l;
                    }
                    if (HP >= 2 || half == 0) {
                        float2* dst = reinterpret_cast<float2*>(a.part_o + idx * D + sub * DPL);
                        #pragma unroll
                        for (int i = 0; i < DPL / 2; ++i) dst[i] = o[i];
                    }
                }
            }
            if (!(meta.flags & F_SINGLE)) {
                // publish the partials, then take a ticket; the last partition merges
                const int ctx_s = s_ctx[meta.s];
                const int np = nparts_of(ctx_s - attend_first(ctx_s, a.window, a.B < CT ? a.B : CT),
                                         part_of(P_eff, a, meta.s));
                ticket_issue(a, tk, shk, meta.p, np, lane);
            }
        }
    }
    ticket_resolve<D, GE>(a, tk, lane);
}

template <typename C>
int launch_typed(const kv_pool* pool, AttnArgs args, const AttnPlan& plan, unsigned* counters,
                 cudaStream_t stream) {
    // the shared-memory opt-in is a per-device function attribute
    static unsigned long long attr_done = 0;
    const unsigned long long bit = 1ull << (pool->device & 63);
    if (!(attr_done & bit)) {
        if (cudaFuncSetAttribute(attention_partition_kernel<C>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return KV_ERR_CUDA;
        // the whole unified L1 / shared array as shared memory, so C::CPS CTAs fit per SM
        if (C::CPS > 1 && cudaFuncSetAttribute(attention_partition_kernel<C>,
                                               cudaFuncAttributePreferredSharedMemoryCarveout,
                                               cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            return KV_ERR_CUDA;
        attr_done |= bit;
    }
    const int total = args.batch;
    const size_t qrow = static_cast<size_t>(args.H) * C::GO * C::D * sizeof(typename C::QT);
    for (int s0 = 0, sub = 0; s0 < total; s0 += kMaxBatch, ++sub) {
        AttnArgs sa = args;
        sa.batch = total - s0 < kMaxBatch ? total - s0 : kMaxBatch;
        sa.q = static_cast<const char*>(args.q) + s0 * qrow;
        sa.out = static_cast<char*>(args.out) +
                 static_cast<int64_t>(s0) * args.H * C::GO * C::D * (args.out_f16 ? 2 : 4);
        sa.tables = args.tables + static_cast<int64_t>(s0) * args.max_blocks;
        sa.lens = args.lens + s0;
        if (args.k_new) {
            const int64_t nofs = static_cast<int64_t>(s0) * args.H * C::D * args.in_bytes;
            sa.k_new = args.k_new + nofs;
            sa.v_new = args.v_new + nofs;
        }
        const int64_t pofs = static_cast<int64_t>(s0) * args.H * C::GO * args.max_parts;
        if (args.part_ml) {
            sa.part_ml = args.part_ml + 2 * pofs;
            sa.part_o = args.part_o + pofs * C::D;
            sa.arrivals = args.arrivals + static_cast<int64_t>(s0) * args.H;
            if (args.grp_arrivals) sa.grp_arrivals = args.grp_arrivals + static_cast<int64_t>(s0) * args.H * args.n_grp;
        }
        sa.s_fine = args.s_fine - s0 > 0 ? args.s_fine - s0 : 0;
        sa.s_base = s0;
        sa.counter = counters + sub;
        sa.exit_counter = counters + kMaxSub + sub;
        const int64_t upper = static_cast<int64_t>(sa.batch) * (args.H / C::KVH) * args.max_parts;
        int64_t grid = (upper + C::NR - 1) / C::NR;
        if (grid > static_cast<int64_t>(pool->num_sms) * C::CPS) grid = static_cast<int64_t>(pool->num_sms) * C::CPS;
        if (grid < 1) grid = 1;
        if (plan.flags & KV_DECODE_PDL) {
            // may begin while the previous kernel on the stream finishes (see the kernel)
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(static_cast<unsigned>(grid));
            cfg.blockDim = dim3(C::THREADS);
            cfg.dynamicSmemBytes = C::SMEM;
            cfg.stream = stream;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaLaunchKernelEx(&cfg, attention_partition_kernel<C>, sa) != cudaSuccess) {
                cudaGetLastError();
                return KV_ERR_CUDA;
            }
        } else {
            attention_partition_kernel<C><<<static_cast<int>(grid), C::THREADS, C::SMEM, stream>>>(sa);
        }
        if (cudaGetLastError() != cudaSuccess) return KV_ERR_CUDA;
    }
    return KV_OK;
}

}  // namespace
}  // namespace kvp
