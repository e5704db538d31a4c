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
// * Work items are (sequence, head, partition) triples; a partition is P tokens
//   (split-context, flash-decoding style).  Items are handed out dynamically with one
//   atomic counter, so ragged batches balance.
// * Each CTA is persistent (one per SM): warp NC is a producer, warps 0..NC-1 are
//   consumers.  The producer streams each item as chunks of CT = 32 tokens: for every
//   physical block in the chunk it issues one 1-D bulk copy (cp.async.bulk, the TMA
//   engine) of the contiguous (block, head) K tile and one of the V tile into the
//   consumer's shared-memory ring, completing on an mbarrier.  The block-table entries
//   of an item are loaded one item ahead by the 32 producer lanes.
// * A consumer owns NSW ring stages.  Per chunk: each lane holds head_dim/32 dims of q;
//   32 partial dot products are transpose-reduced across the warp so that lane t ends
//   with token t's score; fp32 online softmax (log2 domain) with a running max; the
//   V tile is accumulated in fp32 with p_t broadcast by shuffle.  ("KV Cache篇" §6.3:
//   tiles in on-chip SRAM, softmax kept in on-chip state.)
// * A sequence that fits one partition is normalised and written directly; longer
//   ones write (m, l, o) partials merged by reduce_kernel (exact log-sum-exp merge).
//
// No tensor cores: one query row per head is a matrix-vector product bound by HBM.

#include <math_constants.h>

#include "kvp_internal.cuh"

namespace kvp {
namespace {

constexpr int CT = 32;             // tokens per chunk: lane t <-> token t after the reduce
constexpr int kMaxBatch = 1024;    // sequences per launch (prefix table in shared memory)
constexpr int kMaxSub = 64;        // launches per call -> batch <= 65536
constexpr unsigned FULL = 0xffffffffu;

enum : int { F_FIRST = 1, F_LAST = 2, F_TERM = 4, F_SINGLE = 8 };

struct __align__(16) Meta {
    int s, h, p, ntok;      // item (sequence, head, partition); valid tokens in the chunk
    int flags, scidx, pad0, pad1;   // scidx: 2 bits per block = (id & 3) for FP8 scales
};

constexpr int round_up(int a, int b) { return (a + b - 1) / b * b; }

template <int D_, typename KV_, typename QT_>
struct Cfg {
    static constexpr int D = D_;
    using KV = KV_;
    using QT = QT_;
    static constexpr int ESZ = sizeof(KV);
    static constexpr int DPL = D / 32;                    // dims per lane
    static constexpr bool FP8 = (ESZ == 1);
    static constexpr int ROW = D * ESZ;                   // bytes of one token row of one head
    static constexpr int KV_BYTES = CT * ROW;             // bytes of K (or V) per chunk
    static constexpr int Q_BYTES = D * sizeof(QT);
    static constexpr int SC_BYTES = FP8 ? 2 * 4 * 16 : 0; // <= 4 blocks per chunk, K and V
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = KV_BYTES;
    static constexpr int Q_OFF = 2 * KV_BYTES;
    static constexpr int SC_OFF = Q_OFF + Q_BYTES;
    static constexpr int META_OFF = SC_OFF + SC_BYTES;
    static constexpr int STAGE = round_up(META_OFF + (int)sizeof(Meta), 128);
    static constexpr int NC = STAGE <= 9 * 1024 ? 8 : (STAGE <= 17 * 1024 ? 4 : 3);
    static constexpr int NSW = STAGE <= 17 * 1024 ? 3 : 2;
    static constexpr int THREADS = (NC + 1) * 32;
    static constexpr int BAR_OFF = NC * NSW * STAGE;
    static constexpr int PREFIX_OFF = BAR_OFF + 2 * NC * NSW * 8;
    static constexpr int PSTATE_OFF = PREFIX_OFF + 2 * kMaxBatch * 4;
    static constexpr int SMEM = PSTATE_OFF + 2 * NC * 32;
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    static_assert(Q_OFF % 16 == 0 && SC_OFF % 16 == 0 && META_OFF % 16 == 0, "alignment");
};

struct AttnArgs {
    const char* kpool;
    const char* vpool;
    const float* kscale;
    const float* vscale;
    const void* q;
    float* out;
    const int32_t* tables;
    const int32_t* lens;
    float* part_ml;        // [batch*H*max_parts][2]  (m in log2 units, l)
    float* part_o;         // [batch*H*max_parts][D]  unnormalised
    unsigned* counter;
    int* err;
    int batch, H, B, max_blocks, ctx_limit, P, max_parts, num_blocks;
    float qscale;          // scale * log2(e)
};

__device__ __forceinline__ int nparts_of(int ctx, int P) { return ctx <= P ? 1 : (ctx + P - 1) / P; }

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

// lane's DPL elements of one row -> floats
template <typename C>
__device__ __forceinline__ void load_row(const char* row, int lane, float (&x)[C::DPL]) {
    using KV = typename C::KV;
    const char* p = row + lane * C::DPL * C::ESZ;
    if constexpr (C::ESZ == 4) {
        if constexpr (C::DPL == 4) {
            float4 v = *reinterpret_cast<const float4*>(p);
            x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
        } else {
            float2 v = *reinterpret_cast<const float2*>(p);
            x[0] = v.x; x[1] = v.y;
        }
    } else if constexpr (C::ESZ == 2) {
        if constexpr (C::DPL == 4) {
            uint2 v = *reinterpret_cast<const uint2*>(p);
            float2 a = __half22float2(*reinterpret_cast<__half2*>(&v.x));
            float2 b = __half22float2(*reinterpret_cast<__half2*>(&v.y));
            x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
        } else {
            uint32_t v = *reinterpret_cast<const uint32_t*>(p);
            float2 a = __half22float2(*reinterpret_cast<__half2*>(&v));
            x[0] = a.x; x[1] = a.y;
        }
    } else {
        if constexpr (C::DPL == 4) {
            uint32_t v = *reinterpret_cast<const uint32_t*>(p);
            float2 a = e4m3x2_to_float2(static_cast<uint16_t>(v & 0xffffu));
            float2 b = e4m3x2_to_float2(static_cast<uint16_t>(v >> 16));
            x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
        } else {
            uint16_t v = *reinterpret_cast<const uint16_t*>(p);
            float2 a = e4m3x2_to_float2(v);
            x[0] = a.x; x[1] = a.y;
        }
    }
    (void)sizeof(KV);
}

template <typename C>
__device__ __forceinline__ void load_q(const char* qrow, int lane, float qs, float (&x)[C::DPL]) {
    using QT = typename C::QT;
    const QT* p = reinterpret_cast<const QT*>(qrow) + lane * C::DPL;
    #pragma unroll
    for (int i = 0; i < C::DPL; ++i) x[i] = static_cast<float>(p[i]) * qs;
}

// Item decode shared by the producer: (s, h, p) of compact item index `it`.
struct __align__(16) Item {
    int s, h, p, tok0, ntok, nchunks, single, valid;
};
static_assert(sizeof(Item) == 32, "producer state slot");

__device__ __forceinline__ Item decode_item(int it, int n_items, const int* s_ctx, const int* s_end,
                                            int batch, int H, int P) {
    Item r{};
    r.valid = it < n_items;
    if (!r.valid) return r;
    int lo = 0, hi = batch - 1;          // first s with s_end[s] > it
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (s_end[mid] > it) hi = mid; else lo = mid + 1;
    }
    const int s = lo;
    const int start = s ? s_end[s - 1] : 0;
    const int ctx = s_ctx[s];
    const int np = nparts_of(ctx, P);
    const int rr = it - start;
    r.s = s;
    r.h = rr / np;
    r.p = rr - r.h * np;
    r.tok0 = r.p * P;
    r.ntok = min(P, ctx - r.tok0);
    r.nchunks = r.ntok > 0 ? (r.ntok + CT - 1) / CT : 1;
    r.single = np == 1;
    return r;
}

template <typename C>
__global__ void __launch_bounds__(C::THREADS, 1) attention_partition_kernel(AttnArgs a) {
    constexpr int NC = C::NC, NSW = C::NSW, D = C::D;
    extern __shared__ __align__(128) char smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);   // full[NC*NSW], empty[NC*NSW]
    int* s_ctx = reinterpret_cast<int*>(smem + C::PREFIX_OFF);
    int* s_end = s_ctx + kMaxBatch;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- prologue: clamp lengths, items per sequence, inclusive prefix
    for (int s = tid; s < a.batch; s += C::THREADS) {
        int c = a.lens[s];
        if (c < 0 || c > a.ctx_limit) {
            if (blockIdx.x == 0) atomicOr(a.err, KV_DEVERR_CONTEXT);
            c = c < 0 ? 0 : a.ctx_limit;
        }
        s_ctx[s] = c;
        s_end[s] = a.H * nparts_of(c, a.P);
    }
    if (tid == 0) {
        for (int i = 0; i < 2 * NC * NSW; ++i) mbar_init(smem_u32(&bars[i]), 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {
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

    auto full_bar = [&](int w, int st) { return smem_u32(&bars[w * NSW + st]); };
    auto empty_bar = [&](int w, int st) { return smem_u32(&bars[NC * NSW + w * NSW + st]); };
    auto stage_ptr = [&](int w, int st) { return smem + (w * NSW + st) * C::STAGE; };

    if (warp == NC) {
        // ================================================================ producer
        // Per consumer stream: the item being streamed (cur) and the next one (nxt),
        // kept in shared memory (warp-uniform values); each lane keeps the physical id
        // of item block `lane` for cur and nxt in registers.
        Item* cur = reinterpret_cast<Item*>(smem + C::PSTATE_OFF);
        Item* nxt = cur + NC;
        unsigned pending = 0;                          // lane 0: next item index (in flight)
        if (lane == 0) pending = atomicAdd(a.counter, 1u);
        int cur_id[NC], nxt_id[NC], chunk[NC], fills[NC];

        auto acquire = [&](Item* slot) -> int {
            const int idx = static_cast<int>(__shfl_sync(FULL, pending, 0));
            if (lane == 0) pending = atomicAdd(a.counter, 1u);
            const Item it = decode_item(idx, n_items, s_ctx, s_end, a.batch, a.H, a.P);
            int id = 0;
            if (it.valid) {
                const int nblk = (it.ntok + a.B - 1) / a.B;
                if (lane < nblk)
                    id = a.tables[static_cast<int64_t>(it.s) * a.max_blocks + it.tok0 / a.B + lane];
            }
            if (lane == 0) *slot = it;
            __syncwarp();
            return id;
        };

        #pragma unroll
        for (int w = 0; w < NC; ++w) {
            cur_id[w] = acquire(&cur[w]);
            nxt_id[w] = acquire(&nxt[w]);
            chunk[w] = 0;
            fills[w] = 0;
        }
        unsigned alive = (1u << NC) - 1u;
        bool failed = false;
        const int CB = CT / a.B;                        // blocks per full chunk
        const uint32_t tile = static_cast<uint32_t>(a.B) * C::ROW;
        while (alive && !failed) {
            #pragma unroll
            for (int w = 0; w < NC; ++w) {
                if (!(alive & (1u << w)) || failed) continue;
                const int st = fills[w] % NSW;
                const uint32_t par = ((fills[w] / NSW) & 1) ^ 1;
                if (!mbar_wait_bounded(empty_bar(w, st), par, a.err)) { failed = true; continue; }
                char* stg = stage_ptr(w, st);
                Meta* meta = reinterpret_cast<Meta*>(stg + C::META_OFF);
                const uint32_t fb = full_bar(w, st);
                const Item it = cur[w];
                if (!it.valid) {
                    if (lane == 0) {
                        meta->flags = F_TERM;
                        mbar_arrive(fb);
                    }
                    alive &= ~(1u << w);
                } else {
                    const int c = chunk[w];
                    const int nt = min(CT, it.ntok - c * CT);      // 0 only for an empty sequence
                    const int nblk = nt > 0 ? (nt + a.B - 1) / a.B : 0;
                    // block ids of this chunk: item block c*CB + j lives in producer lane c*CB + j
                    int id = __shfl_sync(FULL, cur_id[w], (c * CB + lane) & 31);
                    if (lane < nblk && (id < 0 || id >= a.num_blocks)) {
                        atomicOr(a.err, KV_DEVERR_BLOCK_ID);
                        id = 0;
                    }
                    int scidx = 0;
                    if constexpr (C::FP8) {
                        const int bits = lane < nblk ? ((id & 3) << (2 * lane)) : 0;
                        scidx = __reduce_or_sync(FULL, bits);
                    }
                    const bool with_q = (c == 0) && nt > 0;
                    const uint32_t bytes = nblk * (2 * tile + (C::FP8 ? 32u : 0u)) +
                                           (with_q ? C::Q_BYTES : 0);
                    if (lane == 0) {
                        meta->s = it.s;
                        meta->h = it.h;
                        meta->p = it.p;
                        meta->ntok = nt;
                        meta->flags = (c == 0 ? F_FIRST : 0) | (c == it.nchunks - 1 ? F_LAST : 0) |
                                      (it.single ? F_SINGLE : 0);
                        meta->scidx = scidx;
                        if (bytes) mbar_arrive_expect_tx(fb, bytes);
                        else mbar_arrive(fb);
                    }
                    __syncwarp();
                    if (lane < nblk) {
                        const int64_t toff = (static_cast<int64_t>(id) * a.H + it.h) * tile;
                        const uint32_t dst = smem_u32(stg) + lane * tile;
                        bulk_g2s(dst + C::K_OFF, a.kpool + toff, tile, fb);
                        bulk_g2s(dst + C::V_OFF, a.vpool + toff, tile, fb);
                        if constexpr (C::FP8) {
                            const uint32_t sc = smem_u32(stg) + C::SC_OFF + lane * 16;
                            bulk_g2s(sc, a.kscale + (id & ~3), 16, fb);
                            bulk_g2s(sc + 64, a.vscale + (id & ~3), 16, fb);
                        }
                    }
                    if (with_q && lane == 0) {
                        const char* qsrc = static_cast<const char*>(a.q) +
                                           (static_cast<int64_t>(it.s) * a.H + it.h) * C::Q_BYTES;
                        bulk_g2s(smem_u32(stg) + C::Q_OFF, qsrc, C::Q_BYTES, fb);
                    }
                    if (++chunk[w] == it.nchunks) {
                        const Item n = nxt[w];
                        __syncwarp();
                        if (lane == 0) cur[w] = n;
                        cur_id[w] = nxt_id[w];
                        chunk[w] = 0;
                        if (n.valid) {
                            nxt_id[w] = acquire(&nxt[w]);
                        } else {
                            __syncwarp();
                        }
                    }
                }
                ++fills[w];
                __syncwarp();
            }
        }
        // Drain: every fill this warp issued has landed before the CTA may exit.
        #pragma unroll
        for (int w = 0; w < NC; ++w) {
            for (int st = 0; st < NSW && st < fills[w]; ++st) {
                const int last = fills[w] - 1 - ((fills[w] - 1 - st) % NSW);
                mbar_wait_bounded(full_bar(w, st), (last / NSW) & 1, a.err);
            }
        }
        return;
    }

    // ==================================================================== consumer
    const int w = warp;
    float qf[C::DPL], acc[C::DPL];
    float m = -CUDART_INF_F, lsum = 0.f;
    #pragma unroll
    for (int i = 0; i < C::DPL; ++i) { qf[i] = 0.f; acc[i] = 0.f; }

    for (int j = 0;; ++j) {
        const int st = j % NSW;
        const uint32_t par = (j / NSW) & 1;
        const uint32_t fb = full_bar(w, st);
        if (!mbar_wait_bounded(fb, par, a.err)) {
            mbar_wait_bounded(fb, par, a.err);      // let copies in flight land, then leave
            break;
        }
        const char* stg = stage_ptr(w, st);
        const Meta meta = *reinterpret_cast<const Meta*>(stg + C::META_OFF);
        if (meta.flags & F_TERM) break;
        const int nt = meta.ntok;
        if (meta.flags & F_FIRST) {
            m = -CUDART_INF_F;
            lsum = 0.f;
            #pragma unroll
            for (int i = 0; i < C::DPL; ++i) acc[i] = 0.f;
            if (nt > 0) load_q<C>(stg + C::Q_OFF, lane, a.qscale, qf);
        }
        if (nt > 0) {
            const char* K = stg + C::K_OFF;
            const char* V = stg + C::V_OFF;
            float part[CT];
            #pragma unroll
            for (int t = 0; t < CT; ++t) {
                float kx[C::DPL];
                load_row<C>(K + t * C::ROW, lane, kx);
                float d = 0.f;
                #pragma unroll
                for (int i = 0; i < C::DPL; ++i) d = fmaf(qf[i], kx[i], d);
                part[t] = d;
            }
            // transpose-reduce: after the loop lane t holds the full dot product of token t
            #pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                const bool upper = (lane & off) != 0;
                #pragma unroll
                for (int i = 0; i < off; ++i) {
                    const float send = upper ? part[i] : part[i + off];
                    const float keep = upper ? part[i + off] : part[i];
                    part[i] = keep + __shfl_xor_sync(FULL, send, off);
                }
            }
            float x = part[0];
            float vs = 1.f;
            if constexpr (C::FP8) {
                const int blk = lane / a.B;                 // block of token `lane` in the chunk
                const int sub = (meta.scidx >> (2 * blk)) & 3;
                const float* sc = reinterpret_cast<const float*>(stg + C::SC_OFF);
                x *= sc[blk * 4 + sub];
                vs = sc[16 + blk * 4 + sub];
            }
            x = lane < nt ? x : -CUDART_INF_F;
            const float m_new = fmaxf(m, warp_max(x));
            const float corr = ex2_approx(m - m_new);
            const float pr = ex2_approx(x - m_new);
            lsum = fmaf(lsum, corr, pr);
            #pragma unroll
            for (int i = 0; i < C::DPL; ++i) acc[i] *= corr;
            const float pv = pr * vs;
            if (nt == CT) {
                #pragma unroll
                for (int t = 0; t < CT; ++t) {
                    const float pt = __shfl_sync(FULL, pv, t);
                    float vx[C::DPL];
                    load_row<C>(V + t * C::ROW, lane, vx);
                    #pragma unroll
                    for (int i = 0; i < C::DPL; ++i) acc[i] = fmaf(pt, vx[i], acc[i]);
                }
            } else {
                #pragma unroll
                for (int t = 0; t < CT; ++t) {
                    if (t < nt) {
                        const float pt = __shfl_sync(FULL, pv, t);
                        float vx[C::DPL];
                        load_row<C>(V + t * C::ROW, lane, vx);
                        #pragma unroll
                        for (int i = 0; i < C::DPL; ++i) acc[i] = fmaf(pt, vx[i], acc[i]);
                    }
                }
            }
            m = m_new;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(w, st));
        if (meta.flags & F_LAST) {
            const float l = warp_sum(lsum);
            const int64_t sh = static_cast<int64_t>(meta.s) * a.H + meta.h;
            if (meta.flags & F_SINGLE) {
                float* o = a.out + sh * D + lane * C::DPL;
                const float inv = nt > 0 ? 1.f / l : 0.f;   // empty sequence -> zeros
                #pragma unroll
                for (int i = 0; i < C::DPL; ++i) o[i] = nt > 0 ? acc[i] * inv : 0.f;
            } else {
                const int64_t idx = sh * a.max_parts + meta.p;
                if (lane == 0) {
                    a.part_ml[2 * idx] = m;
                    a.part_ml[2 * idx + 1] = l;
                }
                float* o = a.part_o + idx * D + lane * C::DPL;
                #pragma unroll
                for (int i = 0; i < C::DPL; ++i) o[i] = acc[i];
            }
        }
    }
}

// Merge the partials of every (sequence, head) split into more than one partition:
// M = max m_p, L = sum l_p 2^(m_p - M), out = sum o_p 2^(m_p - M) / L.
template <int D>
__global__ void __launch_bounds__(256) attention_reduce_kernel(AttnArgs a) {
    constexpr int DPL = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (gw >= static_cast<int64_t>(a.batch) * a.H) return;
    const int s = static_cast<int>(gw / a.H);
    int ctx = a.lens[s];
    ctx = ctx < 0 ? 0 : (ctx > a.ctx_limit ? a.ctx_limit : ctx);
    const int np = nparts_of(ctx, a.P);
    if (np <= 1) return;
    const int64_t base = gw * a.max_parts;
    float mx = -CUDART_INF_F;
    for (int p = lane; p < np; p += 32) mx = fmaxf(mx, a.part_ml[2 * (base + p)]);
    mx = warp_max(mx);
    float L = 0.f, acc[DPL];
    #pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
    for (int p = 0; p < np; ++p) {
        const float wgt = ex2_approx(a.part_ml[2 * (base + p)] - mx);
        L = fmaf(a.part_ml[2 * (base + p) + 1], wgt, L);
        const float* o = a.part_o + (base + p) * D + lane * DPL;
        #pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] = fmaf(wgt, o[i], acc[i]);
    }
    const float inv = 1.f / L;
    float* out = a.out + gw * D + lane * DPL;
    #pragma unroll
    for (int i = 0; i < DPL; ++i) out[i] = acc[i] * inv;
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
        attr_done |= bit;
    }
    const int total = args.batch;
    const size_t qrow = static_cast<size_t>(args.H) * C::D * sizeof(typename C::QT);
    for (int s0 = 0, sub = 0; s0 < total; s0 += kMaxBatch, ++sub) {
        AttnArgs sa = args;
        sa.batch = total - s0 < kMaxBatch ? total - s0 : kMaxBatch;
        sa.q = static_cast<const char*>(args.q) + s0 * qrow;
        sa.out = args.out + static_cast<int64_t>(s0) * args.H * C::D;
        sa.tables = args.tables + static_cast<int64_t>(s0) * args.max_blocks;
        sa.lens = args.lens + s0;
        const int64_t pofs = static_cast<int64_t>(s0) * args.H * args.max_parts;
        if (args.part_ml) {
            sa.part_ml = args.part_ml + 2 * pofs;
            sa.part_o = args.part_o + pofs * C::D;
        }
        sa.counter = counters + sub;
        const int64_t upper = static_cast<int64_t>(sa.batch) * args.H * args.max_parts;
        int64_t grid = (upper + C::NC - 1) / C::NC;
        if (grid > pool->num_sms) grid = pool->num_sms;
        if (grid < 1) grid = 1;
        attention_partition_kernel<C><<<static_cast<int>(grid), C::THREADS, C::SMEM, stream>>>(sa);
        if (cudaGetLastError() != cudaSuccess) return KV_ERR_CUDA;
    }
    if (plan.max_parts > 1) {
        const int64_t warps = static_cast<int64_t>(total) * args.H;
        const int blocks = static_cast<int>((warps + 7) / 8);
        attention_reduce_kernel<C::D><<<blocks, 256, 0, stream>>>(args);
        if (cudaGetLastError() != cudaSuccess) return KV_ERR_CUDA;
    }
    return KV_OK;
}

template <typename C>
int consumers_of() { return C::NC; }

int consumers_for(const kv_pool_desc& d) {
    if (d.dtype == KV_F32) return d.head_dim == 128 ? consumers_of<Cfg<128, float, float>>()
                                                    : consumers_of<Cfg<64, float, float>>();
    if (d.dtype == KV_F16) return d.head_dim == 128 ? consumers_of<Cfg<128, __half, __half>>()
                                                    : consumers_of<Cfg<64, __half, __half>>();
    return d.head_dim == 128 ? consumers_of<Cfg<128, uint8_t, __half>>()
                             : consumers_of<Cfg<64, uint8_t, __half>>();
}

constexpr size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

int plan_attention(const kv_pool* pool, int batch, int max_context, int partition_tokens,
                   AttnPlan* plan) {
    const kv_pool_desc& d = pool->desc;
    if (batch < 0 || max_context < 0 || batch > kMaxBatch * kMaxSub) return KV_ERR_INVALID_ARG;
    const int cap = 32 * d.block_size;             // one producer lane per block of a partition
    const int nc = consumers_for(d);
    int P;
    if (partition_tokens > 0) {
        if (partition_tokens % CT != 0 || partition_tokens > cap) return KV_ERR_INVALID_ARG;
        P = partition_tokens;
    } else if (partition_tokens == 0) {
        const int64_t units = static_cast<int64_t>(batch > 0 ? batch : 1) * d.num_heads;
        const int64_t target = 4ll * pool->num_sms * nc;     // >= 4 items per consumer warp
        int64_t parts = (target + units - 1) / units;
        if (parts < 1) parts = 1;
        int64_t p = (max_context + parts - 1) / parts;
        p = (p + CT - 1) / CT * CT;
        if (p < CT) p = CT;
        if (p > cap) p = cap;
        P = static_cast<int>(p);
    } else {
        return KV_ERR_INVALID_ARG;
    }
    plan->partition = P;
    plan->max_parts = max_context <= P ? 1 : (max_context + P - 1) / P;
    plan->consumers = nc;
    size_t ws = 256;                                // kMaxSub work counters
    if (plan->max_parts > 1) {
        const size_t n = static_cast<size_t>(batch) * d.num_heads * plan->max_parts;
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
    const kv_pool_desc& d = pool->desc;
    if (batch == 0) return KV_OK;
    char* ws = static_cast<char*>(workspace);
    unsigned* counters = reinterpret_cast<unsigned*>(ws);
    const int nsub = (batch + kMaxBatch - 1) / kMaxBatch;
    if (cudaMemsetAsync(counters, 0, nsub * sizeof(unsigned), stream) != cudaSuccess) return KV_ERR_CUDA;

    AttnArgs a{};
    a.kpool = static_cast<const char*>(pool->k_layers[layer]);
    a.vpool = static_cast<const char*>(pool->v_layers[layer]);
    a.kscale = pool->k_scales ? pool->k_scales[layer] : nullptr;
    a.vscale = pool->v_scales ? pool->v_scales[layer] : nullptr;
    a.q = q;
    a.out = out;
    a.tables = block_tables;
    a.lens = context_lens;
    if (plan.max_parts > 1) {
        const size_t n = static_cast<size_t>(batch) * d.num_heads * plan.max_parts;
        a.part_ml = reinterpret_cast<float*>(ws + 256);
        a.part_o = reinterpret_cast<float*>(ws + 256 + align256(n * 2 * sizeof(float)));
    }
    a.err = pool->d_err;
    a.batch = batch;
    a.H = d.num_heads;
    a.B = d.block_size;
    a.max_blocks = max_blocks;
    const int64_t lim_tables = static_cast<int64_t>(max_blocks) * d.block_size;
    a.ctx_limit = static_cast<int>(lim_tables < max_context ? lim_tables : max_context);
    a.P = plan.partition;
    a.max_parts = plan.max_parts;
    a.num_blocks = d.num_blocks;
    a.qscale = scale * 1.4426950408889634f;        // log2(e): softmax evaluated with 2^x

    if (d.dtype == KV_F32) {
        if (d.head_dim == 128) return launch_typed<Cfg<128, float, float>>(pool, a, plan, counters, stream);
        return launch_typed<Cfg<64, float, float>>(pool, a, plan, counters, stream);
    }
    if (d.dtype == KV_F16) {
        if (d.head_dim == 128) return launch_typed<Cfg<128, __half, __half>>(pool, a, plan, counters, stream);
        return launch_typed<Cfg<64, __half, __half>>(pool, a, plan, counters, stream);
    }
    if (d.head_dim == 128) return launch_typed<Cfg<128, uint8_t, __half>>(pool, a, plan, counters, stream);
    return launch_typed<Cfg<64, uint8_t, __half>>(pool, a, plan, counters, stream);
}

}  // namespace kvp
