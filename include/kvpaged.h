/*
 * kvpaged — single-token decode attention over a block-paged KV cache (GB300, sm_103a).
 *
 * C ABI.  Plain pointers and sizes only.  Every device buffer is owned by the
 * caller; the library never frees caller memory.  Every call returns 0 on
 * success or a negative kv_status; no C++ exception crosses this boundary.
 * Device calls are asynchronous on the given stream and never synchronise,
 * except kv_get_device_error.
 *
 * Sources (web pages, cited by title and section):
 *   [KV Cache篇]      "大模型推理加速——KV Cache篇"
 *   [KV缓存机制解析]  "KV缓存机制解析：优化大型语言模型推理性能"
 *   [PagedAttention]  "KV Cache与PagedAttention：大模型推理显存优化方案"
 *
 * Pool layout (per layer, chosen for this library):
 *   K, V: [num_blocks][num_heads][block_size][head_dim] elements of `dtype`.
 *   One (block, head) tile is block_size*head_dim contiguous elements, so a
 *   tile moves as one bulk copy.  Slot id = physical_block * block_size + offset.
 *   FP8 pools add per-layer scale arrays k_scale[], v_scale[]: one float32 per
 *   physical block (shared by all heads), capacity rounded up to a multiple of 4
 *   floats, 16-byte aligned.  Stored value = e4m3 code * scale.
 */
#ifndef KVPAGED_H
#define KVPAGED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported from libkvpaged.so (built with hidden default visibility). */
#if defined(__GNUC__)
#define KV_API __attribute__((visibility("default")))
#else
#define KV_API
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* kv_stream_t;

typedef enum {
    KV_OK = 0,
    KV_ERR_INVALID_ARG = -1,  /* bad pointer, size, alignment, layer, dtype or shape  */
    KV_ERR_NO_BLOCKS = -2,    /* allocator: free list too short; state left unchanged */
    KV_ERR_STATE = -3,        /* allocator: unknown/freed sequence, refcount misuse     */
    KV_ERR_CUDA = -4,         /* a CUDA runtime call failed (launch, query, memcpy)     */
    KV_ERR_DEVICE = -5,       /* kv_get_device_error found a device-side error bit      */
    KV_ERR_UNSUPPORTED = -6   /* valid request this library version does not implement  */
} kv_status;

typedef enum { KV_F32 = 0, KV_F16 = 1, KV_FP8_E4M3 = 2 } kv_dtype;

/* Device-side error bits (kv_get_device_error).  Kernels never trap: they set a
 * bit, skip or clamp the offending access, and finish. */
enum {
    KV_DEVERR_SLOT = 1,        /* slot_mapping entry >= num_blocks*block_size           */
    KV_DEVERR_BLOCK_ID = 2,    /* block table / copy pair id outside [0, num_blocks)    */
    KV_DEVERR_CONTEXT = 4,     /* context_len < 0, > max_blocks*block_size or > max_context */
    KV_DEVERR_TIMEOUT = 8,     /* a bounded mbarrier wait ran out (about one second)    */
    KV_DEVERR_PREFIX = 16      /* a prefix group broke its rules (attended without sharing) */
};

typedef struct {
    int num_layers;   /* >= 1, <= 4096                              */
    int num_blocks;   /* physical blocks per layer, >= 1            */
    int block_size;   /* B: 8, 16 or 32 tokens                      */
    int num_heads;    /* H: 1 .. 256                                */
    int head_dim;     /* d: 64 or 128                               */
    kv_dtype dtype;   /* element type of the pool                   */
} kv_pool_desc;

typedef struct kv_pool kv_pool;    /* opaque; bound to the device current at creation */
typedef struct kv_alloc kv_alloc;  /* opaque; host memory only                        */

typedef struct {
    int num_blocks;        /* pool size                                                 */
    int free_blocks;       /* on the free list                                          */
    int shared_blocks;     /* reference count > 1                                       */
    int num_seqs;          /* live sequences                                            */
    int64_t used_slots;    /* sum over live sequences of their length                   */
    int64_t wasted_slots;  /* sum over live sequences of n_blocks*B - length (tail waste,
                              counted per sequence; [PagedAttention] §2.2)              */
} kv_alloc_stats_t;

/* ---------------------------------------------------------------- misc */

/* Static string for a kv_status value.  Never NULL. */
KV_API const char* kv_status_str(int status);

/* Library ABI version (major*100 + minor). */
KV_API int kv_version(void);

/* ---------------------------------------------------------------- pool */

/* Wrap caller-owned device memory as a paged KV pool.
 *   desc        shape and dtype (validated: see kv_pool_desc).
 *   k_layers, v_layers  host arrays of desc->num_layers device pointers, each to
 *               num_blocks*num_heads*block_size*head_dim elements, 16-byte aligned.
 *   k_scales, v_scales  FP8 only: host arrays of num_layers device pointers to float32
 *               [round_up(num_blocks, 4)], 16-byte aligned; must be NULL otherwise.
 *   out         receives the handle.
 * The pool keeps copies of the pointers, not the memory.  It allocates one small
 * device word for device error bits (its only allocation).
 * Paged storage of the cache: [PagedAttention] §2.1 and §3.1 (global block pool). */
KV_API int kv_pool_create(const kv_pool_desc* desc, void* const* k_layers, void* const* v_layers,
                   float* const* k_scales, float* const* v_scales, kv_pool** out);

/* Release the handle (not the caller's memory).  Synchronises nothing; the caller
 * must not destroy a pool with work still queued on it. */
KV_API int kv_pool_destroy(kv_pool* pool);

/* Copy of the descriptor the pool was created with. */
KV_API int kv_pool_get_desc(const kv_pool* pool, kv_pool_desc* desc);

/* Fast paths the pool was set up with, as bit flags in *flags.
 *   KV_FEATURE_TENSOR_MAPS  fp16 or FP8 pool with head_dim 128: every layer has
 *                           128-byte-swizzled tensor maps of its K and V pools, and
 *                           grouped-query decode (2, 4 or 8 query heads per KV head) runs
 *                           its scores and P V on the tensor cores (FP8: the K and V
 *                           fragments are converted exactly from the E4M3 codes in
 *                           registers).  Without it the same calls run on the CUDA cores
 *                           with identical semantics. */
#define KV_FEATURE_TENSOR_MAPS 1u
KV_API int kv_pool_features(const kv_pool* pool, unsigned* flags);

/* Read (and if clear != 0, reset) the pool's device error bits.  Enqueues a copy on
 * `stream` and synchronises that stream.  Returns KV_ERR_DEVICE if any bit is set
 * (bits in *code), else KV_OK with *code = 0. */
KV_API int kv_get_device_error(kv_pool* pool, kv_stream_t stream, int clear, int* code);

/* Self-test of the kernels' bounded waits (no counterpart on the pages).  Launches one warp
 * on `stream` that waits on a shared-memory mbarrier nothing arrives at, through the same
 * bounded wait every kernel wait uses, with a limit of limit_ns nanoseconds instead of the
 * kernels' one second.  The wait gives up, sets KV_DEVERR_TIMEOUT in the pool's error word
 * and the kernel returns normally: the context stays usable.  limit_ns in [1, 1e9], else
 * KV_ERR_INVALID_ARG.  Asynchronous; read the bit with kv_get_device_error. */
KV_API int kv_selftest_wait_timeout(kv_pool* pool, uint64_t limit_ns, kv_stream_t stream);

/* ---------------------------------------------------------------- append */

/* Write num_tokens new tokens' K and V into their slots for one layer.
 *   k, v           device, [num_tokens][num_heads][head_dim] of in_dtype, 16-byte aligned.
 *                  in_dtype must equal the pool dtype for F32/F16 pools; an FP8 pool
 *                  takes F16 or F32 input and stores
 *                  e4m3 = round-nearest-even-satfinite(fp32(x) / scale[block]), where
 *                  scale[block] is the value already in the layer's scale array
 *                  (the caller sets a fresh block's scale before appending into it).
 *   slot_mapping   device int64 [num_tokens]; slot < 0 means "skip this token".
 * Token i, head h lands at block slot/B, offset slot%B.  Out-of-range slots set
 * KV_DEVERR_SLOT and are skipped.  Bit-exact copy for F32/F16.
 * The cache write of [KV Cache篇] §3.1 (cache_k[:, start_pos] = xk) and
 * write_KV_to_block of [PagedAttention] §3.3. */
KV_API int kv_append(kv_pool* pool, int layer, const void* k, const void* v, kv_dtype in_dtype,
              const int64_t* slot_mapping, int num_tokens, kv_stream_t stream);

/* ---------------------------------------------------------------- copy-on-write */

/* For each pair (src, dst) in pairs (device int32 [num_pairs][2]) copy the whole
 * physical block src onto dst — K and V, every head, all B slots, and for FP8
 * pools both scales — in every layer of [layer_begin, layer_end).  Bit-exact.
 * dst blocks must be distinct and must not appear as a src (result undefined
 * otherwise).  Ids outside [0, num_blocks) set KV_DEVERR_BLOCK_ID and are skipped.
 * copy_block of [PagedAttention] §3.3 (batched, as its "批量处理多个块的CoW" asks). */
KV_API int kv_copy_blocks(kv_pool* pool, const int32_t* pairs, int num_pairs, int layer_begin,
                   int layer_end, kv_stream_t stream);

/* ---------------------------------------------------------------- swap to host memory */

/* Bytes of the host image of num_blocks blocks over layers [layer_begin, layer_end):
 * num_blocks * layers * 2 * (num_heads*block_size*head_dim*element bytes), plus for FP8
 * pools num_blocks * layers * 2 * 4 bytes of scales.  0 on invalid arguments. */
KV_API size_t kv_swap_bytes(const kv_pool* pool, int num_blocks, int layer_begin, int layer_end);

/* Copy the listed physical blocks (device int32 blocks[num_blocks]) of every layer in
 * [layer_begin, layer_end) (at most 64 layers per call) into host_dst: host memory the GPU
 * can address, 16-byte aligned, of kv_swap_bytes bytes — pinned memory (cudaHostAlloc /
 * cudaHostRegister), or on systems with coherent pageable-memory access (e.g. Grace with
 * NVLink-C2C) any host memory; anything else gives KV_ERR_INVALID_ARG.
 * Image layout: for block i, layer l: the K block then the V block (raw [H][B][d]); after
 * all blocks, for FP8 pools, per block and layer the K then the V scale (float32).  One
 * kernel moves everything through the device mapping.  Asynchronous: host_dst is complete
 * when the stream reaches this point.  Ids outside the pool set KV_DEVERR_BLOCK_ID and are
 * skipped.  With the allocator the caller then releases the blocks (kv_alloc_seq_free) to
 * preempt a sequence.
 * Cold blocks moved to CPU memory: [KV缓存机制解析] §6.1 (缓存分块加载) and
 * [PagedAttention] §7.2 (冷块交换到CPU内存). */
KV_API int kv_swap_out(kv_pool* pool, const int32_t* blocks, int num_blocks, int layer_begin, int layer_end,
                       void* host_dst, kv_stream_t stream);

/* The reverse: write an image made by kv_swap_out into the listed (freshly allocated)
 * physical blocks, bit-exact.  Same rules. */
KV_API int kv_swap_in(kv_pool* pool, const void* host_src, const int32_t* blocks, int num_blocks,
                      int layer_begin, int layer_end, kv_stream_t stream);

/* ---------------------------------------------------------------- decode attention */

/* Bytes of device workspace paged_decode_attention needs for these arguments
 * (0 on invalid arguments).  partition_tokens as in paged_decode_attention.  Arguments
 * whose split-context work would exceed 2^30 items per launch of 1024 sequences
 * (min(batch, 1024) x num_heads x ceil(max_context / partition)) are invalid here and in
 * every decode entry point. */
KV_API size_t paged_decode_workspace_size(const kv_pool* pool, int batch, int max_context,
                                   int partition_tokens);

/* Largest batch of one decode-attention call (every entry point); a larger batch is
 * refused with KV_ERR_INVALID_ARG before anything is launched. */
#define KV_MAX_DECODE_BATCH 65536

/* out[s,h,:] = softmax(scale * q[s,h,:] . K_s^T) . V_s  over the first
 * context_lens[s] tokens of sequence s, for every sequence s and head h, read
 * through block_tables.  One query token per sequence (decode); batch 0 ..
 * KV_MAX_DECODE_BATCH.
 *   q             device [batch][num_heads][head_dim]: float32 for F32 pools, float16
 *                 for F16 and FP8 pools; 16-byte aligned.
 *   out           device float32 [batch][num_heads][head_dim] (written, not accumulated).
 *   block_tables  device int32 [batch][max_blocks_per_seq]; entry j of row s is the
 *                 physical block of tokens [j*B, (j+1)*B) of sequence s.
 *   context_lens  device int32 [batch]; includes the token appended this step.
 *                 0 gives out = 0.  Values above min(max_blocks_per_seq*B, max_context)
 *                 are clamped and set KV_DEVERR_CONTEXT.
 *   max_context   host upper bound of context_lens (sizes the split-context workspace).
 *   scale         score multiplier, usually 1/sqrt(head_dim); finite and > 0.
 *   partition_tokens  0 = library choice (about 8 work items per consumer warp, one
 *                 round for grouped-query launches, 256 to 1024 tokens; with 512 or
 *                 more and several rounds of items, the last sequences of the batch
 *                 take half of it; at 256, the kernel splits into 192-token partitions
 *                 when the actual lengths still give every item its own consumer warp,
 *                 and the workspace is sized for that); else tokens per split-context
 *                 partition, a multiple of 32.  Sequences longer than one partition are
 *                 split into equal parts of at most that many tokens, attended per
 *                 partition and merged exactly (log-sum-exp) in the same launch by the
 *                 warp that finishes the last partition of that sequence and head.
 *   workspace     device, >= paged_decode_workspace_size(...) bytes, 256-byte aligned,
 *                 contents need not be initialised; not shared between concurrent calls.
 * Arithmetic: fp32 scores, fp32 online softmax, fp32 accumulation of V.  For F16 and
 * FP8 pools the products are of fp16 operands (q, K and V elements as fp16; E4M3 codes
 * convert to fp16 exactly) accumulated in fp32, and the softmax weights enter the V
 * products as fp16 (relative rounding 2^-11; below 2^8 by the running maximum).  With
 * the FP8 V scale folded into those weights, v_scale values must stay below 255.
 * F32 pools: fp32 operands throughout.
 * The cached decode step of [KV Cache篇] §3.1 / [KV缓存机制解析] §5.1 over the
 * block-table gather of [PagedAttention] §3.2, with [KV Cache篇] §6.3's tiling. */
KV_API int paged_decode_attention(kv_pool* pool, int layer, const void* q, float* out,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, int batch, int max_context,
                           float scale, int partition_tokens, void* workspace,
                           size_t workspace_bytes, kv_stream_t stream);

/* One decode step of a layer in one launch: append each sequence's newest token, then
 * attend (the fused append + attention of the decode loop).  For every sequence s with
 * n = context_lens[s] >= 1, token n-1 is the token produced this step: its K and V
 * (k_new, v_new: device [batch][num_heads][head_dim] of in_dtype, 16-byte aligned; dtype
 * rules as kv_append) are stored into the slot block_tables[s][(n-1)/B]*B + (n-1)%B of
 * every head, and out is what paged_decode_attention returns over the updated cache.
 * The pool bytes written and the output are identical to kv_append followed by
 * paged_decode_attention.  Requirement: the block receiving a sequence's new token must
 * not be shared with another sequence of the batch (copy-on-write already done, as the
 * host allocator guarantees); a sequence with context_len 0 appends nothing.  All other
 * arguments, the workspace and the errors are those of paged_decode_attention.
 * The write-then-read order of [KV Cache篇] §3.1 and the batched cache update of
 * [KV缓存机制解析] §6.2, done inside the attention kernel by the warp that owns the
 * sequence's last chunk. */
KV_API int paged_decode_attention_append(kv_pool* pool, int layer, const void* q, const void* k_new,
                                         const void* v_new, kv_dtype in_dtype, float* out,
                                         const int32_t* block_tables, int max_blocks_per_seq,
                                         const int32_t* context_lens, int batch, int max_context,
                                         float scale, int partition_tokens, void* workspace,
                                         size_t workspace_bytes, kv_stream_t stream);

/* Grouped-query (GQA) and multi-query (MQA) decode attention: num_q_heads query heads
 * share the pool's num_heads KV heads; query head j reads KV head j / G with
 * G = num_q_heads / num_heads in {1, 2, 4, 8} (G > 1: fp16 and FP8 pools).  Each K/V tile
 * is read once for its G query heads.
 *   q    device [batch][num_q_heads][head_dim] (as paged_decode_attention).
 *   out  device float32 [batch][num_q_heads][head_dim].
 *   k_new, v_new  NULL, or the newest token's K/V [batch][num_heads][head_dim] of in_dtype
 *        appended first exactly as paged_decode_attention_append does.
 * Everything else as paged_decode_attention; the workspace size comes from
 * paged_decode_workspace_size_gqa.  [KV Cache篇] §6.2 (MQA/GQA: KV heads shared by
 * groups of query heads, fewer bytes read). */
KV_API size_t paged_decode_workspace_size_gqa(const kv_pool* pool, int batch, int num_q_heads,
                                              int max_context, int partition_tokens);
KV_API int paged_decode_attention_gqa(kv_pool* pool, int layer, const void* q, int num_q_heads,
                                      const void* k_new, const void* v_new, kv_dtype in_dtype,
                                      float* out, const int32_t* block_tables, int max_blocks_per_seq,
                                      const int32_t* context_lens, int batch, int max_context,
                                      float scale, int partition_tokens, void* workspace,
                                      size_t workspace_bytes, kv_stream_t stream);

/* Every option of one decode-attention launch in one struct (field meanings as in the
 * entry points above).
 *   num_q_heads  0 = the pool's num_heads; else a multiple (grouped-query, as
 *                paged_decode_attention_gqa).
 *   k_new, v_new NULL, or the newest token's K/V (fused append, as
 *                paged_decode_attention_append; in_dtype ignored when NULL).
 *   window       0 = the whole context; W > 0: sliding-window decode — each query attends
 *                only to the last W tokens of its sequence (all of them when shorter), as the
 *                rolling-window cache of [KV缓存机制解析] §8 keeps the most recent tokens.
 *                Blocks lying wholly before position context_len - W are never read, so the
 *                host may release them (kv_alloc_seq_trim) and leave their table entries -1.
 *   flags        0, or a sum of the bits below (any other bit: KV_ERR_INVALID_ARG):
 *     KV_DECODE_WORKSPACE_ZEROED  the workspace's counters are already zero, so the call
 *                does not clear them (one cudaMemsetAsync less per call).  True for a
 *                workspace zero-filled once after allocation and used since only by decode
 *                calls of this library of one shape (the same layer pool geometry, batch,
 *                num_q_heads, max_context, partition_tokens and window; context_lens,
 *                tables, q and the layer may change) that left no device error bit: every
 *                launch leaves its counters zero when it completes.  A call of another
 *                shape places its counters elsewhere in the workspace, possibly where the
 *                previous shape kept its partials: zero-fill the workspace again before
 *                such a call, and after a device error, before passing this flag.
 *     KV_DECODE_PDL  launch with programmatic dependent launch: the kernel may be scheduled
 *                while the previous kernel on the stream is still finishing; it reads no
 *                global memory (inputs, pool or workspace) before that kernel has completed
 *                and its writes are visible, except as the two EARLY flags below allow.  Saves the launch gap between back-to-back
 *                kernels (with KV_DECODE_WORKSPACE_ZEROED no clearing copy sits between
 *                two consecutive decode calls).  Also valid inside stream capture.
 *     KV_DECODE_EARLY_TABLES  (with KV_DECODE_PDL; ignored without it) context_lens and
 *                block_tables were written before the previous kernel on the stream
 *                started (for instance host copies issued before a step's layer loop), so
 *                the kernel may read them, and the first block ids they point to, while
 *                that kernel is still finishing.  q, k_new, v_new, out and the workspace
 *                are still read and written only after it has completed (the pool too,
 *                unless KV_DECODE_EARLY_POOL).
 *     KV_DECODE_EARLY_POOL  (with KV_DECODE_PDL and KV_DECODE_EARLY_TABLES; ignored
 *                otherwise) the previous kernel on the stream writes no K/V pool row this
 *                call reads, except each sequence's last two rows, context_len - 2 and
 *                context_len - 1 (the token a fused decode step of the same layer appended
 *                just before, and this call's own slot).  Then the first K/V tiles (whole
 *                chunks below those rows) are fetched while that kernel is still
 *                finishing.  True in a model's layer loop (the kernel before a layer's
 *                attention does not write its pool) and in a loop of fused decode steps
 *                over one layer; false right after kv_copy_blocks, kv_swap_in or kv_append
 *                into rows this call reads.
 *     KV_DECODE_OUT_F16  out is float16 [batch][num_q_heads][head_dim] instead of float32:
 *                each element is the float32 result rounded to nearest even (beyond the
 *                float16 range: +-inf), as the attention output of [KV Cache篇] §3.1 is cast
 *                back to the query's type.  Partials and their merge stay float32; only the
 *                final store is rounded, so the value equals the float32 call's, rounded.
 *   out          device float32 [batch][num_q_heads][head_dim], or float16 with
 *                KV_DECODE_OUT_F16; 16-byte aligned.
 *   prefix_groups, num_prefix_groups  NULL and 0, or shared prompt prefixes: device int32
 *                [num_prefix_groups][3] of (first, count, shared_tokens), 4-byte aligned.  The
 *                `count` sequences first .. first+count-1 of the batch (2 to 8 of them) hold the
 *                same physical blocks in their first shared_tokens / block_size table entries: the
 *                candidates of parallel sampling forked from one prompt, which share its blocks
 *                until they write into them ([PagedAttention] §5.1).  Every (block, head) tile of
 *                that prefix is then read once for the query rows of all `count` members (their
 *                scores and P V on the tensor cores) instead of once per member; each member's
 *                tokens after the prefix are attended on their own and the parts merge exactly
 *                (log-sum-exp).  The result is the call's result without groups, up to rounding.
 *                Rules: groups sorted by `first` and disjoint; shared_tokens a multiple of
 *                block_size, at most every member's context_len (at most context_len - 1 with
 *                k_new: the appended token lies in a block of the member's own); a group may not
 *                span a multiple of 1024 sequences.  A group breaking them is attended without
 *                sharing and sets KV_DEVERR_PREFIX.  That the members' table entries agree is the
 *                caller's promise (the first member's entries are read).  Under
 *                KV_DECODE_EARLY_TABLES the groups count as tables.  num_prefix_groups <= batch.
 *                Needs an fp16 or FP8 pool with head_dim 128 (KV_FEATURE_TENSOR_MAPS),
 *                num_q_heads equal to num_heads and window 0, else KV_ERR_UNSUPPORTED.  The
 *                workspace size depends on whether groups are given (not on their contents):
 *                paged_decode_workspace_size_ex reads num_prefix_groups.  Partitioning with
 *                groups: partition_tokens 0 = about 8 partitions of max_context, 64 to 1024
 *                tokens; an explicit value must be at least ceil(max_context / 31) rounded up to
 *                a multiple of 32 (a member has at most 32 partitions). */
#define KV_DECODE_WORKSPACE_ZEROED 1u
#define KV_DECODE_PDL 2u
#define KV_DECODE_EARLY_TABLES 4u
#define KV_DECODE_OUT_F16 8u
#define KV_DECODE_EARLY_POOL 16u
typedef struct {
    int layer;
    const void* q;
    int num_q_heads;
    const void* k_new;
    const void* v_new;
    kv_dtype in_dtype;
    void* out;
    const int32_t* block_tables;
    int max_blocks_per_seq;
    const int32_t* context_lens;
    int batch;
    int max_context;
    int window;
    float scale;
    int partition_tokens;
    void* workspace;
    size_t workspace_bytes;
    kv_stream_t stream;
    unsigned flags;
    const int32_t* prefix_groups;
    int num_prefix_groups;
} kv_decode_args;

/* Workspace bytes for paged_decode_attention_ex with these arguments (0 on invalid ones). */
KV_API size_t paged_decode_workspace_size_ex(const kv_pool* pool, const kv_decode_args* args);

/* Decode attention with every option of kv_decode_args; errors as paged_decode_attention. */
KV_API int paged_decode_attention_ex(kv_pool* pool, const kv_decode_args* args);

/* One decode step of a batch, driven from the host in one call: the write-then-read step of
 * [PagedAttention] §3.3 (allocate or copy-on-write, write the new token, attend) for every
 * sequence of a batch, through the host allocator and one layer's fused call.
 *   1. kv_alloc_decode_step(alloc, seqs, n, ...) reserves each sequence's next slot, planning
 *      a block copy where the slot lies in a shared block (all or nothing);
 *   2. the block tables, context lengths and planned copy pairs are written into the
 *      caller's host staging buffer `staging` (int32 [n*max_blocks + n + 2*n]: tables
 *      [n][max_blocks] padded with -1, lengths [n], pairs [n][2]; page-locked for the copy
 *      to be asynchronous), which is copied whole to `dev_meta` (device, same layout);
 *   3. `inputs_bytes` bytes are copied from host `inputs_h` to device `inputs_d` (the caller
 *      packs the step's q, k_new and v_new there; may be 0).  When the inputs lie at the
 *      same offset after `staging` and after `dev_meta`, at most 256 bytes past the staging
 *      data, steps 2 and 3 are one copy of both (and of the padding between them);
 *   4. the planned block copies run over every layer of the pool (kv_copy_blocks);
 *   5. paged_decode_attention_ex(pool, args) runs the step's fused append + attention;
 *   6. `out_bytes` bytes of args->out are copied back to host `out_h` (may be 0).
 * args must describe this batch: batch == n, block_tables == dev_meta (tables part),
 * context_lens == dev_meta + n*max_blocks, max_blocks_per_seq == max_blocks, k_new and v_new
 * set (the step appends its token), and neither KV_DECODE_EARLY_TABLES nor
 * KV_DECODE_EARLY_POOL (the tables are copied just before the call);
 * otherwise KV_ERR_INVALID_ARG with nothing reserved.  A sequence whose table would exceed
 * max_blocks after the step is refused the same way.  Every device operation is issued
 * on args->stream and nothing synchronises, so a caller keeps one staging buffer per step
 * in flight (a copy reads it later).  Returns the number of planned block copies (>= 0) or
 * a negative kv_status: KV_ERR_STATE / KV_ERR_NO_BLOCKS from step 1 leave the allocator
 * unchanged and issue nothing; a failure after step 1 (a CUDA call, the attention's own
 * argument checks) returns its status with the slots already reserved. */
KV_API int kv_decode_step(kv_alloc* alloc, kv_pool* pool, const int32_t* seqs, int n, int max_blocks,
                          int32_t* staging, int32_t* dev_meta, const void* inputs_h, void* inputs_d,
                          size_t inputs_bytes, void* out_h, size_t out_bytes, const kv_decode_args* args);

/* Size of the library's fixed device scratch array used by paged_decode_attention_static. */
#define KV_STATIC_SCRATCH_BYTES (16u << 20)

/* paged_decode_attention without a workspace argument and without any allocation: for
 * callers that cannot call cudaMalloc (a plugin whose host application owns all device
 * memory and gives it no allocator; a serving loop that forbids device allocation once
 * it runs, since cudaMalloc can synchronise the device or fail late).  The pages have no
 * counterpart of this entry point: it only changes where the scratch memory comes from.
 * Arguments and results are those of paged_decode_attention, minus workspace and
 * workspace_bytes.  The scratch (work counters and split-context partials) is a
 * file-scope device array of KV_STATIC_SCRATCH_BYTES that every GPU loading the library
 * holds until the process exits.
 *   - The first call on a device looks up the array's device address (once per device,
 *     with that device current); make that first call before any stream capture.  The
 *     address belongs to the device's context: the first call after cudaDeviceReset
 *     replaced that context looks it up again (so does every call if the context's id
 *     cannot be read).
 *   - It runs the plain call only: no launch flags (no programmatic dependent launch, no
 *     early tables or tiles, float32 output), and there is no fused-append, grouped-query
 *     or sliding-window form of it.
 *   - The pool's device must be the current device (else KV_ERR_INVALID_ARG).
 *   - If the scratch these arguments need (paged_decode_workspace_size) exceeds
 *     KV_STATIC_SCRATCH_BYTES the call is refused with KV_ERR_INVALID_ARG and nothing
 *     is launched; a larger partition_tokens needs less scratch.
 *   - All calls share the array and it keeps the last call's contents; the counters
 *     that must start at zero are cleared by every call.  Calls whose kernels overlap on
 *     the GPU (other streams, other host threads) race on it: serialise them.
 *   - Calls no cudaMalloc, cudaFree or allocating library routine. */
KV_API int paged_decode_attention_static(kv_pool* pool, int layer, const void* q, float* out,
                                         const int32_t* block_tables, int max_blocks_per_seq,
                                         const int32_t* context_lens, int batch, int max_context,
                                         float scale, int partition_tokens, kv_stream_t stream);

/* ---------------------------------------------------------------- host block allocator */
/* Host memory only; not thread-safe (the caller serialises).  Block ids are the
 * physical ids of a kv_pool of the same num_blocks and block_size.
 * Free list, first-fit allocation, per-block reference counts and copy-on-write:
 * [PagedAttention] §3.1 and §3.3. */

/* free_order: NULL for 0..num_blocks-1, else a permutation of the physical ids giving
 * the initial free list, head first.  Allocation pops the head; a block whose count
 * reaches 0 is pushed back on the head. */
KV_API int kv_alloc_create(int num_blocks, int block_size, const int32_t* free_order, kv_alloc** out);
KV_API int kv_alloc_destroy(kv_alloc* a);

/* New empty sequence (length 0, no blocks). */
KV_API int kv_alloc_seq_new(kv_alloc* a, int* seq_id);

/* New sequence sharing every block of `parent` (each reference count + 1), same length. */
KV_API int kv_alloc_seq_fork(kv_alloc* a, int parent, int* child);

/* Reserve slots for the next `count` tokens of `seq` (count >= 1).  slots_out: host
 * int64 [count].  A new block is taken whenever the length is a multiple of B.  If the
 * first token lands in a block with reference count > 1, a copy is planned:
 * cow_pair_out (host int32 [2]) receives (src, dst), the sequence's table points at dst
 * and src's count drops by one; otherwise cow_pair_out = (-1, -1).  The caller copies
 * (kv_copy_blocks) before writing.  Fails with KV_ERR_NO_BLOCKS, state unchanged, when
 * the free list is too short for the whole request. */
KV_API int kv_alloc_append_slots(kv_alloc* a, int seq, int count, int64_t* slots_out,
                          int32_t* cow_pair_out);

/* One decode step's slots for a batch: reserve the next slot of each of the n sequences
 * seqs[0..n-1] (host int32), in order, exactly as n calls kv_alloc_append_slots(seq, 1)
 * would.  slots_out: host int64 [n]; cow_pairs_out: host int32 [n][2] receives the planned
 * block copies (src, dst) in order, *n_cow their number (the caller runs kv_copy_blocks on
 * them before the step writes).  The whole step is checked first: an unknown sequence gives
 * KV_ERR_STATE and a free list too short for every block the step takes gives
 * KV_ERR_NO_BLOCKS, with the state unchanged in both cases.  The per-step write path of
 * [PagedAttention] §3.3 (write_to_block) for a batch; one call instead of one per sequence. */
KV_API int kv_alloc_decode_step(kv_alloc* a, const int32_t* seqs, int n, int64_t* slots_out,
                                int32_t* cow_pairs_out, int* n_cow);

/* Sliding window: release every block of `seq` that lies wholly before token keep_from
 * (count - 1, back to the free list at 0) and set its table entry to -1; later entries
 * keep their logical positions and the length is unchanged.  *released (may be NULL)
 * receives the number of table entries cleared.  Idempotent. */
KV_API int kv_alloc_seq_trim(kv_alloc* a, int seq, int64_t keep_from, int* released);

/* Drop the sequence: every block's count - 1, blocks reaching 0 return to the free list. */
KV_API int kv_alloc_seq_free(kv_alloc* a, int seq);

/* Length and block count of a live sequence. */
KV_API int kv_alloc_seq_info(const kv_alloc* a, int seq, int* length, int* n_blocks);

/* The sequence's block table (host int32, cap entries available); *n_blocks = its length. */
KV_API int kv_alloc_block_table(const kv_alloc* a, int seq, int32_t* out, int cap, int* n_blocks);

/* Padded tables for a batch: tables (host int32 [n][max_blocks], unused entries -1)
 * and context_lens (host int32 [n]).  KV_ERR_INVALID_ARG if a table exceeds max_blocks. */
KV_API int kv_alloc_build_tables(const kv_alloc* a, const int32_t* seqs, int n, int32_t* tables,
                          int max_blocks, int32_t* context_lens);

/* Reference count of one physical block. */
KV_API int kv_alloc_ref_count(const kv_alloc* a, int block, int* ref);

/* Current free list, head first (cap entries available); *n = its length. */
KV_API int kv_alloc_free_list(const kv_alloc* a, int32_t* out, int cap, int* n);

KV_API int kv_alloc_stats(const kv_alloc* a, kv_alloc_stats_t* stats);

#ifdef __cplusplus
}
#endif

#endif /* KVPAGED_H */
