// Host block allocator: free list, per-block reference counts, per-sequence block
// tables, fork (sharing) and copy-on-write planning.
//
// "KV Cache与PagedAttention：大模型推理显存优化方案" §3.1 gives a global physical
// block pool managed through a free structure and first-fit allocation; with
// fixed-size blocks first fit is "take the first free block", so the free list is a
// stack whose top is the list head.  §3.3 gives the reference-count rule: a write
// into a block whose count is > 1 first allocates a new block, copies, decrements
// the old count and repoints the table.  The copy itself is device work
// (kv_copy_blocks); here it is only planned.  §5.1 (parallel sampling) shares a
// prompt's blocks among candidates: that is kv_alloc_seq_fork.

#include <algorithm>
#include <climits>
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/kvpaged.h"

struct kv_alloc {
    int num_blocks = 0;
    int block_size = 0;
    std::vector<int32_t> free_stack;   // back() is the free-list head
    std::vector<int32_t> ref;          // per physical block
    struct Seq {
        std::vector<int32_t> table;
        int64_t len = 0;
    };
    std::unordered_map<int, Seq> seqs;
    int next_id = 0;
};

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Blocks needed to append `count` tokens to `s`: new logical blocks plus one for a
// planned copy when the first write lands in a shared, partially filled block.
int64_t blocks_needed(const kv_alloc* a, const kv_alloc::Seq& s, int64_t count) {
    const int64_t B = a->block_size;
    int64_t need = ceil_div(s.len + count, B) - ceil_div(s.len, B);
    if (s.len % B != 0 && a->ref[s.table.back()] > 1) need += 1;
    return need;
}

int32_t pop_free(kv_alloc* a) {
    int32_t b = a->free_stack.back();
    a->free_stack.pop_back();
    a->ref[b] = 1;
    return b;
}

int release(kv_alloc* a, int32_t b) {
    if (a->ref[b] <= 0) return KV_ERR_STATE;
    if (--a->ref[b] == 0) a->free_stack.push_back(b);
    return KV_OK;
}

}  // namespace

extern "C" {

int kv_alloc_create(int num_blocks, int block_size, const int32_t* free_order, kv_alloc** out) {
    if (!out || num_blocks <= 0 || block_size <= 0) return KV_ERR_INVALID_ARG;
    *out = nullptr;
    kv_alloc* a = new (std::nothrow) kv_alloc;
    if (!a) return KV_ERR_INVALID_ARG;
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->ref.assign(num_blocks, 0);
    a->free_stack.resize(num_blocks);
    if (free_order) {
        std::vector<char> seen(num_blocks, 0);
        for (int i = 0; i < num_blocks; ++i) {
            int32_t b = free_order[i];
            if (b < 0 || b >= num_blocks || seen[b]) { delete a; return KV_ERR_INVALID_ARG; }
            seen[b] = 1;
            a->free_stack[num_blocks - 1 - i] = b;   // free_order[0] ends on top
        }
    } else {
        for (int i = 0; i < num_blocks; ++i) a->free_stack[num_blocks - 1 - i] = i;
    }
    *out = a;
    return KV_OK;
}

int kv_alloc_destroy(kv_alloc* a) {
    if (!a) return KV_ERR_INVALID_ARG;
    delete a;
    return KV_OK;
}

int kv_alloc_seq_new(kv_alloc* a, int* seq_id) {
    if (!a || !seq_id) return KV_ERR_INVALID_ARG;
    int id = a->next_id++;
    a->seqs.emplace(id, kv_alloc::Seq{});
    *seq_id = id;
    return KV_OK;
}

int kv_alloc_seq_fork(kv_alloc* a, int parent, int* child) {
    if (!a || !child) return KV_ERR_INVALID_ARG;
    auto it = a->seqs.find(parent);
    if (it == a->seqs.end()) return KV_ERR_STATE;
    kv_alloc::Seq s = it->second;
    for (int32_t b : s.table)
        if (b >= 0) a->ref[b] += 1;                  // entries a window trimmed are -1
    int id = a->next_id++;
    a->seqs.emplace(id, std::move(s));
    *child = id;
    return KV_OK;
}

int kv_alloc_append_slots(kv_alloc* a, int seq, int count, int64_t* slots_out,
                          int32_t* cow_pair_out) {
    if (!a || !slots_out || !cow_pair_out || count <= 0) return KV_ERR_INVALID_ARG;
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end()) return KV_ERR_STATE;
    kv_alloc::Seq& s = it->second;
    if (blocks_needed(a, s, count) > (int64_t)a->free_stack.size()) return KV_ERR_NO_BLOCKS;
    const int64_t B = a->block_size;
    cow_pair_out[0] = -1;
    cow_pair_out[1] = -1;
    for (int i = 0; i < count; ++i) {
        if (s.len % B == 0) {
            s.table.push_back(pop_free(a));            // a new logical block
        } else if (a->ref[s.table.back()] > 1) {       // only possible for i == 0
            int32_t src = s.table.back();
            int32_t dst = pop_free(a);
            a->ref[src] -= 1;                          // other sharers keep it (count >= 1)
            s.table.back() = dst;
            cow_pair_out[0] = src;
            cow_pair_out[1] = dst;
        }
        slots_out[i] = (int64_t)s.table[s.len / B] * B + s.len % B;
        s.len += 1;
    }
    return KV_OK;
}

int kv_alloc_decode_step(kv_alloc* a, const int32_t* seqs, int n, int64_t* slots_out, int32_t* cow_pairs_out,
                         int* n_cow) {
    if (!a || n < 0 || (n > 0 && (!seqs || !slots_out || !cow_pairs_out)) || !n_cow) return KV_ERR_INVALID_ARG;
    *n_cow = 0;
    // every sequence must exist, and the free list must hold every block the step takes:
    // a new block where the length is a multiple of B, or a copy where the last block is
    // still shared (the last of its sharers in this step writes in place)
    std::unordered_map<int32_t, int> ref_left;
    int64_t need = 0;
    const int64_t B = a->block_size;
    for (int i = 0; i < n; ++i) {
        auto it = a->seqs.find(seqs[i]);
        if (it == a->seqs.end()) return KV_ERR_STATE;
        const kv_alloc::Seq& s = it->second;
        if (s.len % B == 0) {
            ++need;
        } else {
            const int32_t last = s.table.back();
            auto r = ref_left.find(last);
            int& left = r == ref_left.end() ? (ref_left[last] = a->ref[last]) : r->second;
            if (left > 1) {
                ++need;
                --left;
            }
        }
    }
    if (need > (int64_t)a->free_stack.size()) return KV_ERR_NO_BLOCKS;
    for (int i = 0; i < n; ++i) {
        int32_t pair[2];
        const int rc = kv_alloc_append_slots(a, seqs[i], 1, slots_out + i, pair);
        if (rc != KV_OK) return rc;                    // not reached: checked above
        if (pair[0] >= 0) {
            cow_pairs_out[2 * *n_cow] = pair[0];
            cow_pairs_out[2 * *n_cow + 1] = pair[1];
            *n_cow += 1;
        }
    }
    return KV_OK;
}

int kv_alloc_seq_free(kv_alloc* a, int seq) {
    if (!a) return KV_ERR_INVALID_ARG;
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end()) return KV_ERR_STATE;
    int rc = KV_OK;
    for (int32_t b : it->second.table)
        if (b >= 0 && release(a, b) != KV_OK) rc = KV_ERR_STATE;
    a->seqs.erase(it);
    return rc;
}

int kv_alloc_seq_trim(kv_alloc* a, int seq, int64_t keep_from, int* released) {
    if (!a || keep_from < 0) return KV_ERR_INVALID_ARG;
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end()) return KV_ERR_STATE;
    kv_alloc::Seq& s = it->second;
    // the block that receives the next token must stay: keep_from may not pass the length
    if (keep_from > s.len) return KV_ERR_INVALID_ARG;
    const int64_t whole = keep_from / a->block_size;      // blocks ending at or before keep_from
    int n = 0, rc = KV_OK;
    for (int64_t j = 0; j < whole && j < (int64_t)s.table.size(); ++j) {
        if (s.table[j] < 0) continue;
        if (release(a, s.table[j]) != KV_OK) rc = KV_ERR_STATE;
        s.table[j] = -1;
        ++n;
    }
    if (released) *released = n;
    return rc;
}

int kv_alloc_seq_info(const kv_alloc* a, int seq, int* length, int* n_blocks) {
    if (!a || !length || !n_blocks) return KV_ERR_INVALID_ARG;
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end()) return KV_ERR_STATE;
    *length = (int)it->second.len;
    *n_blocks = (int)it->second.table.size();
    return KV_OK;
}

int kv_alloc_block_table(const kv_alloc* a, int seq, int32_t* out, int cap, int* n_blocks) {
    if (!a || !n_blocks || cap < 0 || (cap > 0 && !out)) return KV_ERR_INVALID_ARG;
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end()) return KV_ERR_STATE;
    const auto& t = it->second.table;
    *n_blocks = (int)t.size();
    if ((int)t.size() > cap) return KV_ERR_INVALID_ARG;
    std::copy(t.begin(), t.end(), out);
    return KV_OK;
}

int kv_alloc_build_tables(const kv_alloc* a, const int32_t* seqs, int n, int32_t* tables,
                          int max_blocks, int32_t* context_lens) {
    if (!a || n < 0 || max_blocks <= 0 || (n > 0 && (!seqs || !tables || !context_lens)))
        return KV_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        auto it = a->seqs.find(seqs[i]);
        if (it == a->seqs.end()) return KV_ERR_STATE;
        const auto& t = it->second.table;
        if ((int)t.size() > max_blocks || it->second.len > INT32_MAX) return KV_ERR_INVALID_ARG;
        int32_t* row = tables + (int64_t)i * max_blocks;
        std::fill(row, row + max_blocks, -1);
        std::copy(t.begin(), t.end(), row);
        context_lens[i] = (int32_t)it->second.len;
    }
    return KV_OK;
}

int kv_alloc_ref_count(const kv_alloc* a, int block, int* ref) {
    if (!a || !ref || block < 0 || block >= a->num_blocks) return KV_ERR_INVALID_ARG;
    *ref = a->ref[block];
    return KV_OK;
}

int kv_alloc_free_list(const kv_alloc* a, int32_t* out, int cap, int* n) {
    if (!a || !n || cap < 0 || (cap > 0 && !out)) return KV_ERR_INVALID_ARG;
    *n = (int)a->free_stack.size();
    if (*n > cap) return KV_ERR_INVALID_ARG;
    std::copy(a->free_stack.rbegin(), a->free_stack.rend(), out);
    return KV_OK;
}

int kv_alloc_stats(const kv_alloc* a, kv_alloc_stats_t* st) {
    if (!a || !st) return KV_ERR_INVALID_ARG;
    st->num_blocks = a->num_blocks;
    st->free_blocks = (int)a->free_stack.size();
    st->shared_blocks = (int)std::count_if(a->ref.begin(), a->ref.end(), [](int32_t r) { return r > 1; });
    st->num_seqs = (int)a->seqs.size();
    int64_t used = 0, waste = 0;
    for (const auto& kv : a->seqs) {
        const int64_t trimmed = std::count(kv.second.table.begin(), kv.second.table.end(), -1);
        used += kv.second.len - trimmed * a->block_size;  // tokens still held in live blocks
        waste += (int64_t)kv.second.table.size() * a->block_size - kv.second.len;
    }
    st->used_slots = used;
    st->wasted_slots = waste;
    return KV_OK;
}

}  // extern "C"
