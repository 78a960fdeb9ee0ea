// Host block allocator: free stack, per-sequence block tables, reference
// counts and copy-on-write.  Semantics are documented in include/pkv.h.
//
// "PagedAttention (vLLM) -- Virtual memory cho AI", section "Co che Block
// Table": blocks are handed out only when a token needs one and freed blocks
// are reused at once without defragmentation; section "Copy-on-Write cho Beam
// Search": branches share prefix blocks and split a block when they diverge.
#include "pkv.h"

#include <algorithm>
#include <climits>
#include <new>
#include <unordered_map>
#include <vector>

struct pkv_allocator {
    struct Seq {
        std::vector<int32_t> table;
        int64_t tokens = 0;
    };
    int num_blocks = 0;
    int block_size = 0;
    std::vector<int32_t> free_stack;  // back() is handed out next
    std::vector<int32_t> refcnt;
    std::unordered_map<int64_t, Seq> seqs;

    int32_t take() {
        int32_t b = free_stack.back();
        free_stack.pop_back();
        refcnt[b] = 1;
        return b;
    }
    void release(int32_t b) {
        if (--refcnt[b] == 0) free_stack.push_back(b);
    }
};

extern "C" {

pkv_allocator *block_allocator_create(int num_blocks, int block_size) {
    if (num_blocks < 1 || block_size < 1) return nullptr;
    pkv_allocator *a = new (std::nothrow) pkv_allocator();
    if (!a) return nullptr;
    try {
        a->num_blocks = num_blocks;
        a->block_size = block_size;
        a->refcnt.assign(num_blocks, 0);
        a->free_stack.resize(num_blocks);
        for (int i = 0; i < num_blocks; ++i) a->free_stack[i] = num_blocks - 1 - i;
    } catch (...) {
        delete a;
        return nullptr;
    }
    return a;
}

void block_allocator_destroy(pkv_allocator *a) { delete a; }

pkv_status block_allocator_add_seq(pkv_allocator *a, int64_t seq, int64_t num_tokens) {
    if (!a || num_tokens < 0 || a->seqs.count(seq)) return PKV_ERR_INVALID;
    const int64_t need = (num_tokens + a->block_size - 1) / a->block_size;
    if (need > (int64_t)a->free_stack.size()) return PKV_ERR_OOM;
    try {
        pkv_allocator::Seq s;
        s.table.reserve((size_t)need + 1);
        s.tokens = num_tokens;
        auto it = a->seqs.emplace(seq, std::move(s)).first;
        for (int64_t i = 0; i < need; ++i) it->second.table.push_back(a->take());
    } catch (...) {
        return PKV_ERR_INVALID;
    }
    return PKV_OK;
}

pkv_status block_allocator_append_slot(pkv_allocator *a, int64_t seq, int64_t *slot_out,
                                       int32_t *cow_src_out, int32_t *cow_dst_out) {
    if (!a) return PKV_ERR_INVALID;
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end()) return PKV_ERR_INVALID;
    pkv_allocator::Seq &s = it->second;
    const int64_t offset = s.tokens % a->block_size;
    int32_t src = -1, dst = -1;
    if (offset == 0) {
        // last block full (or none yet): a fresh block for this token
        if (a->free_stack.empty()) return PKV_ERR_OOM;
        try {
            s.table.push_back(-1);
        } catch (...) {
            return PKV_ERR_INVALID;
        }
        s.table.back() = a->take();
    } else if (a->refcnt[s.table.back()] > 1) {
        // shared, partially filled last block: copy it before writing
        if (a->free_stack.empty()) return PKV_ERR_OOM;
        src = s.table.back();
        dst = a->take();
        a->refcnt[src] -= 1;
        s.table.back() = dst;
    }
    const int64_t slot = (int64_t)s.table.back() * a->block_size + offset;
    s.tokens += 1;
    if (slot_out) *slot_out = slot;
    if (cow_src_out) *cow_src_out = src;
    if (cow_dst_out) *cow_dst_out = dst;
    return PKV_OK;
}

pkv_status block_allocator_append_slots(pkv_allocator *a, const int64_t *seqs, int n,
                                        int64_t *slots_out, int64_t *cow_pairs_out,
                                        int *n_cow_out) {
    if (!a || n < 0 || (n > 0 && (!seqs || !slots_out || !cow_pairs_out))) return PKV_ERR_INVALID;
    // validate and count the blocks this step needs before changing anything
    int64_t need = 0;
    try {
        std::unordered_map<int64_t, char> seen;
        seen.reserve((size_t)n * 2);
        for (int i = 0; i < n; ++i) {
            auto it = a->seqs.find(seqs[i]);
            if (it == a->seqs.end() || !seen.emplace(seqs[i], 1).second) return PKV_ERR_INVALID;
            const pkv_allocator::Seq &s = it->second;
            if (s.tokens % a->block_size == 0 || a->refcnt[s.table.back()] > 1) ++need;
        }
    } catch (...) {
        return PKV_ERR_INVALID;
    }
    if (need > (int64_t)a->free_stack.size()) return PKV_ERR_OOM;
    int ncow = 0;
    for (int i = 0; i < n; ++i) {
        int32_t src = -1, dst = -1;
        const pkv_status st = block_allocator_append_slot(a, seqs[i], &slots_out[i], &src, &dst);
        if (st != PKV_OK) return st;  // unreachable after the checks above
        if (src >= 0) {
            cow_pairs_out[2 * ncow] = src;
            cow_pairs_out[2 * ncow + 1] = dst;
            ++ncow;
        }
    }
    if (n_cow_out) *n_cow_out = ncow;
    return PKV_OK;
}

pkv_status block_allocator_fork(pkv_allocator *a, int64_t parent, int64_t child) {
    if (!a || parent == child) return PKV_ERR_INVALID;
    auto it = a->seqs.find(parent);
    if (it == a->seqs.end() || a->seqs.count(child)) return PKV_ERR_INVALID;
    try {
        pkv_allocator::Seq copy = it->second;  // copy before emplace may rehash
        for (int32_t b : copy.table) a->refcnt[b] += 1;
        a->seqs.emplace(child, std::move(copy));
    } catch (...) {
        return PKV_ERR_INVALID;
    }
    return PKV_OK;
}

pkv_status block_allocator_free_seq(pkv_allocator *a, int64_t seq) {
    if (!a) return PKV_ERR_INVALID;
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end()) return PKV_ERR_INVALID;
    for (int32_t b : it->second.table) a->release(b);
    a->seqs.erase(it);
    return PKV_OK;
}

pkv_status block_allocator_block_table(const pkv_allocator *a, int64_t seq, int32_t *out,
                                       int cap, int *n_out) {
    if (!a) return PKV_ERR_INVALID;
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end()) return PKV_ERR_INVALID;
    const auto &t = it->second.table;
    if ((int64_t)t.size() > (int64_t)cap || (!out && !t.empty())) return PKV_ERR_INVALID;
    std::copy(t.begin(), t.end(), out);
    if (n_out) *n_out = (int)t.size();
    return PKV_OK;
}

pkv_status block_allocator_block_tables(const pkv_allocator *a, const int64_t *seqs, int n,
                                        int32_t *out, int cap, int32_t pad,
                                        int32_t *seq_lens_out) {
    if (!a || n < 0 || cap < 0 || (n > 0 && (!seqs || !out))) return PKV_ERR_INVALID;
    for (int i = 0; i < n; ++i) {  // validate everything before writing
        auto it = a->seqs.find(seqs[i]);
        if (it == a->seqs.end() || (int64_t)it->second.table.size() > (int64_t)cap ||
            it->second.tokens > INT32_MAX)
            return PKV_ERR_INVALID;
    }
    for (int i = 0; i < n; ++i) {
        const auto &s = a->seqs.find(seqs[i])->second;
        int32_t *row = out + (int64_t)i * cap;
        std::copy(s.table.begin(), s.table.end(), row);
        std::fill(row + s.table.size(), row + cap, pad);
        if (seq_lens_out) seq_lens_out[i] = (int32_t)s.tokens;
    }
    return PKV_OK;
}

pkv_status block_allocator_prefix_groups(const pkv_allocator *a, const int64_t *seqs, int n,
                                        int32_t *group_offsets_out, int32_t *prefix_lens_out,
                                        int *num_groups_out) {
    if (!a || n < 0 || (n > 0 && (!seqs || !group_offsets_out || !prefix_lens_out)) || !num_groups_out)
        return PKV_ERR_INVALID;
    std::vector<const pkv_allocator::Seq *> ss((size_t)n);
    for (int i = 0; i < n; ++i) {
        auto it = a->seqs.find(seqs[i]);
        if (it == a->seqs.end()) return PKV_ERR_INVALID;
        ss[i] = &it->second;
    }
    const int64_t B = a->block_size;
    const int64_t align = B > 16 ? B : 16;  // whole 16-token tiles and whole blocks
    int g = 0;
    group_offsets_out[0] = 0;
    for (int i = 0; i < n;) {
        // leading full blocks identical in the run of sequences starting at i
        int64_t common = ss[i]->tokens / B;
        int j = i + 1;
        while (j < n) {
            const auto &lt = ss[i]->table, &t = ss[j]->table;
            int64_t c = 0;
            const int64_t lim = std::min<int64_t>(common, ss[j]->tokens / B);
            while (c < lim && lt[(size_t)c] == t[(size_t)c]) ++c;
            if (c == 0) break;
            common = c;
            ++j;
        }
        const int64_t shared = j - i > 1 ? common * B / align * align : 0;
        prefix_lens_out[g] = (int32_t)shared;
        group_offsets_out[g + 1] = j;
        ++g;
        i = j;
    }
    *num_groups_out = g;
    return PKV_OK;
}

pkv_status block_allocator_slots(const pkv_allocator *a, int64_t seq, int64_t start,
                                 int64_t count, int64_t *out) {
    if (!a || start < 0 || count < 0 || (count > 0 && !out)) return PKV_ERR_INVALID;
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end() || start + count > it->second.tokens) return PKV_ERR_INVALID;
    const auto &t = it->second.table;
    const int64_t B = a->block_size;
    for (int64_t i = 0; i < count; ++i) {
        const int64_t pos = start + i;
        out[i] = (int64_t)t[(size_t)(pos / B)] * B + pos % B;
    }
    return PKV_OK;
}

int64_t block_allocator_num_tokens(const pkv_allocator *a, int64_t seq) {
    if (!a) return -1;
    auto it = a->seqs.find(seq);
    return it == a->seqs.end() ? -1 : it->second.tokens;
}

int block_allocator_num_free(const pkv_allocator *a) {
    return a ? (int)a->free_stack.size() : -1;
}

int block_allocator_refcount(const pkv_allocator *a, int32_t block) {
    if (!a || block < 0 || block >= a->num_blocks) return -1;
    return a->refcnt[block];
}

pkv_status block_allocator_waste(const pkv_allocator *a, int64_t *used_tokens,
                                 int64_t *allocated_slots) {
    if (!a) return PKV_ERR_INVALID;
    // occupancy of each live block: the most any holder has written into it
    std::vector<int32_t> fill(a->num_blocks, -1);
    const int64_t B = a->block_size;
    for (const auto &kv : a->seqs) {
        const auto &s = kv.second;
        for (size_t i = 0; i < s.table.size(); ++i) {
            const int64_t used = std::min<int64_t>(B, std::max<int64_t>(0, s.tokens - (int64_t)i * B));
            int32_t &f = fill[s.table[i]];
            f = std::max<int32_t>(f, (int32_t)used);
        }
    }
    int64_t used = 0, alloc = 0;
    for (int32_t f : fill) {
        if (f >= 0) {
            used += f;
            alloc += B;
        }
    }
    if (used_tokens) *used_tokens = used;
    if (allocated_slots) *allocated_slots = alloc;
    return PKV_OK;
}

}  // extern "C"
