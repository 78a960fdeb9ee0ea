// Host block allocator: free stack, per-sequence block tables, reference
// counts, copy-on-write and a prefix cache of full prompt blocks.  Semantics
// are documented in include/pkv.h.
//
// "PagedAttention (vLLM) -- Virtual memory cho AI", section "Co che Block
// Table": blocks are handed out only when a token needs one and freed blocks
// are reused at once without defragmentation; section "Copy-on-Write cho Beam
// Search": branches share prefix blocks and split a block when they diverge.
// "vLLM PagedAttention: Buoc dot pha ve thong luong suy luan LLM", list of
// advanced features, "Prefix caching": the KV cache of a prompt prefix shared
// by several requests is reused instead of recomputed.
#include "pkv.h"

#include <algorithm>
#include <climits>
#include <cstring>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

namespace {
// FNV-1a over the parent prefix hash and a block's token ids: a deterministic
// 64-bit digest of the whole token prefix up to and including the block.
uint64_t prefix_hash(uint64_t parent, const int32_t *tokens, int n) {
    uint64_t h = 1469598103934665603ull;
    auto mix = [&h](uint64_t v, int bytes) {
        for (int i = 0; i < bytes; ++i) {
            h ^= (v >> (8 * i)) & 0xffu;
            h *= 1099511628211ull;
        }
    };
    mix(parent, 8);
    for (int i = 0; i < n; ++i) mix((uint32_t)tokens[i], 4);
    return h;
}
constexpr uint64_t kRootHash = 0x9e3779b97f4a7c15ull;  // parent of a prompt's first block
}  // namespace

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

    // Prefix cache: full prompt blocks registered under the hash of their whole
    // token prefix.  A registered block whose last holder goes away stays
    // registered and joins `evictable` (front = released longest ago); it is
    // handed out again, losing its registration, only when the free stack is
    // empty.
    std::unordered_map<uint64_t, int32_t> cache;    // prefix hash -> block
    std::vector<char> cached;                        // block is registered
    std::vector<uint64_t> key, parent;               // its prefix hash, its parent's
    std::vector<int32_t> toks;                       // its block_size token ids
    std::list<int32_t> evictable;
    std::vector<std::list<int32_t>::iterator> ev_pos;
    int64_t hits = 0, misses = 0;

    int64_t available() const { return (int64_t)free_stack.size() + (int64_t)evictable.size(); }
    void unregister(int32_t b) {
        cache.erase(key[b]);
        cached[b] = 0;
    }
    int32_t take() {  // callers checked available() > 0
        int32_t b;
        if (!free_stack.empty()) {
            b = free_stack.back();
            free_stack.pop_back();
        } else {
            b = evictable.front();
            evictable.pop_front();
            unregister(b);
        }
        refcnt[b] = 1;
        return b;
    }
    void release(int32_t b) {
        if (--refcnt[b] == 0 && !cached[b]) free_stack.push_back(b);
    }
    void park(int32_t b) {  // a registered block without holders
        evictable.push_back(b);
        ev_pos[b] = std::prev(evictable.end());
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
        a->cached.assign(num_blocks, 0);
        a->key.assign(num_blocks, 0);
        a->parent.assign(num_blocks, 0);
        a->toks.assign((size_t)num_blocks * block_size, 0);
        a->ev_pos.resize(num_blocks);
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
    if (need > a->available()) return PKV_ERR_OOM;
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
        if (a->available() == 0) return PKV_ERR_OOM;
        try {
            s.table.push_back(-1);
        } catch (...) {
            return PKV_ERR_INVALID;
        }
        s.table.back() = a->take();
    } else if (a->refcnt[s.table.back()] > 1) {
        // shared, partially filled last block: copy it before writing
        if (a->available() == 0) return PKV_ERR_OOM;
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

// One token for each of n distinct sequences; with `tables`, also the
// incremental update of the caller's dense tables (row i of `cap` entries
// belongs to seqs[i]): only the entry of the block that holds the new token is
// written, and lens[i] gets the new token count.
static pkv_status append_step(pkv_allocator *a, const int64_t *seqs, int n, int32_t *tables, int cap, int32_t *lens,
                              int64_t *slots_out, int64_t *cow_pairs_out, int *n_cow_out) {
    // validate and count the blocks this step needs before changing anything
    int64_t need = 0;
    try {
        std::unordered_map<int64_t, char> seen;
        seen.reserve((size_t)n * 2);
        for (int i = 0; i < n; ++i) {
            auto it = a->seqs.find(seqs[i]);
            if (it == a->seqs.end() || !seen.emplace(seqs[i], 1).second) return PKV_ERR_INVALID;
            const pkv_allocator::Seq &s = it->second;
            if (tables && s.tokens / a->block_size >= cap) return PKV_ERR_INVALID;  // the row cannot hold it
            if (s.tokens % a->block_size == 0 || a->refcnt[s.table.back()] > 1) ++need;
        }
    } catch (...) {
        return PKV_ERR_INVALID;
    }
    if (need > a->available()) return PKV_ERR_OOM;
    int ncow = 0;
    for (int i = 0; i < n; ++i) {
        int32_t src = -1, dst = -1;
        int64_t slot = -1;
        const pkv_status st = block_allocator_append_slot(a, seqs[i], &slot, &src, &dst);
        if (st != PKV_OK) return st;  // unreachable after the checks above
        slots_out[i] = slot;
        if (src >= 0) {
            cow_pairs_out[2 * ncow] = src;
            cow_pairs_out[2 * ncow + 1] = dst;
            ++ncow;
        }
        if (tables) {
            const int64_t tokens = a->seqs.find(seqs[i])->second.tokens;  // after the append
            tables[(int64_t)i * cap + (tokens - 1) / a->block_size] = (int32_t)(slot / a->block_size);
            if (lens) lens[i] = (int32_t)tokens;
        }
    }
    if (n_cow_out) *n_cow_out = ncow;
    return PKV_OK;
}

pkv_status block_allocator_append_slots(pkv_allocator *a, const int64_t *seqs, int n,
                                        int64_t *slots_out, int64_t *cow_pairs_out,
                                        int *n_cow_out) {
    if (!a || n < 0 || (n > 0 && (!seqs || !slots_out || !cow_pairs_out))) return PKV_ERR_INVALID;
    return append_step(a, seqs, n, nullptr, 0, nullptr, slots_out, cow_pairs_out, n_cow_out);
}

pkv_status block_allocator_append_step(pkv_allocator *a, const int64_t *seqs, int n, int32_t *tables, int cap,
                                       int32_t *seq_lens, int64_t *slots_out, int64_t *cow_pairs_out,
                                       int *n_cow_out) {
    if (!a || n < 0 || cap < 1 ||
        (n > 0 && (!seqs || !tables || !seq_lens || !slots_out || !cow_pairs_out)))
        return PKV_ERR_INVALID;
    return append_step(a, seqs, n, tables, cap, seq_lens, slots_out, cow_pairs_out, n_cow_out);
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
    const auto &t = it->second.table;
    for (int32_t b : t) a->release(b);
    // registered blocks left without holders become evictable, the last block
    // of the prefix first (evicted before the blocks it extends)
    for (size_t i = t.size(); i-- > 0;)
        if (a->refcnt[t[i]] == 0 && a->cached[t[i]]) a->park(t[i]);
    a->seqs.erase(it);
    return PKV_OK;
}

pkv_status block_allocator_extend(pkv_allocator *a, int64_t seq, int64_t count, int64_t *slots_out,
                                  int32_t *cow_src_out, int32_t *cow_dst_out) {
    if (!a || count < 0 || (count > 0 && !slots_out)) return PKV_ERR_INVALID;
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end()) return PKV_ERR_INVALID;
    pkv_allocator::Seq &s = it->second;
    const int B = a->block_size;
    const bool shared_partial = s.tokens % B != 0 && a->refcnt[s.table.back()] > 1;
    const int64_t need = (s.tokens + count + B - 1) / B - (s.tokens + B - 1) / B + (shared_partial && count > 0);
    if (need > a->available()) return PKV_ERR_OOM;  // nothing changed
    try {
        s.table.reserve(s.table.size() + (size_t)need);
    } catch (...) {
        return PKV_ERR_INVALID;
    }
    int32_t src = -1, dst = -1;
    for (int64_t i = 0; i < count; ++i) {
        int32_t cs = -1, cd = -1;
        const pkv_status st = block_allocator_append_slot(a, seq, &slots_out[i], &cs, &cd);
        if (st != PKV_OK) return st;  // cannot happen: blocks were counted above
        if (cs >= 0) {
            src = cs;
            dst = cd;
        }
    }
    if (cow_src_out) *cow_src_out = src;
    if (cow_dst_out) *cow_dst_out = dst;
    return PKV_OK;
}

pkv_status block_allocator_truncate(pkv_allocator *a, int64_t seq, int64_t num_tokens) {
    if (!a) return PKV_ERR_INVALID;
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end()) return PKV_ERR_INVALID;
    pkv_allocator::Seq &s = it->second;
    if (num_tokens < 0 || num_tokens > s.tokens) return PKV_ERR_INVALID;
    const int B = a->block_size;
    const size_t keep = (size_t)((num_tokens + B - 1) / B);
    // blocks wholly past the new end: released in table order, registered ones
    // left without holders parked last block first (as when a sequence is freed)
    for (size_t i = keep; i < s.table.size(); ++i) a->release(s.table[i]);
    for (size_t i = s.table.size(); i-- > keep;)
        if (a->refcnt[s.table[i]] == 0 && a->cached[s.table[i]]) a->park(s.table[i]);
    s.table.resize(keep);
    s.tokens = num_tokens;
    // a registered block that is now this holder's partially filled last block
    // would be written in place by the next append: it loses its registration
    if (keep > 0 && num_tokens % B != 0) {
        const int32_t b = s.table.back();
        if (a->cached[b] && a->refcnt[b] == 1) a->unregister(b);
    }
    return PKV_OK;
}

pkv_status block_allocator_add_seq_cached(pkv_allocator *a, int64_t seq, const int32_t *tokens,
                                          int64_t num_tokens, int64_t *cached_tokens_out) {
    if (!a || num_tokens < 0 || (num_tokens > 0 && !tokens) || a->seqs.count(seq)) return PKV_ERR_INVALID;
    const int B = a->block_size;
    const int64_t nfull = num_tokens / B, need = (num_tokens + B - 1) / B;
    // leading full blocks already registered (exact token match)
    std::vector<int32_t> hit;
    std::vector<uint64_t> keys((size_t)nfull);
    uint64_t h = kRootHash;
    bool missed = false;
    for (int64_t i = 0; i < nfull; ++i) {
        const int32_t *bt = tokens + i * B;
        const uint64_t k = prefix_hash(h, bt, B);
        keys[(size_t)i] = k;
        if (!missed) {
            auto c = a->cache.find(k);
            if (c != a->cache.end() && a->parent[c->second] == h &&
                std::memcmp(&a->toks[(size_t)c->second * B], bt, (size_t)B * sizeof(int32_t)) == 0)
                hit.push_back(c->second);
            else
                missed = true;
        }
        h = k;
    }
    int64_t revived = 0;  // hits that are evictable now and leave the pool
    for (int32_t b : hit) revived += a->refcnt[b] == 0;
    if (need - (int64_t)hit.size() > a->available() - revived) return PKV_ERR_OOM;
    try {
        pkv_allocator::Seq s;
        s.table.reserve((size_t)need + 1);
        s.tokens = num_tokens;
        auto it = a->seqs.emplace(seq, std::move(s)).first;
        auto &table = it->second.table;
        for (int32_t b : hit) {
            if (a->refcnt[b] == 0) a->evictable.erase(a->ev_pos[b]);
            a->refcnt[b] += 1;
            table.push_back(b);
        }
        uint64_t ph = hit.empty() ? kRootHash : keys[hit.size() - 1];
        for (int64_t i = (int64_t)hit.size(); i < need; ++i) {
            const int32_t b = a->take();
            table.push_back(b);
            if (i < nfull && !a->cache.count(keys[(size_t)i])) {  // register the new full block
                a->cache.emplace(keys[(size_t)i], b);
                a->cached[b] = 1;
                a->key[b] = keys[(size_t)i];
                a->parent[b] = ph;
                std::memcpy(&a->toks[(size_t)b * B], tokens + i * B, (size_t)B * sizeof(int32_t));
            }
            if (i < nfull) ph = keys[(size_t)i];
        }
    } catch (...) {
        return PKV_ERR_INVALID;
    }
    a->hits += (int64_t)hit.size();
    a->misses += nfull - (int64_t)hit.size();
    if (cached_tokens_out) *cached_tokens_out = (int64_t)hit.size() * B;
    return PKV_OK;
}

pkv_status block_allocator_cache_stats(const pkv_allocator *a, int64_t *hits, int64_t *misses,
                                       int *cached_blocks, int *evictable_blocks) {
    if (!a) return PKV_ERR_INVALID;
    if (hits) *hits = a->hits;
    if (misses) *misses = a->misses;
    if (cached_blocks) *cached_blocks = (int)a->cache.size();
    if (evictable_blocks) *evictable_blocks = (int)a->evictable.size();
    return PKV_OK;
}

pkv_status block_allocator_cache_clear(pkv_allocator *a) {
    if (!a) return PKV_ERR_INVALID;
    // unreferenced registered blocks go back to the free stack, oldest first;
    // registered blocks still held keep their blocks but leave the cache
    for (int32_t b : a->evictable) {
        a->cached[b] = 0;
        a->free_stack.push_back(b);
    }
    a->evictable.clear();
    for (auto &kv : a->cache) a->cached[kv.second] = 0;
    a->cache.clear();
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
    return a ? (int)a->available() : -1;
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
