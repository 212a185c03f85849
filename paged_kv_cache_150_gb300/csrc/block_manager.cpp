// Host block manager: free list, refcounts, block tables, fork and
// copy-on-write.  Pure host code; it feeds block tables and slot mappings to
// the kernels.
//
// Follows "10 PagedAttention" (PidokuInfra), section 4 "Tiny example"
// (stack of free ids, Allocate/Free/Fork/BlocksNeeded/AppendToken/
// PhysicalIndex) and "04 · PagedAttention" (nano-vLLM Deep Dive), section 6
// "Copy-on-write block sharing" and section 7 "The BlockManager in code"
// (refcount > 1 means copy before writing; allocation failure is reported,
// not raised).  Every failing call leaves the state unchanged.
//
// Prefix caching ("10 PagedAttention" section 5, "The relationship to prefix
// caching"; nano-vLLM's hash_to_block): full prompt blocks are registered
// under a chained hash (64-bit FNV-1a over the parent block's hash, 8 bytes
// little-endian, then the block's token ids, 4 bytes little-endian each; the
// parent of block 0 is 0), and a new prompt reuses the blocks of its longest
// registered prefix (refcount + 1).  A hit also compares the token ids.  By
// default a block leaves the map when its refcount reaches 0.  With retention
// (the eviction of the pages' hands-on exercise, "10 PagedAttention" section
// 10 A) it stays registered as evictable, in order of release (a freed
// sequence's blocks from its last to its first): a later hit revives it, and
// allocation takes free blocks first, then evicts the least recently
// released.
#include <cstdint>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"

struct pa_bm {
    int32_t num_blocks = 0;
    int32_t block_size = 0;
    std::vector<int32_t> free;     // stack; back() is the top
    std::vector<int32_t> ref;      // refcount per block, 0 when free
    struct Seq {
        bool live = false;
        int32_t len = 0;
        std::vector<int32_t> table;
    };
    std::vector<Seq> seqs;          // indexed by sequence id
    // prefix cache
    std::unordered_map<uint64_t, int32_t> cached;  // chained hash -> block
    std::vector<uint64_t> block_hash;               // per block, valid when registered
    std::vector<char> registered;
    std::vector<int32_t> block_tokens;              // B token ids per registered block
    int64_t hits = 0, lookups = 0;
    // retention: registered blocks at refcount 0, least recently released first
    bool retain = false;
    std::list<int32_t> lru;
    std::vector<std::list<int32_t>::iterator> lru_it;  // sized once retention is first switched on
    std::vector<int32_t> scratch;

    void unregister(int32_t b) {
        cached.erase(block_hash[b]);
        registered[b] = 0;
    }
    bool is_registered(int32_t b) const { return !registered.empty() && registered[b]; }
    void release(int32_t b) {  // refcount reached 0, not retained
        free.push_back(b);
        if (is_registered(b)) unregister(b);
    }
    void make_evictable(int32_t b) { lru_it[b] = lru.insert(lru.end(), b); }
    void revive(int32_t b) { lru.erase(lru_it[b]); }  // a hit on an evictable block
    // The least recently released evictable block goes back on the free stack.
    void evict_oldest() {
        const int32_t b = lru.front();
        lru.pop_front();
        unregister(b);
        free.push_back(b);
    }
    // Blocks an allocation may use: free ones and evictable ones.
    int64_t available() const { return (int64_t)free.size() + (int64_t)lru.size(); }
    // Evict the least recently released blocks onto the free stack until it
    // holds n (the caller has checked available() >= n).
    void reserve(size_t n) {
        while (free.size() < n && !lru.empty()) evict_oldest();
    }

    int32_t blocks_needed(int64_t tokens) const {
        return (int32_t)((tokens + block_size - 1) / block_size);
    }
    Seq *get(int32_t s) {
        return (s >= 0 && s < (int32_t)seqs.size() && seqs[s].live) ? &seqs[s] : nullptr;
    }
    const Seq *get(int32_t s) const {
        return (s >= 0 && s < (int32_t)seqs.size() && seqs[s].live) ? &seqs[s] : nullptr;
    }
    // Top n ids in stack order; the caller has checked available() >= n.
    void take(int32_t n, std::vector<int32_t> &out) {
        reserve((size_t)n);
        const size_t first = free.size() - (size_t)n;
        for (size_t i = first; i < free.size(); ++i) {
            out.push_back(free[i]);
            ref[free[i]] = 1;
        }
        free.resize(first);
    }
    int32_t pop_one() {
        reserve(1);
        const int32_t b = free.back();
        free.pop_back();
        ref[b] = 1;
        return b;
    }
    int32_t slot(const Seq &s, int32_t pos) const {
        return s.table[pos / block_size] * block_size + pos % block_size;
    }
};

// Sizes a new manager and fills its free stack (the caller's order, or ids
// from num_blocks-1 down to 0); a bad order leaves num_blocks = -1.
static void fill_new(pa_bm *bm, int32_t num_blocks, int32_t block_size, const int32_t *free_order) {
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->ref.assign((size_t)num_blocks, 0);
    bm->free.reserve((size_t)num_blocks);
    if (free_order) {
        std::vector<char> seen((size_t)num_blocks, 0);
        for (int32_t i = 0; i < num_blocks; ++i) {
            const int32_t b = free_order[i];
            if (b < 0 || b >= num_blocks || seen[b]) {
                bm->num_blocks = -1;
                return;
            }
            seen[b] = 1;
            bm->free.push_back(b);
        }
    } else {
        for (int32_t b = num_blocks - 1; b >= 0; --b) bm->free.push_back(b);
    }
}

extern "C" pa_bm_t *pa_bm_create(int32_t num_blocks, int32_t block_size, const int32_t *free_order) {
    if (num_blocks < 0 || block_size <= 0) return nullptr;
    if ((int64_t)num_blocks * block_size >= ((int64_t)1 << 31)) return nullptr;
    pa_bm *bm = new (std::nothrow) pa_bm();
    if (!bm) return nullptr;
    try {
        fill_new(bm, num_blocks, block_size, free_order);
    } catch (const std::bad_alloc &) {
        delete bm;
        return nullptr;
    }
    if (bm->num_blocks < 0) {  // a bad free order
        delete bm;
        return nullptr;
    }
    return bm;
}

extern "C" void pa_bm_destroy(pa_bm_t *bm) { delete bm; }

extern "C" pa_status_t pa_bm_new_seq(pa_bm_t *bm, int32_t num_tokens, int32_t *seq_out) try {
    if (!bm || num_tokens < 0 || !seq_out) return PA_ERR_INVALID_ARG;
    const int32_t n = bm->blocks_needed(num_tokens);
    if ((int64_t)n > bm->available()) return PA_ERR_NO_BLOCKS;
    pa_bm::Seq s;
    s.live = true;
    s.len = num_tokens;
    s.table.reserve((size_t)n);
    bm->take(n, s.table);
    bm->seqs.push_back(std::move(s));
    *seq_out = (int32_t)bm->seqs.size() - 1;
    return PA_OK;
} catch (const std::bad_alloc &) {
    return PA_ERR_HOST_MEMORY;
}

extern "C" pa_status_t pa_bm_fork(pa_bm_t *bm, int32_t parent, int32_t *child_out) try {
    if (!bm || !child_out) return PA_ERR_INVALID_ARG;
    const pa_bm::Seq *p = bm->get(parent);
    if (!p) return PA_ERR_INVALID_ARG;
    pa_bm::Seq c;
    c.live = true;
    c.len = p->len;
    c.table = p->table;
    for (int32_t b : c.table) bm->ref[b] += 1;
    bm->seqs.push_back(std::move(c));
    *child_out = (int32_t)bm->seqs.size() - 1;
    return PA_OK;
} catch (const std::bad_alloc &) {
    return PA_ERR_HOST_MEMORY;
}

extern "C" pa_status_t pa_bm_free_seq(pa_bm_t *bm, int32_t seq) try {
    if (!bm) return PA_ERR_INVALID_ARG;
    pa_bm::Seq *s = bm->get(seq);
    if (!s) return PA_ERR_INVALID_ARG;
    // Retained blocks enter the eviction order from the sequence's last block
    // to its first: prefix matching stops at a prompt's first miss, so a
    // prompt should lose its tail before its head.
    std::vector<int32_t> &kept = bm->scratch;
    kept.clear();
    for (int32_t b : s->table) {
        if (--bm->ref[b] != 0) continue;
        if (bm->retain && bm->is_registered(b))
            kept.push_back(b);
        else
            bm->release(b);
    }
    for (size_t i = kept.size(); i-- > 0;) bm->make_evictable(kept[i]);
    s->table.clear();
    s->table.shrink_to_fit();
    s->live = false;
    s->len = 0;
    return PA_OK;
} catch (const std::bad_alloc &) {
    return PA_ERR_HOST_MEMORY;
}

extern "C" pa_status_t pa_bm_append_tokens(pa_bm_t *bm, int32_t seq, int32_t count, int32_t *slots_out,
                                           int32_t *cow_pairs_out, int32_t *num_pairs_out) try {
    if (!bm || count < 0 || (count > 0 && !slots_out)) return PA_ERR_INVALID_ARG;
    pa_bm::Seq *s = bm->get(seq);
    if (!s) return PA_ERR_INVALID_ARG;
    if ((int64_t)s->len + count > INT32_MAX) return PA_ERR_INVALID_ARG;
    if (num_pairs_out) *num_pairs_out = 0;
    if (count == 0) return PA_OK;
    const int32_t pos0 = s->len;
    const int32_t B = bm->block_size;
    // Blocks this append needs: new blocks past the table, plus one private
    // copy when the first token lands in a partly filled shared block.
    const bool cow = (pos0 % B != 0) && bm->ref[s->table[pos0 / B]] > 1;
    const int64_t grow = (int64_t)bm->blocks_needed((int64_t)pos0 + count) - (int64_t)s->table.size();
    if (cow && !cow_pairs_out) return PA_ERR_INVALID_ARG;
    if ((int64_t)cow + grow > bm->available()) return PA_ERR_NO_BLOCKS;
    if (cow) {
        const int32_t old = s->table[pos0 / B];
        const int32_t fresh = bm->pop_one();
        bm->ref[old] -= 1;
        s->table[pos0 / B] = fresh;
        cow_pairs_out[0] = old;
        cow_pairs_out[1] = fresh;
        if (num_pairs_out) *num_pairs_out = 1;
    }
    for (int32_t i = 0; i < count; ++i) {
        const int32_t pos = pos0 + i;
        if (pos % B == 0) s->table.push_back(bm->pop_one());
        slots_out[i] = bm->slot(*s, pos);
    }
    s->len = pos0 + count;
    return PA_OK;
} catch (const std::bad_alloc &) {
    return PA_ERR_HOST_MEMORY;
}

extern "C" pa_status_t pa_bm_append_token(pa_bm_t *bm, int32_t seq, int32_t *slot_out, int32_t *cow_src,
                                          int32_t *cow_dst) {
    if (!slot_out) return PA_ERR_INVALID_ARG;
    int32_t pair[2] = {-1, -1};
    int32_t np = 0;
    const pa_status_t st = pa_bm_append_tokens(bm, seq, 1, slot_out, pair, &np);
    if (st != PA_OK) return st;
    if (cow_src) *cow_src = np ? pair[0] : -1;
    if (cow_dst) *cow_dst = np ? pair[1] : -1;
    return PA_OK;
}

extern "C" pa_status_t pa_bm_seq_len(const pa_bm_t *bm, int32_t seq, int32_t *len_out,
                                     int32_t *num_blocks_out) {
    if (!bm) return PA_ERR_INVALID_ARG;
    const pa_bm::Seq *s = bm->get(seq);
    if (!s) return PA_ERR_INVALID_ARG;
    if (len_out) *len_out = s->len;
    if (num_blocks_out) *num_blocks_out = (int32_t)s->table.size();
    return PA_OK;
}

extern "C" pa_status_t pa_bm_block_table(const pa_bm_t *bm, int32_t seq, int32_t *out, int32_t capacity,
                                         int32_t *len_out) {
    if (!bm || capacity < 0 || (capacity > 0 && !out)) return PA_ERR_INVALID_ARG;
    const pa_bm::Seq *s = bm->get(seq);
    if (!s) return PA_ERR_INVALID_ARG;
    const int32_t n = (int32_t)s->table.size();
    if (len_out) *len_out = n;
    if (n > capacity) return PA_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i) out[i] = s->table[i];
    return PA_OK;
}

extern "C" pa_status_t pa_bm_physical_index(const pa_bm_t *bm, int32_t seq, int32_t pos, int32_t *slot_out) {
    if (!bm || !slot_out) return PA_ERR_INVALID_ARG;
    const pa_bm::Seq *s = bm->get(seq);
    if (!s || pos < 0 || pos / bm->block_size >= (int32_t)s->table.size()) return PA_ERR_INVALID_ARG;
    *slot_out = bm->slot(*s, pos);
    return PA_OK;
}

extern "C" pa_status_t pa_bm_refcount(const pa_bm_t *bm, int32_t block, int32_t *ref_out) {
    if (!bm || !ref_out || block < 0 || block >= bm->num_blocks) return PA_ERR_INVALID_ARG;
    *ref_out = bm->ref[block];
    return PA_OK;
}

extern "C" pa_status_t pa_bm_stats(const pa_bm_t *bm, int32_t *free_out, int32_t *used_out,
                                   int32_t *shared_out) {
    if (!bm) return PA_ERR_INVALID_ARG;
    int32_t shared = 0;
    for (int32_t r : bm->ref) shared += r > 1;
    if (free_out) *free_out = (int32_t)bm->available();  // evictable blocks count as free
    if (used_out) *used_out = bm->num_blocks - (int32_t)bm->available();
    if (shared_out) *shared_out = shared;
    return PA_OK;
}

extern "C" pa_status_t pa_bm_export(const pa_bm_t *bm, const int32_t *seqs, int32_t n, int32_t max_blocks,
                                    int32_t *tables_out, int32_t *lens_out) {
    if (!bm || n < 0 || max_blocks <= 0 || (n > 0 && (!seqs || !tables_out || !lens_out)))
        return PA_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i) {
        const pa_bm::Seq *s = bm->get(seqs[i]);
        if (!s || (int32_t)s->table.size() > max_blocks) return PA_ERR_INVALID_ARG;
    }
    for (int32_t i = 0; i < n; ++i) {
        const pa_bm::Seq *s = bm->get(seqs[i]);
        int32_t *row = tables_out + (int64_t)i * max_blocks;
        const int32_t nb = (int32_t)s->table.size();
        for (int32_t j = 0; j < max_blocks; ++j) row[j] = j < nb ? s->table[j] : -1;
        lens_out[i] = s->len;
    }
    return PA_OK;
}

namespace {
constexpr uint64_t kFnvOffset = 0xCBF29CE484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001B3ull;

uint64_t block_chain_hash(uint64_t parent, const int32_t *tokens, int32_t B) {
    uint64_t h = kFnvOffset;
    for (int i = 0; i < 8; ++i) {
        h ^= (parent >> (8 * i)) & 0xFFu;
        h *= kFnvPrime;
    }
    for (int32_t t = 0; t < B; ++t) {
        const uint32_t v = (uint32_t)tokens[t];
        for (int i = 0; i < 4; ++i) {
            h ^= (v >> (8 * i)) & 0xFFu;
            h *= kFnvPrime;
        }
    }
    return h;
}
}  // namespace

extern "C" pa_status_t pa_bm_new_seq_cached(pa_bm_t *bm, const int32_t *token_ids, int32_t num_tokens,
                                            int32_t *seq_out, int32_t *num_cached_tokens_out) try {
    if (!bm || num_tokens < 0 || (num_tokens > 0 && !token_ids) || !seq_out) return PA_ERR_INVALID_ARG;
    const int32_t B = bm->block_size;
    const int32_t n_full = num_tokens / B;
    if (bm->registered.empty()) {
        bm->registered.assign((size_t)bm->num_blocks, 0);
        bm->block_hash.assign((size_t)bm->num_blocks, 0);
        bm->block_tokens.assign((size_t)bm->num_blocks * B, 0);
    }
    std::vector<uint64_t> hashes((size_t)n_full);
    uint64_t parent = 0;
    for (int32_t j = 0; j < n_full; ++j) parent = hashes[j] = block_chain_hash(parent, token_ids + (int64_t)j * B, B);
    std::vector<int32_t> table;
    int64_t lookups = 0;
    for (int32_t j = 0; j < n_full; ++j) {
        ++lookups;
        auto it = bm->cached.find(hashes[j]);
        if (it == bm->cached.end()) break;
        const int32_t b = it->second;
        bool same = true;
        for (int32_t t = 0; t < B && same; ++t)
            same = bm->block_tokens[(int64_t)b * B + t] == token_ids[(int64_t)j * B + t];
        if (!same) break;
        table.push_back(b);
    }
    const int32_t reused = (int32_t)table.size();
    const int32_t need = bm->blocks_needed(num_tokens) - reused;
    int64_t revived = 0;  // hits on evictable blocks leave the evictable pool
    for (int32_t b : table) revived += bm->ref[b] == 0 ? 1 : 0;
    if ((int64_t)need > bm->available() - revived) return PA_ERR_NO_BLOCKS;
    for (int32_t b : table) {
        if (bm->ref[b] == 0) bm->revive(b);
        bm->ref[b] += 1;
    }
    bm->take(need, table);
    for (int32_t j = reused; j < n_full; ++j) {
        const int32_t b = table[j];
        bm->cached[hashes[j]] = b;
        bm->block_hash[b] = hashes[j];
        bm->registered[b] = 1;
        for (int32_t t = 0; t < B; ++t) bm->block_tokens[(int64_t)b * B + t] = token_ids[(int64_t)j * B + t];
    }
    bm->lookups += lookups;
    bm->hits += reused;
    pa_bm::Seq s;
    s.live = true;
    s.len = num_tokens;
    s.table = std::move(table);
    bm->seqs.push_back(std::move(s));
    *seq_out = (int32_t)bm->seqs.size() - 1;
    if (num_cached_tokens_out) *num_cached_tokens_out = reused * B;
    return PA_OK;
} catch (const std::bad_alloc &) {
    return PA_ERR_HOST_MEMORY;
}

extern "C" pa_status_t pa_bm_slots(const pa_bm_t *bm, int32_t seq, int32_t first_pos, int32_t count,
                                   int32_t *slots_out) {
    if (!bm || count < 0 || first_pos < 0 || (count > 0 && !slots_out)) return PA_ERR_INVALID_ARG;
    const pa_bm::Seq *s = bm->get(seq);
    if (!s || (int64_t)first_pos + count > s->len) return PA_ERR_INVALID_ARG;
    for (int32_t i = 0; i < count; ++i) slots_out[i] = bm->slot(*s, first_pos + i);
    return PA_OK;
}

extern "C" pa_status_t pa_bm_set_prefix_retention(pa_bm_t *bm, int32_t on) try {
    if (!bm) return PA_ERR_INVALID_ARG;
    if (on && bm->lru_it.empty()) bm->lru_it.resize((size_t)bm->num_blocks);
    if (!on)  // the evictable blocks become plain free blocks, oldest first
        while (!bm->lru.empty()) bm->evict_oldest();
    bm->retain = on != 0;
    return PA_OK;
} catch (const std::bad_alloc &) {
    return PA_ERR_HOST_MEMORY;
}

extern "C" pa_status_t pa_bm_evictable(const pa_bm_t *bm, int32_t *count_out) {
    if (!bm || !count_out) return PA_ERR_INVALID_ARG;
    *count_out = (int32_t)bm->lru.size();
    return PA_OK;
}

extern "C" pa_status_t pa_bm_cache_stats(const pa_bm_t *bm, int32_t *cached_blocks_out, int64_t *hits_out,
                                         int64_t *lookups_out) {
    if (!bm) return PA_ERR_INVALID_ARG;
    if (cached_blocks_out) *cached_blocks_out = (int32_t)bm->cached.size();
    if (hits_out) *hits_out = bm->hits;
    if (lookups_out) *lookups_out = bm->lookups;
    return PA_OK;
}
