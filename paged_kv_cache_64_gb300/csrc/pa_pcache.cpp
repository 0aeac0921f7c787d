// Prefix-caching block pool (host side), the allocator's automatic prefix
// caching: "2.1 PagedAttention" (infra-guide), section 9 (the V1
// KVCacheManager / BlockPool split, the doubly linked free queue, reference
// counts, touch on a hit, free order), and "PagedAttention: Treating KV
// Memory Like Virtual Memory", section "A separate mechanism: automatic
// prefix caching" (block hash chain, block-aligned matches, no copy on a
// hit, LRU by free-queue order, cache_salt on the first block).
//
// Blocks are in use (refcount > 0) or in the free queue, an intrusive doubly
// linked list over the block ids: new blocks come off the head, a hit block
// is unlinked from anywhere in O(1), freed blocks without a hash are linked
// at the head and hashed ones at the tail.  A block is hashed when it fills
// (FNV-1a 64 over the previous hash, or the salt for a request's first block,
// and the block's token ids); a hash table maps each cached hash to its
// block, whose previous hash and token ids are kept so that a hit is
// verified exactly.  Taking a cached block from the queue evicts its hash.
// The pool is single-threaded; every failing call leaves it unchanged.
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"

namespace {

constexpr uint64_t kFnvOffset = 14695981039346656037ull;
constexpr uint64_t kFnvPrime = 1099511628211ull;

uint64_t fnv_bytes(uint64_t h, uint64_t v, int nbytes) {
    for (int i = 0; i < nbytes; ++i) {
        h ^= (v >> (8 * i)) & 0xffu;
        h *= kFnvPrime;
    }
    return h;
}

uint64_t hash_block(uint64_t prev, const int32_t *tokens, int n) {
    uint64_t h = fnv_bytes(kFnvOffset, prev, 8);
    for (int i = 0; i < n; ++i) h = fnv_bytes(h, (uint64_t)(uint32_t)tokens[i], 4);
    return h;
}

struct Request {
    std::vector<int32_t> table;
    std::vector<int32_t> tokens;
    std::vector<uint64_t> chain;  // hashes of the request's full blocks
    uint64_t salt = 0;
};

}  // namespace

struct pa_pcache {
    int num_blocks = 0;
    int block_size = 0;
    // free queue: head / tail and links, -1 = none
    int head = -1, tail = -1;
    std::vector<int32_t> next, prev;
    std::vector<uint8_t> in_free;
    int num_free = 0;
    std::vector<int32_t> refs;
    std::vector<uint8_t> hashed;
    std::vector<uint64_t> hash, prev_hash;
    std::vector<int32_t> content;  // [num_blocks][block_size] token ids of cached blocks
    std::unordered_map<uint64_t, int32_t> cached;
    std::unordered_map<int64_t, Request> reqs;

    void link_tail(int b) {
        prev[b] = tail;
        next[b] = -1;
        if (tail >= 0) next[tail] = b; else head = b;
        tail = b;
        in_free[b] = 1;
        ++num_free;
    }
    void link_head(int b) {
        next[b] = head;
        prev[b] = -1;
        if (head >= 0) prev[head] = b; else tail = b;
        head = b;
        in_free[b] = 1;
        ++num_free;
    }
    void unlink(int b) {
        if (prev[b] >= 0) next[prev[b]] = next[b]; else head = next[b];
        if (next[b] >= 0) prev[next[b]] = prev[b]; else tail = prev[b];
        prev[b] = next[b] = -1;
        in_free[b] = 0;
        --num_free;
    }
    // the cached block holding (p, tokens), or -1; h receives the hash
    int find(uint64_t p, const int32_t *tokens, uint64_t *h) const {
        *h = hash_block(p, tokens, block_size);
        auto it = cached.find(*h);
        if (it == cached.end()) return -1;
        const int b = it->second;
        if (prev_hash[b] != p ||
            std::memcmp(&content[(size_t)b * block_size], tokens, sizeof(int32_t) * block_size))
            return -1;
        return b;
    }
    int lookup(const int32_t *tokens, int n, uint64_t salt, std::vector<int32_t> *hits) const {
        const int maxb = n > 0 ? (n - 1) / block_size : 0;
        uint64_t p = salt;
        int count = 0;
        for (int i = 0; i < maxb; ++i) {
            uint64_t h;
            const int b = find(p, tokens + (size_t)i * block_size, &h);
            if (b < 0) break;
            if (hits) hits->push_back(b);
            p = h;
            ++count;
        }
        return count;
    }
    int take() {
        const int b = head;
        unlink(b);
        if (hashed[b]) {  // evicted: the block is about to hold new content
            cached.erase(hash[b]);
            hashed[b] = 0;
        }
        refs[b] = 1;
        return b;
    }
    // block i of request r has just filled
    void register_block(Request &r, int i) {
        const uint64_t p = i > 0 ? r.chain[i - 1] : r.salt;
        const int32_t *toks = &r.tokens[(size_t)i * block_size];
        uint64_t h;
        const int found = find(p, toks, &h);
        r.chain.push_back(h);
        const int b = r.table[i];
        if (found < 0 && cached.find(h) == cached.end()) {
            cached.emplace(h, b);
            hashed[b] = 1;
            hash[b] = h;
            prev_hash[b] = p;
            std::memcpy(&content[(size_t)b * block_size], toks, sizeof(int32_t) * block_size);
        }
    }
};

extern "C" {

pa_status pa_pcache_create(int num_blocks, int block_size, const int32_t *free_order,
                           pa_pcache **out) {
    if (!out || num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID;
    if ((size_t)num_blocks * (size_t)block_size > ((size_t)1 << 34)) return PA_ERR_INVALID;
    pa_pcache *pc = new (std::nothrow) pa_pcache;
    if (!pc) return PA_ERR_INVALID;
    try {
        pc->num_blocks = num_blocks;
        pc->block_size = block_size;
        pc->next.assign(num_blocks, -1);
        pc->prev.assign(num_blocks, -1);
        pc->in_free.assign(num_blocks, 0);
        pc->refs.assign(num_blocks, 0);
        pc->hashed.assign(num_blocks, 0);
        pc->hash.assign(num_blocks, 0);
        pc->prev_hash.assign(num_blocks, 0);
        pc->content.assign((size_t)num_blocks * block_size, 0);
    } catch (...) {
        delete pc;
        return PA_ERR_INVALID;
    }
    for (int i = 0; i < num_blocks; ++i) {
        const int b = free_order ? free_order[i] : i;
        if (b < 0 || b >= num_blocks || pc->in_free[b]) {
            delete pc;
            return PA_ERR_INVALID;
        }
        pc->link_tail(b);
    }
    *out = pc;
    return PA_OK;
}

void pa_pcache_destroy(pa_pcache *pc) { delete pc; }

uint64_t pa_pcache_hash_block(uint64_t prev, const int32_t *tokens, int n) {
    return hash_block(prev, tokens, n < 0 ? 0 : n);
}

pa_status pa_pcache_lookup(const pa_pcache *pc, const int32_t *tokens, int n, uint64_t salt,
                           int *num_blocks_out) {
    if (!pc || n < 0 || (n > 0 && !tokens) || !num_blocks_out) return PA_ERR_INVALID;
    *num_blocks_out = pc->lookup(tokens, n, salt, nullptr);
    return PA_OK;
}

pa_status pa_pcache_add(pa_pcache *pc, int64_t seq_id, const int32_t *tokens, int n,
                        uint64_t salt, int *num_cached_out, int64_t *slots_out) {
    if (!pc || n < 0 || (n > 0 && (!tokens || !slots_out)) || !num_cached_out)
        return PA_ERR_INVALID;
    if (pc->reqs.count(seq_id)) return PA_ERR_INVALID;
    const int B = pc->block_size;
    std::vector<int32_t> hits;
    try {
        hits.reserve((size_t)n / B + 1);
    } catch (...) {
        return PA_ERR_INVALID;
    }
    pc->lookup(tokens, n, salt, &hits);
    const int need = (n + B - 1) / B - (int)hits.size();
    int free_hits = 0;
    for (int b : hits) free_hits += pc->refs[b] == 0;
    if (need > pc->num_free - free_hits) return PA_ERR_OUT_OF_BLOCKS;
    Request *rp = nullptr;
    try {  // every allocation before the pool changes
        rp = &pc->reqs.emplace(seq_id, Request()).first->second;
        rp->table.reserve((size_t)(n + B - 1) / B + 1);
        rp->chain.reserve((size_t)n / B + 1);
        rp->tokens.assign(tokens, tokens + n);
    } catch (...) {
        pc->reqs.erase(seq_id);
        return PA_ERR_INVALID;
    }
    Request &r = *rp;
    r.salt = salt;
    for (int b : hits) {  // touch: nothing is copied
        if (pc->refs[b] == 0) pc->unlink(b);
        ++pc->refs[b];
        r.table.push_back(b);
        r.chain.push_back(pc->hash[b]);
    }
    for (int i = 0; i < need; ++i) r.table.push_back(pc->take());
    for (int i = (int)hits.size(); i < n / B; ++i) pc->register_block(r, i);
    for (int p = 0; p < n; ++p) slots_out[p] = (int64_t)r.table[p / B] * B + p % B;
    *num_cached_out = (int)hits.size() * B;
    return PA_OK;
}

pa_status pa_pcache_append(pa_pcache *pc, int64_t seq_id, int32_t token, int64_t *slot_out) {
    if (!pc || !slot_out) return PA_ERR_INVALID;
    auto it = pc->reqs.find(seq_id);
    if (it == pc->reqs.end()) return PA_ERR_NOT_FOUND;
    Request &r = it->second;
    const int B = pc->block_size;
    const int L = (int)r.tokens.size();
    if (L % B == 0 && pc->num_free == 0) return PA_ERR_OUT_OF_BLOCKS;
    try {
        r.tokens.reserve(L + 1);
        if (L % B == 0) r.table.reserve(r.table.size() + 1);
    } catch (...) {
        return PA_ERR_INVALID;
    }
    if (L % B == 0) r.table.push_back(pc->take());
    r.tokens.push_back(token);
    if ((L + 1) % B == 0) pc->register_block(r, L / B);
    *slot_out = (int64_t)r.table[L / B] * B + L % B;
    return PA_OK;
}

pa_status pa_pcache_free(pa_pcache *pc, int64_t seq_id) {
    if (!pc) return PA_ERR_INVALID;
    auto it = pc->reqs.find(seq_id);
    if (it == pc->reqs.end()) return PA_ERR_NOT_FOUND;
    const std::vector<int32_t> &t = it->second.table;
    // tail first; unhashed blocks to the head (the first one freed ends up
    // first), hashed ones to the tail in the order they are freed
    std::vector<int32_t> no_hash;
    for (size_t k = t.size(); k-- > 0;) {
        const int b = t[k];
        if (--pc->refs[b] == 0) {
            if (pc->hashed[b]) pc->link_tail(b);
            else no_hash.push_back(b);
        }
    }
    for (size_t k = no_hash.size(); k-- > 0;) pc->link_head(no_hash[k]);
    pc->reqs.erase(it);
    return PA_OK;
}

pa_status pa_pcache_block_table(const pa_pcache *pc, int64_t seq_id, int32_t *out, int cap,
                                int *n_out) {
    if (!pc || !n_out || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID;
    auto it = pc->reqs.find(seq_id);
    if (it == pc->reqs.end()) return PA_ERR_NOT_FOUND;
    const std::vector<int32_t> &t = it->second.table;
    *n_out = (int)t.size();
    if ((int)t.size() > cap) return PA_ERR_INVALID;
    for (size_t i = 0; i < t.size(); ++i) out[i] = t[i];
    return PA_OK;
}

pa_status pa_pcache_len(const pa_pcache *pc, int64_t seq_id, int64_t *len_out) {
    if (!pc || !len_out) return PA_ERR_INVALID;
    auto it = pc->reqs.find(seq_id);
    if (it == pc->reqs.end()) return PA_ERR_NOT_FOUND;
    *len_out = (int64_t)it->second.tokens.size();
    return PA_OK;
}

int pa_pcache_num_free(const pa_pcache *pc) { return pc ? pc->num_free : -1; }

pa_status pa_pcache_free_queue(const pa_pcache *pc, int32_t *out, int cap, int *n_out) {
    if (!pc || !n_out || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID;
    *n_out = pc->num_free;
    if (pc->num_free > cap) return PA_ERR_INVALID;
    int i = 0;
    for (int b = pc->head; b >= 0; b = pc->next[b]) out[i++] = b;
    return PA_OK;
}

int pa_pcache_refcount(const pa_pcache *pc, int block) {
    if (!pc || block < 0 || block >= pc->num_blocks) return -1;
    return pc->refs[block];
}

pa_status pa_pcache_block_hash(const pa_pcache *pc, int block, uint64_t *hash_out,
                               int *cached_out) {
    if (!pc || !hash_out || !cached_out || block < 0 || block >= pc->num_blocks)
        return PA_ERR_INVALID;
    *cached_out = pc->hashed[block];
    *hash_out = pc->hashed[block] ? pc->hash[block] : 0;
    return PA_OK;
}

}  // extern "C"
