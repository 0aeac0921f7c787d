// Host block allocator behind the pa_alloc_* / pa_seq_* entry points.
//
// Block-manager semantics of "Why AI servers waste memory, and how paging
// fixes it" (spicyshark.co): sections "The idea: a block table" (steps 1-5),
// "A hand-worked example" (free list taken from the front, freed blocks
// appended at the back, in table order), "The real implementation" (append
// with the copy-on-write branch, the up-front free-list check, free that
// returns a block only at refcount zero) and "Sharing a prefix with
// copy-on-write" (fork copies the table and adds one reference per block).
// The same protocol is given as formulas in "PagedAttention and Virtual
// Memory Management ..." (llms.blog) section 5.
//
// Data layout: the free list is a ring buffer of block ids (FIFO); tables are
// std::vector<int32_t> keyed by a 64-bit sequence id.  Every operation checks
// first and then mutates, so a failing call changes nothing.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"

namespace {

struct Sequence {
    std::vector<int32_t> table;
    int64_t tokens = 0;
};

}  // namespace

struct pa_alloc {
    int num_blocks = 0;
    int block_size = 0;
    // FIFO ring of free block ids: [head, head + count) modulo num_blocks.
    std::vector<int32_t> ring;
    int head = 0;
    int count = 0;
    std::vector<int32_t> refs;
    std::unordered_map<int64_t, Sequence> seqs;

    int32_t pop_front() {
        int32_t b = ring[head];
        head = (head + 1) % num_blocks;
        --count;
        refs[b] = 1;
        return b;
    }
    void push_back(int32_t b) {
        ring[(head + count) % num_blocks] = b;
        ++count;
    }
    // Blocks an append of n tokens to s would take from the free list.
    int64_t blocks_needed(const Sequence &s, int64_t n) const {
        if (n <= 0) return 0;
        int64_t B = block_size;
        int64_t first = s.tokens, last = s.tokens + n - 1;
        // positions p in [first, last] with p % B == 0
        int64_t fresh = last / B - (first + B - 1) / B + 1;
        if (fresh < 0) fresh = 0;
        bool cow = (first % B != 0) && refs[s.table.back()] > 1;
        return fresh + (cow ? 1 : 0);
    }
};

extern "C" {

pa_status pa_alloc_create(int num_blocks, int block_size, const int32_t *free_order,
                          pa_alloc **out) {
    if (!out || num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID;
    *out = nullptr;
    pa_alloc *a = new (std::nothrow) pa_alloc();
    if (!a) return PA_ERR_INVALID;
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->ring.resize(num_blocks);
    a->refs.assign(num_blocks, 0);
    if (free_order) {
        std::vector<char> seen(num_blocks, 0);
        for (int i = 0; i < num_blocks; ++i) {
            int32_t b = free_order[i];
            if (b < 0 || b >= num_blocks || seen[b]) {
                delete a;
                return PA_ERR_INVALID;
            }
            seen[b] = 1;
            a->ring[i] = b;
        }
    } else {
        for (int i = 0; i < num_blocks; ++i) a->ring[i] = i;
    }
    a->head = 0;
    a->count = num_blocks;
    *out = a;
    return PA_OK;
}

void pa_alloc_destroy(pa_alloc *a) { delete a; }

pa_status pa_seq_add(pa_alloc *a, int64_t seq_id) {
    if (!a) return PA_ERR_INVALID;
    if (a->seqs.count(seq_id)) return PA_ERR_NOT_FOUND;
    a->seqs.emplace(seq_id, Sequence());
    return PA_OK;
}

pa_status pa_seq_append(pa_alloc *a, int64_t seq_id, int n_tokens, int64_t *slots_out,
                        int64_t *cow_pair_out, int *n_cow_out) {
    if (!a || n_tokens < 0 || (n_tokens > 0 && !slots_out)) return PA_ERR_INVALID;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
    Sequence &s = it->second;
    if (a->blocks_needed(s, n_tokens) > a->count) return PA_ERR_OUT_OF_BLOCKS;
    int n_cow = 0;
    const int64_t B = a->block_size;
    for (int i = 0; i < n_tokens; ++i) {
        int64_t offset = s.tokens % B;
        if (offset == 0) {
            s.table.push_back(a->pop_front());
        } else if (a->refs[s.table.back()] > 1) {
            int32_t old_blk = s.table.back();
            int32_t new_blk = a->pop_front();
            a->refs[old_blk] -= 1;
            s.table.back() = new_blk;
            if (cow_pair_out) {
                cow_pair_out[0] = old_blk;
                cow_pair_out[1] = new_blk;
            }
            ++n_cow;
        }
        slots_out[i] = (int64_t)s.table.back() * B + offset;
        s.tokens += 1;
    }
    if (n_cow_out) *n_cow_out = n_cow;
    return PA_OK;
}

pa_status pa_seq_fork(pa_alloc *a, int64_t parent, int64_t child) {
    if (!a) return PA_ERR_INVALID;
    auto it = a->seqs.find(parent);
    if (it == a->seqs.end() || a->seqs.count(child)) return PA_ERR_NOT_FOUND;
    Sequence copy = it->second;
    for (int32_t b : copy.table) a->refs[b] += 1;
    a->seqs.emplace(child, std::move(copy));
    return PA_OK;
}

pa_status pa_seq_free(pa_alloc *a, int64_t seq_id) {
    if (!a) return PA_ERR_INVALID;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
    for (int32_t b : it->second.table) {
        a->refs[b] -= 1;
        if (a->refs[b] == 0) a->push_back(b);
    }
    a->seqs.erase(it);
    return PA_OK;
}

pa_status pa_seq_len(const pa_alloc *a, int64_t seq_id, int64_t *len_out) {
    if (!a || !len_out) return PA_ERR_INVALID;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
    *len_out = it->second.tokens;
    return PA_OK;
}

pa_status pa_seq_block_table(const pa_alloc *a, int64_t seq_id, int32_t *out, int cap,
                             int *n_out) {
    if (!a || !n_out || cap < 0) return PA_ERR_INVALID;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
    const std::vector<int32_t> &t = it->second.table;
    *n_out = (int)t.size();
    if ((int64_t)t.size() > cap || (!out && !t.empty())) return PA_ERR_INVALID;
    if (!t.empty()) std::memcpy(out, t.data(), t.size() * sizeof(int32_t));
    return PA_OK;
}

pa_status pa_alloc_export(const pa_alloc *a, const int64_t *seq_ids, int n, int32_t *tables_out,
                          int max_blocks_per_seq, int32_t *lens_out) {
    if (!a || n < 0 || max_blocks_per_seq < 0) return PA_ERR_INVALID;
    if (n > 0 && (!seq_ids || !lens_out || (max_blocks_per_seq > 0 && !tables_out)))
        return PA_ERR_INVALID;
    for (int i = 0; i < n; ++i) {  // check everything before writing anything
        auto it = a->seqs.find(seq_ids[i]);
        if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
        if ((int64_t)it->second.table.size() > max_blocks_per_seq) return PA_ERR_INVALID;
        if (it->second.tokens > INT32_MAX) return PA_ERR_INVALID;
    }
    for (int i = 0; i < n; ++i) {
        const Sequence &s = a->seqs.find(seq_ids[i])->second;
        int32_t *row = tables_out + (int64_t)i * max_blocks_per_seq;
        size_t k = s.table.size();
        if (k) std::memcpy(row, s.table.data(), k * sizeof(int32_t));
        for (int64_t j = (int64_t)k; j < max_blocks_per_seq; ++j) row[j] = 0;
        lens_out[i] = (int32_t)s.tokens;
    }
    return PA_OK;
}

int pa_alloc_num_free(const pa_alloc *a) { return a ? a->count : -1; }

pa_status pa_alloc_free_list(const pa_alloc *a, int32_t *out, int cap, int *n_out) {
    if (!a || !n_out || cap < 0) return PA_ERR_INVALID;
    *n_out = a->count;
    if (a->count > cap || (!out && a->count > 0)) return PA_ERR_INVALID;
    for (int i = 0; i < a->count; ++i) out[i] = a->ring[(a->head + i) % a->num_blocks];
    return PA_OK;
}

int pa_block_refcount(const pa_alloc *a, int block) {
    if (!a || block < 0 || block >= a->num_blocks) return -1;
    return a->refs[block];
}

// Whole blocks every sequence reaches through the same table entries (the
// cascade's shared prefix), capped by the shortest sequence.
pa_status pa_shared_prefix_len(const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *seq_lens, int num_seqs, int block_size,
                               int *prefix_len_out) {
    if (num_seqs < 0 || max_blocks_per_seq < 0 || block_size < 1 || !prefix_len_out)
        return PA_ERR_INVALID;
    if (num_seqs == 0) {
        *prefix_len_out = 0;
        return PA_OK;
    }
    if (!block_tables || !seq_lens) return PA_ERR_INVALID;
    int min_len = seq_lens[0];
    for (int i = 0; i < num_seqs; ++i) {
        if (seq_lens[i] < 0) return PA_ERR_INVALID;
        min_len = seq_lens[i] < min_len ? seq_lens[i] : min_len;
    }
    const int nb = std::min(min_len / block_size, max_blocks_per_seq);
    int n = 0;
    for (; n < nb; ++n) {
        const int32_t b0 = block_tables[n];
        bool same = true;
        for (int i = 1; i < num_seqs && same; ++i)
            same = block_tables[(int64_t)i * max_blocks_per_seq + n] == b0;
        if (!same) break;
    }
    *prefix_len_out = n * block_size;
    return PA_OK;
}

}  // extern "C"
