// Parameters and helpers shared by the two decode kernels (CUDA-core and
// tensor-core) and the split-KV reduce.
#pragma once

#include <stdint.h>

#include <utility>

#include "pa_common.cuh"

namespace pa {

constexpr int kUnit = 16;                   // positions per pipeline stage / TMA box
constexpr float kLazyRescale = 8.0f;        // base-2 units
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kSinglePassTokens = 1 << 30;  // "partition" covering any sequence

struct DecodeParams {
    void *out;                   // [S][Hq][D] (mode 0) or nullptr
    const uint16_t *q;           // [S][Hq][D]
    const uint16_t *k_pool;      // [NB][Hkv][B][D]
    const uint16_t *v_pool;
    const int32_t *block_tables; // [S][max_blocks_per_seq]
    const int32_t *seq_lens;     // [S]
    float *part_m;               // [S][Hq][NP]
    float *part_l;               // [S][Hq][NP]
    float *part_o;               // [S][Hq][NP][D]
    int *err;
    int num_seqs;
    int num_blocks;
    int max_blocks_per_seq;
    int max_seq_len;
    int num_q_heads;
    int num_kv_heads;
    int group;                   // G
    int block_size;
    int log2_block;
    int partition_tokens;        // P, multiple of kUnit
    int num_partitions;          // NP (partial slots per (sequence, query head))
    // Consecutive partitions one CTA computes (tensor-core kernel; 0 or 1:
    // one).  Each still gets its own partial; grid.x = ceil(NP / span).
    int span;
    // Compact grid (decode mode, no cascade, batches of up to
    // kCompactMaxSeqs): a 1-D grid whose CTAs map, in order, onto the work
    // items that exist (see compact_item), so CTAs with nothing to do come
    // last and are dispatched after every CTA with work.  0: 3-D grid; 1:
    // items sequence by sequence; 2: full chunks first (see compact_find).
    int compact;
    float scale_log2;            // scale * log2(e)
    int mode;                    // 0: decode (direct output when 1 partition), 1: partials only
    // Fused cache write of each sequence's newest token (pa_decode_step), or nullptr.
    const uint16_t *k_new;       // [S][Hkv][D]
    const uint16_t *v_new;
    const int64_t *slot_mapping; // [S]
    // Fused split-KV combine (nullptr when the launch does not combine):
    // arrival counters [S][Hkv] (the last chunk to arrive combines) and ready
    // flags [S][Hkv][ws_parts] (the last chunk waits for the others' flags;
    // only when every CTA of the launch is resident, see finish_item).  A
    // flag holds the call's epoch once its chunk's partials are published.
    unsigned long long *counters;
    unsigned int *flags;
    unsigned int epoch;          // tag of this call (never 0)
    int one_wave;                // 3-D grid: every CTA of the launch fits on the GPU at once
    // Sub-range of each sequence (the tail of a cascade step): positions
    // [len_offset, seq_lens[i]) read through block-table entries from
    // table_offset on; partials go to slot part_base + part of a workspace laid
    // out with ws_parts slots per (sequence, query head).
    int len_offset;
    int table_offset;
    int ws_parts;
    int part_base;
    // Cascade tail: slots [0, prefix_parts) of each row already hold the
    // shared prefix's partials (written by an earlier launch); the item's own
    // partials follow at part_base == prefix_parts, and the CTA that finishes
    // the item combines all of them into the output.
    int prefix_parts;
    // Cascade tail launched right after the prefix pass, which lets it start
    // at once: its wait for the previous kernel is put off until it reads the
    // prefix's partials (the prefix pass's only output).
    int late_wait;
    // FP8 pools (E4M3 codes): fl32(1 / scale) of each pool for the fused
    // write, and the V scale applied to the output (the K scale is folded
    // into scale_log2).
    float k_inv;
    float v_inv;
    float v_scale;
};

// Length of sequence i, clamped to what the launch covers; a value out of
// range is a bad index.
__device__ __forceinline__ int checked_len(const int32_t *seq_lens, int i, int max_seq_len,
                                           int table_cap, int *err, bool report) {
    int L = seq_lens[i];
    const int cap = max_seq_len < table_cap ? max_seq_len : table_cap;
    if (L < 0 || L > cap) {
        if (report) record_error(err, PA_ERR_BAD_INDEX);
        L = L < 0 ? 0 : cap;
    }
    return L;
}

// Programmatic dependent launch: wait for the previous kernel on the stream
// (and its memory) before touching global memory that it may write; let the
// next one start its prologue once this one is past its main loop (the
// cascade's prefix pass lets its tail pass start as soon as it holds its
// TMEM).  No-ops without the launch attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Length of the attended range of sequence `seq` (seq_lens minus
// len_offset), clamped to what the launch and the block table cover; a value
// out of range is a bad index.
__device__ __forceinline__ int item_len(const DecodeParams &p, int seq, bool report) {
    int L = p.seq_lens[seq] - p.len_offset;
    const int table_cap = (p.max_blocks_per_seq - p.table_offset) * p.block_size;
    int cap = p.max_seq_len - p.len_offset;
    if (table_cap < cap) cap = table_cap;
    if (cap < 0) cap = 0;
    if (L < 0 || L > cap) {
        if (report) record_error(p.err, PA_ERR_BAD_INDEX);
        L = L < 0 ? 0 : cap;
    }
    return L;
}

constexpr int kCompactMaxSeqs = 128;

constexpr int kCompactGroups = kCompactMaxSeqs / 32;

// Lengths of the sequences of a compact launch (at most kCompactMaxSeqs):
// lane j loads those of sequences j, 32 + j, 64 + j, 96 + j together (one
// memory round trip), -1 past the batch.
__device__ __forceinline__ void compact_lens(const DecodeParams &p, int *len) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 0; k < kCompactGroups; ++k) {
        const int s = 32 * k + lane;
        len[k] = s < p.num_seqs ? item_len(p, s, false) : -1;
    }
}

// Work item `c` of a compact grid, from the lengths compact_lens loaded.
// The items are the chunks of span * P positions of each sequence (at least
// one, so a zero-length sequence still has its CTA), each split over the KV
// heads: c = item * Hkv + kvh, sequence by sequence (p.compact == 1), or
// (p.compact == 2, grids the hardware schedules over several waves) every
// full chunk first, sequence by sequence, then each sequence's last, shorter
// chunk, so that the short items fill the end of the launch (longest first
// is the better order for a greedy schedule; this is the part of it that
// costs nothing).  A sequence's last chunk has the highest item index of its
// chunks either way.  *total is set to the number of items times Hkv (the
// launch's work, whatever c is).  Every thread of a warp calls it
// (converged); it scans the lengths 32 at a time (inclusive warp prefix
// sums) and returns false for c past the last item.
__device__ __forceinline__ bool compact_find(const DecodeParams &p, const int *len, int c, int *seq,
                                             int *chunk, int *kvh, int *total) {
    const int lane = threadIdx.x & 31;
    const int item = c / p.num_kv_heads;
    const int chunk_tok = p.partition_tokens * (p.span > 1 ? p.span : 1);
    auto scan = [&](int n) -> int {  // inclusive prefix sum over the warp
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, n, off);
            if (lane >= off) n += t;
        }
        return n;
    };
    bool found = false;
    if (p.compact != 2) {
        int base = 0;  // items of the sequences before this group of 32
#pragma unroll
        for (int k = 0; k < kCompactGroups; ++k) {
            const int s0 = 32 * k;
            if (s0 >= p.num_seqs) break;
            const int L = len[k];
            const int n = L < 0 ? 0 : (L == 0 ? 1 : (L - 1) / chunk_tok + 1);
            const int incl = scan(n);
            const int group_total = base + __shfl_sync(0xffffffffu, incl, 31);
            if (!found && item < group_total) {
                const unsigned m = __ballot_sync(0xffffffffu, base + incl > item);
                const int l = __ffs(m) - 1;
                *seq = s0 + l;
                *chunk = item - (base + __shfl_sync(0xffffffffu, incl - n, l));
                *kvh = c - item * p.num_kv_heads;
                found = true;
            }
            base = group_total;
        }
        *total = base * p.num_kv_heads;
        return found;
    }
    // full chunks first, then each sequence's shorter last chunk
    int nf_total = 0;  // full chunks of the sequences before this group of 32
#pragma unroll
    for (int k = 0; k < kCompactGroups; ++k) {
        const int s0 = 32 * k;
        if (s0 >= p.num_seqs) break;
        const int n = len[k] < 0 ? 0 : len[k] / chunk_tok;
        const int incl = scan(n);
        const int group_total = nf_total + __shfl_sync(0xffffffffu, incl, 31);
        if (!found && item < group_total) {
            const unsigned m = __ballot_sync(0xffffffffu, nf_total + incl > item);
            const int l = __ffs(m) - 1;
            *seq = s0 + l;
            *chunk = item - (nf_total + __shfl_sync(0xffffffffu, incl - n, l));
            found = true;
        }
        nf_total = group_total;
    }
    int np_total = 0;  // last chunks of the sequences before this group of 32
#pragma unroll
    for (int k = 0; k < kCompactGroups; ++k) {
        const int s0 = 32 * k;
        if (s0 >= p.num_seqs) break;
        const int L = len[k];
        const int n = (L == 0 || (L > 0 && L % chunk_tok != 0)) ? 1 : 0;
        const int incl = scan(n);
        const int group_total = np_total + __shfl_sync(0xffffffffu, incl, 31);
        const int pi = item - nf_total;  // rank among the last chunks
        if (!found && pi >= 0 && pi < group_total) {
            const unsigned m = __ballot_sync(0xffffffffu, np_total + incl > pi);
            const int l = __ffs(m) - 1;
            *seq = s0 + l;
            *chunk = __shfl_sync(0xffffffffu, L < 0 ? 0 : L / chunk_tok, l);  // after its full ones
            found = true;
        }
        np_total = group_total;
    }
    *kvh = c - item * p.num_kv_heads;
    *total = (nf_total + np_total) * p.num_kv_heads;
    return found;
}

// Work item of CTA `c` of a compact grid (lengths loaded here).
__device__ __forceinline__ bool compact_item(const DecodeParams &p, int c, int *seq, int *chunk,
                                             int *kvh) {
    int len[kCompactGroups];
    compact_lens(p, len);
    int total;
    return compact_find(p, len, c, seq, chunk, kvh, &total);
}

// Grid of a decode launch: chunks x KV heads x sequences, or the same count
// as a 1-D compact grid.
inline dim3 decode_grid(const DecodeParams &p, int chunks, int num_kv_heads, int num_seqs) {
    if (p.compact) return dim3((unsigned)((int64_t)chunks * num_kv_heads * num_seqs));
    return dim3((unsigned)chunks, (unsigned)num_kv_heads, (unsigned)num_seqs);
}

// Block-table entries of the attended range of `seq`.
__device__ __forceinline__ const int32_t *seq_table(const DecodeParams &p, int seq) {
    return p.block_tables + (int64_t)seq * p.max_blocks_per_seq + p.table_offset;
}

// Workspace row of partial `part` of (seq, query head h).
__device__ __forceinline__ int64_t part_row(const DecodeParams &p, int seq, int h, int part) {
    return ((int64_t)seq * p.num_q_heads + h) * p.ws_parts + p.part_base + part;
}

// Fused cache write (pa_decode_step): the CTA that owns the newest position
// L-1 of (seq, kvh) first writes that token's K and V into its slot, so the
// copies it issues afterwards read it.  The slot must be the one the block
// table gives for position L-1; otherwise nothing is written and a bad index
// is recorded.  Threads [0, D/4) take one 16-byte piece each; the caller
// synchronises the CTA before its copies start.
template <int D>
__device__ __forceinline__ void fused_cache_write(const DecodeParams &p, int seq, int kvh, int L) {
    constexpr int pieces = D / 8;
    const int t = threadIdx.x;
    if (t >= 2 * pieces) return;
    const int pos = L - 1;
    const bool is_v = t >= pieces;
    const int c = t % pieces;
    // the table entry, the slot and the token's piece are loaded together
    const uint4 *src = reinterpret_cast<const uint4 *>(
                           (is_v ? p.v_new : p.k_new) + ((int64_t)seq * p.num_kv_heads + kvh) * D) +
                       c;
    const uint4 val = *src;
    const int phys = seq_table(p, seq)[pos >> p.log2_block];
    const int off = pos & (p.block_size - 1);
    const int64_t slot = p.slot_mapping[seq];
    if ((unsigned)phys >= (unsigned)p.num_blocks || slot != (int64_t)phys * p.block_size + off) {
        if (t == 0) record_error(p.err, PA_ERR_BAD_INDEX);
        return;
    }
    uint4 *dst = reinterpret_cast<uint4 *>(const_cast<uint16_t *>(is_v ? p.v_pool : p.k_pool) +
                                           (((int64_t)phys * p.num_kv_heads + kvh) * p.block_size +
                                            off) * D) +
                 c;
    *dst = val;
    // make the generic-proxy store visible to the bulk-copy (async) proxy
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

constexpr int kFuseMaxParts = 8;  // combine inside the decode kernel up to this many partitions

// Compare-and-swap with acquire-release semantics at GPU scope: the
// caller's earlier writes (and those its CTA barrier ordered before it) are
// visible to whoever reads the swapped value, and the caller's later reads
// see what the writers of earlier values published.
__device__ __forceinline__ unsigned long long atom_cas_acq_rel(unsigned long long *p,
                                                               unsigned long long cmp,
                                                               unsigned long long val) {
    unsigned long long old;
    asm volatile("atom.acq_rel.gpu.global.cas.b64 %0, [%1], %2, %3;"
                 : "=l"(old)
                 : "l"(p), "l"(cmp), "l"(val)
                 : "memory");
    return old;
}

// Epoch-tagged arrival counter of the fused combine: true in exactly one CTA,
// the last of `expected` to arrive in this call.  The word holds the call's
// epoch (high half) and its count (low half); a stale or garbage word counts
// as zero.  The last arrival swaps in the reset value (epoch, 0), so graph
// replays of one call start from zero again.  Every arrival first tries the
// swap a last arrival would make (the word then holds (epoch, expected - 1)),
// so the last CTA usually needs one round trip; the others learn the word's
// value from the failed swap and retry.
__device__ __forceinline__ bool arrive_last(unsigned long long *ctr, unsigned int epoch,
                                            int expected, int *err) {
    const unsigned long long tag = (unsigned long long)epoch << 32;
    unsigned long long old = tag | (unsigned long long)(expected - 1);
    for (int it = 0; it < (1 << 16); ++it) {
        const unsigned long long cnt = ((old >> 32) == epoch) ? (old & 0xffffffffull) : 0ull;
        const bool last = cnt + 1 == (unsigned long long)expected;
        const unsigned long long prev = atom_cas_acq_rel(ctr, old, last ? tag : (tag | (cnt + 1)));
        if (prev == old) return last;
        old = prev;
    }
    record_error(err, PA_ERR_DEVICE_TIMEOUT);
    return false;
}

// Ready flags of the fused combine: a release store (the writer's earlier
// stores, and those its CTA barrier ordered before it, are visible to whoever
// acquires the value), and a bounded acquire wait for a value.
__device__ __forceinline__ void flag_release(unsigned int *f, unsigned int v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned int flag_acquire(const unsigned int *f) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    return v;
}
__device__ __forceinline__ bool flag_wait(const unsigned int *f, unsigned int v) {
    if (flag_acquire(f) == v) return true;
    const unsigned long long t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (flag_acquire(f) == v) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// 16-byte global -> shared copy through L2 only (cp.async.cg), and the wait
// for every copy this thread has committed.
__device__ __forceinline__ void cp_async16_cg(void *smem_dst, const void *gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gmem_src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
}

// Most partials one combine merges (the cascade's prefix chunks plus the
// tail's partitions); the host keeps every launch within it.
constexpr int kCombineMaxParts = 256;

// Split-KV step 3 inside the CTA that finishes (seq, kvh): for each of its
// G heads, over the slots [0, np) of the row, M = max_k m_k,
// w_k = l_k 2^(m_k - M) / sum_j l_j 2^(m_j - M), out = sum_k w_k O_k.  All
// `nthreads` threads of the CTA call it.  `scratch` is 16-byte aligned
// shared memory the CTA no longer needs, `scratch_bytes` of it, at least
// 2 * G * np floats.  Partials are read through L2 (other CTAs wrote them).
// When every O row fits in the scratch after the (m, l) pairs, the rows are
// copied in (cp.async) together with the (m, l) loads, so the merge costs
// one round of loads; otherwise four O rows per thread are kept in flight
// after the weights are known.
template <bool BF16, int D>
__device__ void fused_combine(const DecodeParams &p, int seq, int kvh, int np, float *scratch,
                              int scratch_bytes, int nthreads) {
    const int G = p.group;
    const int tid = threadIdx.x;
    const int64_t row0 = ((int64_t)seq * p.num_q_heads + (int64_t)kvh * G) * p.ws_parts;
    float *ms = scratch, *ws = scratch + G * np;
    const int buf_off = (2 * G * np + 3) & ~3;  // floats; rows [k][g][D] after (m, l)
    float *buf = scratch + buf_off;
    const bool staged = (int64_t)(buf_off + np * G * D) * 4 <= (int64_t)scratch_bytes;
    if (staged) {
        const int n16 = np * G * (D / 4);
        for (int i = tid; i < n16; i += nthreads) {
            const int x4 = i % (D / 4), r = i / (D / 4);  // r = k * G + g
            const int k = r / G, g = r - k * G;
            cp_async16_cg(buf + r * D + x4 * 4,
                          p.part_o + (row0 + (int64_t)g * p.ws_parts + k) * D + x4 * 4);
        }
    }
    for (int i = tid; i < G * np; i += nthreads) {
        const int g = i / np, k = i - g * np;
        ms[i] = __ldcg(p.part_m + row0 + (int64_t)g * p.ws_parts + k);
        ws[i] = __ldcg(p.part_l + row0 + (int64_t)g * p.ws_parts + k);
    }
    if (staged) cp_async_commit_wait_all();
    __syncthreads();
    if (tid < G) {
        float M = -INFINITY;
        for (int k = 0; k < np; ++k) M = fmaxf(M, ms[tid * np + k]);
        float tot = 0.f;
        for (int k = 0; k < np; ++k) {
            const float mk = ms[tid * np + k];
            const float w = (mk == -INFINITY) ? 0.f : ws[tid * np + k] * fast_exp2(mk - M);
            ws[tid * np + k] = w;
            tot += w;
        }
        const float inv = tot > 0.f ? 1.0f / tot : 0.f;
        for (int k = 0; k < np; ++k) ws[tid * np + k] *= inv;
    }
    __syncthreads();
    if (staged) {
        for (int item = tid; item < G * (D / 8); item += nthreads) {
            const int g = item / (D / 8);
            const int x0 = (item % (D / 8)) * 8;
            const float *w = ws + g * np;
            float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int k = 0; k < np; ++k) {
                const float4 *src = reinterpret_cast<const float4 *>(buf + (k * G + g) * D + x0);
                const float4 a = src[0], b = src[1];
                const float wk = w[k];
                o[0] += wk * a.x; o[1] += wk * a.y; o[2] += wk * a.z; o[3] += wk * a.w;
                o[4] += wk * b.x; o[5] += wk * b.y; o[6] += wk * b.z; o[7] += wk * b.w;
            }
            uint16_t *out = static_cast<uint16_t *>(p.out) +
                            ((int64_t)seq * p.num_q_heads + kvh * G + g) * D + x0;
            *reinterpret_cast<uint4 *>(out) =
                make_uint4(narrow2<BF16>(o[0], o[1]), narrow2<BF16>(o[2], o[3]),
                           narrow2<BF16>(o[4], o[5]), narrow2<BF16>(o[6], o[7]));
        }
        return;
    }
    for (int item = tid; item < G * (D / 8); item += nthreads) {
        const int g = item / (D / 8);
        const int x0 = (item % (D / 8)) * 8;
        const float *src = p.part_o + (row0 + (int64_t)g * p.ws_parts) * D + x0;
        const float *w = ws + g * np;
        float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        int k = 0;
        for (; k + 4 <= np; k += 4) {
            float4 a[4], b[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                a[j] = __ldcg(reinterpret_cast<const float4 *>(src + (int64_t)(k + j) * D));
                b[j] = __ldcg(reinterpret_cast<const float4 *>(src + (int64_t)(k + j) * D) + 1);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float wk = w[k + j];
                o[0] += wk * a[j].x; o[1] += wk * a[j].y; o[2] += wk * a[j].z; o[3] += wk * a[j].w;
                o[4] += wk * b[j].x; o[5] += wk * b[j].y; o[6] += wk * b[j].z; o[7] += wk * b[j].w;
            }
        }
        for (; k < np; ++k) {
            const float4 a = __ldcg(reinterpret_cast<const float4 *>(src + (int64_t)k * D));
            const float4 b = __ldcg(reinterpret_cast<const float4 *>(src + (int64_t)k * D) + 1);
            const float wk = w[k];
            o[0] += wk * a.x; o[1] += wk * a.y; o[2] += wk * a.z; o[3] += wk * a.w;
            o[4] += wk * b.x; o[5] += wk * b.y; o[6] += wk * b.z; o[7] += wk * b.w;
        }
        uint16_t *out = static_cast<uint16_t *>(p.out) +
                        ((int64_t)seq * p.num_q_heads + kvh * G + g) * D + x0;
        *reinterpret_cast<uint4 *>(out) = make_uint4(narrow2<BF16>(o[0], o[1]), narrow2<BF16>(o[2], o[3]),
                                                     narrow2<BF16>(o[4], o[5]), narrow2<BF16>(o[6], o[7]));
    }
}

// End of a CTA that wrote the partials of chunk `chunk` of (seq, kvh), an
// item of `nchunks` chunks; one CTA of the item combines them.
//  - use_flags (every CTA of the launch is resident at once): every chunk
//    but the last publishes its partials by a release store of the call's
//    epoch into its flag and is done; the last chunk's CTA, which has the
//    item's highest block index, waits for the other flags (acquire;
//    bounded), clears them for the next call on this workspace (a graph
//    replay repeats the epoch), and combines.  The waiting CTA holds its
//    slot, which is why this needs the whole launch resident.
//  - otherwise, with counters (p.counters): the last chunk to arrive
//    combines (arrive_last).
//  - a cascade tail of one partition (neither), or an empty tail: combine at
//    once.
// The combined slots are the prefix's and the item's: [0, prefix_parts +
// nparts_seq).  Called by every thread of the CTA; scratch and scratch_bytes
// as in fused_combine.  Ordering: the CTA barrier puts every thread's
// partial stores before thread 0's release (flag store or counter swap);
// the combiner acquires, and the next barrier orders its CTA's reads of the
// partials after that.
template <bool BF16, int D>
__device__ void finish_item(const DecodeParams &p, int seq, int kvh, int nparts_seq, int chunk,
                            int nchunks, bool use_flags, float *scratch, int scratch_bytes) {
    __shared__ int all_ready;
    __syncthreads();
    if (nparts_seq > 0 && p.counters != nullptr && !use_flags) {
        if (threadIdx.x == 0)
            all_ready = arrive_last(p.counters + (int64_t)seq * p.num_kv_heads + kvh, p.epoch,
                                    nchunks, p.err);
        __syncthreads();
        if (!all_ready) return;
    } else if (nparts_seq > 0 && p.flags != nullptr) {
        unsigned int *flag = p.flags + ((int64_t)seq * p.num_kv_heads + kvh) * p.ws_parts;
        if (chunk + 1 < nchunks) {
            if (threadIdx.x == 0) flag_release(flag + chunk, p.epoch);
            return;
        }
        if (threadIdx.x < 32) {
            bool ok = true;
            for (int k = threadIdx.x; k < nchunks - 1; k += 32) {
                if (flag_wait(flag + k, p.epoch))
                    flag[k] = 0u;
                else
                    ok = false;
            }
            ok = __all_sync(0xffffffffu, ok);
            if (threadIdx.x == 0) {
                all_ready = ok;
                if (!ok) record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
            }
        }
        __syncthreads();
        if (!all_ready) return;
    }
    fused_combine<BF16, D>(p, seq, kvh, p.prefix_parts + nparts_seq, scratch, scratch_bytes,
                           blockDim.x);
}

// Kernel launch with programmatic stream serialization allowed (PDL).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Tensor-core decode (pa_decode_tc.cu).
bool tc_supported(int head_dim, int group);
int tc_ctas_per_sm(bool bf16, int head_dim);
pa_status launch_decode_tc(const DecodeParams &prm, bool bf16, int head_dim, int num_partitions,
                           int num_kv_heads, int num_seqs, cudaStream_t stream);

// Tensor-core decode over E4M3 pools (pa_decode_tc_fp8.cu).
bool fp8_supported(int head_dim, int group);
int fp8_ctas_per_sm(bool bf16, int head_dim, int group);
pa_status launch_decode_fp8(const DecodeParams &prm, bool bf16, int head_dim, int num_partitions,
                            int num_kv_heads, int num_seqs, cudaStream_t stream);

// Prefix pass of the shared-prefix (cascade) decode (pa_cascade.cu): the
// positions [0, prefix_len) that every sequence reaches through the same
// block-table entries (sequence 0's row gives them), attended once per KV
// head by the query rows of all sequences.  Leaves the (m, l, O) partial of
// chunk c of each (sequence, query head) in workspace slot c.
struct CascadeParams {
    const uint16_t *q;           // [S][Hq][D]
    const int32_t *block_tables; // [S][max_blocks_per_seq]
    const int32_t *seq_lens;     // [S] (checked: >= prefix_len)
    float *part_m;               // [S][Hq][ws_parts]
    float *part_l;
    float *part_o;               // [S][Hq][ws_parts][D]
    int *err;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int group;
    int num_blocks;
    int max_blocks_per_seq;
    int block_size;
    int log2_block;
    int prefix_len;              // a multiple of block_size, > 0
    int chunk_tokens;            // a multiple of 128
    int num_chunks;              // a multiple of cluster (trailing chunks may be empty)
    int cluster;                 // CTAs of consecutive chunks merged in one cluster (1, 2, 4, 8)
    int ws_parts;                // the merged partial of cluster c goes to slot c
    float scale_log2;
};

// Chunking of the prefix pass: chunk length (a multiple of 128 positions),
// number of chunks and cluster size, spreading the pass over about one CTA
// per SM of the current device.  The pass leaves num_chunks / cluster
// partials per (sequence, query head).
struct CascadeChunks {
    int chunk_tokens;
    int num_chunks;
    int cluster;
};
CascadeChunks cascade_chunks(int prefix_len, int num_rows, int num_kv_heads, int head_dim,
                             bool bf16);
pa_status launch_cascade_prefix(const CascadeParams &cp, const void *k_pool, const void *v_pool,
                                bool bf16, int head_dim, cudaStream_t stream);

}  // namespace pa
