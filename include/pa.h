/*
 * pa.h - C ABI of the paged KV-cache library (paged decode attention,
 * cache write, block copy, host block allocator) for NVIDIA GB300 (sm_103a).
 *
 * Conventions for every entry point:
 *  - Plain C types only.  "Device" pointers are CUDA global-memory addresses
 *    owned by the caller (the library never frees or keeps them); "host"
 *    pointers are ordinary CPU memory.  No entry point allocates device
 *    memory: scratch space for split-KV comes from a caller-provided
 *    workspace.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream of the current device).  Device entry points enqueue work on it
 *    and return after launch, without synchronising.
 *  - Shapes and arguments are validated on the host before any launch;
 *    invalid ones return PA_ERR_INVALID and launch nothing.  Combinations of
 *    (head_dim, block_size, G) that are not compiled in return
 *    PA_ERR_UNSUPPORTED.  Launch failures return PA_ERR_CUDA.
 *  - Index values read on the device (block-table entries, slots, copy
 *    pairs, sequence lengths) are range-checked inside the kernels: a bad
 *    value is never dereferenced; the kernel records PA_ERR_BAD_INDEX in a
 *    per-device error word and skips or clamps the access.  Bounded waits
 *    that run out record PA_ERR_DEVICE_TIMEOUT.  pa_check_error reads the
 *    word.  Kernels never trap.
 *  - Element type of K/V/q/out is given by pa_dtype (16-bit IEEE half or
 *    bfloat16); arithmetic is fp32 with fp32 accumulation; outputs are
 *    rounded to nearest even.
 *
 * Memory layout (all dense, row-major, no padding):
 *    K / V pool       [num_blocks][num_kv_heads][block_size][head_dim]
 *    q, out           [num_seqs][num_q_heads][head_dim]
 *    block_tables     int32 [num_seqs][max_blocks_per_seq]
 *    seq_lens         int32 [num_seqs]
 *    k_new, v_new     [num_tokens][num_kv_heads][head_dim]
 *    slot_mapping     int64 [num_tokens]   (slot = block * block_size + offset)
 *    block_mapping    int64 [num_pairs][2] (src, dst)
 *
 * Sources for the operations (page title, section):
 *  [P1] "PagedAttention: Treating KV Memory Like Virtual Memory"
 *       (lenatriestounderstand.com)
 *  [P2] "Why AI servers waste memory, and how paging fixes it" (spicyshark.co)
 *  [P3] "PagedAttention and Virtual Memory Management: Mathematical
 *       Foundations of Non-Contiguous KV-Cache Allocation, Dynamic Block
 *       Translation, and Copy-on-Write Forking Mechanics" (llms.blog)
 *  [P4] "2.1 PagedAttention" (infra-guide)
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID = 1,       /* bad argument or shape; nothing changed / launched */
    PA_ERR_OUT_OF_BLOCKS = 2, /* allocator: not enough free blocks; nothing changed */
    PA_ERR_UNSUPPORTED = 3,   /* shape combination not compiled in */
    PA_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    PA_ERR_DEVICE_TIMEOUT = 5,/* a bounded device wait ran out (reported by pa_check_error) */
    PA_ERR_BAD_INDEX = 6,     /* an out-of-range index was met on the device (pa_check_error) */
    PA_ERR_NOT_FOUND = 7,     /* allocator: unknown sequence id, or id already in use */
    PA_ERR_TOO_LARGE = 8      /* pa_decode_static_scratch: partials exceed the fixed scratch */
} pa_status;

typedef enum { PA_F16 = 0, PA_BF16 = 1 } pa_dtype;

/* Library version (major*10000 + minor*100 + patch). */
int pa_version(void);

/* Human-readable name of a status code (static string). */
const char *pa_status_string(pa_status s);

/* ------------------------------------------------------------------------
 * pa_cache_write (reshape_and_cache)
 *
 * For every new token t and KV head h:
 *   K_pool[slot/B][h][slot%B][:] = k_new[t][h][:]   (same for V)
 * with slot = slot_mapping[t] and B = block_size.  A negative slot means
 * "skip this token".  A slot >= num_blocks*block_size is a bad index: it is
 * not written and PA_ERR_BAD_INDEX is recorded.  Pure copy, bit-exact.
 *   [P2] "The real implementation" (append writes k, v at the offset of the
 *   last block); [P3] section 5, case 1 (write into slot o = t mod B of block
 *   p); [P4] section 5 (physical_block_number, physical_block_offset).
 * Arguments: k_new, v_new, slot_mapping, k_pool, v_pool are device pointers;
 * num_tokens >= 0 (0 launches nothing); head_dim in {64, 128};
 * block_size > 0.  Pools are updated in place.
 * ---------------------------------------------------------------------- */
pa_status pa_cache_write(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                         int num_tokens, void *k_pool, void *v_pool, int num_blocks,
                         int num_kv_heads, int head_dim, int block_size, pa_dtype dtype,
                         void *stream);

/* ------------------------------------------------------------------------
 * pa_copy_blocks (copy-on-write block duplication)
 *
 * For each pair (src, dst) of block_mapping, in every layer l < num_layers,
 * for both pools:  pool_l[dst][:] = pool_l[src][:]  (the whole block:
 * num_kv_heads*block_size*head_dim elements = block_bytes bytes).
 *   [P2] "The real implementation", the copy-on-write branch of append (the
 *   whole block is copied); [P3] section 5 case 2 step 2 (copies the first o
 *   token vectors: the extra slots copied here are never read).
 * Pairs are independent: a dst must not also appear as a src or as another
 * pair's dst in the same call (the allocator never produces that).  An index
 * outside [0, num_blocks) is a bad index (pair skipped, PA_ERR_BAD_INDEX).
 * Arguments: k_pools, v_pools are HOST arrays of num_layers DEVICE pointers
 * (1 <= num_layers <= 1024); block_mapping is a DEVICE int64 array
 * [num_pairs][2]; num_pairs >= 0 (0 launches nothing); block_bytes > 0 and a
 * multiple of 16; every pool pointer 16-byte aligned.
 * ---------------------------------------------------------------------- */
pa_status pa_copy_blocks(void *const *k_pools, void *const *v_pools, int num_layers,
                         const int64_t *block_mapping, int num_pairs, int num_blocks,
                         size_t block_bytes, void *stream);

/* ------------------------------------------------------------------------
 * pa_decode (single-query paged decode attention with grouped-query heads)
 *
 * For sequence i (L_i = seq_lens[i] tokens), query head h, G =
 * num_q_heads/num_kv_heads, kv = h / G, T_i = block_tables[i]:
 *   K_i[p] = K_pool[T_i[p / B]][kv][p % B][:],  p < L_i   (same for V)
 *   s_p    = scale * dot(q[i][h], K_i[p])
 *   out[i][h][:] = sum_p softmax(s)_p * V_i[p][:]
 * L_i = 0 gives a zero row.  Slots past L_i are never read into the result,
 * whatever they hold (NaN included).
 *   [P1] "How the kernel reads a block table" (tiles, running max and sum,
 *   address = block_table[i / B] * block stride + (i mod B) * slot stride);
 *   [P3] section 4 (Vectorized Address Computation; Fused PagedAttention
 *   Algorithm with online softmax; Parallel Partitioning, steps 1-3);
 *   [P2] "Reading through the table".
 *
 * Long sequences are split into partitions of P tokens (split-KV: P3 section
 * 4, Parallel Partitioning, step 2), each producing (m_k, l_k, O_k), then
 * combined by the cross-partition reduce (step 3).  partition_tokens:
 *   -1  single pass (one work unit per (sequence, KV head); no workspace)
 *    0  automatic choice from the shapes and the GPU's SM count
 *   >0  P = partition_tokens (must be a multiple of block_size)
 * With P > 0 or automatic, workspace must hold at least
 * pa_decode_workspace_size(...) bytes (device memory, 256-byte aligned); it
 * is scratch, overwritten on every call, and may be NULL when the size is 0.
 * It needs no initialisation: besides the partials it holds one arrival
 * counter per (sequence, KV head) and one ready flag per partial, tagged
 * with a per-call epoch so that stale contents read as zero; when a
 * sequence has at most 8 partials one CTA of the launch combines them (one
 * launch), otherwise a separate combine kernel runs.  When a CTA computes
 * several consecutive partitions (see pa_set_decode_span), it combines them
 * as it goes (the online softmax's rescale is the combine formula) and
 * leaves one partial for its span.  Launches use programmatic dependent launch: each
 * kernel waits for the previous work on the stream before reading memory.
 *
 * Arguments (device pointers unless stated):
 *   out, q                 [num_seqs][num_q_heads][head_dim]
 *   k_pool, v_pool         [num_blocks][num_kv_heads][block_size][head_dim]
 *   block_tables           int32 [num_seqs][max_blocks_per_seq]; entries
 *                          must lie in [0, num_blocks) for the blocks a
 *                          sequence uses (checked: PA_ERR_BAD_INDEX)
 *   seq_lens               int32 [num_seqs]; 0 <= L_i <= max_seq_len and
 *                          L_i <= max_blocks_per_seq*block_size (checked)
 *   max_seq_len            host int, an upper bound of every L_i (sizes the
 *                          launch); 0 is allowed
 *   head_dim in {64,128}; block_size in {16,32}; 1 <= G <= 8; scale finite.
 *   num_seqs and num_kv_heads at most 65535 (PA_ERR_INVALID above: a larger
 *   batch is split into several calls by the caller).
 *   q, out, pools and workspace 16-byte aligned.
 * ---------------------------------------------------------------------- */
pa_status pa_decode(void *out, const void *q, const void *k_pool, const void *v_pool,
                    int num_blocks, const int32_t *block_tables, int max_blocks_per_seq,
                    const int32_t *seq_lens, int max_seq_len, int num_seqs, int num_q_heads,
                    int num_kv_heads, int head_dim, int block_size, float scale,
                    int partition_tokens, void *workspace, size_t workspace_bytes,
                    pa_dtype dtype, void *stream);

/* ------------------------------------------------------------------------
 * pa_decode_step: one decode step, fused.  For every sequence i its newest
 * token (position seq_lens[i]-1) is first written into the cache exactly as
 * pa_cache_write would write k_new[i], v_new[i] at slot_mapping[i]; then
 * pa_decode runs over seq_lens[i] positions, new token included.  Both happen
 * inside one kernel: the CTA that reads position seq_lens[i]-1 writes it
 * first.  slot_mapping[i] must be the slot the block table gives for that
 * position (block_tables[i][(L-1)/B]*B + (L-1)%B); a different slot is
 * reported as PA_ERR_BAD_INDEX and that token is not written.  Sequences
 * with seq_lens[i] = 0 write nothing.  The pools are updated in place.
 *   k_new, v_new: [num_seqs][num_kv_heads][head_dim] (device); slot_mapping:
 *   int64 [num_seqs] (device).  Other arguments as pa_decode.
 * ---------------------------------------------------------------------- */
pa_status pa_decode_step(void *out, const void *q, const void *k_new, const void *v_new,
                         const int64_t *slot_mapping, void *k_pool, void *v_pool, int num_blocks,
                         const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *seq_lens, int max_seq_len, int num_seqs, int num_q_heads,
                         int num_kv_heads, int head_dim, int block_size, float scale,
                         int partition_tokens, void *workspace, size_t workspace_bytes,
                         pa_dtype dtype, void *stream);

/* ------------------------------------------------------------------------
 * pa_decode_cascade: pa_decode (or, with k_new != NULL, pa_decode_step) for
 * a batch whose sequences share a prefix, computed as a cascade.  The result
 * is the same attention as pa_decode's (within the output tolerance).
 *
 * Sequences forked from one prompt point the first entries of their block
 * tables at the same physical blocks ([P1] "The same trick for the cache";
 * [P2] "Sharing a prefix with copy-on-write"; [P3] section 5, page-table
 * duplication on a fork).  With P = prefix_len positions (a whole number of
 * blocks) shared by every sequence of the batch:
 *   1. prefix pass: for each KV head, the q rows of ALL sequences of its
 *      group attend to positions [0, P) once, as dense products on the
 *      tensor cores (tcgen05), reading the shared blocks through sequence
 *      0's table; the positions are cut into chunks, each leaving a partial
 *      (m, l, O) per (sequence, query head) in the workspace;
 *   2. tail pass: each sequence attends to its own positions [P, L_i)
 *      (through table entries P/B onwards), as pa_decode does, writes that
 *      partial next to the prefix's, and combines all of them with the
 *      split-KV log-sum-exp merge ([P3] section 4, Parallel Partitioning,
 *      step 3).  softmax over [0, L_i) equals that merge of the two ranges.
 * Requirements (checked on the device, PA_ERR_BAD_INDEX when violated, the
 * output then being unspecified): for every sequence i, seq_lens[i] >= P and
 * block_tables[i][b] == block_tables[0][b] for b < P / block_size.
 * prefix_len must be a multiple of block_size, <= max_seq_len and
 * <= max_blocks_per_seq*block_size (else PA_ERR_INVALID); prefix_len = 0
 * is plain pa_decode / pa_decode_step with partition_tokens = 0.
 * k_new, v_new, slot_mapping: NULL for a plain decode, or the newest tokens
 * as in pa_decode_step; their positions must lie in the tails (the tail
 * pass, which writes them, may run while the prefix pass is still reading
 * the prefix).
 * workspace: pa_decode_cascade_workspace_size(...) bytes of device memory,
 * 256-byte aligned, scratch (no initialisation needed).  Other arguments as
 * pa_decode.
 * ---------------------------------------------------------------------- */
pa_status pa_decode_cascade(void *out, const void *q, const void *k_new, const void *v_new,
                            const int64_t *slot_mapping, void *k_pool, void *v_pool,
                            int num_blocks, const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *seq_lens, int max_seq_len, int num_seqs,
                            int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                            float scale, int prefix_len, void *workspace, size_t workspace_bytes,
                            pa_dtype dtype, void *stream);

/* ------------------------------------------------------------------------
 * pa_shared_prefix_len: the prefix_len pa_decode_cascade can be given for a
 * batch (host-side planning; no device work).  Counts the leading block-table
 * entries b that every sequence holds in common (block_tables[i][b] ==
 * block_tables[0][b] for all i: forks of one prompt, [P2] "Sharing a prefix
 * with copy-on-write"), capped by the shortest sequence's whole blocks
 * (min seq_lens / block_size) and by max_blocks_per_seq, and writes that
 * count times block_size to *prefix_len_out.  An empty batch gives 0.
 *   block_tables: int32 [num_seqs][max_blocks_per_seq], HOST memory;
 *   seq_lens: int32 [num_seqs], HOST memory; neither is modified.
 * Errors: PA_ERR_INVALID (nothing written) for num_seqs < 0,
 * max_blocks_per_seq < 0, block_size < 1, a null prefix_len_out, null
 * arrays with num_seqs > 0, or a negative length.
 * ---------------------------------------------------------------------- */
pa_status pa_shared_prefix_len(const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *seq_lens, int num_seqs, int block_size,
                               int *prefix_len_out);

/* Bytes of workspace pa_decode_cascade needs for these shapes on the current
 * CUDA device (the prefix chunking follows its SM count); 0 for invalid
 * arguments. */
size_t pa_decode_cascade_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                        int head_dim, int block_size, int max_seq_len,
                                        int prefix_len, pa_dtype dtype);

/* ------------------------------------------------------------------------
 * FP8 KV cache (a variant).  [P3] section 1 gives b = 1 byte per element for
 * FP8 in the KV-size formula and nothing more; the format and the scale are
 * this library's conventions: pools hold OCP E4M3 codes (1 sign, 4 exponent
 * bits with bias 7, 3 mantissa bits, subnormals, no infinities, S.1111.111
 * NaN, largest finite 448), one byte per element, in the same
 * [num_blocks][num_kv_heads][block_size][head_dim] layout, and each pool has
 * one scale: element = scale * code value.
 *
 * pa_cache_write_fp8: pa_cache_write into E4M3 pools.  Each element x of
 * k_new / v_new (16-bit, dtype) becomes the code nearest (ties to even) to
 * the fp32 product x * fl32(1 / scale), saturating at +-448.  Other
 * arguments as pa_cache_write; scales finite and > 0.
 * ---------------------------------------------------------------------- */
pa_status pa_cache_write_fp8(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                             int num_tokens, void *k_pool, void *v_pool, int num_blocks,
                             int num_kv_heads, int head_dim, int block_size, float k_scale,
                             float v_scale, pa_dtype dtype, void *stream);

/* pa_decode over E4M3 pools: out[i][h] = sum_p softmax(s)_p * v_scale * V_i[p]
 * with s_p = scale * dot(q[i][h], k_scale * K_i[p]) (code values).  q and out
 * are 16-bit (dtype).  With k_new != NULL, each sequence's newest token is
 * first quantised and written as pa_cache_write_fp8 would (the fused step of
 * pa_decode_step).  The tensor-core kernel takes the codes as they are as
 * E4M3 operands of q.K^T and P.V, with q and P as sums of four E5M2 terms
 * each and fp32 accumulation.
 * head_dim in {64, 128}, G <= 8, block_size in {16, 32}; partition_tokens
 * and workspace as pa_decode (size from pa_decode_fp8_workspace_size). */
pa_status pa_decode_fp8(void *out, const void *q, const void *k_new, const void *v_new,
                        const int64_t *slot_mapping, void *k_pool, void *v_pool, int num_blocks,
                        const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *seq_lens, int max_seq_len, int num_seqs, int num_q_heads,
                        int num_kv_heads, int head_dim, int block_size, float scale,
                        float k_scale, float v_scale, int partition_tokens, void *workspace,
                        size_t workspace_bytes, pa_dtype dtype, void *stream);

size_t pa_decode_fp8_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                    int head_dim, int block_size, int max_seq_len,
                                    int partition_tokens, pa_dtype dtype);

/* Partition size pa_decode uses for these shapes when partition_tokens = 0
 * (-1 means it will run single pass).  Needs the current CUDA device. */
int pa_decode_auto_partition(int num_seqs, int num_kv_heads, int max_seq_len, int head_dim,
                             int block_size, int group_size, pa_dtype dtype);
/* Positions each split-KV partial of pa_decode (fp8 = 0) or pa_decode_fp8
 * (fp8 = 1) covers for these shapes and partition_tokens (0 = automatic):
 * the partition size times the partitions one CTA merges (see
 * pa_set_decode_span), or -1 for single pass.  The decode writes
 * ceil(max_seq_len / this) partials per (sequence, query head) and combines
 * them inside the launch when there are at most 8.  -2 for unsupported or
 * invalid shapes.  Needs the current CUDA device. */
int pa_decode_partial_tokens(int num_seqs, int num_kv_heads, int max_seq_len, int head_dim,
                             int block_size, int group_size, int partition_tokens, pa_dtype dtype,
                             int fp8);
/* The same for pa_decode_fp8 (E4M3 pools; the same choice as pa_decode). */
int pa_decode_fp8_auto_partition(int num_seqs, int num_kv_heads, int max_seq_len, int head_dim,
                                 int block_size, int group_size, pa_dtype dtype);

/* Decode kernel selection, process-wide, for every later call:
 *   0 automatic (default): the tensor-core kernel (tcgen05 MMAs, TMA tensor
 *     copies) wherever it applies (head_dim 64/128, G <= 8), else the
 *     CUDA-core kernel (packed fp32 FMAs);
 *   1 always the CUDA-core kernel;  2 always the tensor-core kernel.
 * Both compute the same result to within the output tolerance.  Returns the
 * previous setting, or -1 (nothing changed) for an invalid value.  Not
 * synchronised with decode calls running on other host threads. */
int pa_set_decode_impl(int impl);
int pa_get_decode_impl(void);

/* Split-KV partitions one tensor-core CTA computes, process-wide, for every
 * later call: 0 automatic (default: several consecutive partitions a CTA
 * when partitions are short and the grid keeps at least two waves of CTAs),
 * n >= 1 that many wherever partitions are a multiple of 128 positions (1
 * elsewhere).  pa_decode_partitions writes each partition's own (m, l, O)
 * partial; the decode entry points merge a CTA's partitions into one
 * partial.  The result is the same for any setting (within the output
 * tolerance).  Returns the previous setting, or -1 (nothing changed) for a
 * negative value.  Not synchronised with decode calls running on other host
 * threads. */
int pa_set_decode_span(int span);

/* Resident CTAs per SM of the decode kernel that these shapes select
 * (occupancy query on the current device; 0 if unsupported). */
int pa_decode_ctas_per_sm(int head_dim, int group_size, pa_dtype dtype);

/* Bytes of workspace pa_decode / pa_decode_partitions need for these
 * shapes; 0 for single pass.  partition_tokens as in pa_decode (0 = auto,
 * resolved as pa_decode would with the same arguments). */
size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                int block_size, int max_seq_len, int partition_tokens,
                                pa_dtype dtype);

/* ------------------------------------------------------------------------
 * pa_decode_partitions (split-KV step 2 on its own)
 *
 * Computes, for every sequence i, query head h and partition k <
 * NP = ceil(max_seq_len / P), over positions [k*P, min((k+1)*P, L_i)):
 *   m[i][h][k] = max_p s_p * log2(e)       (fp32, base-2 units)
 *   l[i][h][k] = sum_p 2^(s_p*log2(e) - m)  (fp32)
 *   O[i][h][k][:] = sum_p 2^(s_p*log2(e) - m) V_i[p] / l   (fp32)
 * Partitions that start at or past L_i hold m = -inf, l = 0, O = 0.
 * Workspace layout (from its start, each array 256-byte aligned):
 *   m  float [num_seqs][num_q_heads][NP]
 *   l  float [num_seqs][num_q_heads][NP]
 *   O  float [num_seqs][num_q_heads][NP][head_dim]
 *   arrival counters  uint64 [num_seqs][num_kv_heads]  (pa_decode only)
 *   ready flags  uint32 [num_seqs][num_kv_heads][NP]  (pa_decode only)
 *   [P3] section 4, "Parallel Partitioning Across GPU Warps", step 2.
 * partition_tokens must be > 0 here.  Other arguments as pa_decode.
 * ---------------------------------------------------------------------- */
pa_status pa_decode_partitions(const void *q, const void *k_pool, const void *v_pool,
                               int num_blocks, const int32_t *block_tables,
                               int max_blocks_per_seq, const int32_t *seq_lens, int max_seq_len,
                               int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                               int block_size, float scale, int partition_tokens,
                               void *workspace, size_t workspace_bytes, pa_dtype dtype,
                               void *stream);

/* ------------------------------------------------------------------------
 * pa_split_kv_reduce (split-KV step 3 on its own)
 *
 * Reads the partials that pa_decode_partitions wrote (same workspace
 * layout, same partition_tokens and max_seq_len) and writes, per (i, h):
 *   M = max_k m_k ;  w_k = l_k * 2^(m_k - M) ;  out = sum_k w_k O_k / sum_k w_k
 * over the partitions k < ceil(L_i / P); L_i = 0 gives zeros.
 *   [P3] section 4, "Parallel Partitioning Across GPU Warps", step 3
 *   (m_global = max m_k, l_global = sum l_k e^(m_k - m_global),
 *    O = sum_k l_k e^(m_k - m_global) / l_global * O_k), in base 2.
 * ---------------------------------------------------------------------- */
pa_status pa_split_kv_reduce(void *out, const void *workspace, size_t workspace_bytes,
                             const int32_t *seq_lens, int max_seq_len, int num_seqs,
                             int num_q_heads, int head_dim, int partition_tokens, pa_dtype dtype,
                             void *stream);

/* ------------------------------------------------------------------------
 * pa_decode_static_scratch: pa_decode for callers that cannot allocate.
 *
 * Some callers of this library cannot hand it a workspace: an inference
 * engine that has already given (nearly) all device memory to its KV-cache
 * pool and its weights, or a latency-critical decode loop that must not
 * call cudaMalloc (it can synchronise the device and can fail under memory
 * pressure), or a foreign-language host that reaches the library only
 * through this C ABI with no allocator of its own.  This entry point
 * computes exactly what pa_decode computes, with the same arguments minus
 * the workspace, and allocates nothing: its split-KV partials live in one
 * file-scope device array of PA_STATIC_SCRATCH_BYTES bytes that every GPU
 * holds from the moment the library is loaded until the process exits.
 * The pages have no counterpart to this entry point.
 *  - A request whose partials need more than PA_STATIC_SCRATCH_BYTES
 *    (pa_decode_workspace_size with the same arguments) is rejected with
 *    PA_ERR_TOO_LARGE before anything is launched; pick a larger
 *    partition_tokens (fewer partials) or -1 (single pass, no scratch).
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.  The address is kept for the life of the
 *    process (as is the error word's, for every entry point): after a
 *    cudaDeviceReset it would be stale, so resetting a device while this
 *    library is loaded is not supported.
 *  - Every call on a device shares the one array, and it keeps whatever the
 *    last call left there.  Nothing in it needs to start at zero: every
 *    partial the combine step reads is written earlier in the same call.
 *    Calls whose kernels overlap on the GPU (different streams, no ordering
 *    between them) race on the array and give wrong results; order them.
 * ---------------------------------------------------------------------- */
#define PA_STATIC_SCRATCH_BYTES ((size_t)16 << 20)

pa_status pa_decode_static_scratch(void *out, const void *q, const void *k_pool,
                                   const void *v_pool, int num_blocks,
                                   const int32_t *block_tables, int max_blocks_per_seq,
                                   const int32_t *seq_lens, int max_seq_len, int num_seqs,
                                   int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, float scale, int partition_tokens,
                                   pa_dtype dtype, void *stream);

/* ------------------------------------------------------------------------
 * pa_check_error: synchronises `stream`, then reads and clears the current
 * device's error word.  Returns PA_OK, PA_ERR_BAD_INDEX,
 * PA_ERR_DEVICE_TIMEOUT, or PA_ERR_CUDA if the synchronisation failed.
 * ---------------------------------------------------------------------- */
pa_status pa_check_error(void *stream);

/* ------------------------------------------------------------------------
 * pa_selftest_wait_timeout: exercises the bounded-wait error path.  Launches
 * one CTA that waits on a shared-memory mbarrier no thread ever arrives on,
 * with the same bounded wait the decode pipeline uses; after the library's
 * wait limit (about one second) the kernel gives up, records
 * PA_ERR_DEVICE_TIMEOUT in the error word and returns.  The GPU context
 * stays usable.  Read the result with pa_check_error.  (Diagnostic entry
 * point; the pages have no counterpart.)
 * ---------------------------------------------------------------------- */
pa_status pa_selftest_wait_timeout(void *stream);

/* ========================================================================
 * Host block allocator (CPU only; no device calls).
 *
 * Semantics ([P2] "The idea: a block table", "A hand-worked example", "The
 * real implementation", "Sharing a prefix with copy-on-write"; [P3]
 * section 5; [P4] sections 3, 6 and 9.3):
 *  - num_blocks blocks of block_size slots; a FIFO free list (take from the
 *    front, freed blocks join the back, in table order); freed blocks are
 *    not cleared.  The initial order is 0..num_blocks-1 unless given.
 *  - each sequence has a block table and a token count; position p is slot
 *    p % B of block table[p / B]; flat slot = block * B + offset.
 *  - append: when the count is a multiple of B (incl. 0) a block is taken
 *    and appended; else if the last block is shared (refcount > 1) a block
 *    is taken, the old block's count drops by one, the table points at the
 *    new block and the pair (old, new) is reported for pa_copy_blocks
 *    (copy-on-write).  Multi-token appends are all or nothing.
 *  - fork: child gets the parent's table and count; each block gains a
 *    reference.  free: each block loses one; at zero it joins the free list.
 * Every failing call returns an error and leaves the state unchanged.  An
 * allocator object is not thread-safe: one thread at a time.
 * ===================================================================== */
typedef struct pa_alloc pa_alloc;

/* free_order: NULL, or a host array holding a permutation of
 * 0..num_blocks-1 that sets the initial free-list order. */
pa_status pa_alloc_create(int num_blocks, int block_size, const int32_t *free_order,
                          pa_alloc **out);
void pa_alloc_destroy(pa_alloc *a);

/* New empty sequence (PA_ERR_NOT_FOUND if the id is in use). */
pa_status pa_seq_add(pa_alloc *a, int64_t seq_id);

/* Append n_tokens >= 0 tokens.  slots_out (host, may be NULL if n_tokens
 * is 0) receives each token's flat slot.  cow_pair_out (host, 2 entries)
 * receives (src, dst) when a copy-on-write happened; *n_cow_out (host) is
 * set to 0 or 1.  PA_ERR_OUT_OF_BLOCKS when the blocks needed exceed the
 * free list (nothing changes). */
pa_status pa_seq_append(pa_alloc *a, int64_t seq_id, int n_tokens, int64_t *slots_out,
                        int64_t *cow_pair_out, int *n_cow_out);

pa_status pa_seq_fork(pa_alloc *a, int64_t parent, int64_t child);
pa_status pa_seq_free(pa_alloc *a, int64_t seq_id);

/* Token count of a sequence. */
pa_status pa_seq_len(const pa_alloc *a, int64_t seq_id, int64_t *len_out);

/* Copy a sequence's block table into out (host, cap entries).  *n_out gets
 * the table length; PA_ERR_INVALID if cap is too small (nothing written). */
pa_status pa_seq_block_table(const pa_alloc *a, int64_t seq_id, int32_t *out, int cap,
                             int *n_out);

/* Export tables and lengths of n sequences into a dense int32
 * [n][max_blocks_per_seq] array (host; unused entries set to 0) and an
 * int32 [n] length array (host).  PA_ERR_INVALID if a table is longer than
 * max_blocks_per_seq or a length does not fit in int32. */
pa_status pa_alloc_export(const pa_alloc *a, const int64_t *seq_ids, int n,
                          int32_t *tables_out, int max_blocks_per_seq, int32_t *lens_out);

int pa_alloc_num_free(const pa_alloc *a);

/* Free list, front first (host, cap entries); *n_out gets its length. */
pa_status pa_alloc_free_list(const pa_alloc *a, int32_t *out, int cap, int *n_out);

/* Reference count of a block (-1 if out of range). */
int pa_block_refcount(const pa_alloc *a, int block);

/* ------------------------------------------------------------------------
 * Prefix-caching block pool (host): the allocator with automatic prefix
 * caching.  [P4] section 9 (KVCacheManager over BlockPool: get_computed_blocks,
 * allocate_slots, free in reverse order; the doubly linked free queue;
 * get_new_blocks / free_blocks / touch with reference counts); [P1] "A
 * separate mechanism: automatic prefix caching" (block hash chain over the
 * previous block's hash and the block's token ids, block-aligned matches,
 * nothing copied on a hit, cached blocks evicted oldest-first) and "Where the
 * analogy stops" (cache_salt mixed into the first block's hash).
 *
 * Every block is in use (refcount > 0) or in the free queue.  New blocks come
 * off the queue's head; taking a cached block evicts its hash.  A request's
 * block fills -> it is hashed: FNV-1a 64 (offset basis 0xcbf29ce484222325,
 * prime 0x100000001b3) over the previous block's hash (the request's salt for
 * its first block) as 8 little-endian bytes, then each token id as 4
 * little-endian bytes; it is cached under that hash unless a block already
 * holds the same content.  A lookup matches the longest run of a prompt's
 * leading full blocks whose chain is cached (stored token ids and previous
 * hash compared, so a hash collision only costs a hit), at most
 * (n - 1) / block_size blocks: the last prompt token is always computed.
 * Freeing visits the request's blocks tail first; each loses a reference;
 * blocks reaching zero go to the queue's head when unhashed (the first one
 * freed becomes the head) and to its tail when hashed (LRU eviction).  Only
 * full blocks are shared, so no block is ever copied.  Single-threaded;
 * every failing call leaves the pool unchanged.  All pointers are host.
 * ---------------------------------------------------------------------- */
typedef struct pa_pcache pa_pcache;

/* num_blocks >= 1, block_size >= 1; free_order: NULL (0 .. num_blocks-1) or
 * a permutation of the block ids, the initial queue from the head. */
pa_status pa_pcache_create(int num_blocks, int block_size, const int32_t *free_order,
                           pa_pcache **out);
void pa_pcache_destroy(pa_pcache *pc);

/* The block hash above, for n token ids after `prev`. */
uint64_t pa_pcache_hash_block(uint64_t prev, const int32_t *tokens, int n);

/* Number of leading full blocks of the n-token prompt that are cached
 * (get_computed_blocks); nothing changes. */
pa_status pa_pcache_lookup(const pa_pcache *pc, const int32_t *tokens, int n, uint64_t salt,
                           int *num_blocks_out);

/* New request seq_id with its n-token prompt: the cached run is shared
 * (touch: references, no copy), the rest of the prompt gets new blocks, and
 * the prompt's newly full blocks are hashed.  *num_cached_out = tokens found
 * (a multiple of block_size); slots_out[p] (n entries) = slot of prompt
 * position p (block * block_size + offset); the caller writes K/V for
 * positions >= *num_cached_out.  PA_ERR_OUT_OF_BLOCKS if the queue (after
 * the hits are taken out of it) is too short; PA_ERR_INVALID for a
 * duplicate id. */
pa_status pa_pcache_add(pa_pcache *pc, int64_t seq_id, const int32_t *tokens, int n,
                        uint64_t salt, int *num_cached_out, int64_t *slots_out);

/* One generated token: its slot; a block that fills is hashed.
 * PA_ERR_NOT_FOUND for an unknown id, PA_ERR_OUT_OF_BLOCKS when a block is
 * needed and the queue is empty. */
pa_status pa_pcache_append(pa_pcache *pc, int64_t seq_id, int32_t token, int64_t *slot_out);

/* End of a request: its blocks freed tail first (see above). */
pa_status pa_pcache_free(pa_pcache *pc, int64_t seq_id);

/* Block table of a request into out (cap entries); *n_out gets its length;
 * PA_ERR_INVALID if cap is too small (nothing written). */
pa_status pa_pcache_block_table(const pa_pcache *pc, int64_t seq_id, int32_t *out, int cap,
                                int *n_out);

/* Tokens of a request (prompt and generated). */
pa_status pa_pcache_len(const pa_pcache *pc, int64_t seq_id, int64_t *len_out);

int pa_pcache_num_free(const pa_pcache *pc);

/* Free queue, head first (cap entries); *n_out gets its length;
 * PA_ERR_INVALID if cap is too small. */
pa_status pa_pcache_free_queue(const pa_pcache *pc, int32_t *out, int cap, int *n_out);

/* Reference count of a block (-1 if out of range). */
int pa_pcache_refcount(const pa_pcache *pc, int block);

/* Whether a block is cached and under which hash (0 when not). */
pa_status pa_pcache_block_hash(const pa_pcache *pc, int block, uint64_t *hash_out,
                               int *cached_out);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
