// Parameters and helpers shared by the two decode kernels (CUDA-core and
// tensor-core) and the split-KV reduce.
#pragma once

#include <stdint.h>

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
    int num_blocks;
    int max_blocks_per_seq;
    int max_seq_len;
    int num_q_heads;
    int num_kv_heads;
    int group;                   // G
    int block_size;
    int log2_block;
    int partition_tokens;        // P, multiple of kUnit
    int num_partitions;          // NP (grid.x)
    float scale_log2;            // scale * log2(e)
    int mode;                    // 0: decode (direct output when 1 partition), 1: partials only
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

// Tensor-core decode (pa_decode_tc.cu).
bool tc_supported(int head_dim, int group);
int tc_ctas_per_sm(bool bf16, int head_dim);
pa_status launch_decode_tc(const DecodeParams &prm, bool bf16, int head_dim, int num_partitions,
                           int num_kv_heads, int num_seqs, cudaStream_t stream);

}  // namespace pa
