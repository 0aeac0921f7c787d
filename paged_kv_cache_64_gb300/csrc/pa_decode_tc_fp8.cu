// Tensor-core paged decode over E4M3 pools: the E4M3 variants of the kernel
// in pa_decode_tc.cuh (K and V tiles as 8-bit operands, q and P as E5M2
// terms; one byte a K or V element moved) with operands of 8 heads, and the
// host side of all E4M3 variants (those of 4 heads are in
// pa_decode_tc_fp8_g4.cu).
#include <cuda.h>  // CUtensorMap and its enums only

#include <cstdint>

#include "pa_decode_tc.cuh"

namespace pa {

TcKernel tc8_pick8(bool bf16, int D, bool span, bool compact, int *smem, int *cols) {
    return tc8_pick<8>(bf16, D, span, compact, smem, cols);
}

// The variant for head size D and a group of `group` query heads: E4M3
// operands of 4 heads (up to 4) or 8.
static TcKernel pick_tc8(bool bf16, int D, int group, int *smem, int *cols, bool span = false,
                         bool compact = false) {
    return group <= 4 ? tc8_pick4(bf16, D, span, compact, smem, cols)
                      : tc8_pick8(bf16, D, span, compact, smem, cols);
}

bool fp8_supported(int head_dim, int group) { return tc_supported(head_dim, group); }

int fp8_ctas_per_sm(bool bf16, int head_dim, int group) {
    int smem = 0, cols = 0;
    TcKernel k = pick_tc8(bf16, head_dim, group, &smem, &cols);
    return tc_occupancy(k, smem, cols);
}

pa_status launch_decode_fp8(const DecodeParams &prm, bool bf16, int head_dim, int num_partitions,
                            int num_kv_heads, int num_seqs, cudaStream_t stream) {
    if (num_seqs == 0) return PA_OK;
    int smem = 0, cols = 0;
    TcKernel k = pick_tc8(bf16, head_dim, prm.group, &smem, &cols, prm.span > 1, prm.compact != 0);
    const int64_t rows = (int64_t)prm.num_blocks * num_kv_heads * prm.block_size;
    // both pools land swizzled: K as the K-major A operand of q.K^T, V as the
    // MN-major A operand (V^T) of P.V
    CUtensorMap mk, mv;
    if (!pool_tensor_map_fp8(&mk, prm.k_pool, rows, head_dim, true) ||
        !pool_tensor_map_fp8(&mv, prm.v_pool, rows, head_dim, true))
        return PA_ERR_CUDA;
    return launch_tc_kernel(k, smem, fp8_ctas_per_sm(bf16, head_dim, prm.group), prm, mk, mv,
                            num_partitions, num_kv_heads, num_seqs, stream);
}

}  // namespace pa
