// Tensor-core paged decode over E4M3 pools: the E4M3 variants of the kernel
// in pa_decode_tc.cuh (K and V tiles as 8-bit operands, q and P as E5M2
// terms; one byte a K or V element moved) and their host side.
#include <cuda.h>  // CUtensorMap and its enums only

#include <cstdint>

#include "pa_decode_tc.cuh"

namespace pa {

template <int D, bool SPAN, bool COMPACT>
static TcKernel tc8_variant(bool bf16) {
    return bf16 ? paged_decode_tc_kernel<true, D, SPAN, COMPACT, true>
                : paged_decode_tc_kernel<false, D, SPAN, COMPACT, true>;
}

static TcKernel pick_tc8(bool bf16, int D, int *smem, bool span = false, bool compact = false) {
    *smem = D == 128 ? TcShape<128, true>::SMEM_BYTES : TcShape<64, true>::SMEM_BYTES;
    if (D == 128)
        return span ? (compact ? tc8_variant<128, true, true>(bf16) : tc8_variant<128, true, false>(bf16))
                    : (compact ? tc8_variant<128, false, true>(bf16) : tc8_variant<128, false, false>(bf16));
    return span ? (compact ? tc8_variant<64, true, true>(bf16) : tc8_variant<64, true, false>(bf16))
                : (compact ? tc8_variant<64, false, true>(bf16) : tc8_variant<64, false, false>(bf16));
}

bool fp8_supported(int head_dim, int group) { return tc_supported(head_dim, group); }

int fp8_ctas_per_sm(bool bf16, int head_dim, int /*group*/) {
    int smem = 0;
    TcKernel k = pick_tc8(bf16, head_dim, &smem);
    return tc_occupancy(k, smem, TcShape<64, true>::COLS);
}

pa_status launch_decode_fp8(const DecodeParams &prm, bool bf16, int head_dim, int num_partitions,
                            int num_kv_heads, int num_seqs, cudaStream_t stream) {
    if (num_seqs == 0) return PA_OK;
    int smem = 0;
    TcKernel k = pick_tc8(bf16, head_dim, &smem, prm.span > 1, prm.compact != 0);
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
