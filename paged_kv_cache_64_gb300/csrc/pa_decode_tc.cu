// Tensor-core paged decode: host side of the 16-bit-pool variants (the
// kernel template is in pa_decode_tc.cuh), the TMA descriptors of the pools
// and the launch shared with the E4M3-pool variants.
#include <cuda.h>  // CUtensorMap and its enums only; the encoder comes from the driver at run time

#include <cstdint>
#include <mutex>

#include "pa_decode_tc.cuh"

namespace pa {

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn tensor_map_encoder() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// The pool [NB][Hkv][B][d] viewed as a 2-D tensor of NB*Hkv*B rows of d
// elements; boxes of 16 rows x 64 columns, 128-byte swizzle.
bool pool_tensor_map(CUtensorMap *map, const void *pool, int64_t rows, int D, bool bf16) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kUnit};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
               const_cast<void *>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// An E4M3 pool [NB][Hkv][B][d] (one byte per element) viewed the same way;
// boxes of 16 rows x d bytes, row-major or swizzled as a K-major operand.
bool pool_tensor_map_fp8(CUtensorMap *map, const void *pool, int64_t rows, int D, bool swizzle) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D};
    const cuuint32_t box[2] = {(cuuint32_t)D, (cuuint32_t)kUnit};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(pool), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               !swizzle ? CU_TENSOR_MAP_SWIZZLE_NONE
                        : (D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B),
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool SPAN, bool COMPACT>
static TcKernel tc_variant(bool bf16) {
    return bf16 ? paged_decode_tc_kernel<true, D, SPAN, COMPACT, 0>
                : paged_decode_tc_kernel<false, D, SPAN, COMPACT, 0>;
}

static TcKernel pick_tc(bool bf16, int D, int *smem, bool span = false, bool compact = false) {
    *smem = D == 128 ? TcShape<128, 0>::SMEM_BYTES : TcShape<64, 0>::SMEM_BYTES;
    if (D == 128)
        return span ? (compact ? tc_variant<128, true, true>(bf16) : tc_variant<128, true, false>(bf16))
                    : (compact ? tc_variant<128, false, true>(bf16) : tc_variant<128, false, false>(bf16));
    return span ? (compact ? tc_variant<64, true, true>(bf16) : tc_variant<64, true, false>(bf16))
                : (compact ? tc_variant<64, false, true>(bf16) : tc_variant<64, false, false>(bf16));
}

bool tc_supported(int head_dim, int group) {
    return (head_dim == 64 || head_dim == 128) && group >= 1 && group <= kTcG;
}

// Resident CTAs per SM, from the kernel's own footprint: the runtime's
// occupancy query answers 1 for kernels that allocate TMEM, while the
// hardware co-schedules as many as registers, shared memory and TMEM allow.
// A warp's registers come from one of the 4 sub-partitions (16K registers
// each).
int tc_occupancy(TcKernel k, int smem, int tmem_cols) {
    if (!ensure_smem_attr(reinterpret_cast<const void *>(k), smem)) return 1;
    int dev = 0, smem_sm = 0, reserved = 0;
    cudaFuncAttributes a;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) !=
            cudaSuccess ||
        cudaFuncGetAttributes(&a, k) != cudaSuccess)
        return 1;
    const int by_smem = smem_sm / (smem + reserved);
    const int regs = (a.numRegs + 7) / 8 * 8;
    const int warps_per_subpartition = 16384 / (regs * 32);
    const int by_regs = 4 * warps_per_subpartition / tc_warps<false>();
    const int by_tmem = 512 / tmem_cols;
    int n = by_smem < by_regs ? by_smem : by_regs;
    n = n < by_tmem ? n : by_tmem;
    return n > 0 ? n : 1;
}

int tc_ctas_per_sm(bool bf16, int head_dim) {
    int smem = 0;
    TcKernel k = pick_tc(bf16, head_dim, &smem);
    return tc_occupancy(k, smem, TcShape<64, 0>::COLS);
}

pa_status launch_tc_kernel(TcKernel k, int smem, int ctas_per_sm, const DecodeParams &prm,
                           const CUtensorMap &mk, const CUtensorMap &mv, int num_partitions,
                           int num_kv_heads, int num_seqs, cudaStream_t stream) {
    if (!ensure_smem_attr(reinterpret_cast<const void *>(k), smem)) return PA_ERR_CUDA;
    dim3 grid = decode_grid(prm, num_partitions, num_kv_heads, num_seqs);
    DecodeParams p = prm;
    if (p.compact) {
        // Compact grids whose upper bound (every sequence at the longest
        // length) is within four waves: one CTA a resident slot, each taking
        // every gridDim.x-th item, so that the CTAs a short batch does not
        // need are never launched (each would hold a slot for a memory round
        // trip only to find nothing to do, at the end of the launch).  Larger
        // grids keep one item a CTA, balanced by the hardware scheduler.
        // Grids the hardware schedules over more than four waves take their
        // full chunks first and the sequences' shorter last chunks at the end
        // (compact_find), which evens out the last wave.
        const unsigned slots = (unsigned)(sm_count() * ctas_per_sm);
        if (p.span <= 1 && slots > 0 && grid.x > slots && grid.x <= 4 * slots) grid.x = slots;
        p.one_wave = p.span <= 1 && slots > 0 && grid.x <= slots;
        p.compact = slots > 0 && grid.x > 4 * slots ? 2 : 1;
    }
    const int threads = 32 * (prm.span > 1 ? tc_warps<true>() : tc_warps<false>());
    if (launch_pdl(k, grid, dim3(threads), (size_t)smem, stream, p, mk, mv) != cudaSuccess)
        return PA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status launch_decode_tc(const DecodeParams &prm, bool bf16, int head_dim, int num_partitions,
                           int num_kv_heads, int num_seqs, cudaStream_t stream) {
    if (num_seqs == 0) return PA_OK;
    int smem = 0;
    TcKernel k = pick_tc(bf16, head_dim, &smem, prm.span > 1, prm.compact != 0);
    const int64_t rows = (int64_t)prm.num_blocks * num_kv_heads * prm.block_size;
    CUtensorMap mk, mv;
    if (!pool_tensor_map(&mk, prm.k_pool, rows, head_dim, bf16) ||
        !pool_tensor_map(&mv, prm.v_pool, rows, head_dim, bf16))
        return PA_ERR_CUDA;
    return launch_tc_kernel(k, smem, tc_ctas_per_sm(bf16, head_dim), prm, mk, mv, num_partitions,
                            num_kv_heads, num_seqs, stream);
}

}  // namespace pa
