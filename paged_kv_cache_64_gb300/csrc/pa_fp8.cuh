// E4M3 / E5M2 helpers shared by the decode kernels over E4M3 pools: the
// 8-bit operand layouts the TMA copies write, the conversions of the q and P
// splits, and the fused write of the newest token into E4M3 pools.
#pragma once
#include <cstdint>
#include <cstring>

#include "pa_common.cuh"
#include "pa_decode.cuh"
#include "pa_tcgen05.cuh"

namespace pa {

// Byte offset of element (row, k) in a K-major E4M3 operand of D-byte rows
// stored in swizzled atoms of 8 rows (the layout the TMA copy writes): the
// 16-byte chunk c of row r sits at chunk c ^ (r & 7) for d = 128 (128-byte
// swizzle) and c ^ ((r >> 1) & 3) for d = 64 (64-byte swizzle).
template <int D>
__device__ __forceinline__ uint32_t e4m3_operand_offset(int row, int k) {
    const int sw = D == 128 ? (row & 7) : ((row >> 1) & 3);
    return (uint32_t)((row >> 3) * 8 * D + (row & 7) * D + ((((k >> 4) ^ sw)) << 4) + (k & 15));
}

template <int D>
__device__ __forceinline__ uint64_t e4m3_operand_desc(uint32_t saddr) {
    return D == 128 ? sw128_desc(saddr, 16, 8 * D) : sw64_desc(saddr, 16, 8 * D);
}

// Two fp32 values to two E5M2 codes (the first in the low byte), nearest
// with ties to even, saturating at +-57344 (PTX cvt.rn.satfinite.e5m2x2.f32).
__device__ __forceinline__ uint32_t e5m2x2_from_f32(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// The same from two f16 values (low half first; PTX cvt.rn.satfinite.e5m2x2.f16x2).
__device__ __forceinline__ uint32_t e5m2x2_from_f16x2(uint32_t h) {
    uint16_t r;
    asm("cvt.rn.satfinite.e5m2x2.f16x2 %0, %1;" : "=h"(r) : "r"(h));
    return r;
}

// Two E5M2 codes (low byte first) to two f16 values, exactly (PTX
// cvt.rn.f16x2.e5m2x2: every E5M2 value is an f16 value).
__device__ __forceinline__ uint32_t f16x2_from_e5m2x2(uint16_t c) {
    uint32_t r;
    asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(r) : "h"(c));
    return r;
}

// a - b on packed f16 pairs.
__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// 2^e for e in [-126, 127], exactly.
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// Two E5M2 codes (low byte first) back to fp32, exactly.
__device__ __forceinline__ float2 e5m2x2_to_f32(uint32_t codes) {
    const uint32_t h = f16x2_from_e5m2x2((uint16_t)codes);
    __half2 hh;
    memcpy(&hh, &h, 4);
    return __half22float2(hh);
}

// Fused cache write of the newest token into the E4M3 pools: quantise its K
// and V (x * inv_scale in fp32, nearest code) and store them at its slot,
// which must be the slot the block table gives for position L-1.  Threads
// [0, 2 * d/16) take 16 elements each.
template <bool BF16, int D>
__device__ __forceinline__ void fused_cache_write_fp8(const DecodeParams &p, int seq, int kvh,
                                                      int L) {
    constexpr int chunks = D / 16;
    const int t = threadIdx.x;
    if (t >= 2 * chunks) return;
    const int pos = L - 1;
    const int phys = seq_table(p, seq)[pos >> p.log2_block];
    const int off = pos & (p.block_size - 1);
    const int64_t slot = p.slot_mapping[seq];
    if ((unsigned)phys >= (unsigned)p.num_blocks || slot != (int64_t)phys * p.block_size + off) {
        if (t == 0) record_error(p.err, PA_ERR_BAD_INDEX);
        return;
    }
    const bool is_v = t >= chunks;
    const int c = t % chunks;
    const uint4 *src = reinterpret_cast<const uint4 *>(
                           (is_v ? p.v_new : p.k_new) + ((int64_t)seq * p.num_kv_heads + kvh) * D) +
                       2 * c;
    const uint4 q = quantize16_e4m3<BF16>(src[0], src[1], is_v ? p.v_inv : p.k_inv);
    const uint8_t *pool = reinterpret_cast<const uint8_t *>(is_v ? p.v_pool : p.k_pool);
    uint4 *dst = reinterpret_cast<uint4 *>(const_cast<uint8_t *>(pool) +
                                           (((int64_t)phys * p.num_kv_heads + kvh) * p.block_size +
                                            off) * D) +
                 c;
    *dst = q;
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

}  // namespace pa
