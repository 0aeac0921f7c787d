// Paged decode over an FP8 KV cache for GB300 (sm_103a).
//
// The pools hold OCP E4M3 codes (one byte per element), one scale per K or V
// pool: element = scale * code value ("b = 1 for FP8" in the KV-size formula
// of "PagedAttention and Virtual Memory Management: Mathematical Foundations
// ..." (llms.blog), section 1; the format and the scale are this library's
// conventions).
// Same computation as the tensor-core kernel in pa_decode_tc.cu (whose header
// describes the products, the roles and the online softmax), with half the
// K/V bytes moved.  Per tile of 128 positions:
//
//   S^T[128 pos x N] = K_codes[128 x d] . Qs^T[d x N]       kind::f8f6f4, E4M3 x E5M2
//   d = 128: O^T[128 x N] = V_codes^T[128 x 128 pos] . Ps^T  kind::f8f6f4, E4M3 x E5M2
//   d = 64:  O^T[128 x 16] = V16^T[128 x 128 pos] . P16^T    kind::f16 (rows 64.. zero)
//
// with N = 16 for groups of up to 4 query heads, 32 for up to 8 (four E5M2
// terms a head).
// q.K^T reads the E4M3 K tile exactly as the TMA copy lands it (K-major,
// swizzled), so K is never converted.  Its other operand, Qs, holds each query
// head as four E5M2 terms: with 2^e_g the power of two that brings head g's
// largest |q| into [2^14, 2^15), q_g * 2^e_g = t1 + t2 + t3 + t4, t1 the
// nearest E5M2 value, t2 that of the remainder, and so on (each remainder is
// exact in fp32).  A 16-bit q has at most 11 significant bits and the four
// terms carry 12, so the sum equals q * 2^e_g except for the part of an
// element below E5M2's subnormal quantum 2^-16 (under 2^-31 of the head's
// largest), and the four S columns of a head add up, times 2^-e_g, to q.K^T
// within fp32 rounding.  E5M2 rather than E4M3 terms: the same bits per term
// but a floor 2^14 times lower, so a q row whose elements span more than
// 2^17 keeps its small elements (three E4M3 terms lose everything under
// 2^-17 of the largest, which moves scores measurably when those elements
// meet large keys).
// At d = 128 P.V reads V the same way: the staged V tile (128-byte swizzle)
// is V^T as an MN-major operand, and P is split like q (Ps: four E5M2 terms
// per head of P times 2^k, the power of two that brings the tile's largest P
// into [2^14, 2^15), rounded to f16 first; the tile's O is scaled back by
// 2^-k), so nothing is converted and the tensor cores run 8 instructions a
// tile.  Stale V rows of the last tile are zeroed in the staged tile before
// P.V (0 * NaN would poison the product).  At d = 64 a V row is 64 bytes,
// half an MN-major atom, so converter warps widen V exactly to f16
// (cvt.rn.f16x2.e4m3x2: every E4M3 value is an f16 value) into a zero-padded
// V^T operand instead.  The K scale is folded into the softmax scale, the V
// scale into the output.
// Separate K and V staging rings (5 and 7 tiles at d = 128: a K slot frees
// when its q.K^T has run, a V slot only after P.V; 6 and 10 at d = 64) are
// the large buffers, each filled in tile order by its own producer at
// d = 128.  Two softmax warpgroups take alternate tiles (even tiles with S
// buffer 0, odd ones with S buffer 1; P and O double-buffered per group),
// each with its own running maximum, sum and accumulator; the groups merge
// their states at the end of each split-KV partition the CTA computes.
// Roles: 0 producer (K at d = 128), 1 TMEM owner and MMA issuer (of group
// A's tiles at d = 128), 2..5 and 6..9 softmax / epilogue groups A and B (A
// also builds Qs); at d = 128 also 10 the V producer and 11 the MMA issuer of
// group B's tiles, at d = 64 10..15 V converters.
#include <cuda.h>  // CUtensorMap and its enums only; the encoder comes from the driver at run time

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "pa_common.cuh"
#include "pa_decode.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int kF8Tile = 128;       // positions per tile (MMA M of q.K^T)
constexpr int kF8N = 16;           // MMA N of P.V in f16: the query heads of a group, zero-padded
constexpr int kF8G = 8;            // largest group the kernel serves
constexpr int kF8Conv0 = 10;       // first converter warp (f16 P.V only)
constexpr int kF8VProd = 10;       // the V producer warp (E4M3 P.V only)
constexpr int kF8Issuer1 = 11;     // the odd tiles' MMA issuer (E4M3 P.V only)
constexpr int kF8ConvWarps = 6;    // converter warps (V)

constexpr int kF8MaxRing = 12;     // slots of a staging ring

enum F8Bar {
    // the f16 V operand buffers of d = 64
    kVOpFull0 = 0, kVOpFull1, kVOpEmpty0, kVOpEmpty1, kQReady,
    kSFull0, kSFull1, kSEmpty0, kSEmpty1,
    kPFull0, kOFull0 = kPFull0 + 4, kOEmpty0 = kOFull0 + 4,  // 4 of each: tile t uses 2*(t&1) + ((t>>1)&1)
    // the K and V staging rings, kF8MaxRing of each
    kKFull0 = kOEmpty0 + 4,
    kKEmpty0 = kKFull0 + kF8MaxRing,
    kVFull0 = kKEmpty0 + kF8MaxRing,
    kVEmpty0 = kVFull0 + kF8MaxRing,
    kNumF8Bars = kVEmpty0 + kF8MaxRing
};

template <int D, int GM>
struct F8Shape {
    // d = 128: P.V on E4M3 codes too (V^T straight from the staged tile, P as
    // four E5M2 terms); d = 64: V widened to f16 by converter warps
    static constexpr bool DIRECT = D == 128;
    // GM (4 or 8): the heads a KV head's group may have.  The E5M2 operands
    // hold four terms per head in rows t * GM + g: QN rows (the MMA N).
    // TMEM: S of each softmax group at 0 and QN, O of tile t at
    // 2 * QN + QN * (2 * (t & 1) + ((t >> 1) & 1)) (two per group).
    static constexpr int NTERM = 4;  // E5M2 terms of a q or P value
    static constexpr int QN = NTERM * GM;
    static_assert(QN == 16 || QN == 32, "MMA N");
    static constexpr int S0 = 0, O0 = 2 * QN;
    static constexpr int COLS = 6 * QN <= 128 ? 128 : 256;
    // d = 128: producer K, even tiles' issuer, 8 softmax, producer V, odd
    // tiles' issuer;
    // d = 64: producer, MMA issuer, 8 softmax, 6 converters (4 per
    // sub-partition, 128 registers)
    static constexpr int WARPS = DIRECT ? 12 : 16;
    static constexpr int THREADS = WARPS * 32;
    static constexpr int SLAB = kF8Tile * 128;        // one 64-dim f16 slab of a tile: 16 KiB
    static constexpr int V_BYTES = 2 * SLAB;          // V^T is M = 128 dims; d = 64 pads with zeros
    static constexpr int STG_BYTES = kF8Tile * D;     // E4M3 tile of K (or V): 128 rows of d bytes
    // K tiles and Qs: K-major 8-bit operands of d-byte rows, in atoms of 8 rows
    // (128-byte swizzle for d = 128, 64-byte for d = 64)
    static constexpr int Q_BYTES = QN * D;
    // P^T: 16 rows of 128 f16 positions, or up to 32 rows of 128 E5M2 positions
    static constexpr int P_BYTES = 4096;
    // Staging rings of E4M3 tiles: a K slot is free once q.K^T has read it,
    // a V slot only once P.V (d = 128) or the converters (d = 64) have, so
    // the V ring is the deeper one.
    static constexpr int NK = DIRECT ? 5 : 6;
    static constexpr int NV = DIRECT ? 7 : 10;
    static constexpr int NVB = DIRECT ? 0 : 2;        // f16 V operand buffers
    static constexpr int OFF_STG = 0;                 // K slots, then V slots
    static constexpr int OFF_VSTG = OFF_STG + NK * STG_BYTES;
    static constexpr int OFF_V = OFF_VSTG + NV * STG_BYTES;
    static constexpr int OFF_Q = OFF_V + NVB * V_BYTES;
    static constexpr int OFF_P = OFF_Q + Q_BYTES;     // four buffers: two per softmax group
    static constexpr int OFF_RED = OFF_P + 4 * P_BYTES;
    // per softmax group: two tile-max buffers and the final sums
    static constexpr int RED_BYTES = 2 * 3 * 4 * kF8N * 4;
    // per head: softmax scale (log2 units, K scale included) times 2^-e_g
    static constexpr int OFF_QMUL = OFF_RED + RED_BYTES;
    // group B's state for a partition's merge: acc [G][D], then m_run,
    // m_true, l, failed; two buffers (partition parity)
    static constexpr int OFF_XCH = OFF_QMUL + kF8G * 4;
    static constexpr int XCH_BYTES = kF8G * D * 4 + 4 * kF8G * 4;
    static constexpr int OFF_BAR = OFF_XCH + 2 * XCH_BYTES;
    static constexpr int OFF_MISC = OFF_BAR + kNumF8Bars * 8;
    // MISC: TMEM address, abort flag, then the issuers' progress (d = 128)
    static constexpr int SMEM_BYTES = OFF_MISC + 32 + 1024;  // + slack to align the base to 1 KiB
    static_assert(OFF_V % 1024 == 0 && OFF_Q % 1024 == 0 && OFF_P % 1024 == 0, "atom alignment");
    static_assert(STG_BYTES % 1024 == 0, "TMA swizzle alignment");
    static_assert(NK <= kF8MaxRing && NV <= kF8MaxRing, "ring barriers");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert((NK + NV) * STG_BYTES >= 2 * kF8G * kCombineMaxParts * 4,
                  "combine scratch in the staging rings");
};

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

// Named barrier `id` over `n` threads (ids 1..3 are the softmax groups' own
// and their joint one; 0 is __syncthreads).
__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

template <bool BF16>
__device__ __forceinline__ uint16_t narrow_f16(float x) {
    __half h = __float2half_rn(x);
    uint16_t u;
    memcpy(&u, &h, 2);
    return u;
}

template <bool BF16>
__device__ __forceinline__ uint16_t narrow_out(float x) {
    if constexpr (BF16) {
        __nv_bfloat16 h = __float2bfloat16_rn(x);
        uint16_t u;
        memcpy(&u, &h, 2);
        return u;
    } else {
        return narrow_f16<false>(x);
    }
}

template <bool BF16, int D, int GM>
__global__ void __launch_bounds__(F8Shape<D, GM>::THREADS, 1)
    paged_decode_fp8_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmap_k,
                            const __grid_constant__ CUtensorMap tmap_v) {
    using S = F8Shape<D, GM>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + S::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::OFF_MISC + 8);
    // d = 128: per softmax group, q.K^T and P.V MMAs issued so far
    volatile int *progress = reinterpret_cast<volatile int *>(smem + S::OFF_MISC + 16);
    float *red = reinterpret_cast<float *>(smem + S::OFF_RED);
    float *qmul = reinterpret_cast<float *>(smem + S::OFF_QMUL);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.group;
    const int P = p.partition_tokens;
    if (threadIdx.x == 0) {  // descriptors are kernel parameters: fetch them early
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    pdl_wait();  // inputs may come from the previous kernel on the stream
    int part, kvh, seq;  // split-KV chunk (span of partitions), KV head, sequence
    if (p.compact) {
        if (!compact_item(p, blockIdx.x, &seq, &part, &kvh)) return;  // past the last item
    } else {
        part = blockIdx.x;
        kvh = blockIdx.y;
        seq = blockIdx.z;
    }
    const int L = item_len(p, seq, threadIdx.x == 0 && part == 0 && kvh == 0);
    const int nparts_seq = L == 0 ? 0 : (L - 1) / P + 1;
    // partitions [part0, part0 + R) of the sequence: this CTA's span
    const int R = p.span > 1 ? p.span : 1;
    const int part0 = part * R;
    const int start = part0 * P;
    if (start >= L) {  // empty partitions: as in the other decode kernels
        if (p.mode == 0) {
            if (part == 0) {
                uint32_t *o = reinterpret_cast<uint32_t *>(p.out);
                const int64_t base = ((int64_t)seq * p.num_q_heads + (int64_t)kvh * G) * D / 2;
                for (int i = threadIdx.x; i < G * D / 2; i += blockDim.x) o[base + i] = 0u;
            }
        } else {
            for (int j = 0; j < R && part0 + j < p.num_partitions; ++j)
                for (int g = 0; g < G; ++g) {
                    const int64_t row = part_row(p, seq, kvh * G + g, part0 + j);
                    if (threadIdx.x == 0) {
                        p.part_m[row] = -INFINITY;
                        p.part_l[row] = 0.f;
                    }
                    for (int x = threadIdx.x; x < D; x += blockDim.x) p.part_o[row * D + x] = 0.f;
                }
        }
        return;
    }
    const int part_end = (part0 + R < nparts_seq) ? part0 + R : nparts_seq;  // past the last
    const int end = (part_end * P < L) ? part_end * P : L;
    const int nunits = (end - start + kUnit - 1) / kUnit;
    const int ntiles = (end - start + kF8Tile - 1) / kF8Tile;
    const bool direct = (p.mode == 0) && (nparts_seq <= 1);
    // tiles per partition (an even number when the span has several; the
    // host guarantees it), else all of them
    const int tpp = R > 1 ? P / kF8Tile : ntiles;

    if (p.k_new != nullptr && part_end == nparts_seq) fused_cache_write_fp8<BF16, D>(p, seq, kvh, L);
    if (threadIdx.x == 0) {
        // kVOpFull: the converter warps; kQReady, kSEmpty, kPFull, kOEmpty:
        // the 4 warps of a softmax group; kKFull, kVFull: the producer's
        // expect-tx arrival; kKEmpty: the commit of q.K^T; kVEmpty: the commit
        // of P.V (d = 128) or the converter warps (d = 64)
        const int counts[kKFull0] = {kF8ConvWarps, kF8ConvWarps, 1, 1, 4, 1, 1, 4, 4,
                                     4, 4, 4, 4, 1, 1, 1, 1, 4, 4, 4, 4};
        for (int b = 0; b < kKFull0; ++b) mbar_init(&bar[b], counts[b]);
        for (int b = 0; b < kF8MaxRing; ++b) {
            mbar_init(&bar[kKFull0 + b], 1);
            mbar_init(&bar[kKEmpty0 + b], 1);
            mbar_init(&bar[kVFull0 + b], 1);
            mbar_init(&bar[kVEmpty0 + b], S::DIRECT ? 1 : kF8ConvWarps);
        }
        *abort_flag = 0;
        for (int i = 0; i < 4; ++i) progress[i] = 0;
        mbar_init_fence();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, S::COLS);
        tmem_relinquish();
    }
    if constexpr (!S::DIRECT) {
        // rows 64..127 of both V^T operand buffers: zero once, never written again
        for (int vb = 0; vb < S::NVB; ++vb) {
            uint4 *z = reinterpret_cast<uint4 *>(smem + S::OFF_V + vb * S::V_BYTES + S::SLAB);
            for (int i = threadIdx.x; i < S::SLAB / 16; i += S::THREADS) z[i] = make_uint4(0, 0, 0, 0);
        }
        fence_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 || (S::DIRECT && warp == kF8VProd)) {
        // ---------------------------------------------------------- producers
        // d = 128: warp 0 copies the K tiles and warp kF8VProd the V tiles,
        // each in tile order as its ring's slots free up (K runs ahead: its
        // slots free up first); d = 64: warp 0 copies K then V of each tile.
        // Lane j of the window holds the pool row of unit w + j, 32 units (4
        // tiles) a window; the block-table entries of the next window are
        // loaded when a window opens, so no copy waits for a table load.
        const int kv0 = (S::DIRECT && warp != 0) ? 1 : 0;
        const int kv1 = S::DIRECT ? kv0 : 1;
        const int32_t *table = seq_table(p, seq);
        auto table_entry = [&](int u) -> int {
            return u < nunits ? __ldg(table + ((start + u * kUnit) >> p.log2_block)) : 0;
        };
        auto unit_row = [&](int u, int phys) -> int {  // first row of unit u in [NB*Hkv*B, d]
            if (u >= nunits) return 0;
            if ((unsigned)phys >= (unsigned)p.num_blocks) {
                if (kv0 == 0) record_error(p.err, PA_ERR_BAD_INDEX);
                phys = 0;
            }
            const int pos = start + u * kUnit;
            return (phys * p.num_kv_heads + kvh) * p.block_size + (pos & (p.block_size - 1));
        };
        int w = -32, rows = 0, next = table_entry(lane);
        bool ok = true;
        for (int t = 0; t < ntiles && ok; ++t) {
            if (8 * t >= w + 32) {  // windows open in order: w + 32 == 8 * t
                w = 8 * t;
                rows = unit_row(w + lane, next);
                next = table_entry(w + 32 + lane);
            }
            const int nu = (nunits - 8 * t < 8) ? nunits - 8 * t : 8;
            const int r0 = __shfl_sync(kFullMask, rows, (8 * t - w + lane) & 31);
            for (int kv = kv0; kv <= kv1; ++kv) {
                const int n = kv ? S::NV : S::NK;
                const int slot = t % n;
                if (t >= n) {  // the slot's readers are done with its previous tile
                    const bool done =
                        mbar_wait(&bar[(kv ? kVEmpty0 : kKEmpty0) + slot], ((t / n) - 1) & 1);
                    if (!__all_sync(kFullMask, done)) {
                        ok = false;
                        break;
                    }
                }
                uint64_t *full = &bar[(kv ? kVFull0 : kKFull0) + slot];
                uint8_t *dst = smem + (kv ? S::OFF_VSTG : S::OFF_STG) + slot * S::STG_BYTES;
                if (lane == 0) mbar_arrive_expect_tx(full, nu * kUnit * D);
                // lane j < nu copies unit j of the tile: one instruction
                // issues the tile's copies
                if (lane < nu) tma_load_2d(dst + lane * kUnit * D, kv ? &tmap_v : &tmap_k, 0, r0, full);
                __syncwarp();
            }
        }
        if (!ok && lane == 0) {
            record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
        }
    } else if (!S::DIRECT && warp >= kF8Conv0) {
      if constexpr (!S::DIRECT) {
        // ---------------------------------------------------------- V converters
        // E4M3 staging (row-major) -> f16 V^T operand (MN-major, 128-byte
        // swizzle).  Item = (row, 16 codes); every load of a thread is issued
        // before the first conversion.  Rows past the end of the range get
        // zeros (0 * NaN would poison P.V).
        constexpr int NCT = kF8ConvWarps * 32;
        constexpr int NITEMS = kF8Tile * (D / 16);
        constexpr int NIT = (NITEMS + NCT - 1) / NCT;
        const int ct = threadIdx.x - kF8Conv0 * 32;
        bool ok = true;
        for (int t = 0; t < ntiles && ok; ++t) {
            const int nvalid = (end - start - t * kF8Tile < kF8Tile) ? end - start - t * kF8Tile
                                                                      : kF8Tile;
            const int slot = t % S::NV;
            const int stg = S::OFF_VSTG + slot * S::STG_BYTES;
            const int ob = t % S::NVB;
            const int op_off = S::OFF_V + ob * S::V_BYTES;
            ok = __all_sync(kFullMask, mbar_wait(&bar[kVFull0 + slot], (t / S::NV) & 1)) &&
                 (t < S::NVB ||
                  __all_sync(kFullMask, mbar_wait(&bar[kVOpEmpty0 + ob], ((t / S::NVB) - 1) & 1)));
            if (!ok) break;
            uint4 raw[NIT];
#pragma unroll
            for (int i = 0; i < NIT; ++i) {
                const int it = ct + NCT * i;
                const int row = it / (D / 16), c = it % (D / 16);
                raw[i] = (it >= NITEMS || row >= nvalid)
                             ? make_uint4(0, 0, 0, 0)  // code 0 is +0
                             : *reinterpret_cast<const uint4 *>(smem + stg + row * D + c * 16);
            }
#pragma unroll
            for (int i = 0; i < NIT; ++i) {
                const int it = ct + NCT * i;
                if (it >= NITEMS) break;
                const int row = it / (D / 16), c = it % (D / 16);
                const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
                uint32_t h[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    h[2 * j] = f16x2_from_e4m3x2((uint16_t)(w[j] & 0xffffu));
                    h[2 * j + 1] = f16x2_from_e4m3x2((uint16_t)(w[j] >> 16));
                }
                *reinterpret_cast<uint4 *>(smem + op_off + sw128_offset(row, c * 16, S::SLAB)) =
                    make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4 *>(smem + op_off + sw128_offset(row, c * 16 + 8, S::SLAB)) =
                    make_uint4(h[4], h[5], h[6], h[7]);
            }
            fence_async_smem();  // generic-proxy writes, read by the tensor cores
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bar[kVOpFull0 + ob]);
                mbar_arrive(&bar[kVEmpty0 + slot]);
            }
        }
        if (!ok && lane == 0) {
            record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
        }
      }
    } else if (warp == 1 || (S::DIRECT && warp == kF8Issuer1)) {
        // ---------------------------------------------------------- MMA issue
        // (d = 128: warp 1 for the even tiles and warp kF8Issuer1 for the odd
        // ones; d = 64: every MMA from warp 1)
        if (lane == 0) {
            constexpr uint32_t idesc_qk = e4m3_e5m2_idesc(kF8Tile, S::QN, false);
            constexpr uint32_t idesc_pv = f16_idesc(false, true, false, 128, kF8N);
            constexpr uint32_t idesc_pv8 = e4m3_e5m2_idesc(128, S::QN, true);  // V^T MN-major
            const uint32_t sbase = smem_addr(smem);
            // q.K^T of tile t (its K landed, its S buffer read by the softmax)
            auto issue_qk = [&](int t) -> bool {
                const int b = t & 1, slot = t % S::NK;
                if (!mbar_wait(&bar[kKFull0 + slot], (t / S::NK) & 1)) return false;
                if (t >= 2 && !mbar_wait(&bar[kSEmpty0 + b], ((t >> 1) - 1) & 1)) return false;
                tc_fence_after();
                const uint32_t kaddr = sbase + S::OFF_STG + slot * S::STG_BYTES;
#pragma unroll
                for (int ks = 0; ks < D / 32; ++ks)  // 32 codes (bytes) of d per MMA
                    tc_mma_f8(tmem + S::S0 + S::QN * b, e4m3_operand_desc<D>(kaddr + ks * 32),
                              e4m3_operand_desc<D>(sbase + S::OFF_Q + ks * 32), idesc_qk, ks > 0);
                tc_commit(&bar[kSFull0 + b]);
                tc_commit(&bar[kKEmpty0 + slot]);
                return true;
            };
            // P.V of tile t (its V landed or converted, its P written, its O
            // buffer accumulated from tile t-4)
            auto issue_pv = [&](int t) -> bool {
                const int b = 2 * (t & 1) + ((t >> 1) & 1);  // P and O buffer
                if (!mbar_wait(&bar[S::DIRECT ? kVFull0 + t % S::NV : kVOpFull0 + (t & 1)],
                               S::DIRECT ? (t / S::NV) & 1 : (t >> 1) & 1))
                    return false;
                if (!mbar_wait(&bar[kPFull0 + b], (t >> 2) & 1)) return false;
                if (t >= 4 && !mbar_wait(&bar[kOEmpty0 + b], ((t >> 2) - 1) & 1)) return false;
                tc_fence_after();
                if constexpr (S::DIRECT) {
                    // V^T straight from the staged tile: MN-major, 8-position
                    // atoms 1024 bytes apart, 32 positions per MMA
                    const int slot = t % S::NV;
                    const uint32_t vaddr = sbase + S::OFF_VSTG + slot * S::STG_BYTES;
#pragma unroll
                    for (int ks = 0; ks < kF8Tile / 32; ++ks)
                        tc_mma_f8(tmem + S::O0 + S::QN * b, sw128_desc(vaddr + ks * 4096, 16, 1024),
                                  sw128_desc(sbase + S::OFF_P + b * S::P_BYTES + ks * 32, 16, 1024),
                                  idesc_pv8, ks > 0);
                    tc_commit(&bar[kOFull0 + b]);
                    tc_commit(&bar[kVEmpty0 + slot]);
                } else {
#pragma unroll
                    for (int ks = 0; ks < kF8Tile / 16; ++ks) {
                        const uint32_t voff = ks * 2048;  // 16 positions = two 8-row groups
                        const uint32_t poff = b * S::P_BYTES + (ks >> 2) * (kF8N * 128) + (ks & 3) * 32;
                        tc_mma(tmem + S::O0 + S::QN * b,
                               sw128_desc(sbase + S::OFF_V + (t & 1) * S::V_BYTES + voff, S::SLAB, 1024),
                               sw128_desc(sbase + S::OFF_P + poff, 16, 1024), idesc_pv, ks > 0);
                    }
                    tc_commit(&bar[kOFull0 + b]);
                    tc_commit(&bar[kVOpEmpty0 + (t & 1)]);
                }
                return true;
            };
            // Fixed order q.K^T 0, 1, then q.K^T t+2 and P.V t: q.K^T of tile
            // t+2 only needs the softmax to have read S of tile t (the first
            // thing it does with tile t), so a softmax group finds its next S
            // ready when it has written P of this tile.
            bool ok = true;
            if constexpr (S::DIRECT) {
                // One issuer per softmax group (warp 1: even tiles, warp
                // kF8Issuer1: odd ones), each in its tiles' order: q.K^T of
                // the group's first tile, then q.K^T of tile t+2 and P.V of
                // tile t.  The groups only share the staging rings, whose
                // slots alternate between them: before q.K^T of tile t the
                // other group must have issued q.K^T of every tile up to
                // t - NK and P.V of every tile up to t - NV, so those tiles
                // have landed and the parity tests on the slots of t can
                // only mean t's copies.
                const int g = warp == 1 ? 0 : 1, o = 1 - g;
                auto other_covers = [&](int t) -> bool {
                    const unsigned long long t0 = global_timer_ns();
                    for (;;) {
                        // the other group's next tile to issue, q.K^T and P.V
                        const int nq = o + 2 * progress[2 * o], nv = o + 2 * progress[2 * o + 1];
                        if (nq > t - S::NK && nv > t - S::NV) return true;
                        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
                    }
                };
                auto qk = [&](int t) -> bool {
                    if (!other_covers(t) || !issue_qk(t)) return false;
                    progress[2 * g] = progress[2 * g] + 1;
                    return true;
                };
                ok = mbar_wait(&bar[kQReady], 0) && (g >= ntiles || qk(g));
                for (int t = g; ok && t < ntiles; t += 2) {
                    ok = (t + 2 >= ntiles || qk(t + 2)) && issue_pv(t);
                    if (ok) progress[2 * g + 1] = progress[2 * g + 1] + 1;
                }
            } else {
                ok = mbar_wait(&bar[kQReady], 0) && issue_qk(0) && (ntiles < 2 || issue_qk(1));
                for (int t = 0; ok && t < ntiles; ++t)
                    ok = (t + 2 >= ntiles || issue_qk(t + 2)) && issue_pv(t);
            }
            if (!ok) {
                record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
            }
        }
    } else {
        // ---------------------------------------------------------- softmax / epilogue
        const int grp = (warp - 2) >> 2;         // 0: even tiles, 1: odd tiles
        const int sw = (warp - 2) & 3;           // warp within the group
        const int quad = warp & 3;               // TMEM lane quadrant this warp may access
        const int r = quad * 32 + lane;          // TMEM lane: position (S) or dimension (O)
        const int st = sw * 32 + lane;           // 0..127 within the group
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        float *gred = red + grp * (3 * 4 * kF8N);  // this group's exchange area
        float *xch = reinterpret_cast<float *>(smem + S::OFF_XCH);

        if (grp == 0) {
            // Qs: head g's q times 2^e_g as four E5M2 terms in rows t * GM + g
            // (t = 0..3) of a QN-row K-major operand (the rows of absent heads
            // zero).  Thread (g, j) takes EPT elements.
            constexpr int TPH = 128 / GM, EPT = D / TPH;  // threads per head, elements each
            const int g = st / TPH, j = st % TPH;
            float x[EPT];
#pragma unroll
            for (int e = 0; e < EPT; ++e) x[e] = 0.f;
            if (g < G) {
                const uint16_t *src =
                    p.q + ((int64_t)seq * p.num_q_heads + (int64_t)kvh * G + g) * D + j * EPT;
                uint32_t w[EPT / 2];
                if constexpr (EPT == 8) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(src);
                    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
                } else if constexpr (EPT == 4) {
                    const uint2 v = *reinterpret_cast<const uint2 *>(src);
                    w[0] = v.x; w[1] = v.y;
                } else {
                    w[0] = *reinterpret_cast<const uint32_t *>(src);
                }
#pragma unroll
                for (int e = 0; e < EPT / 2; ++e) {
                    const float2 f = widen2<BF16>(w[e]);
                    x[2 * e] = f.x;
                    x[2 * e + 1] = f.y;
                }
            }
            float amax = 0.f;
#pragma unroll
            for (int e = 0; e < EPT; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
            for (int off = TPH / 2; off >= 1; off >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, off));
            // 2^e_g brings amax into [2^14, 2^15): e_g = 14 - floor(log2 amax)
            int eg = 0;
            if (amax > 0.f) {
                const int ex = (int)((__float_as_uint(amax) >> 23) & 0xffu) - 127;
                eg = 14 - (ex < -126 ? -126 : ex);
                eg = eg < -120 ? -120 : (eg > 120 ? 120 : eg);
            }
            const float up = exp2i(eg);
            uint32_t code[S::NTERM][(EPT + 3) / 4];  // EPT codes per term, 4 per word
#pragma unroll
            for (int t = 0; t < S::NTERM; ++t)
#pragma unroll
                for (int w4 = 0; w4 < (EPT + 3) / 4; ++w4) code[t][w4] = 0u;
#pragma unroll
            for (int e2 = 0; e2 < EPT / 2; ++e2) {  // element pairs
                float a = x[2 * e2] * up, b = x[2 * e2 + 1] * up;
#pragma unroll
                for (int t = 0; t < S::NTERM; ++t) {
                    const uint32_t c = e5m2x2_from_f32(a, b);
                    const float2 back = e5m2x2_to_f32(c);
                    a -= back.x;  // exact: the remainder is representable
                    b -= back.y;
                    code[t][e2 >> 1] |= c << (16 * (e2 & 1));
                }
            }
#pragma unroll
            for (int t = 0; t < S::NTERM; ++t) {
                const int row = GM * t + g;
                uint8_t *dst = smem + S::OFF_Q + e4m3_operand_offset<D>(row, j * EPT);
                if constexpr (EPT == 8) {
                    *reinterpret_cast<uint2 *>(dst) = make_uint2(code[t][0], code[t][1]);
                } else if constexpr (EPT == 4) {
                    *reinterpret_cast<uint32_t *>(dst) = code[t][0];
                } else {
                    *reinterpret_cast<uint16_t *>(dst) = (uint16_t)code[t][0];
                }
            }
            if (j == 0) qmul[g] = g < G ? p.scale_log2 * exp2i(-eg) : 0.f;
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[kQReady]);
        }
        named_bar(3, 256);  // qmul is written
        float qm[GM];
#pragma unroll
        for (int g = 0; g < GM; ++g) qm[g] = qmul[g];

        float m_run[GM], m_true[GM], l_part[GM], acc[GM], alpha_prev[GM];
        // 2^-k of the previous tile's P scale (E4M3 P only)
        float kinv_prev[GM];
#pragma unroll
        for (int g = 0; g < GM; ++g) {
            m_run[g] = -INFINITY;
            m_true[g] = -INFINITY;
            l_part[g] = 0.f;
            acc[g] = 0.f;
            alpha_prev[g] = 1.f;
            kinv_prev[g] = 1.f;
        }
        bool failed = false;
        // O of tile k (one of this group's two buffers) into the accumulator
        auto accumulate = [&](int k) -> bool {
            const int ob = 2 * grp + ((k >> 1) & 1);
            const bool landed = mbar_wait(&bar[kOFull0 + ob], (k >> 2) & 1);
            if (!__all_sync(kFullMask, landed)) return false;
            tc_fence_after();
            float o[16];
            tmem_load16(tmem + lane_addr + S::O0 + S::QN * ob, o);
            if constexpr (S::DIRECT) {
                // a head's four P terms are four columns: add them, undo the
                // tile's power-of-two P scale
                float o34[16];
                if constexpr (GM == 8) tmem_load16(tmem + lane_addr + S::O0 + S::QN * ob + 16, o34);
#pragma unroll
                for (int g = 0; g < GM; ++g)
                    o[g] = (GM == 8 ? (o[g] + o[GM + g]) + (o34[g] + o34[GM + g])
                                    : (o[g] + o[GM + g]) + (o[2 * GM + g] + o[3 * GM + g])) *
                           kinv_prev[g];
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[kOEmpty0 + ob]);
#pragma unroll
            for (int g = 0; g < GM; ++g) acc[g] = acc[g] * alpha_prev[g] + o[g];
            return true;
        };

        int last = -1;
        // Partition by partition of the CTA's span (one partition unless
        // p.span > 1): tiles [j * tpp, (j + 1) * tpp) of partition j, every
        // other one this group's.  Both groups meet at each partition's end,
        // whether or not they had a tile in it.
        const int nspan = part_end - part0;
        for (int j = 0; j < nspan; ++j) {
            const int t1 = ((j + 1) * tpp < ntiles) ? (j + 1) * tpp : ntiles;
            for (int i = j * tpp + grp; i < t1; i += 2) {
              const bool landed = !failed && mbar_wait(&bar[kSFull0 + grp], (i >> 1) & 1);
              const bool ok = __all_sync(kFullMask, landed);
              float s[GM];
              if (ok) {
                  tc_fence_after();
                  float t12[16], t34[16];
                  tmem_load16(tmem + lane_addr + S::S0 + S::QN * grp, t12);
                  if constexpr (GM == 8) tmem_load16(tmem + lane_addr + S::S0 + S::QN * grp + 16, t34);
                  tc_fence_before();
                  __syncwarp();
                  if (lane == 0) mbar_arrive(&bar[kSEmpty0 + grp]);
  #pragma unroll
                  for (int g = 0; g < GM; ++g)
                      s[g] = GM == 8 ? (t12[g] + t12[GM + g]) + (t34[g] + t34[GM + g])
                                     : (t12[g] + t12[GM + g]) + (t12[2 * GM + g] + t12[3 * GM + g]);
              } else {
  #pragma unroll
                  for (int g = 0; g < GM; ++g) s[g] = 0.f;
              }
              const int tile0 = start + i * kF8Tile;
              const int nvalid = (end - tile0 < kF8Tile) ? end - tile0 : kF8Tile;
              const bool valid = r < nvalid;
              // tile max of each head over the 128 positions: a halving
              // butterfly over the warp (each exchange hands the partner the
              // heads it keeps), after which lane L holds head (L >> 2) & 7
              float *tmax = gred + ((i >> 1) & 1) * (4 * kF8N);
  #pragma unroll
              for (int g = 0; g < GM; ++g) s[g] = valid ? s[g] * qm[g] : -INFINITY;  // select: NaN-safe
              {
                  // GM = 8: lane L ends with head (L >> 2) & 7; GM = 4: (L >> 3) & 3
                  float v4[4], v2[2];
                  if constexpr (GM == 8) {
                      const bool b4 = lane & 16;
  #pragma unroll
                      for (int j = 0; j < 4; ++j)
                          v4[j] = fmaxf(b4 ? s[4 + j] : s[j],
                                        __shfl_xor_sync(kFullMask, b4 ? s[j] : s[4 + j], 16));
                  } else {
  #pragma unroll
                      for (int j = 0; j < 4; ++j) v4[j] = s[j];
                  }
                  constexpr int o2 = GM == 8 ? 8 : 16, o1 = o2 / 2;
                  const bool c2 = lane & o2, c1 = lane & o1;
  #pragma unroll
                  for (int j = 0; j < 2; ++j)
                      v2[j] = fmaxf(c2 ? v4[2 + j] : v4[j],
                                    __shfl_xor_sync(kFullMask, c2 ? v4[j] : v4[2 + j], o2));
                  float v = fmaxf(c1 ? v2[1] : v2[0], __shfl_xor_sync(kFullMask, c1 ? v2[0] : v2[1], o1));
  #pragma unroll
                  for (int off = o1 / 2; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(kFullMask, v, off));
                  constexpr int sh = GM == 8 ? 2 : 3;
                  if ((lane & ((1 << sh) - 1)) == 0) tmax[sw * kF8N + ((lane >> sh) & (GM - 1))] = v;
              }
              if (lane == 0) tmax[sw * kF8N + kF8N - 1] = ok ? 1.f : 0.f;  // column 15: health flag
              named_bar(1 + grp, 128);
              bool all_ok = true;
  #pragma unroll
              for (int w = 0; w < 4; ++w) all_ok &= tmax[w * kF8N + kF8N - 1] != 0.f;
              if (!all_ok) {
                  failed = true;
                  break;
              }
              bool need = false;
              float mx[GM];
  #pragma unroll
              for (int g = 0; g < GM; ++g) {
                  mx[g] = fmaxf(fmaxf(tmax[g], tmax[kF8N + g]),
                                fmaxf(tmax[2 * kF8N + g], tmax[3 * kF8N + g]));
                  need |= (g < G) && (mx[g] > m_run[g] + kLazyRescale);
              }
              float alpha[GM];
  #pragma unroll
              for (int g = 0; g < GM; ++g) {
                  alpha[g] = 1.f;
                  if (need) {  // group-uniform
                      const float mn = fmaxf(m_run[g], mx[g]);
                      alpha[g] = fast_exp2(m_run[g] - mn);
                      m_run[g] = mn;
                      l_part[g] *= alpha[g];
                  }
                  m_true[g] = fmaxf(m_true[g], mx[g]);
              }
              // E5M2 P: each head's P is taken times 2^k, the power of two that
              // brings the tile's largest P into [2^14, 2^15), so that its four
              // E5M2 terms keep 12 bits of every value down to 2^-21 of that
              // largest, and lose less than 2^-31 of it below (the sum l keeps
              // the unscaled values)
              float pv[GM], kinv[GM];
  #pragma unroll
              for (int g = 0; g < GM; ++g) {
                  pv[g] = 0.f;
                  kinv[g] = 1.f;
                  if (g < G) {
                      float pg = fast_exp2(s[g] - m_run[g]);  // masked: 2^-inf = 0
                      l_part[g] += pg;
                      if constexpr (S::DIRECT) {
                          const float dm = mx[g] - m_run[g];  // <= lazy-rescale threshold
                          int k = 0;
                          if (dm > -INFINITY) {
                              k = 14 - __float2int_rd(dm);
                              k = k > 126 ? 126 : k;
                          }
                          kinv[g] = exp2i(-k);
                          pg *= exp2i(k);  // exact: a power of two, k >= 6
                      }
                      pv[g] = pg;
                  }
              }
              // P buffer of this tile: last read by P.V of tile i-4, whose O this
              // group accumulated (after waiting for it) two tiles ago
              uint8_t *pbuf = smem + S::OFF_P + (2 * grp + ((i >> 1) & 1)) * S::P_BYTES;
              if constexpr (S::DIRECT) {
                  // P^T as four E5M2 terms of P rounded to f16 (11 significant
                  // bits: the terms hold it exactly down to E5M2's subnormal
                  // range), split in packed f16 pairs: rows t*GM + g (t = term,
                  // g = head), 128 positions of one byte, K-major with 128-byte
                  // swizzle
  #pragma unroll
                  for (int g = 0; g < GM; g += 2) {
                      uint32_t h = narrow2<false>(pv[g], pv[g + 1]);
  #pragma unroll
                      for (int t = 0; t < S::NTERM; ++t) {
                          const uint32_t c = e5m2x2_from_f16x2(h);
                          h = hsub2_bits(h, f16x2_from_e5m2x2((uint16_t)c));  // exact
                          pbuf[e4m3_operand_offset<128>(GM * t + g, r)] = (uint8_t)(c & 0xffu);
                          pbuf[e4m3_operand_offset<128>(GM * t + g + 1, r)] = (uint8_t)(c >> 8);
                      }
                  }
                  if (!valid) {
                      // Stale rows of the last tile: P is 0 there but V must be
                      // finite (0 * NaN would poison the product), so zero them
                      // once the V tile has landed (its slot cannot move on
                      // before P.V of this tile, which waits for this P).
                      const int slot = i % S::NV;
                      if (mbar_wait(&bar[kVFull0 + slot], (i / S::NV) & 1)) {
                          uint4 *vrow = reinterpret_cast<uint4 *>(smem + S::OFF_VSTG +
                                                                  slot * S::STG_BYTES + r * D);
  #pragma unroll
                          for (int c = 0; c < D / 16; ++c) vrow[c] = make_uint4(0, 0, 0, 0);
                      } else {
                          failed = true;
                      }
                  }
              } else {
                  // P^T (16 rows = heads, 128 positions) in the operand layout, f16
  #pragma unroll
                  for (int g = 0; g < kF8N; ++g)
                      *reinterpret_cast<uint16_t *>(pbuf + sw128_offset(g, r, kF8N * 128)) =
                          narrow_f16<false>(g < GM ? pv[g] : 0.f);
              }
              fence_async_smem();
              __syncwarp();
              if (lane == 0) mbar_arrive(&bar[kPFull0 + 2 * grp + ((i >> 1) & 1)]);
              // this group's previous tile, while P.V of this one runs
              if (last >= 0 && !accumulate(last)) failed = true;
  #pragma unroll
              for (int g = 0; g < GM; ++g) {
                  alpha_prev[g] = alpha[g];
                  kinv_prev[g] = kinv[g];
              }
              last = i;
            }
            if (!failed && last >= 0 && !accumulate(last)) failed = true;
            last = -1;
            // l over the group's 128 position-threads, per head
            float *lsum = gred + 2 * (4 * kF8N);
#pragma unroll
            for (int g = 0; g < GM; ++g) {
                float v = l_part[g];
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(kFullMask, v, off);
                if (lane == 0) lsum[sw * kF8N + g] = v;
            }
            named_bar(1 + grp, 128);
            float lt[GM];
#pragma unroll
            for (int g = 0; g < GM; ++g)
                lt[g] = lsum[g] + lsum[kF8N + g] + lsum[2 * kF8N + g] + lsum[3 * kF8N + g];
            // group B hands its state to group A (two exchange buffers, by
            // partition parity: B may write the next one while A still reads)
            float *xacc = xch + (j & 1) * (S::XCH_BYTES / 4);  // [kF8G][D]
            float *xm = xacc + kF8G * D;                       // m_run, m_true, l, failed
            if (grp == 1) {
                if (r < D) {
#pragma unroll
                    for (int g = 0; g < GM; ++g) xacc[g * D + r] = acc[g];
                }
                if (st == 0) {
#pragma unroll
                    for (int g = 0; g < GM; ++g) {
                        xm[g] = m_run[g];
                        xm[kF8G + g] = m_true[g];
                        xm[2 * kF8G + g] = lt[g];
                    }
                    xm[3 * kF8G] = failed ? 1.f : 0.f;
                }
            }
            named_bar(3, 256);
            if (grp == 0) {
                failed |= xm[3 * kF8G] != 0.f;
                if (failed) {
                    if (st == 0) {
                        record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
                        *abort_flag = 1;
                    }
                } else if (r < D) {
#pragma unroll
                    for (int g = 0; g < GM; ++g) {
                        if (g >= G) break;
                        // merge of the two groups' partial softmaxes
                        const float mb = xm[g];
                        const float M = fmaxf(m_run[g], mb);
                        const float sa = fast_exp2(m_run[g] - M);
                        const float sb = mb == -INFINITY ? 0.f : fast_exp2(mb - M);
                        const float l = lt[g] * sa + xm[2 * kF8G + g] * sb;
                        const float a = acc[g] * sa + xacc[g * D + r] * sb;
                        const float mt = fmaxf(m_true[g], xm[kF8G + g]);
                        const float o = a / l * p.v_scale;  // V elements are v_scale * codes
                        const int h = kvh * G + g;
                        if (direct) {
                            uint16_t *out = static_cast<uint16_t *>(p.out);
                            out[((int64_t)seq * p.num_q_heads + h) * D + r] = narrow_out<BF16>(o);
                        } else {
                            const int64_t row = part_row(p, seq, h, part0 + j);
                            p.part_o[row * D + r] = o;
                            if (r == 0) {
                                p.part_m[row] = mt;
                                p.part_l[row] = l * fast_exp2(M - mt);
                            }
                        }
                    }
                }
            }
            if (j + 1 < nspan) {  // a fresh running state for the next partition
#pragma unroll
                for (int g = 0; g < GM; ++g) {
                    m_run[g] = -INFINITY;
                    m_true[g] = -INFINITY;
                    l_part[g] = 0.f;
                    acc[g] = 0.f;
                    alpha_prev[g] = 1.f;
                    kinv_prev[g] = 1.f;
                }
            }
        }
    }

    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        // let copies and MMAs still in flight finish before shared memory and
        // TMEM are released (each wait is bounded)
        const int last = ntiles - 1;
        (void)mbar_wait(&bar[kKFull0 + last % S::NK], (last / S::NK) & 1);
        (void)mbar_wait(&bar[kVFull0 + last % S::NV], (last / S::NV) & 1);
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, S::COLS);
    }
    if (!direct && !*abort_flag && p.counters != nullptr)
        finish_item<BF16, D>(p, seq, kvh, nparts_seq, part, (nparts_seq + R - 1) / R, p.one_wave,
                             reinterpret_cast<float *>(smem + S::OFF_STG),
                             (S::NK + S::NV) * S::STG_BYTES);
}

using F8Kernel = void (*)(const DecodeParams, const CUtensorMap, const CUtensorMap);

struct F8Pick {
    F8Kernel fn;
    int smem, threads, cols;
};

template <int D, int GM>
F8Pick pick_fp8_shape(bool bf16) {
    using S = F8Shape<D, GM>;
    return {bf16 ? paged_decode_fp8_kernel<true, D, GM> : paged_decode_fp8_kernel<false, D, GM>,
            S::SMEM_BYTES, S::THREADS, S::COLS};
}

// The instantiation for head size D and a group of `group` query heads
// (up to 4, or up to 8).
F8Pick pick_fp8(bool bf16, int D, int group) {
    if (D == 128) return group <= 4 ? pick_fp8_shape<128, 4>(bf16) : pick_fp8_shape<128, 8>(bf16);
    return group <= 4 ? pick_fp8_shape<64, 4>(bf16) : pick_fp8_shape<64, 8>(bf16);
}

}  // namespace

bool fp8_supported(int head_dim, int group) {
    return (head_dim == 64 || head_dim == 128) && group >= 1 && group <= kF8G;
}

// Resident CTAs per SM from the kernel's footprint (shared memory, registers
// per sub-partition, TMEM), as for the 16-bit tensor-core kernel.
int fp8_ctas_per_sm(bool bf16, int head_dim, int group) {
    const F8Pick f = pick_fp8(bf16, head_dim, group);
    const F8Kernel k = f.fn;
    const int smem = f.smem, threads = f.threads;
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
    const int by_smem = smem_sm / (smem + (int)a.sharedSizeBytes + reserved);
    const int regs = (a.numRegs + 7) / 8 * 8;
    const int warps_per_subpartition = 16384 / (regs * 32);
    const int by_regs = 4 * warps_per_subpartition / (threads / 32);
    const int by_tmem = 512 / f.cols;
    int n = by_smem < by_regs ? by_smem : by_regs;
    n = n < by_tmem ? n : by_tmem;
    return n > 0 ? n : 1;
}

pa_status launch_decode_fp8(const DecodeParams &prm, bool bf16, int head_dim, int num_partitions,
                            int num_kv_heads, int num_seqs, cudaStream_t stream) {
    if (num_seqs == 0) return PA_OK;
    const F8Pick f = pick_fp8(bf16, head_dim, prm.group);
    const F8Kernel k = f.fn;
    const int smem = f.smem, threads = f.threads;
    if (!ensure_smem_attr(reinterpret_cast<const void *>(k), smem)) return PA_ERR_CUDA;
    const int64_t rows = (int64_t)prm.num_blocks * num_kv_heads * prm.block_size;
    CUtensorMap mk, mv;
    // K lands swizzled (the q.K^T operand); V too at d = 128 (the MN-major
    // P.V operand), row-major at d = 64 (the converters' input)
    if (!pool_tensor_map_fp8(&mk, prm.k_pool, rows, head_dim, true) ||
        !pool_tensor_map_fp8(&mv, prm.v_pool, rows, head_dim, head_dim == 128))
        return PA_ERR_CUDA;
    const dim3 grid = decode_grid(prm, num_partitions, num_kv_heads, num_seqs);
    if (launch_pdl(k, grid, dim3((unsigned)threads), (size_t)smem, stream, prm, mk, mv) != cudaSuccess)
        return PA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
