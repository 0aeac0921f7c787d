// Paged decode over an FP8 KV cache for GB300 (sm_103a).
//
// The pools hold OCP E4M3 codes (one byte per element), one scale per K or V
// pool: element = scale * code value ("b = 1 for FP8" in the KV-size formula
// of "PagedAttention and Virtual Memory Management: Mathematical Foundations
// ..." (llms.blog), section 1; format and scale are this build's readings).
// Same computation as the tensor-core kernel in pa_decode_tc.cu (whose header
// describes the products, the roles and the online softmax), with half the
// K/V bytes moved:
//   - the producer's TMA copies land the E4M3 tiles in a staging buffer
//     (row-major, 16 rows of d bytes per box);
//   - converter warps (three for K, three for V) widen them exactly to f16 (PTX
//     cvt.rn.f16x2.e4m3x2: every E4M3 value is an f16 value) into the
//     128-byte-swizzled K and V operand tiles, zeroing V rows past the end;
//   - the MMAs run in kind::f16 with f16 operands (q converted to f16, P
//     written as f16); the K scale is folded into the softmax scale and the V
//     scale into the output.
// The staging buffer is a ring of several tiles (one CTA per SM holds it),
// so the copies run that many tiles ahead of the conversion and the
// products: the bytes in flight per SM, not the conversion, set the rate.
// Two softmax warpgroups take alternate tiles (even tiles with S, P and O
// buffers 0, odd tiles with buffers 1), each with its own running maximum,
// sum and accumulator, merged at the end, so two tiles' softmax run at once.
// Roles (16 warps): 0 producer, 1 TMEM owner and MMA issuer, 2..5 and 6..9
// softmax / epilogue groups A and B, 10..12 K converters, 13..15 V
// converters.
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
constexpr int kF8N = 16;           // MMA N: the query heads of a group, zero-padded
constexpr int kF8G = 8;            // largest group the kernel serves
constexpr int kF8Warps = 16;  // 4 per SM sub-partition: up to 128 registers a thread
constexpr int kF8Threads = kF8Warps * 32;
constexpr int kF8Cols = 64;        // TMEM columns: S x2 and O x2, 16 fp32 columns each
constexpr int kF8S0 = 0, kF8O0 = 32;
constexpr int kF8Conv0 = 10;       // first converter warp
constexpr int kF8ConvWarps = 3;    // converter warps for K, and as many for V

constexpr int kF8MaxStages = 8;

enum F8Bar {
    kKFull0 = 0, kKFull1, kVFull0, kVFull1, kKEmpty0, kKEmpty1, kVEmpty0, kVEmpty1, kQReady,
    kSFull0, kSFull1, kSEmpty0, kSEmpty1, kPFull0, kPFull1, kOFull0, kOFull1, kOEmpty0, kOEmpty1,
    kStgFull0,                                // kF8MaxStages of each
    kStgEmpty0 = kStgFull0 + kF8MaxStages,
    kNumF8Bars = kStgEmpty0 + kF8MaxStages
};

template <int D>
struct F8Shape {
    static constexpr int KH = D / 64;                 // 64-dim (128-byte) f16 slabs along d
    static constexpr int SLAB = kF8Tile * 128;        // one slab of a tile: 16 KiB
    static constexpr int K_BYTES = KH * SLAB;
    static constexpr int V_BYTES = 2 * SLAB;          // V^T is M = 128 dims; d = 64 pads with zeros
    static constexpr int Q_BYTES = KH * kF8N * 128;   // q as a 16-row K-major operand
    static constexpr int P_BYTES = 2 * kF8N * 128;    // P^T: 16 rows x 128 positions (two atoms)
    static constexpr int STG_BYTES = kF8Tile * D;     // E4M3 tile of K (or V), row-major
    static constexpr int NSTG = D == 128 ? 2 : 4;     // staging ring: tiles in flight
    static constexpr int NVB = 2;                     // V operand buffers (K has two)
    // K and V operand tiles, two of each: tile t converts into buffer t & 1
    // while the tensor cores still read the other
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + 2 * K_BYTES;
    static constexpr int OFF_Q = OFF_V + NVB * V_BYTES;
    static constexpr int OFF_P = OFF_Q + Q_BYTES;     // two buffers
    static constexpr int OFF_STG = OFF_P + 2 * P_BYTES;  // stage s: K at s * 2 * STG, V after it
    static constexpr int OFF_RED = OFF_STG + NSTG * 2 * STG_BYTES;
    // per softmax group: two tile-max buffers and the final sums
    static constexpr int RED_BYTES = 2 * 3 * 4 * kF8N * 4;
    // group B's state for the final merge: acc [G][D], then m_run, m_true, l
    static constexpr int OFF_XCH = OFF_RED + RED_BYTES;
    static constexpr int XCH_BYTES = kF8G * D * 4 + 4 * kF8G * 4;
    static constexpr int OFF_BAR = OFF_XCH + XCH_BYTES;
    static constexpr int OFF_MISC = OFF_BAR + kNumF8Bars * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack to align the base to 1 KiB
    static_assert(OFF_V % 1024 == 0 && OFF_Q % 1024 == 0 && OFF_P % 1024 == 0, "atom alignment");
    static_assert(OFF_STG % 128 == 0 && STG_BYTES % 128 == 0, "TMA destinations");
    static_assert(NSTG <= kF8MaxStages, "stage barriers");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(K_BYTES >= 2 * kF8G * kCombineMaxParts * 4, "combine scratch in the K tile");
};

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

template <bool BF16, int D>
__global__ void __launch_bounds__(kF8Threads, 1)
    paged_decode_fp8_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmap_k,
                            const __grid_constant__ CUtensorMap tmap_v) {
    using S = F8Shape<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + S::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::OFF_MISC + 8);
    float *red = reinterpret_cast<float *>(smem + S::OFF_RED);

    const int part = blockIdx.x, kvh = blockIdx.y, seq = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.group;
    const int P = p.partition_tokens;
    if (threadIdx.x == 0) {  // descriptors are kernel parameters: fetch them early
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    pdl_wait();  // inputs may come from the previous kernel on the stream
    const int L = item_len(p, seq, threadIdx.x == 0 && part == 0 && kvh == 0);
    const int nparts_seq = L == 0 ? 0 : (L - 1) / P + 1;
    const int start = part * P;
    if (start >= L) {  // empty partition: as in the other decode kernels
        if (p.mode == 0) {
            if (part == 0) {
                uint32_t *o = reinterpret_cast<uint32_t *>(p.out);
                const int64_t base = ((int64_t)seq * p.num_q_heads + (int64_t)kvh * G) * D / 2;
                for (int i = threadIdx.x; i < G * D / 2; i += blockDim.x) o[base + i] = 0u;
            }
        } else {
            for (int g = 0; g < G; ++g) {
                const int64_t row = part_row(p, seq, kvh * G + g, part);
                if (threadIdx.x == 0) {
                    p.part_m[row] = -INFINITY;
                    p.part_l[row] = 0.f;
                }
                for (int x = threadIdx.x; x < D; x += blockDim.x) p.part_o[row * D + x] = 0.f;
            }
        }
        return;
    }
    const int end = (start + P < L) ? start + P : L;
    const int nunits = (end - start + kUnit - 1) / kUnit;
    const int ntiles = (end - start + kF8Tile - 1) / kF8Tile;
    const bool direct = (p.mode == 0) && (nparts_seq <= 1);

    if (p.k_new != nullptr && part == nparts_seq - 1) fused_cache_write_fp8<BF16, D>(p, seq, kvh, L);
    if (threadIdx.x == 0) {
        // kKFull / kVFull: the converter warps of K / V; kQReady, kSEmpty,
        // kPFull, kOEmpty: the 4 warps of a softmax group
        const int counts[kStgFull0] = {kF8ConvWarps, kF8ConvWarps, kF8ConvWarps, kF8ConvWarps,
                                       1, 1, 1, 1, 4, 1, 1, 4, 4, 4, 4, 1, 1, 4, 4};
        for (int b = 0; b < kStgFull0; ++b) mbar_init(&bar[b], counts[b]);
        for (int b = 0; b < kF8MaxStages; ++b) {
            mbar_init(&bar[kStgFull0 + b], 1);   // the producer's expect-tx arrival
            mbar_init(&bar[kStgEmpty0 + b], 2 * kF8ConvWarps);  // every converter warp
        }
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kF8Cols);
        tmem_relinquish();
    }
    if constexpr (D == 64) {
        // rows 64..127 of both V^T operand buffers: zero once, never written again
        for (int vb = 0; vb < S::NVB; ++vb) {
            uint4 *z = reinterpret_cast<uint4 *>(smem + S::OFF_V + vb * S::V_BYTES + S::SLAB);
            for (int i = threadIdx.x; i < S::SLAB / 16; i += kF8Threads) z[i] = make_uint4(0, 0, 0, 0);
        }
        fence_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        const int32_t *table = seq_table(p, seq);
        bool ok = true;
        for (int u0 = 0; u0 < nunits && ok; u0 += 32) {  // 32 units = 4 tiles
            const int u = u0 + lane;
            int row0 = 0;  // first row of the unit in the 2-D view [NB*Hkv*B, d]
            if (u < nunits) {
                const int pos = start + u * kUnit;
                int phys = table[pos >> p.log2_block];
                if ((unsigned)phys >= (unsigned)p.num_blocks) {
                    record_error(p.err, PA_ERR_BAD_INDEX);
                    phys = 0;
                }
                row0 = (phys * p.num_kv_heads + kvh) * p.block_size + (pos & (p.block_size - 1));
            }
            for (int t = u0 / 8; t < ntiles && t < (u0 + 32) / 8; ++t) {
                const int nu = (nunits - 8 * t < 8) ? nunits - 8 * t : 8;
                const int sg = t % S::NSTG;
                if (t >= S::NSTG) {  // the converters have read this stage's previous tile
                    const bool done = mbar_wait(&bar[kStgEmpty0 + sg], ((t / S::NSTG) - 1) & 1);
                    if (!__all_sync(kFullMask, done)) {
                        ok = false;
                        break;
                    }
                }
                uint64_t *full = &bar[kStgFull0 + sg];
                uint8_t *stg = smem + S::OFF_STG + sg * 2 * S::STG_BYTES;
                if (lane == 0) mbar_arrive_expect_tx(full, nu * 2 * kUnit * D);
                // lane j < nu copies unit j of the tile (K and V): one
                // instruction issues the tile's copies
                const int r0 = __shfl_sync(kFullMask, row0, (8 * t - u0 + lane) & 31);
                if (lane < nu) {
                    tma_load_2d(stg + lane * kUnit * D, &tmap_k, 0, r0, full);
                    tma_load_2d(stg + S::STG_BYTES + lane * kUnit * D, &tmap_v, 0, r0, full);
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) {
            record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
        }
    } else if (warp >= kF8Conv0) {
        // ---------------------------------------------------------- converters
        // E4M3 staging -> f16 operand tiles, K by warps 10..12 and V by warps
        // 13..15, each group at its own pace (K of the next tiles converts
        // while V waits for the previous P.V).  Item = (row, 16 codes); every
        // load of a thread is issued before the first conversion.  Rows past
        // the end of the range get zeros in V (0 * NaN would poison P.V) and
        // are masked in S.
        constexpr int NCT = kF8ConvWarps * 32;                 // threads per group
        constexpr int NITEMS = kF8Tile * (D / 16);
        constexpr int NIT = (NITEMS + NCT - 1) / NCT;
        const bool is_v = warp >= kF8Conv0 + kF8ConvWarps;
        const int ct = threadIdx.x - (kF8Conv0 + (is_v ? kF8ConvWarps : 0)) * 32;
        bool ok = true;
        for (int t = 0; t < ntiles && ok; ++t) {
            const int nvalid = (end - start - t * kF8Tile < kF8Tile) ? end - start - t * kF8Tile
                                                                      : kF8Tile;
            const int sg = t % S::NSTG;
            const int stg = S::OFF_STG + sg * 2 * S::STG_BYTES + (is_v ? S::STG_BYTES : 0);
            const int nb = is_v ? S::NVB : 2;  // operand buffers
            const int ob = t % nb;
            const int op_off = is_v ? S::OFF_V + ob * S::V_BYTES : S::OFF_K + ob * S::K_BYTES;
            ok = __all_sync(kFullMask, mbar_wait(&bar[kStgFull0 + sg], (t / S::NSTG) & 1)) &&
                 (t < nb || __all_sync(kFullMask, mbar_wait(&bar[(is_v ? kVEmpty0 : kKEmpty0) + ob],
                                                             ((t / nb) - 1) & 1)));
            if (!ok) break;
            uint4 raw[NIT];
#pragma unroll
            for (int i = 0; i < NIT; ++i) {
                const int it = ct + NCT * i;
                const int row = it / (D / 16), c = it % (D / 16);
                raw[i] = (it >= NITEMS || (is_v && row >= nvalid))
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
                mbar_arrive(&bar[(is_v ? kVFull0 : kKFull0) + ob]);
                mbar_arrive(&bar[kStgEmpty0 + sg]);
            }
        }
        if (!ok && lane == 0) {
            record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc_qk = f16_idesc(false, false, false, kF8Tile, kF8N);
            constexpr uint32_t idesc_pv = f16_idesc(false, true, false, 128, kF8N);
            const uint32_t sbase = smem_addr(smem);
            bool ok = mbar_wait(&bar[kQReady], 0);
            // Whichever is ready first: q.K^T of tile nq once its K has landed
            // and its S buffer is free, or P.V of tile nv once its V, P and O
            // buffer are.  q.K^T of the next tile therefore runs while the
            // softmax works on this one, instead of waiting behind this P.V.
            int nq = 0, nv = 0;
            unsigned long long since = global_timer_ns();
            unsigned spins = 0;
            while (ok && nv < ntiles) {
                bool moved = false;
                if (nq < ntiles && mbar_test_wait(&bar[kKFull0 + (nq & 1)], (nq >> 1) & 1) &&
                    (nq < 2 || mbar_test_wait(&bar[kSEmpty0 + (nq & 1)], ((nq >> 1) - 1) & 1))) {
                    const int b = nq & 1;
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t koff = (ks >> 2) * S::SLAB + (ks & 3) * 32;
                        const uint32_t qoff = (ks >> 2) * (kF8N * 128) + (ks & 3) * 32;
                        tc_mma(tmem + kF8S0 + 16 * b,
                               sw128_desc(sbase + S::OFF_K + b * S::K_BYTES + koff, 16, 1024),
                               sw128_desc(sbase + S::OFF_Q + qoff, 16, 1024), idesc_qk, ks > 0);
                    }
                    tc_commit(&bar[kSFull0 + b]);
                    tc_commit(&bar[kKEmpty0 + b]);
                    ++nq;
                    moved = true;
                }
                if (nv < nq && mbar_test_wait(&bar[kVFull0 + nv % S::NVB], (nv / S::NVB) & 1) &&
                    mbar_test_wait(&bar[kPFull0 + (nv & 1)], (nv >> 1) & 1) &&
                    (nv < 2 || mbar_test_wait(&bar[kOEmpty0 + (nv & 1)], ((nv >> 1) - 1) & 1))) {
                    const int b = nv & 1;
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < kF8Tile / 16; ++ks) {
                        const uint32_t voff = ks * 2048;  // 16 positions = two 8-row groups
                        const uint32_t poff = b * S::P_BYTES + (ks >> 2) * (kF8N * 128) + (ks & 3) * 32;
                        tc_mma(tmem + kF8O0 + 16 * b,
                               sw128_desc(sbase + S::OFF_V + (nv % S::NVB) * S::V_BYTES + voff,
                                          S::SLAB, 1024),
                               sw128_desc(sbase + S::OFF_P + poff, 16, 1024), idesc_pv, ks > 0);
                    }
                    tc_commit(&bar[kOFull0 + b]);
                    tc_commit(&bar[kVEmpty0 + nv % S::NVB]);
                    ++nv;
                    moved = true;
                }
                if (moved) {
                    since = global_timer_ns();
                } else if ((++spins & 31) == 0 && global_timer_ns() - since > kWaitLimitNs) {
                    ok = false;
                }
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
            // q of the group of heads as the K-major B operand in f16 (16
            // rows, 128-byte swizzle), rows >= G zero.  Unscaled: the scales
            // are applied in fp32.
            for (int ci = st; ci < kF8N * (D / 8); ci += 128) {
                const int g = ci / (D / 8), c = ci % (D / 8);
                uint4 v = make_uint4(0, 0, 0, 0);
                if (g < G) {
                    const uint4 raw = *reinterpret_cast<const uint4 *>(
                        p.q + ((int64_t)seq * p.num_q_heads + (int64_t)kvh * G + g) * D + c * 8);
                    if constexpr (BF16) {
                        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
                        uint32_t h[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float2 f = widen2<true>(w[i]);
                            h[i] = narrow2<false>(f.x, f.y);
                        }
                        v = make_uint4(h[0], h[1], h[2], h[3]);
                    } else {
                        v = raw;
                    }
                }
                *reinterpret_cast<uint4 *>(smem + S::OFF_Q + sw128_offset(g, c * 8, kF8N * 128)) = v;
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[kQReady]);
        }

        float m_run[kF8G], m_true[kF8G], l_part[kF8G], acc[kF8G], alpha_prev[kF8G];
#pragma unroll
        for (int g = 0; g < kF8G; ++g) {
            m_run[g] = -INFINITY;
            m_true[g] = -INFINITY;
            l_part[g] = 0.f;
            acc[g] = 0.f;
            alpha_prev[g] = 1.f;
        }
        bool failed = false;
        // O of tile k (this group's buffer) into the accumulator
        auto accumulate = [&](int k) -> bool {
            const bool landed = mbar_wait(&bar[kOFull0 + grp], (k >> 1) & 1);
            if (!__all_sync(kFullMask, landed)) return false;
            tc_fence_after();
            float o[16];
            tmem_load16(tmem + lane_addr + kF8O0 + 16 * grp, o);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[kOEmpty0 + grp]);
#pragma unroll
            for (int g = 0; g < kF8G; ++g) acc[g] = acc[g] * alpha_prev[g] + o[g];
            return true;
        };

        int last = -1;
        for (int i = grp; i < ntiles; i += 2) {
            const bool landed = !failed && mbar_wait(&bar[kSFull0 + grp], (i >> 1) & 1);
            const bool ok = __all_sync(kFullMask, landed);
            float s[16];
            if (ok) {
                tc_fence_after();
                tmem_load16(tmem + lane_addr + kF8S0 + 16 * grp, s);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[kSEmpty0 + grp]);
            } else {
#pragma unroll
                for (int g = 0; g < 16; ++g) s[g] = 0.f;
            }
            const int tile0 = start + i * kF8Tile;
            const int nvalid = (end - tile0 < kF8Tile) ? end - tile0 : kF8Tile;
            const bool valid = r < nvalid;
            // tile max of each head over the 128 positions
            float *tmax = gred + ((i >> 1) & 1) * (4 * kF8N);
#pragma unroll
            for (int g = 0; g < kF8G; ++g) {
                s[g] = valid ? s[g] * p.scale_log2 : -INFINITY;  // select: NaN-safe
                float v = s[g];
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(kFullMask, v, off));
                if (lane == 0) tmax[sw * kF8N + g] = v;
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
            float mx[kF8G];
#pragma unroll
            for (int g = 0; g < kF8G; ++g) {
                mx[g] = fmaxf(fmaxf(tmax[g], tmax[kF8N + g]),
                              fmaxf(tmax[2 * kF8N + g], tmax[3 * kF8N + g]));
                need |= (g < G) && (mx[g] > m_run[g] + kLazyRescale);
            }
            float alpha[kF8G];
#pragma unroll
            for (int g = 0; g < kF8G; ++g) {
                alpha[g] = 1.f;
                if (need) {  // group-uniform
                    const float mn = fmaxf(m_run[g], mx[g]);
                    alpha[g] = fast_exp2(m_run[g] - mn);
                    m_run[g] = mn;
                    l_part[g] *= alpha[g];
                }
                m_true[g] = fmaxf(m_true[g], mx[g]);
            }
            float pv[kF8G];
#pragma unroll
            for (int g = 0; g < kF8G; ++g) {
                pv[g] = 0.f;
                if (g < G) {
                    pv[g] = fast_exp2(s[g] - m_run[g]);  // masked: 2^-inf = 0
                    l_part[g] += pv[g];
                }
            }
            // this group's previous tile: its P.V, which reads the P buffer
            // about to be rewritten, must be complete
            if (last >= 0 && !accumulate(last)) failed = true;
            // P^T (16 rows = heads, 128 positions) in the operand layout, f16
            uint8_t *pbuf = smem + S::OFF_P + grp * S::P_BYTES;
#pragma unroll
            for (int g = 0; g < kF8N; ++g)
                *reinterpret_cast<uint16_t *>(pbuf + sw128_offset(g, r, kF8N * 128)) =
                    narrow_f16<false>(g < kF8G ? pv[g] : 0.f);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[kPFull0 + grp]);
#pragma unroll
            for (int g = 0; g < kF8G; ++g) alpha_prev[g] = alpha[g];
            last = i;
        }
        if (!failed && last >= 0 && !accumulate(last)) failed = true;

        // l over the group's 128 position-threads, per head
        float *lsum = gred + 2 * (4 * kF8N);
#pragma unroll
        for (int g = 0; g < kF8G; ++g) {
            float v = l_part[g];
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(kFullMask, v, off);
            if (lane == 0) lsum[sw * kF8N + g] = v;
        }
        named_bar(1 + grp, 128);
        float lt[kF8G];
#pragma unroll
        for (int g = 0; g < kF8G; ++g)
            lt[g] = lsum[g] + lsum[kF8N + g] + lsum[2 * kF8N + g] + lsum[3 * kF8N + g];
        // group B hands its state to group A
        float *xacc = xch;                  // [kF8G][D]
        float *xm = xch + kF8G * D;         // m_run, m_true, l, failed
        if (grp == 1) {
            if (r < D) {
#pragma unroll
                for (int g = 0; g < kF8G; ++g) xacc[g * D + r] = acc[g];
            }
            if (st == 0) {
#pragma unroll
                for (int g = 0; g < kF8G; ++g) {
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
                for (int g = 0; g < kF8G; ++g) {
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
                        const int64_t row = part_row(p, seq, h, part);
                        p.part_o[row * D + r] = o;
                        if (r == 0) {
                            p.part_m[row] = mt;
                            p.part_l[row] = l * fast_exp2(M - mt);
                        }
                    }
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
        (void)mbar_wait(&bar[kStgFull0 + last % S::NSTG], (last / S::NSTG) & 1);
        (void)mbar_wait(&bar[kVEmpty0 + last % S::NVB], (last / S::NVB) & 1);
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kF8Cols);
    }
    if (!direct && !*abort_flag && p.counters != nullptr)
        finish_item<BF16, D>(p, seq, kvh, nparts_seq, reinterpret_cast<float *>(smem + S::OFF_K));
}

using F8Kernel = void (*)(const DecodeParams, const CUtensorMap, const CUtensorMap);

F8Kernel pick_fp8(bool bf16, int D, int *smem) {
    if (D == 128) {
        *smem = F8Shape<128>::SMEM_BYTES;
        return bf16 ? paged_decode_fp8_kernel<true, 128> : paged_decode_fp8_kernel<false, 128>;
    }
    *smem = F8Shape<64>::SMEM_BYTES;
    return bf16 ? paged_decode_fp8_kernel<true, 64> : paged_decode_fp8_kernel<false, 64>;
}

}  // namespace

bool fp8_supported(int head_dim, int group) {
    return (head_dim == 64 || head_dim == 128) && group >= 1 && group <= kF8G;
}

// Resident CTAs per SM from the kernel's footprint (shared memory, registers
// per sub-partition, TMEM), as for the 16-bit tensor-core kernel.
int fp8_ctas_per_sm(bool bf16, int head_dim) {
    int smem = 0;
    F8Kernel k = pick_fp8(bf16, head_dim, &smem);
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
    const int by_regs = 4 * warps_per_subpartition / kF8Warps;
    const int by_tmem = 512 / kF8Cols;
    int n = by_smem < by_regs ? by_smem : by_regs;
    n = n < by_tmem ? n : by_tmem;
    return n > 0 ? n : 1;
}

pa_status launch_decode_fp8(const DecodeParams &prm, bool bf16, int head_dim, int num_partitions,
                            int num_kv_heads, int num_seqs, cudaStream_t stream) {
    if (num_seqs == 0) return PA_OK;
    int smem = 0;
    F8Kernel k = pick_fp8(bf16, head_dim, &smem);
    if (!ensure_smem_attr(reinterpret_cast<const void *>(k), smem)) return PA_ERR_CUDA;
    const int64_t rows = (int64_t)prm.num_blocks * num_kv_heads * prm.block_size;
    CUtensorMap mk, mv;
    if (!pool_tensor_map_fp8(&mk, prm.k_pool, rows, head_dim) ||
        !pool_tensor_map_fp8(&mv, prm.v_pool, rows, head_dim))
        return PA_ERR_CUDA;
    dim3 grid((unsigned)num_partitions, (unsigned)num_kv_heads, (unsigned)num_seqs);
    if (launch_pdl(k, grid, dim3(kF8Threads), (size_t)smem, stream, prm, mk, mv) != cudaSuccess)
        return PA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
