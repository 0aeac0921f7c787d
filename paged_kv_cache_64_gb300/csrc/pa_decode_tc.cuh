#pragma once
// Tensor-core paged decode for GB300 (sm_103a): the head-group products
// q.K^T and P.V on the 5th-generation tensor cores (tcgen05.mma, fp32
// accumulators in TMEM), K/V tiles moved by 2-D TMA tensor copies with
// 128-byte swizzle.
//
// Same computation as the CUDA-core kernel in pa_decode.cu (see the header
// comment there and the sources cited in pa.h): for each (partition, KV head,
// sequence) the positions [start, end) are gathered through the block table
// and attended by the G query heads of the KV head with an online softmax.
// What changes is who does the arithmetic.  Per tile of 128 positions:
//
//   S^T[128 pos x 16]  = K_tile[128 x d]  . Q^T[d x 16]          (M=128, N=16, K=d)
//   O^T[d(128) x 16]   = V_tile^T[128 x 128 pos] . P^T[128 x 16] (M=128, N=16, K=128)
//
// with the G <= 8 heads of the group in the N columns (zero-padded to 16).
// Tokens on M is the layout that makes both operands of q.K^T and P.V come
// straight from the swizzled K/V tiles (K as a K-major A operand, V as an
// MN-major A operand); the softmax warps read S^T and O^T out of TMEM one
// row (position, or dimension) per thread.
//
// Roles (7 warps; 6 in the variant with several partitions a CTA, whose
// warp 1 issues both products, so that its larger register state still
// fits two CTAs an SM):
//   warp 0      producer: block-table lookups and TMA tensor copies of 16-row
//               boxes (one per 16 positions and 64 dims) into the K and V tiles;
//   warp 1      allocates the 64 TMEM columns; lane 0 issues the q.K^T MMAs
//               and commits their completion to mbarriers;
//   warps 2..5  softmax / epilogue: thread r owns TMEM lane r (position r of a
//               tile for S, dimension r for O); they also write q and P^T into
//               shared memory in the operand layout (K-major, 128-byte swizzle);
//   warp 6      lane 0 issues the P.V MMAs.
// A small tcgen05.mma takes tens of nanoseconds to issue from one thread and
// a tile needs 4 to 8 q.K^T and 8 P.V instructions, so the two products are
// issued from different warps: q.K^T of the next tile never queues behind
// P.V of this one.
// Online softmax with the same lazy rescale as the CUDA-core kernel; the
// accumulator lives in registers (thread = dimension) and takes each tile's
// O^T from a double-buffered TMEM slot.
//
// E4M3 pools (F8G = 4 or 8): the same roles and pipeline on 8-bit operands.
// K and V tiles land as E4M3 codes (16 rows x d bytes a box; 128-byte
// swizzle at d = 128, 64-byte at d = 64) and are the A operands of
// tcgen05.mma kind::f8f6f4 as they are; q and P are the B operands as four
// E5M2 terms of each of F8G heads (rows t * F8G + g, N = 4 * F8G), so a
// head's score and output are the sums of four columns:
//
//   S^T[128 pos x 4*F8G] = K_codes[128 x d] . Qs^T[d x 4*F8G]
//   O^T[d x 4*F8G]       = V_codes^T[d x 128 pos] . Ps^T[128 pos x 4*F8G]
//
// The K scale is folded into the score factor, the V scale into the output.
#include <cuda.h>  // CUtensorMap and its enums only; the encoder comes from the driver at run time

#include <cmath>
#include <cstdint>
#include <cstring>
#include <type_traits>

#include "pa_common.cuh"
#include "pa_decode.cuh"
#include "pa_fp8.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {

constexpr int kTcTile = 128;       // positions per tile (MMA M of q.K^T)
constexpr int kTcN = 16;           // MMA N: the query heads of a group, zero-padded
constexpr int kTcG = 8;            // largest group the kernel serves
constexpr int kTcPvWarp = 6;       // issuer of the P.V MMAs (variants without SPAN)
// Warps of a variant: the P.V issuer's warp is left out of the SPAN one.
template <bool SPAN>
constexpr int tc_warps() {
    return SPAN ? 6 : 7;
}
enum TcBar {
    kQReady = 0,
    kSFull0, kSFull1, kSEmpty0, kSEmpty1, kPFull0, kPFull1, kOFull0, kOFull1, kOEmpty0, kOEmpty1,
    kPreReady,
    kRingBars  // then the staging rings' full and empty barriers (TcShape)
};

// F8G: 0 for 16-bit pools; 4 or 8 for E4M3 pools (one byte an element),
// groups of up to F8G query heads.
template <int D, int F8G>
struct TcShape {
    static constexpr bool F8 = F8G != 0;
    static constexpr int RB = F8 ? D : 2 * D;         // bytes of a K or V row
    static constexpr int KH = D / 64;                 // 16-bit: 64-dim (128-byte) slabs along d
    static constexpr int SLAB = kTcTile * 128;        // 16-bit: one slab of a tile, 16 KiB
    static constexpr int STAGE = kTcTile * RB;        // one staged K or V tile
    // MMA N of both products: the heads zero-padded to 16 (16-bit), or four
    // E5M2 terms of each of F8G heads, rows t * F8G + g (E4M3)
    static constexpr int QN = F8 ? 4 * F8G : kTcN;
    // TMEM: S x2 at column 0, O x2 at 2 * QN, QN fp32 columns each
    static constexpr int COLS = F8 ? 4 * QN : 64;
    static constexpr int S_COL = 0, O_COL = 2 * QN;
    static_assert(4 * QN <= COLS, "TMEM columns");
    // Staging rings (K and V tiles in flight), sized to the shared memory of
    // two CTAs an SM: 16-bit pools three K and three V tiles at d = 64, so a
    // CTA has its next tiles in flight while it computes one (short work
    // items, such as a small model's decode step, are bound by that
    // latency), one of each at d = 128 (two CTAs an SM already keep enough
    // copies in flight for long items, and a second stage would leave one
    // CTA an SM); E4M3 pools, whose tiles take the softmax as long for half
    // the bytes, three K and three V tiles at d = 128, six of each at d = 64.
    // P.V reads V^T as an M = 128 (dims) MN-major operand.  At d = 64 only
    // its first 64 rows are real: rows 64..127 are read from the next STAGE
    // bytes (the next V stage or the first K stage), and only reach TMEM
    // lanes 64..127 of O, which no thread ever writes out.  So the V stages
    // come first at d = 64, K after them, and nothing is zero-padded.
    static constexpr int NK = F8 ? (D == 64 ? 6 : 3) : (D == 64 ? 3 : 1);
    static constexpr int NV = F8 ? (D == 64 ? 6 : 3) : (D == 64 ? 3 : 1);
    // barriers: those of TcBar, then K full, K empty, V full and V empty, CAP
    // of each (CAP >= NK, NV; 3 unless a ring has more slots)
    static constexpr int CAP = NK > 3 || NV > 3 ? (NK > NV ? NK : NV) : 3;
    static constexpr int KFULL = kRingBars, KEMPTY = KFULL + CAP, VFULL = KEMPTY + CAP,
                         VEMPTY = VFULL + CAP, NUM_BARS = VEMPTY + CAP;
    static constexpr int V_BYTES = NV * STAGE;
    static constexpr int K_BYTES = NK * STAGE;
    // q: a QN-row K-major operand (128-byte swizzle; 64-byte for E4M3 at d = 64)
    static constexpr int Q_BYTES = F8 ? QN * D : KH * kTcN * 128;
    // P^T: QN rows x 128 positions, K-major, 128-byte swizzle (16-bit: two
    // atoms of 64 positions; E4M3: one of 128)
    static constexpr int P_BYTES = F8 ? QN * 128 : 2 * kTcN * 128;
    static constexpr int OFF_V = D == 64 ? 0 : K_BYTES;
    static constexpr int OFF_K = D == 64 ? V_BYTES : 0;
    static constexpr int OFF_Q = (D == 64 ? OFF_K + K_BYTES : OFF_V + V_BYTES);
    static constexpr int OFF_P = OFF_Q + Q_BYTES;     // two buffers
    static constexpr int OFF_RED = OFF_P + 2 * P_BYTES;
    static constexpr int RED_BYTES = 3 * 4 * kTcN * 4;  // two tile-max buffers + the final sums
    // E4M3: per head the score factor (softmax scale in log2 units, K scale,
    // 2^-e_g of the q split), then per P buffer the tile's 2^-k_g (P scales)
    // and its online-softmax rescale factors
    static constexpr int OFF_F8 = OFF_RED + RED_BYTES;
    static constexpr int F8_BYTES = 5 * kTcG * 4;
    // cascade tail: the shared prefix's partials merged per head (O, then m,
    // l); none over E4M3 pools (no cascade there)
    static constexpr int OFF_PRE = OFF_F8 + F8_BYTES;
    static constexpr int PRE_BYTES = F8 ? 0 : kTcG * D * 4 + 2 * kTcG * 4;
    // SPAN: a closed partition's per-warp sums and its maxima (m_run,
    // m_true), kept until its partial is written; two buffers (partition
    // parity)
    static constexpr int PEND_FLOATS = 4 * kTcN + 2 * kTcG;
    static constexpr int OFF_PEND = OFF_PRE + PRE_BYTES;
    static constexpr int OFF_BAR = OFF_PEND + 2 * PEND_FLOATS * 4;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    // compact grids: the batch's lengths, kept for the CTA's later items
    static constexpr int OFF_LENS = OFF_MISC + 16;
    static constexpr int SMEM_BYTES = OFF_LENS + kCompactMaxSeqs * 4 + 1024;  // + slack to align the base to 1 KiB
    static_assert(OFF_V % 1024 == 0 && OFF_K % 1024 == 0 && OFF_Q % 1024 == 0 &&
                  OFF_P % 1024 == 0 && STAGE % 1024 == 0, "atom alignment");
    // the last V stage's operand (two STAGEs at d = 64) stays in bounds
    static_assert(OFF_V + (NV - 1) * STAGE + (D == 64 ? 2 : 1) * STAGE <= OFF_BAR,
                  "V^T operand rows in bounds");
    // two CTAs an SM (228 KiB of shared memory, 1 KiB reserved a CTA)
    static_assert(2 * (SMEM_BYTES + 1024) <= 228 * 1024, "two CTAs an SM");
    // the combine's scratch: the staging rings, [0, OFF_Q)
    static_assert(OFF_Q >= 2 * kTcG * kCombineMaxParts * 4, "combine scratch in the rings");
};


// q.K^T of one tile into the S buffer at TMEM address s_tmem: K (kaddr) as
// the K-major A operand, q (qaddr) as the K-major B operand.
template <bool BF16, int D, int F8G>
__device__ __forceinline__ void tc_issue_qk(uint32_t s_tmem, uint32_t kaddr, uint32_t qaddr) {
    using S = TcShape<D, F8G>;
    if constexpr (S::F8) {
        // E4M3 K times the E5M2 terms of q, 32 bytes of d an instruction
        constexpr uint32_t idesc = e4m3_e5m2_idesc(kTcTile, S::QN, false);
#pragma unroll
        for (int ks = 0; ks < D / 32; ++ks)
            tc_mma_f8(s_tmem, e4m3_operand_desc<D>(kaddr + ks * 32),
                      e4m3_operand_desc<D>(qaddr + ks * 32), idesc, ks > 0);
    } else {
        constexpr uint32_t idesc = f16_idesc(BF16, false, false, kTcTile, kTcN);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t koff = (ks >> 2) * S::SLAB + (ks & 3) * 32;
            const uint32_t qoff = (ks >> 2) * (kTcN * 128) + (ks & 3) * 32;
            tc_mma(s_tmem, sw128_desc(kaddr + koff, 16, 1024), sw128_desc(qaddr + qoff, 16, 1024),
                   idesc, ks > 0);
        }
    }
}

// P.V of one tile into the O buffer at o_tmem: the staged V tile (vaddr) as
// V^T, an MN-major A operand of M = 128 dims; P^T (paddr) as the K-major B
// operand.
template <bool BF16, int D, int F8G>
__device__ __forceinline__ void tc_issue_pv(uint32_t o_tmem, uint32_t vaddr, uint32_t paddr) {
    using S = TcShape<D, F8G>;
    if constexpr (S::F8) {
        // 32 positions an instruction: d = 128, one 128-byte atom across M,
        // 8-position groups 1,024 bytes apart; d = 64, two 64-byte atoms
        // across M (the second STAGE bytes on), groups 512 bytes apart
        constexpr uint32_t idesc = e4m3_e5m2_idesc(128, S::QN, true);
#pragma unroll
        for (int ks = 0; ks < kTcTile / 32; ++ks) {
            const uint64_t a = D == 128 ? sw128_desc(vaddr + ks * 4096, 16, 1024)
                                        : sw64_desc(vaddr + ks * 2048, S::STAGE, 512);
            tc_mma_f8(o_tmem, a, sw128_desc(paddr + ks * 32, 16, 1024), idesc, ks > 0);
        }
    } else {
        constexpr uint32_t idesc = f16_idesc(BF16, true, false, 128, kTcN);
#pragma unroll
        for (int ks = 0; ks < kTcTile / 16; ++ks) {
            const uint32_t voff = ks * 2048;  // 16 positions = two 8-row groups
            const uint32_t poff = (ks >> 2) * (kTcN * 128) + (ks & 3) * 32;
            tc_mma(o_tmem, sw128_desc(vaddr + voff, S::SLAB, 1024),
                   sw128_desc(paddr + poff, 16, 1024), idesc, ks > 0);
        }
    }
}

// SPAN: a CTA may compute several consecutive partitions (p.span > 1).
// COMPACT: the launch uses a compact grid (p.compact).  Every variant runs
// two CTAs an SM (shared memory allows no more), so registers are capped for
// two.
template <bool BF16, int D, bool SPAN, bool COMPACT, int F8G>
__global__ void __launch_bounds__(tc_warps<SPAN>() * 32, 2)
    paged_decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmap_k,
                           const __grid_constant__ CUtensorMap tmap_v) {
    using S = TcShape<D, F8G>;
    constexpr bool F8 = S::F8;
    // heads the softmax keeps state for: 8, or the E4M3 operand's F8G
    constexpr int NH = F8 ? F8G : kTcG;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + S::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::OFF_MISC + 8);
    // P.V MMAs issued so far (written by the P.V issuer, read by the q.K^T one)
    volatile int *pv_issued = reinterpret_cast<volatile int *>(smem + S::OFF_MISC + 12);
    float *red = reinterpret_cast<float *>(smem + S::OFF_RED);
    float *f8s = reinterpret_cast<float *>(smem + S::OFF_F8);  // E4M3: score factors, P scales

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.group;
    const int P = p.partition_tokens;
    if (threadIdx.x == 0) {  // descriptors are kernel parameters: fetch them early
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    // The CTA's TMEM columns, for all its items (allocated while an earlier
    // kernel on the stream may still be finishing: it touches no input)
    if (warp == 1) {
        tmem_alloc(tmem_slot, S::COLS);
        tmem_relinquish();
    }
    // Inputs may come from the previous kernel on the stream.  A cascade
    // tail's previous kernel is the prefix pass, whose only output is the
    // prefix's partials: the wait for it is put off until they are read (the
    // prefix pass lets this launch start only after its own wait, so the
    // kernels before it are complete).
    if (!p.late_wait) pdl_wait();

    // One work item: split-KV chunk `part` (a span of partitions) of KV head
    // kvh of sequence seq; `another` when the CTA has a next item.  false when
    // the CTA aborted (a bounded wait gave up).
    auto process = [&](const int seq, const int part, const int kvh, const bool use_flags,
                       const bool another) -> bool {
    const int L = item_len(p, seq, threadIdx.x == 0 && part == 0 && kvh == 0);
    const int nparts_seq = L == 0 ? 0 : (L - 1) / P + 1;
    // partitions [part0, part0 + R) of the sequence: this CTA's span
    const int R = (SPAN && p.span > 1) ? p.span : 1;
    const int part0 = part * R;
    const int start = part0 * P;
    if (start >= L) {  // empty partitions: as in the CUDA-core kernel
        if (p.prefix_parts > 0) {
            // empty cascade tail: the output is the prefix's partials combined
            if (nparts_seq == 0 && part == 0) {
                pdl_wait();
                finish_item<BF16, D>(p, seq, kvh, 0, 0, 1, false, reinterpret_cast<float *>(smem),
                                     S::OFF_Q);
            }
        } else if (p.mode == 0) {
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
        return true;
    }
    const int part_end = (part0 + R < nparts_seq) ? part0 + R : nparts_seq;  // past the last
    const int end = (part_end * P < L) ? part_end * P : L;
    // tiles per partition when the span has several (P is then a multiple of
    // the tile), else never reached
    const int tpp = (SPAN && R > 1) ? P / kTcTile : 1 << 30;
    const int nunits = (end - start + kUnit - 1) / kUnit;
    const int ntiles = (end - start + kTcTile - 1) / kTcTile;
    const bool direct = (p.mode == 0) && (nparts_seq <= 1);
    // single-partition cascade tail: merge the prefix's partials here and
    // write the output directly
    const bool merge_prefix = !F8 && direct && p.prefix_parts > 0;
    float *pre = reinterpret_cast<float *>(smem + S::OFF_PRE);

    // Loads needed after the set-up below are issued first, so they travel
    // while it runs: the producer's first 32 block-table entries (lane j:
    // unit j) and the softmax warps' pieces of q.
    const int32_t *table = seq_table(p, seq);
    int phys_first = 0;
    if (warp == 0 && lane < nunits) phys_first = table[(start + lane * kUnit) >> p.log2_block];
    // 16-byte pieces of q per softmax thread (E4M3 pools: thread st takes
    // kQEpt elements of head st / kQTph, 16, 8 or 4 bytes)
    constexpr int kQPieces = F8 ? 1 : kTcN * (D / 8) / 128;
    constexpr int kQTph = F8 ? 128 / F8G : 1, kQEpt = F8 ? D / kQTph : 8;
    uint4 qv[kQPieces];
#pragma unroll
    for (int j = 0; j < kQPieces; ++j) {
        qv[j] = make_uint4(0, 0, 0, 0);
        const int ci = threadIdx.x - 64 + 128 * j;  // softmax threads: 0..127
        if constexpr (F8) {
            const int g = ci / kQTph, c = ci % kQTph;
            if (warp >= 2 && warp < kTcPvWarp && g < G) {
                const uint16_t *src =
                    p.q + ((int64_t)seq * p.num_q_heads + (int64_t)kvh * G + g) * D + c * kQEpt;
                if constexpr (kQEpt == 8) {
                    qv[j] = *reinterpret_cast<const uint4 *>(src);
                } else if constexpr (kQEpt == 4) {
                    const uint2 v = *reinterpret_cast<const uint2 *>(src);
                    qv[j].x = v.x;
                    qv[j].y = v.y;
                } else {
                    qv[j].x = *reinterpret_cast<const uint32_t *>(src);
                }
            }
        } else {
            const int g = ci / (D / 8), c = ci % (D / 8);
            if (warp >= 2 && warp < kTcPvWarp && g < G)
                qv[j] = *reinterpret_cast<const uint4 *>(
                    p.q + ((int64_t)seq * p.num_q_heads + (int64_t)kvh * G + g) * D + c * 8);
        }
    }
    if (p.k_new != nullptr && part_end == nparts_seq) {
        if constexpr (F8)
            fused_cache_write_fp8<BF16, D>(p, seq, kvh, L);
        else
            fused_cache_write<D>(p, seq, kvh, L);
    }
    if (threadIdx.x == 0) {
        // kQReady, kSEmpty, kPFull, kOEmpty: the 4 softmax warps; the rest one
        // arrival (the producer's expect-tx, an MMA commit, the prefix merge)
        const int counts[kRingBars] = {4, 1, 1, 4, 4, 4, 4, 1, 1, 4, 4, 1};
        for (int b = 0; b < S::NUM_BARS; ++b) mbar_init(&bar[b], b < kRingBars ? counts[b] : 1);
        *abort_flag = 0;
        *pv_issued = 0;
        mbar_init_fence();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        // Windows of 32 units (4 tiles), lane j holding unit j of the window;
        // the next window's table entries are loaded when a window opens.
        const int rows_per_block = p.block_size;
        bool ok = true;
        int phys_cur = phys_first;
        for (int u0 = 0; u0 < nunits && ok; u0 += 32) {  // 32 units = 4 tiles
            const int u = u0 + lane;
            const int phys_next =
                (u + 32 < nunits) ? table[(start + (u + 32) * kUnit) >> p.log2_block] : 0;
            int row0 = 0;  // first row of the unit in the 2-D view [NB*Hkv*B, d]
            if (u < nunits) {
                const int pos = start + u * kUnit;
                int phys = phys_cur;
                if ((unsigned)phys >= (unsigned)p.num_blocks) {
                    record_error(p.err, PA_ERR_BAD_INDEX);
                    phys = 0;
                }
                row0 = (phys * p.num_kv_heads + kvh) * rows_per_block + (pos & (p.block_size - 1));
            }
            for (int t = u0 / 8; t < ntiles && t < (u0 + 32) / 8 && ok; ++t) {
                const int nu = (nunits - 8 * t < 8) ? nunits - 8 * t : 8;
                for (int kv = 0; kv < 2 && ok; ++kv) {
                    const int n = kv ? S::NV : S::NK;  // stages of this ring
                    const int slot = t % n;
                    if (t >= n) {
                        const bool done =
                            mbar_wait(&bar[(kv ? S::VEMPTY : S::KEMPTY) + slot], ((t / n) - 1) & 1);
                        if (!__all_sync(kFullMask, done)) {
                            ok = false;
                            break;
                        }
                    }
                    const int base_off = (kv ? S::OFF_V : S::OFF_K) + slot * S::STAGE;
                    const CUtensorMap *map = kv ? &tmap_v : &tmap_k;
                    uint64_t *full = &bar[(kv ? S::VFULL : S::KFULL) + slot];
                    if (lane == 0) mbar_arrive_expect_tx(full, nu * kUnit * S::RB);
                    // lane j < nu copies unit j of the tile: one instruction issues
                    // the tile's copies (16-bit: one box a 64-dim slab; E4M3:
                    // one box of 16 rows x d bytes)
                    const int r0 = __shfl_sync(kFullMask, row0, (8 * t - u0 + lane) & 31);
                    if (lane < nu) {
                        if constexpr (F8) {
                            tma_load_2d(smem + base_off + lane * (kUnit * D), map, 0, r0, full);
                        } else {
#pragma unroll
                            for (int h = 0; h < S::KH; ++h)
                                tma_load_2d(smem + base_off + h * S::SLAB + lane * 2048, map,
                                            64 * h, r0, full);
                        }
                    }
                    __syncwarp();
                }
            }
            phys_cur = phys_next;
        }
        if (!ok && lane == 0) {
            record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
        }
        if (merge_prefix) {
            // The shared prefix's partials of the group's heads, merged with
            // the online-softmax rescale while the tail is computed, once the
            // prefix pass is complete; four heads per round of loads, lane
            // owns D/32 dims.
            pdl_wait();
            constexpr int V = D / 32;
            const int np = p.prefix_parts;
            const int64_t row0 = ((int64_t)seq * p.num_q_heads + (int64_t)kvh * G) * p.ws_parts;
            for (int g0 = 0; g0 < G; g0 += 4) {
                float M[4], Ls[4], acc[4][V];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    M[j] = -INFINITY;
                    Ls[j] = 0.f;
#pragma unroll
                    for (int v = 0; v < V; ++v) acc[j][v] = 0.f;
                }
                for (int k = 0; k < np; ++k) {
                    float mk[4], lk[4], ov[4][V];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        mk[j] = -INFINITY;
                        lk[j] = 0.f;
#pragma unroll
                        for (int v = 0; v < V; ++v) ov[j][v] = 0.f;
                        if (g0 + j < G) {
                            const int64_t row = row0 + (int64_t)(g0 + j) * p.ws_parts + k;
                            mk[j] = __ldcg(p.part_m + row);
                            lk[j] = __ldcg(p.part_l + row);
                            const float *src = p.part_o + row * D + lane * V;
                            if constexpr (V == 4) {
                                const float4 t = __ldcg(reinterpret_cast<const float4 *>(src));
                                ov[j][0] = t.x; ov[j][1] = t.y; ov[j][2] = t.z; ov[j][3] = t.w;
                            } else {
                                const float2 t = __ldcg(reinterpret_cast<const float2 *>(src));
                                ov[j][0] = t.x; ov[j][1] = t.y;
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (mk[j] == -INFINITY) continue;  // empty partial
                        const float nm = fmaxf(M[j], mk[j]);
                        const float a = fast_exp2(M[j] - nm), b = lk[j] * fast_exp2(mk[j] - nm);
                        Ls[j] = Ls[j] * a + b;
#pragma unroll
                        for (int v = 0; v < V; ++v) acc[j][v] = acc[j][v] * a + b * ov[j][v];
                        M[j] = nm;
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int g = g0 + j;
                    if (g >= G) break;
                    const float inv = Ls[j] > 0.f ? 1.0f / Ls[j] : 0.f;
#pragma unroll
                    for (int v = 0; v < V; ++v) pre[g * D + lane * V + v] = acc[j][v] * inv;
                    if (lane == 0) {
                        pre[kTcG * D + g] = M[j];
                        pre[kTcG * D + kTcG + g] = Ls[j];
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[kPreReady]);
        }
    } else if (warp == 1 && SPAN) {
        // ---------------------------------------------------------- MMA issue
        if (lane == 0) {
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
                // (q.K^T of the last tile only once P.V of every earlier tile
                // is issued: see the stale-row zeroing in the softmax)
                if (nq < ntiles && (nq + 1 < ntiles || nv == nq) &&
                    mbar_test_wait(&bar[S::KFULL + nq % S::NK], (nq / S::NK) & 1) &&
                    (nq < 2 || mbar_test_wait(&bar[kSEmpty0 + (nq & 1)], ((nq >> 1) - 1) & 1))) {
                    const int b = nq & 1;
                    tc_fence_after();
                    tc_issue_qk<BF16, D, F8G>(tmem + S::S_COL + S::QN * b,
                                             sbase + S::OFF_K + (nq % S::NK) * S::STAGE,
                                             sbase + S::OFF_Q);
                    tc_commit(&bar[kSFull0 + b]);
                    tc_commit(&bar[S::KEMPTY + nq % S::NK]);
                    ++nq;
                    moved = true;
                }
                if (nv < nq && mbar_test_wait(&bar[S::VFULL + nv % S::NV], (nv / S::NV) & 1) &&
                    mbar_test_wait(&bar[kPFull0 + (nv & 1)], (nv >> 1) & 1) &&
                    (nv < 2 || mbar_test_wait(&bar[kOEmpty0 + (nv & 1)], ((nv >> 1) - 1) & 1))) {
                    const int b = nv & 1;
                    tc_fence_after();
                    tc_issue_pv<BF16, D, F8G>(tmem + S::O_COL + S::QN * b,
                                             sbase + S::OFF_V + (nv % S::NV) * S::STAGE,
                                             sbase + S::OFF_P + b * S::P_BYTES);
                    tc_commit(&bar[kOFull0 + b]);
                    tc_commit(&bar[S::VEMPTY + nv % S::NV]);
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
    } else if (warp == 1) {
        // ---------------------------------------------------------- q.K^T issue
        if (lane == 0) {
            const uint32_t sbase = smem_addr(smem);
            bool ok = mbar_wait(&bar[kQReady], 0);
            for (int nq = 0; ok && nq < ntiles; ++nq) {
                // tile nq's K has landed and its S buffer has been read
                ok = mbar_wait(&bar[S::KFULL + nq % S::NK], (nq / S::NK) & 1) &&
                     (nq < 2 || mbar_wait(&bar[kSEmpty0 + (nq & 1)], ((nq >> 1) - 1) & 1));
                if (ok && nq > 0 && nq + 1 == ntiles) {
                    // q.K^T of the last tile only once P.V of every earlier tile
                    // is issued (see the stale-row zeroing in the softmax)
                    const unsigned long long t0 = global_timer_ns();
                    while (*pv_issued < nq) {
                        if (global_timer_ns() - t0 > kWaitLimitNs) {
                            ok = false;
                            break;
                        }
                    }
                }
                if (!ok) break;
                const int b = nq & 1;
                tc_fence_after();
                tc_issue_qk<BF16, D, F8G>(tmem + S::S_COL + S::QN * b,
                                         sbase + S::OFF_K + (nq % S::NK) * S::STAGE,
                                         sbase + S::OFF_Q);
                tc_commit(&bar[kSFull0 + b]);
                tc_commit(&bar[S::KEMPTY + nq % S::NK]);
            }
            if (!ok) {
                record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
            }
        }
    } else if (!SPAN && warp == kTcPvWarp) {
        // ---------------------------------------------------------- P.V issue
        if (lane == 0) {
            const uint32_t sbase = smem_addr(smem);
            bool ok = true;
            for (int nv = 0; ok && nv < ntiles; ++nv) {
                // tile nv's V has landed, its P is written, its O buffer has
                // been accumulated from tile nv - 2
                const int b = nv & 1;
                ok = mbar_wait(&bar[S::VFULL + nv % S::NV], (nv / S::NV) & 1) &&
                     mbar_wait(&bar[kPFull0 + b], (nv >> 1) & 1) &&
                     (nv < 2 || mbar_wait(&bar[kOEmpty0 + b], ((nv >> 1) - 1) & 1));
                if (!ok) break;
                tc_fence_after();
                tc_issue_pv<BF16, D, F8G>(tmem + S::O_COL + S::QN * b,
                                         sbase + S::OFF_V + (nv % S::NV) * S::STAGE,
                                         sbase + S::OFF_P + b * S::P_BYTES);
                tc_commit(&bar[kOFull0 + b]);
                tc_commit(&bar[S::VEMPTY + nv % S::NV]);
                *pv_issued = nv + 1;
            }
            if (!ok) {
                record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
            }
        }
    } else {
        // ---------------------------------------------------------- softmax / epilogue
        const int sw = warp - 2;                 // softmax warp 0..3
        const int quad = warp & 3;               // TMEM lane quadrant this warp may access
        const int r = quad * 32 + lane;          // TMEM lane: position (S) or dimension (O)
        const int st = threadIdx.x - 64;         // 0..127
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;

        if constexpr (F8) {
            // Qs: head g's q times 2^e_g as four E5M2 terms in rows t * F8G + g
            // (t = 0..3) of a 4 * F8G-row K-major operand, rows of absent
            // heads zero.  2^e_g brings the head's largest |q| into [2^14, 2^15);
            // each term is the nearest E5M2 value of what the earlier ones
            // left (an exact remainder in fp32).  A 16-bit q has at most 11
            // significant bits and the terms carry 12, so they add up to
            // q * 2^e_g except for the part of an element below E5M2's
            // subnormal quantum (under 2^-31 of the head's largest).
            constexpr int EPT = kQEpt;  // elements a thread (kQTph threads a head)
            const int g = st / kQTph, c = st % kQTph;
            float x[EPT];
            {
                const uint32_t w[4] = {qv[0].x, qv[0].y, qv[0].z, qv[0].w};
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
            for (int off = kQTph / 2; off >= 1; off >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, off));
            int eg = 0;  // 14 - floor(log2 amax), from amax's exponent field
            if (amax > 0.f) {
                const int ex = (int)((__float_as_uint(amax) >> 23) & 0xffu) - 127;
                eg = 14 - (ex < -126 ? -126 : ex);
                eg = eg < -120 ? -120 : (eg > 120 ? 120 : eg);
            }
            const float up = exp2i(eg);
            constexpr int NW = EPT >= 4 ? EPT / 4 : 1;
            uint32_t code[4][NW];  // per term, 4 codes a word
#pragma unroll
            for (int t = 0; t < 4; ++t)
#pragma unroll
                for (int w4 = 0; w4 < NW; ++w4) code[t][w4] = 0u;
#pragma unroll
            for (int e2 = 0; e2 < EPT / 2; ++e2) {  // element pairs
                float a = x[2 * e2] * up, b = x[2 * e2 + 1] * up;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint32_t cd = e5m2x2_from_f32(a, b);
                    const float2 back = e5m2x2_to_f32(cd);
                    a -= back.x;  // exact: the remainder is representable
                    b -= back.y;
                    code[t][e2 >> 1] |= cd << (16 * (e2 & 1));
                }
            }
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                uint8_t *dst = smem + S::OFF_Q + e4m3_operand_offset<D>(F8G * t + g, c * EPT);
                if constexpr (EPT == 8)
                    *reinterpret_cast<uint2 *>(dst) = make_uint2(code[t][0], code[t][1]);
                else if constexpr (EPT == 4)
                    *reinterpret_cast<uint32_t *>(dst) = code[t][0];
                else
                    *reinterpret_cast<uint16_t *>(dst) = (uint16_t)code[t][0];
            }
            // the score factor of head g: softmax scale (log2 units, K scale
            // included) times 2^-e_g
            if (c == 0) f8s[g] = g < G ? p.scale_log2 * exp2i(-eg) : 0.f;
        } else {
            // q of the group as the K-major B operand (16 rows, 128-byte
            // swizzle), rows >= G zero (loaded before the set-up).  Unscaled:
            // the scale is applied to S in fp32.
#pragma unroll
            for (int j = 0; j < kQPieces; ++j) {
                const int ci = st + 128 * j;
                const int g = ci / (D / 8), c = ci % (D / 8);
                *reinterpret_cast<uint4 *>(smem + S::OFF_Q + sw128_offset(g, c * 8, kTcN * 128)) =
                    qv[j];
            }
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kQReady]);
        if constexpr (F8) softmax_bar();  // the score factors are written

        float m_run[kTcG], m_true[kTcG], l_part[kTcG], acc[kTcG], alpha_prev[kTcG];
#pragma unroll
        for (int g = 0; g < NH; ++g) {
            m_run[g] = -INFINITY;
            m_true[g] = -INFINITY;
            l_part[g] = 0.f;
            acc[g] = 0.f;
            alpha_prev[g] = 1.f;
        }
        bool failed = false;
        auto accumulate = [&](int k) -> bool {
            const int b = k & 1;
            const bool landed = mbar_wait(&bar[kOFull0 + b], (k >> 1) & 1);
            if (!__all_sync(kFullMask, landed)) return false;
            tc_fence_after();
            float o[kTcG];
            if constexpr (F8) {
                // a head's four P terms are four columns: add them, undo the
                // tile's power-of-two P scale
                // (16 columns at a time: F8G = 8, terms 0 and 1, then 2 and 3)
                float t[16];
                tmem_load16(tmem + lane_addr + S::O_COL + S::QN * b, t);
#pragma unroll
                for (int g = 0; g < NH; ++g)
                    o[g] = F8G == 8 ? t[g] + t[8 + g] : (t[g] + t[4 + g]) + (t[8 + g] + t[12 + g]);
                if constexpr (F8G == 8) {
                    tmem_load16(tmem + lane_addr + S::O_COL + S::QN * b + 16, t);
#pragma unroll
                    for (int g = 0; g < NH; ++g) o[g] += t[g] + t[8 + g];
                }
                const float *kinv = f8s + kTcG + 2 * kTcG * b;
#pragma unroll
                for (int g = 0; g < NH; ++g) o[g] *= kinv[g];
            } else {
                float t[16];
                tmem_load16(tmem + lane_addr + S::O_COL + 16 * b, t);
#pragma unroll
                for (int g = 0; g < NH; ++g) o[g] = t[g];
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[kOEmpty0 + b]);
            if constexpr (F8) {
                // (tile k's rescale factors wait in shared memory, not in
                // registers)
                const float *alpha_k = f8s + 2 * kTcG + 2 * kTcG * b;
#pragma unroll
                for (int g = 0; g < NH; ++g) acc[g] = acc[g] * alpha_k[g] + o[g];
            } else {
#pragma unroll
                for (int g = 0; g < NH; ++g) acc[g] = acc[g] * alpha_prev[g] + o[g];
            }
            return true;
        };

        float *lsum = red + 2 * (4 * kTcN);
        float *pend = reinterpret_cast<float *>(smem + S::OFF_PEND);
        // SPAN: close partition j without waiting for its last P.V: the
        // per-warp sums and the maxima go to pending buffer j & 1, and the
        // running state starts afresh (acc still takes the last O).
        auto close_partition = [&](int j) {
            float *pb = pend + (j & 1) * S::PEND_FLOATS;
#pragma unroll
            for (int g = 0; g < NH; ++g) {
                float v = l_part[g];
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(kFullMask, v, off);
                if (lane == 0) pb[sw * kTcN + g] = v;
            }
            if (st == 0) {
#pragma unroll
                for (int g = 0; g < NH; ++g) {
                    pb[4 * kTcN + g] = m_run[g];
                    pb[4 * kTcN + kTcG + g] = m_true[g];
                }
            }
#pragma unroll
            for (int g = 0; g < NH; ++g) {
                m_run[g] = -INFINITY;
                m_true[g] = -INFINITY;
                l_part[g] = 0.f;
            }
        };
        // Partial of closed partition j (acc complete), written to slot
        // part0 + j; its pending buffer was filled before a softmax barrier
        // that every thread has passed since.
        auto emit_partial = [&](int j) {
            const float *pb = pend + (j & 1) * S::PEND_FLOATS;
            if (!failed && r < D) {
#pragma unroll
                for (int g = 0; g < NH; ++g) {
                    if (g >= G) break;
                    const float lt = pb[g] + pb[kTcN + g] + pb[2 * kTcN + g] + pb[3 * kTcN + g];
                    const float mr = pb[4 * kTcN + g], mt = pb[4 * kTcN + kTcG + g];
                    const int64_t row = part_row(p, seq, kvh * G + g, part0 + j);
                    // (E4M3: V elements are v_scale times the codes)
                    p.part_o[row * D + r] = F8 ? acc[g] / lt * p.v_scale : acc[g] / lt;
                    if (r == 0) {
                        p.part_m[row] = mt;
                        p.part_l[row] = lt * fast_exp2(mr - mt);
                    }
                }
            }
        };

        // Partition by partition of the CTA's span (one partition without
        // SPAN).  Partitions but the last are closed at their end; the last
        // O of partition j is folded in, and its partial written, during
        // the first tile of partition j+1 (after that tile's P is handed to
        // the MMA), as any tile's O is during the next tile, so the pipeline
        // does not drain at partition ends.
        const int nspan = SPAN ? part_end - part0 : 1;
        for (int j = 0; j < nspan; ++j) {
            const int t_lo = SPAN ? j * tpp : 0;
            const int t_hi = SPAN ? ((j + 1) * tpp < ntiles ? (j + 1) * tpp : ntiles) : ntiles;
            for (int i = t_lo; i < t_hi; ++i) {
              const int b = i & 1;
              const bool landed = !failed && mbar_wait(&bar[kSFull0 + b], (i >> 1) & 1);
              const bool ok = __all_sync(kFullMask, landed);
              float s[16];
              if (ok) {
                  tc_fence_after();
                  if constexpr (F8) {
                      // a head's score is the sum of its four q-term columns
                      // (16 columns at a time: F8G = 8, terms 0 and 1, then 2 and 3)
                      float t[16];
                      tmem_load16(tmem + lane_addr + S::S_COL + S::QN * b, t);
  #pragma unroll
                      for (int g = 0; g < NH; ++g)
                          s[g] = F8G == 8 ? t[g] + t[8 + g] : (t[g] + t[4 + g]) + (t[8 + g] + t[12 + g]);
                      if constexpr (F8G == 8) {
                          tmem_load16(tmem + lane_addr + S::S_COL + S::QN * b + 16, t);
  #pragma unroll
                          for (int g = 0; g < NH; ++g) s[g] += t[g] + t[8 + g];
                      }
  #pragma unroll
                      for (int g = NH; g < 16; ++g) s[g] = 0.f;
                  } else {
                      tmem_load16(tmem + lane_addr + S::S_COL + 16 * b, s);
                  }
                  tc_fence_before();
                  __syncwarp();
                  if (lane == 0) mbar_arrive(&bar[kSEmpty0 + b]);
              } else {
  #pragma unroll
                  for (int g = 0; g < 16; ++g) s[g] = 0.f;
              }
              const int tile0 = start + i * kTcTile;
              const int nvalid = (end - tile0 < kTcTile) ? end - tile0 : kTcTile;
              const bool valid = r < nvalid;
              // tile max of each head over the 128 positions: a halving
              // butterfly over the warp (each exchange hands the partner the
              // heads it keeps; 9 shuffles for 8 heads), after which lane L
              // holds the warp's maximum of head (L >> 2) & 7.  The 16-bit
              // d = 128 3-D-grid variant reduces each head on its own (40
              // shuffles): the butterfly's extra live registers spill at its
              // cap.
              float *tmax = red + b * (4 * kTcN);
  #pragma unroll
              for (int g = 0; g < NH; ++g)
                  s[g] = valid ? s[g] * (F8 ? f8s[g] : p.scale_log2) : -INFINITY;
              if constexpr (!F8 && D == 128 && !SPAN && !COMPACT) {
  #pragma unroll
                  for (int g = 0; g < NH; ++g) {
                      float v = s[g];
  #pragma unroll
                      for (int off = 16; off >= 1; off >>= 1)
                          v = fmaxf(v, __shfl_xor_sync(kFullMask, v, off));
                      if (lane == 0) tmax[sw * kTcN + g] = v;
                  }
              } else if constexpr (NH == 4) {
                  // four heads: lane L ends with head (L >> 3) & 3 (5 shuffles)
                  const bool c2 = lane & 16, c1 = lane & 8;
                  float v2[2];
  #pragma unroll
                  for (int j = 0; j < 2; ++j)
                      v2[j] = fmaxf(c2 ? s[2 + j] : s[j],
                                    __shfl_xor_sync(kFullMask, c2 ? s[j] : s[2 + j], 16));
                  float v = fmaxf(c1 ? v2[1] : v2[0], __shfl_xor_sync(kFullMask, c1 ? v2[0] : v2[1], 8));
                  v = fmaxf(v, __shfl_xor_sync(kFullMask, v, 4));
                  v = fmaxf(v, __shfl_xor_sync(kFullMask, v, 2));
                  v = fmaxf(v, __shfl_xor_sync(kFullMask, v, 1));
                  if ((lane & 7) == 0) tmax[sw * kTcN + ((lane >> 3) & 3)] = v;
              } else {
                  const bool b4 = lane & 16, c2 = lane & 8, c1 = lane & 4;
                  float v4[4], v2[2];
  #pragma unroll
                  for (int j = 0; j < 4; ++j)
                      v4[j] = fmaxf(b4 ? s[4 + j] : s[j],
                                    __shfl_xor_sync(kFullMask, b4 ? s[j] : s[4 + j], 16));
  #pragma unroll
                  for (int j = 0; j < 2; ++j)
                      v2[j] = fmaxf(c2 ? v4[2 + j] : v4[j],
                                    __shfl_xor_sync(kFullMask, c2 ? v4[j] : v4[2 + j], 8));
                  float v = fmaxf(c1 ? v2[1] : v2[0], __shfl_xor_sync(kFullMask, c1 ? v2[0] : v2[1], 4));
                  v = fmaxf(v, __shfl_xor_sync(kFullMask, v, 2));
                  v = fmaxf(v, __shfl_xor_sync(kFullMask, v, 1));
                  if ((lane & 3) == 0) tmax[sw * kTcN + ((lane >> 2) & 7)] = v;
              }
              if (lane == 0) tmax[sw * kTcN + kTcN - 1] = ok ? 1.f : 0.f;  // column 15: health flag
              softmax_bar();
              bool all_ok = true;
  #pragma unroll
              for (int w = 0; w < 4; ++w) all_ok &= tmax[w * kTcN + kTcN - 1] != 0.f;
              if (!all_ok) {
                  failed = true;
                  break;
              }
              bool need = false;
              float mx[kTcG];
  #pragma unroll
              for (int g = 0; g < NH; ++g) {
                  mx[g] = fmaxf(fmaxf(tmax[g], tmax[kTcN + g]),
                                fmaxf(tmax[2 * kTcN + g], tmax[3 * kTcN + g]));
                  need |= (g < G) && (mx[g] > m_run[g] + kLazyRescale);
              }
              float alpha[kTcG];
  #pragma unroll
              for (int g = 0; g < NH; ++g) {
                  alpha[g] = 1.f;
                  if (need) {  // block-uniform
                      const float mn = fmaxf(m_run[g], mx[g]);
                      alpha[g] = fast_exp2(m_run[g] - mn);
                      m_run[g] = mn;
                      l_part[g] *= alpha[g];
                  }
                  m_true[g] = fmaxf(m_true[g], mx[g]);
              }
              uint8_t *pbuf = smem + S::OFF_P + b * S::P_BYTES;
              if constexpr (F8) {
                  // P^T as E5M2 terms: head g's P times 2^k_g, the power of
                  // two that brings the head's largest P of the tile into
                  // [2^14, 2^15), rounded to f16 (11 significant bits), then
                  // split like q into four terms, rows t * F8G + g, 128
                  // positions of one byte (K-major, 128-byte swizzle).  The
                  // terms keep every value down to E5M2's subnormal range
                  // (2^-30 of the tile's largest) exactly; the sum l takes the
                  // unscaled P, and the tile's O columns are scaled back by
                  // 2^-k_g.  Rows of absent heads are left as they are: they
                  // only reach O columns that are never read.
                  float *kinv = f8s + kTcG + 2 * kTcG * b;
  #pragma unroll
                  for (int g = 0; g < NH; ++g) kinv[kTcG + g] = alpha[g];  // (same remark)
  #pragma unroll
                  for (int g = 0; g < NH; g += 2) {
                      if (g >= G) break;
                      float pp[2];
  #pragma unroll
                      for (int h = 0; h < 2; ++h) {
                          float pg = 0.f, ki = 1.f;
                          if (g + h < G) {
                              pg = fast_exp2(s[g + h] - m_run[g + h]);  // masked: 2^-inf = 0
                              l_part[g + h] += pg;
                              const float dm = mx[g + h] - m_run[g + h];  // <= the lazy threshold
                              int k = 0;
                              if (dm > -INFINITY) {
                                  k = 14 - __float2int_rd(dm);
                                  k = k > 126 ? 126 : k;
                              }
                              pg *= exp2i(k);  // exact: a power of two
                              ki = exp2i(-k);
                          }
                          pp[h] = pg;
                          // (every softmax thread stores the same value, and
                          // reads it back after its own store)
                          kinv[g + h] = ki;
                      }
                      uint32_t hv = narrow2<false>(pp[0], pp[1]);
  #pragma unroll
                      for (int t = 0; t < 4; ++t) {
                          const uint32_t cd = e5m2x2_from_f16x2(hv);
                          hv = hsub2_bits(hv, f16x2_from_e5m2x2((uint16_t)cd));  // exact
                          pbuf[e4m3_operand_offset<128>(F8G * t + g, r)] = (uint8_t)(cd & 0xffu);
                          pbuf[e4m3_operand_offset<128>(F8G * t + g + 1, r)] = (uint8_t)(cd >> 8);
                      }
                  }
              } else {
                  // P^T (16 rows = heads, 128 positions) in the operand layout
  #pragma unroll
                  for (int g = 0; g < kTcN; ++g) {
                      float pv = 0.f;
                      if (g < kTcG && g < G) {
                          pv = fast_exp2(s[g] - m_run[g]);  // masked: 2^-inf = 0
                          l_part[g] += pv;
                      }
                      *reinterpret_cast<uint16_t *>(pbuf + sw128_offset(g, r, kTcN * 128)) =
                          narrow1<BF16>(pv);
                  }
              }
              if (!valid) {
                  // Stale rows of the last tile: V must be finite there (0 * NaN
                  // would poison the product), so zero the row once it has landed.
                  // The V stage's previous tile (i - NV) has been consumed
                  // (the MMA issuer holds back q.K^T of the last tile until every
                  // earlier P.V is issued, and tile i's copy waited for that
                  // P.V to finish), so the parity wait below can only mean tile
                  // i's phase.
                  const int vs = i % S::NV;
                  if (mbar_wait(&bar[S::VFULL + vs], (i / S::NV) & 1)) {
                      // (a swizzle only permutes the 16-byte chunks within a row)
                      if constexpr (F8) {
                          uint4 *row = reinterpret_cast<uint4 *>(smem + S::OFF_V + vs * S::STAGE +
                                                                 r * D);
  #pragma unroll
                          for (int c = 0; c < D / 16; ++c) row[c] = make_uint4(0, 0, 0, 0);
                      } else {
  #pragma unroll
                          for (int h = 0; h < S::KH; ++h) {
                              uint4 *row = reinterpret_cast<uint4 *>(
                                  smem + S::OFF_V + vs * S::STAGE + h * S::SLAB + r * 128);
  #pragma unroll
                              for (int c = 0; c < 8; ++c) row[c] = make_uint4(0, 0, 0, 0);
                          }
                      }
                  } else {
                      failed = true;
                  }
              }
              fence_async_smem();
              __syncwarp();
              if (lane == 0) mbar_arrive(&bar[kPFull0 + b]);
              if (i > t_lo) {
                  if (!accumulate(i - 1)) failed = true;
              } else if (SPAN && j > 0) {
                  // partition j-1: its last O, its partial, a fresh acc
                  if (!failed && !accumulate(i - 1)) failed = true;
                  emit_partial(j - 1);
  #pragma unroll
                  for (int g = 0; g < NH; ++g) acc[g] = 0.f;
              }
  #pragma unroll
              for (int g = 0; g < NH; ++g) alpha_prev[g] = alpha[g];
            }
            if (SPAN && j + 1 < nspan)
                close_partition(j);
            else if (!failed && !accumulate(t_hi - 1))
                failed = true;
        }

        // l over the 128 position-threads, per head
#pragma unroll
        for (int g = 0; g < NH; ++g) {
            float v = l_part[g];
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(kFullMask, v, off);
            if (lane == 0) lsum[sw * kTcN + g] = v;
        }
        softmax_bar();
        if (merge_prefix && !failed) {
            const bool ready = mbar_wait(&bar[kPreReady], 0);
            if (!__all_sync(kFullMask, ready)) failed = true;
        }
        if (failed) {
            if (st == 0) {
                record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
            }
        } else if (r < D) {
#pragma unroll
            for (int g = 0; g < NH; ++g) {
                if (g >= G) break;
                const float lt =
                    lsum[g] + lsum[kTcN + g] + lsum[2 * kTcN + g] + lsum[3 * kTcN + g];
                float o = F8 ? acc[g] / lt * p.v_scale : acc[g] / lt;
                const int h = kvh * G + g;
                if (merge_prefix) {
                    // softmax over prefix and tail: the two partials' log-sum-exp merge
                    const float Mp = pre[kTcG * D + g], Lp = pre[kTcG * D + kTcG + g];
                    const float M = fmaxf(m_run[g], Mp);
                    const float wo = fast_exp2(m_run[g] - M);
                    const float wp = (Mp == -INFINITY) ? 0.f : Lp * fast_exp2(Mp - M);
                    o = (acc[g] * wo + wp * pre[g * D + r]) / (lt * wo + wp);
                }
                if (direct) {
                    uint16_t *out = static_cast<uint16_t *>(p.out);
                    out[((int64_t)seq * p.num_q_heads + h) * D + r] = narrow1<BF16>(o);
                } else {
                    const int64_t row = part_row(p, seq, h, part_end - 1);
                    p.part_o[row * D + r] = o;
                    if (r == 0) {
                        p.part_m[row] = m_true[g];
                        p.part_l[row] = lt * fast_exp2(m_run[g] - m_true[g]);
                    }
                }
            }
        }
    }

    if (SPAN && p.mode == 1) {
        // split-KV partitions on their own: the span's partitions past the
        // sequence's end hold the empty partial (-inf, 0, 0)
        for (int j = part_end; j < part0 + R && j < p.num_partitions; ++j)
            for (int g = 0; g < G; ++g) {
                const int64_t row = part_row(p, seq, kvh * G + g, j);
                if (threadIdx.x == 0) {
                    p.part_m[row] = -INFINITY;
                    p.part_l[row] = 0.f;
                }
                for (int x = threadIdx.x; x < D; x += blockDim.x) p.part_o[row * D + x] = 0.f;
            }
    }
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    const bool aborted = *abort_flag != 0;
    if (aborted && threadIdx.x == 0) {
        // let copies and MMAs still in flight finish before shared memory and
        // TMEM are released (each wait is bounded)
        for (int ks = 0; ks < S::NK && ks < ntiles; ++ks) {
            const int tl = ks + S::NK * ((ntiles - 1 - ks) / S::NK);  // last tile of stage ks
            (void)mbar_wait(&bar[S::KFULL + ks], (tl / S::NK) & 1);
        }
        for (int vs = 0; vs < S::NV && vs < ntiles; ++vs) {
            const int tl = vs + S::NV * ((ntiles - 1 - vs) / S::NV);  // last tile of stage vs
            (void)mbar_wait(&bar[S::VFULL + vs], (tl / S::NV) & 1);
            (void)mbar_wait(&bar[S::VEMPTY + vs], (tl / S::NV) & 1);
        }
    }
    if (aborted) return false;
    if (!direct && (p.counters != nullptr || p.prefix_parts > 0)) {
        pdl_wait();  // a cascade tail's combine reads the prefix's partials
        finish_item<BF16, D>(p, seq, kvh, nparts_seq, part, (nparts_seq + R - 1) / R, use_flags,
                             reinterpret_cast<float *>(smem), S::OFF_Q);
    }
    if (another && threadIdx.x == 0) {
        // the last stages' release arrivals (MMA commits nobody waited for)
        // land before the barriers are set up again for the CTA's next item
        for (int ks = 0; ks < S::NK && ks < ntiles; ++ks) {
            const int tl = ks + S::NK * ((ntiles - 1 - ks) / S::NK);
            (void)mbar_wait(&bar[S::KEMPTY + ks], (tl / S::NK) & 1);
        }
        for (int vs = 0; vs < S::NV && vs < ntiles; ++vs) {
            const int tl = vs + S::NV * ((ntiles - 1 - vs) / S::NV);
            (void)mbar_wait(&bar[S::VEMPTY + vs], (tl / S::NV) & 1);
        }
    }
    return true;
    };  // process

    if constexpr (COMPACT && SPAN) {
        // (several partitions a CTA serve long batches, whose compact grids
        // are never capped: one item a CTA)
        int seq = 0, part = 0, kvh = 0;
        if (compact_item(p, blockIdx.x, &seq, &part, &kvh))
            (void)process(seq, part, kvh, false, false);
    } else if constexpr (COMPACT) {
        // Compact grid: CTA b takes items b, b + gridDim.x, ... in order
        // (more than one when the grid was capped at the resident slots).
        // When the grid is resident at once (p.one_wave) and every item has
        // its own CTA, the combine may use ready flags.
        // (the lengths wait in shared memory while an item runs: no registers
        // held across it)
        int *lens_smem = reinterpret_cast<int *>(smem + S::OFF_LENS);
        int seq = 0, part = 0, kvh = 0, total = 0;
        bool more;
        {
            int len[kCompactGroups];
            compact_lens(p, len);
            more = compact_find(p, len, blockIdx.x, &seq, &part, &kvh, &total);
            if (warp == 0) {
#pragma unroll
                for (int k = 0; k < kCompactGroups; ++k) lens_smem[32 * k + lane] = len[k];
            }
        }
        const bool use_flags = p.one_wave && total <= (int)gridDim.x;
        for (int c = blockIdx.x;
             more && process(seq, part, kvh, use_flags, c + (int)gridDim.x < total);) {
            c += gridDim.x;
            more = c < total;
            if (more) {
                int len[kCompactGroups];
#pragma unroll
                for (int k = 0; k < kCompactGroups; ++k) len[k] = lens_smem[32 * k + lane];
                more = compact_find(p, len, c, &seq, &part, &kvh, &total);
            }
        }
    } else {
        (void)process(blockIdx.z, blockIdx.x, blockIdx.y, p.one_wave != 0, false);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(*tmem_slot, S::COLS);
    }
}

// ------------------------------------------------------------------ host side
using TcKernel = void (*)(const DecodeParams, const CUtensorMap, const CUtensorMap);

// Resident CTAs per SM of a variant (shared memory, registers, TMEM columns).
int tc_occupancy(TcKernel k, int smem, int tmem_cols);

// The E4M3 variant for head size D (64 or 128) and E4M3 operands of F8G
// heads (4 or 8): its kernel, shared memory and TMEM columns.  Each F8G's
// variants are instantiated in their own translation unit.
template <int F8G>
TcKernel tc8_pick(bool bf16, int D, bool span, bool compact, int *smem, int *cols) {
    auto v = [&](auto d_const) -> TcKernel {
        constexpr int DD = decltype(d_const)::value;
        *smem = TcShape<DD, F8G>::SMEM_BYTES;
        *cols = TcShape<DD, F8G>::COLS;
        if (span)
            return compact ? (bf16 ? paged_decode_tc_kernel<true, DD, true, true, F8G>
                                   : paged_decode_tc_kernel<false, DD, true, true, F8G>)
                           : (bf16 ? paged_decode_tc_kernel<true, DD, true, false, F8G>
                                   : paged_decode_tc_kernel<false, DD, true, false, F8G>);
        return compact ? (bf16 ? paged_decode_tc_kernel<true, DD, false, true, F8G>
                               : paged_decode_tc_kernel<false, DD, false, true, F8G>)
                       : (bf16 ? paged_decode_tc_kernel<true, DD, false, false, F8G>
                               : paged_decode_tc_kernel<false, DD, false, false, F8G>);
    };
    return D == 128 ? v(std::integral_constant<int, 128>{}) : v(std::integral_constant<int, 64>{});
}
TcKernel tc8_pick4(bool bf16, int D, bool span, bool compact, int *smem, int *cols);
TcKernel tc8_pick8(bool bf16, int D, bool span, bool compact, int *smem, int *cols);

// Launch of a variant over the pools' tensor maps: the grid of decode_grid,
// compact grids capped at the resident slots when that keeps them within
// four waves.
pa_status launch_tc_kernel(TcKernel k, int smem, int ctas_per_sm, const DecodeParams &prm,
                           const CUtensorMap &mk, const CUtensorMap &mv, int num_partitions,
                           int num_kv_heads, int num_seqs, cudaStream_t stream);

}  // namespace pa
