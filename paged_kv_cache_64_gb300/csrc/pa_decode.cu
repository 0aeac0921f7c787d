// Paged decode attention for GB300 (sm_103a): pa_decode, pa_decode_partitions,
// pa_split_kv_reduce.
//
// What is computed (the pages' definition): for sequence i, query head h,
// KV head kv = h / G, positions p < L_i gathered through the block table,
//   out = softmax(scale * q K^T) V
// walked in tiles with a running maximum and sum ("PagedAttention: Treating
// KV Memory Like Virtual Memory", "How the kernel reads a block table";
// "PagedAttention and Virtual Memory Management ..." (llms.blog) section 4,
// "Fused PagedAttention Algorithm"), optionally split into partitions whose
// (m, l, O) partials are combined by a second kernel (same section,
// "Parallel Partitioning Across GPU Warps", steps 2 and 3).
//
// Design (GB300-first, HBM-bound: about G flops per byte of K/V):
//  * One CTA per (partition, KV head, sequence): 4 consumer warps + 1
//    producer warp.  Every query head of the KV head's group is served from
//    the same K/V bytes, so each K/V tile is read from HBM exactly once.
//  * Pipeline stage = 16 consecutive positions of one (block, KV head): a
//    contiguous 16*d*2-byte run in the [block][head][slot][dim] pool, moved
//    by one 1-D bulk copy (TMA engine) for K and one for V into a ring of
//    shared-memory stages, completion tracked by mbarrier transaction bytes.
//    The producer warp reads the block table 32 entries at a time
//    (coalesced) and translates each stage's position: physical block =
//    table[pos >> log2(B)], slot offset = pos & (B - 1).
//  * Consumer warp w takes stages w, w+4, ...  Inside a warp, LT lanes share
//    one token (LT = 8, or 16 when G*d is large); a lane owns d/LT dims in
//    whole 16-byte pieces, so each group of 8 lanes reads one 128-byte
//    row segment: bank-conflict-free LDS.128.
//  * q (pre-scaled by scale*log2 e) lives in registers; dot products use
//    packed fp32x2 FMA (FFMA2); partial sums are combined with a butterfly of
//    warp shuffles; the softmax is base 2 (ex2.approx).
//  * Online softmax with a lazy rescale: the running max m only moves when a
//    new tile's max exceeds it by more than 8 (base-2 units), so the
//    accumulator is rescaled rarely; exp2(s - m) <= 256 keeps fp32 far from
//    overflow.  The true max is tracked separately for the partial outputs.
//  * Masked positions (past L_i in a partial last stage) get score -inf and
//    their V values are replaced by zero with a select, never multiplied
//    by a zero weight, so NaN/Inf in stale slots cannot leak.
//  * Each warp keeps its own (m, l, acc); at the end warps are merged through
//    shared memory with the same rescaling as the cross-partition combine.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>
#include <utility>

#include "pa_common.cuh"
#include "pa_decode.cuh"
#include "pa_internal.h"

namespace pa {

constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;

constexpr int ilog2c(int x) { return x <= 1 ? 0 : 1 + ilog2c(x / 2); }

// Tuning of the G = 8 instantiations (compile-time; defaults measured on
// GB300): heads whose q stays in registers, register cap, rows per chunk,
// ring size.  Other G: q in registers, 168-register cap, 96 KiB ring.
#ifndef PA_G8_QREG
#define PA_G8_QREG 4
#endif
#ifndef PA_G8_MAXREGS
#define PA_G8_MAXREGS 168
#endif
#ifndef PA_G8_ROWS
#define PA_G8_ROWS 1
#endif
#ifndef PA_G8_RING_KB
#define PA_G8_RING_KB 96
#endif
#ifndef PA_RING_KB
#define PA_RING_KB 96
#endif
constexpr int QREG8 = PA_G8_QREG;  // heads whose q stays in registers when G = 8

template <int D, int GP>
struct DecodeShape {
    static constexpr int LT = D / 8;                        // lanes per token: 8 dims each
    static constexpr int TPR = 32 / LT;                     // tokens per warp row
    static constexpr int ROWS = kUnit / TPR;                // rows per stage
    static constexpr int R0 = (GP >= 8) ? PA_G8_ROWS : 16 / GP;  // rows per chunk
    static constexpr int R = (R0 < 1) ? 1 : (R0 > ROWS ? ROWS : R0);
    static constexpr int CHUNKS = ROWS / R;
    static constexpr int NV = R * GP;                       // partial scores per lane
    static constexpr int L2LT = ilog2c(LT), L2NV = ilog2c(NV), L2GP = ilog2c(GP);
    static constexpr int LEVELS = L2LT < L2NV ? L2LT : L2NV;  // reduce-scatter levels
    static constexpr int K = NV >> LEVELS;                  // complete sums kept per lane
    static constexpr int L2K = ilog2c(K);
    static constexpr int SHIFT = L2LT - LEVELS;             // low lane bits: butterfly copies
    static constexpr int TILE_BYTES = kUnit * D * 2;        // one of K or V
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    // Ring of stages: 96 KiB, so that two CTAs share an SM.
    static constexpr int NS = ((GP >= 8) ? PA_G8_RING_KB : PA_RING_KB) * 1024 / STAGE_BYTES;
    static constexpr int RING_BYTES = NS * STAGE_BYTES;
    // q of heads QREG.. lives in shared memory (fp32, pre-scaled) instead of
    // registers, to keep G = 8 under the register cap.
    static constexpr int QREG = (GP >= 8) ? QREG8 : GP;
    static constexpr int QS_OFF = (RING_BYTES + 2 * NS * 8 + 16 + 15) / 16 * 16;
    static constexpr int QS_BYTES = (GP - QREG) * D * 4;
    static constexpr int SMEM_BYTES = QS_OFF + QS_BYTES;
    static_assert(NS % kConsumerWarps == 0, "stages are dealt to warps round robin");
    static_assert(ROWS % R == 0, "chunking");
    static_assert(K <= GP, "a lane's sums belong to one row");
    static_assert(kConsumerWarps * GP * D * 4 + 3 * kConsumerWarps * GP * 4 <= RING_BYTES,
                  "merge scratch must fit in the ring");
    static_assert(2 * 8 * kCombineMaxParts * 4 <= RING_BYTES, "combine scratch must fit in the ring");
};


// Reduce-scatter of NV partial sums over an LT-lane group (lane c in the
// group): after the call, v[0 .. NV >> LEVELS) of lane c hold the complete
// sums of indices ((c >> (log2 LT - LEVELS)) << log2 K) + j.  Each level
// halves the values a lane keeps, trading half with its partner; when NV < LT
// the last levels are a plain butterfly (lanes end with copies).
template <int NV, int LT, int LEVELS>
__device__ __forceinline__ void reduce_scatter(float (&v)[NV], int c) {
#pragma unroll
    for (int lvl = 0; lvl < LEVELS; ++lvl) {
        const int o = LT >> (lvl + 1);
        const int half = NV >> (lvl + 1);
        const bool up = (c & o) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = up ? v[i] : v[i + half];
            const float keep = up ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(kFullMask, send, o);
        }
    }
#pragma unroll
    for (int o = LT >> (LEVELS + 1); o >= 1; o >>= 1) {
#pragma unroll
        for (int j = 0; j < (NV >> LEVELS); ++j) v[j] += __shfl_xor_sync(kFullMask, v[j], o);
    }
}

// Shared-memory load the compiler may not hoist out of the token loop (a
// hoisted copy would put the q of every head back into registers).
__device__ __forceinline__ float4 lds_f4(const float *p) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

// Register cap: <= 168 per thread lets two 5-warp CTAs share an SM (a warp's
// registers come from one of the four 16K-register sub-partitions).
template <int GP>
constexpr int decode_max_regs() { return GP >= 8 ? PA_G8_MAXREGS : 168; }

template <bool BF16, int D, int GP>
__global__ void __launch_bounds__(kDecodeThreads) __maxnreg__(decode_max_regs<GP>())
    paged_decode_kernel(const DecodeParams p) {
    using S = DecodeShape<D, GP>;
    constexpr int LT = S::LT, TPR = S::TPR, R = S::R;
    constexpr int NS = S::NS;

    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *ring = smem;
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + S::RING_BYTES);
    uint64_t *empty_bar = full_bar + NS;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty_bar + NS);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = p.group;
    const int P = p.partition_tokens;

    pdl_wait();  // inputs may come from the previous kernel on the stream
    int part, kvh, seq;  // partition, KV head, sequence
    if (p.compact) {
        if (!compact_item(p, blockIdx.x, &seq, &part, &kvh)) return;  // past the last item
    } else {
        part = blockIdx.x;
        kvh = blockIdx.y;
        seq = blockIdx.z;
    }
    const int L = item_len(p, seq, threadIdx.x == 0 && part == 0 && kvh == 0);
    const int nparts_seq = L == 0 ? 0 : (L - 1) / P + 1;
    const int start = part * P;

    if (start >= L) {
        // Empty partition.  Mode 0: the zero-length sequence's output row is
        // zeros (written by partition 0); nothing else is ever read.  Mode 1:
        // write the empty partial (m = -inf, l = 0, O = 0).  Empty cascade
        // tail: the output is the prefix's partials combined.
        if (p.prefix_parts > 0) {
            if (nparts_seq == 0 && part == 0)
                finish_item<BF16, D>(p, seq, kvh, 0, 0, 1, false, reinterpret_cast<float *>(smem),
                                     S::RING_BYTES);
        } else if (p.mode == 0) {
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
    // a cascade tail writes its partial and merges it with the prefix's
    const bool direct = (p.mode == 0) && (nparts_seq <= 1) && (p.prefix_parts == 0);

    if (p.k_new != nullptr && part == nparts_seq - 1) fused_cache_write<D>(p, seq, kvh, L);
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        *abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();

    // Consumer lanes' softmax state, kept across the final barrier.  After
    // the reduce-scatter a lane owns K complete scores per chunk: heads
    // h0 .. h0+K-1 of one row; slot j of m_run / m_true / l_run is head h0+j.
    constexpr int K = S::K, L2K = S::L2K, SHIFT = S::SHIFT, NV = S::NV;
    constexpr int L2LT = S::L2LT, L2GP = S::L2GP;
    constexpr int ROWBIT0 = SHIFT + L2GP - L2K;  // first lane bit that changes the row
    float m_run[K], m_true[K], l_run[K];
    float2 acc[GP][4];  // the lane's 8 dims, every head of the group
    const int tg = lane / LT;                    // token group within a warp row
    const int c = lane % LT;                     // lane in the group: dims [8c, 8c+8)
    const int vbase = (c >> SHIFT) << L2K;       // first score index v = row*GP + head
    const int my_row = vbase / GP;
    const int h0 = vbase % GP;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer
        const int64_t tile_elems = (int64_t)kUnit * D;
        const int64_t head_elems = (int64_t)p.block_size * D;
        const int64_t block_elems = (int64_t)p.num_kv_heads * head_elems;
        const int32_t *table = seq_table(p, seq);
        bool ok = true;
        for (int u0 = 0; u0 < nunits && ok; u0 += 32) {
            const int u = u0 + lane;
            int phys = 0;
            if (u < nunits) {
                const int pos = start + u * kUnit;
                phys = table[pos >> p.log2_block];
                if ((unsigned)phys >= (unsigned)p.num_blocks) {
                    record_error(p.err, PA_ERR_BAD_INDEX);
                    phys = 0;
                }
            }
            const int cnt = (nunits - u0 < 32) ? nunits - u0 : 32;
            for (int j = 0; j < cnt; ++j) {
                const int uu = u0 + j;
                const int ph = __shfl_sync(kFullMask, phys, j);
                const int stage = uu % NS;
                if (uu >= NS) {
                    // every lane waits; the outcome is made warp-uniform
                    const bool done = mbar_wait(&empty_bar[stage], ((uu / NS) - 1) & 1);
                    if (!__all_sync(kFullMask, done)) {
                        ok = false;
                        break;
                    }
                }
                if (lane == 0) {
                    const int pos = start + uu * kUnit;
                    const int off = pos & (p.block_size - 1);
                    const int64_t elem = (int64_t)ph * block_elems + (int64_t)kvh * head_elems +
                                         (int64_t)off * D;
                    uint8_t *dst = ring + stage * S::STAGE_BYTES;
                    mbar_arrive_expect_tx(&full_bar[stage], 2 * S::TILE_BYTES);
                    bulk_copy_g2s(dst, p.k_pool + elem, S::TILE_BYTES, &full_bar[stage]);
                    bulk_copy_g2s(dst + S::TILE_BYTES, p.v_pool + elem, S::TILE_BYTES,
                                  &full_bar[stage]);
                }
                __syncwarp();
            }
            (void)tile_elems;
        }
        if (!ok && lane == 0) {
            record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
        }
    } else {
        // ------------------------------------------------------ consumers
        const int gbase = tg * LT;
        constexpr int QREG = S::QREG;
        // q of heads >= QREG: fp32 copy in shared memory, filled once
        float *qs = reinterpret_cast<float *>(smem + S::QS_OFF);
        if constexpr (QREG < GP) {
            for (int i = threadIdx.x; i < (GP - QREG) * (D / 8); i += kConsumerWarps * 32) {
                const int g = QREG + i / (D / 8);
                const int x0 = (i % (D / 8)) * 8;
                float f8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                if (g < G) {
                    const uint4 raw = *reinterpret_cast<const uint4 *>(
                        p.q + ((int64_t)seq * p.num_q_heads + (int64_t)kvh * G + g) * D + x0);
                    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 f = widen2<BF16>(w[k]);
                        f8[2 * k] = f.x * p.scale_log2;
                        f8[2 * k + 1] = f.y * p.scale_log2;
                    }
                }
                float4 *dst = reinterpret_cast<float4 *>(qs + (g - QREG) * D + x0);
                dst[0] = make_float4(f8[0], f8[1], f8[2], f8[3]);
                dst[1] = make_float4(f8[4], f8[5], f8[6], f8[7]);
            }
            asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
        }
        float2 q2[QREG > 0 ? QREG : 1][4];  // q of heads < QREG, scaled to base 2
#pragma unroll
        for (int g = 0; g < QREG; ++g) {
            if (g < G) {
                const uint16_t *qrow =
                    p.q + ((int64_t)seq * p.num_q_heads + (int64_t)kvh * G + g) * D;
                const uint4 raw = *reinterpret_cast<const uint4 *>(qrow + c * 8);
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 f = widen2<BF16>(w[k]);
                    q2[g][k] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
                }
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) q2[g][k] = make_float2(0.f, 0.f);
            }
        }
#pragma unroll
        for (int g = 0; g < GP; ++g)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[g][k] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < K; ++j) {
            m_run[j] = -INFINITY;
            m_true[j] = -INFINITY;
            l_run[j] = 0.f;
        }

        for (int u = warp; u < nunits; u += kConsumerWarps) {
            const int stage = u % NS;
            const bool landed = mbar_wait(&full_bar[stage], (u / NS) & 1);
            if (!__all_sync(kFullMask, landed)) {
                if (lane == 0) {
                    record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
                    *abort_flag = 1;
                }
                break;
            }
            const uint8_t *kt = ring + stage * S::STAGE_BYTES;
            const uint8_t *vt = kt + S::TILE_BYTES;
            const int nvalid = end - (start + u * kUnit);  // >= 1
            const bool partial = nvalid < kUnit;

#pragma unroll
            for (int ch = 0; ch < S::CHUNKS; ++ch) {
                // ---- partial dot products over the lane's 8 dims
                float sv[NV];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int t = (ch * R + r) * TPR + tg;
                    const uint4 raw = *reinterpret_cast<const uint4 *>(kt + t * D * 2 + c * 16);
                    const float2 k2[4] = {widen2<BF16>(raw.x), widen2<BF16>(raw.y),
                                          widen2<BF16>(raw.z), widen2<BF16>(raw.w)};
#pragma unroll
                    for (int g = 0; g < GP; ++g) {
                        float2 qg[4];
                        if (g < QREG) {
#pragma unroll
                            for (int k = 0; k < 4; ++k) qg[k] = q2[g < QREG ? g : 0][k];
                        } else {
                            const float4 a0 = lds_f4(qs + (g - QREG) * D + c * 8);
                            const float4 a1 = lds_f4(qs + (g - QREG) * D + c * 8 + 4);
                            qg[0] = make_float2(a0.x, a0.y);
                            qg[1] = make_float2(a0.z, a0.w);
                            qg[2] = make_float2(a1.x, a1.y);
                            qg[3] = make_float2(a1.z, a1.w);
                        }
                        float2 a = __fmul2_rn(qg[0], k2[0]);
                        a = __ffma2_rn(qg[1], k2[1], a);
                        a = __ffma2_rn(qg[2], k2[2], a);
                        a = __ffma2_rn(qg[3], k2[3], a);
                        sv[r * GP + g] = a.x + a.y;
                    }
                }
                // ---- complete sums: lane keeps scores vbase .. vbase+K-1
                reduce_scatter<NV, LT, S::LEVELS>(sv, c);
                if (partial && (ch * R + my_row) * TPR + tg >= nvalid) {
#pragma unroll
                    for (int j = 0; j < K; ++j) sv[j] = -INFINITY;
                }
                // ---- tile max of each head over the warp; lazy rescale
                float mx[K];
                bool need = false;
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    float v = sv[j];
#pragma unroll
                    for (int b = ROWBIT0; b < L2LT; ++b)
                        v = fmaxf(v, __shfl_xor_sync(kFullMask, v, 1 << b));
#pragma unroll
                    for (int o = LT; o < 32; o <<= 1) v = fmaxf(v, __shfl_xor_sync(kFullMask, v, o));
                    mx[j] = v;
                    m_true[j] = fmaxf(m_true[j], v);
                    need |= v > m_run[j] + kLazyRescale;
                }
                if (__any_sync(kFullMask, need)) {
                    float al[K];
#pragma unroll
                    for (int j = 0; j < K; ++j) {
                        const float mn = fmaxf(m_run[j], mx[j]);
                        al[j] = fast_exp2(m_run[j] - mn);
                        m_run[j] = mn;
                        l_run[j] *= al[j];
                    }
#pragma unroll
                    for (int g = 0; g < GP; ++g) {
                        // lane (g >> L2K) << SHIFT holds head g in slot g % K
                        const float a = __shfl_sync(kFullMask, al[g & (K - 1)], (g >> L2K) << SHIFT);
                        const float2 a2 = make_float2(a, a);
#pragma unroll
                        for (int k = 0; k < 4; ++k) acc[g][k] = __fmul2_rn(acc[g][k], a2);
                    }
                }
                float pj[K];
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    pj[j] = fast_exp2(sv[j] - m_run[j]);  // masked: 2^-inf = 0
                    l_run[j] += pj[j];
                }
                // ---- P.V: every lane gathers the weights of its token group
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int t = (ch * R + r) * TPR + tg;
                    uint4 raw = *reinterpret_cast<const uint4 *>(vt + t * D * 2 + c * 16);
                    if (partial && t >= nvalid) raw = make_uint4(0u, 0u, 0u, 0u);
                    const float2 v2[4] = {widen2<BF16>(raw.x), widen2<BF16>(raw.y),
                                          widen2<BF16>(raw.z), widen2<BF16>(raw.w)};
#pragma unroll
                    for (int g = 0; g < GP; ++g) {
                        const int v = r * GP + g;
                        const float pr =
                            __shfl_sync(kFullMask, pj[v & (K - 1)], gbase + ((v >> L2K) << SHIFT));
                        const float2 pp = make_float2(pr, pr);
#pragma unroll
                        for (int k = 0; k < 4; ++k) acc[g][k] = __ffma2_rn(pp, v2[k], acc[g][k]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[stage]);
        }

        // Sum the token groups' accumulators (they share m_run), and each
        // head's l over the lanes that hold it.
#pragma unroll
        for (int o = LT; o < 32; o <<= 1) {
#pragma unroll
            for (int g = 0; g < GP; ++g)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    acc[g][k].x += __shfl_xor_sync(kFullMask, acc[g][k].x, o);
                    acc[g][k].y += __shfl_xor_sync(kFullMask, acc[g][k].y, o);
                }
        }
#pragma unroll
        for (int j = 0; j < K; ++j) {
#pragma unroll
            for (int b = ROWBIT0; b < L2LT; ++b)
                l_run[j] += __shfl_xor_sync(kFullMask, l_run[j], 1 << b);
#pragma unroll
            for (int o = LT; o < 32; o <<= 1) l_run[j] += __shfl_xor_sync(kFullMask, l_run[j], o);
        }
    }

    pdl_trigger();
    __syncthreads();  // ring drained: every issued copy was waited on by a consumer
    if (*abort_flag) {
        // A bounded wait ran out.  Let any copy still in flight land before
        // the CTA's shared memory is released, then stop.
        if (threadIdx.x == 0) {
            for (int s = 0; s < NS; ++s) {
                const int issued = (nunits - s + NS - 1) / NS;  // upper bound of phases
                if (issued > 0) (void)mbar_wait(&full_bar[s], (issued - 1) & 1);
            }
        }
        return;
    }

    // ---------------------------------------------------------- warp merge
    float *red_acc = reinterpret_cast<float *>(ring);                  // [W][GP][D]
    float *red_m = red_acc + kConsumerWarps * GP * D;                  // [W][GP]
    float *red_l = red_m + kConsumerWarps * GP;
    float *red_t = red_l + kConsumerWarps * GP;
    if (warp < kConsumerWarps) {
        if (tg == 0) {
#pragma unroll
            for (int g = 0; g < GP; ++g) {
                float4 *dst = reinterpret_cast<float4 *>(red_acc + (warp * GP + g) * D + c * 8);
                dst[0] = make_float4(acc[g][0].x, acc[g][0].y, acc[g][1].x, acc[g][1].y);
                dst[1] = make_float4(acc[g][2].x, acc[g][2].y, acc[g][3].x, acc[g][3].y);
            }
            if (my_row == 0 && (c & ((1 << SHIFT) - 1)) == 0) {
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    red_m[warp * GP + h0 + j] = m_run[j];
                    red_l[warp * GP + h0 + j] = l_run[j];
                    red_t[warp * GP + h0 + j] = m_true[j];
                }
            }
        }
    }
    __syncthreads();

    constexpr int kPer = 8;  // outputs per thread
    for (int item = threadIdx.x; item < G * (D / kPer); item += blockDim.x) {
        const int g = item / (D / kPer);
        const int x0 = (item % (D / kPer)) * kPer;
        float M = -INFINITY, MT = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            M = fmaxf(M, red_m[w * GP + g]);
            MT = fmaxf(MT, red_t[w * GP + g]);
        }
        float f[kConsumerWarps];
        float lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            f[w] = fast_exp2(red_m[w * GP + g] - M);  // empty warp: exp2(-inf) = 0
            lsum += f[w] * red_l[w * GP + g];
        }
        const float inv = 1.0f / lsum;
        float o[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            float a = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) a += f[w] * red_acc[(w * GP + g) * D + x0 + k];
            o[k] = a * inv;
        }
        const int h = kvh * G + g;
        if (direct) {
            uint4 packed = make_uint4(narrow2<BF16>(o[0], o[1]), narrow2<BF16>(o[2], o[3]),
                                      narrow2<BF16>(o[4], o[5]), narrow2<BF16>(o[6], o[7]));
            uint16_t *out = static_cast<uint16_t *>(p.out);
            *reinterpret_cast<uint4 *>(out + ((int64_t)seq * p.num_q_heads + h) * D + x0) = packed;
        } else {
            const int64_t row = part_row(p, seq, h, part);
            if (x0 == 0) {
                p.part_m[row] = MT;
                p.part_l[row] = lsum * fast_exp2(M - MT);
            }
            float4 *dst = reinterpret_cast<float4 *>(p.part_o + row * D + x0);
            dst[0] = make_float4(o[0], o[1], o[2], o[3]);
            dst[1] = make_float4(o[4], o[5], o[6], o[7]);
        }
    }
    if (!direct && (p.counters != nullptr || p.prefix_parts > 0))
        finish_item<BF16, D>(p, seq, kvh, nparts_seq, part, nparts_seq, false,
                             reinterpret_cast<float *>(smem), S::RING_BYTES);
}

// ------------------------------------------------------------------ reduce
struct ReduceParams {
    void *out;
    const float *part_m;
    const float *part_l;
    const float *part_o;
    const int32_t *seq_lens;
    int *err;
    int num_seqs;
    int num_q_heads;
    int max_seq_len;
    int partition_tokens;
    int num_partitions;
    int skip_single;  // 1: rows of single-partition sequences were written directly
};

constexpr int kReduceWarps = 4;

// One block per (sequence, query head) row: the log-sum-exp merge of the
// row's partials (Parallel Partitioning, step 3).  The block first takes
// the largest m_k, then its warps take every kReduceWarps-th partial, four
// at a time (the loads of four partials in flight per warp, sixteen per
// row), and the warps' sums are added in shared memory.  A lane owns D/32
// consecutive dims.
template <bool BF16, int D>
__global__ void __launch_bounds__(kReduceWarps * 32) split_reduce_kernel(const ReduceParams p) {
    constexpr int V = D / 32, W = kReduceWarps, U = 4;
    __shared__ float s_max[W];
    __shared__ float s_acc[W][D];
    __shared__ float s_l[W];
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = blockIdx.x;
    const int seq = (int)(row / p.num_q_heads);
    const int L = checked_len(p.seq_lens, seq, p.max_seq_len, p.max_seq_len, p.err, false);
    const int np = L == 0 ? 0 : (L - 1) / p.partition_tokens + 1;
    if (p.skip_single && np <= 1) return;
    uint16_t *out = static_cast<uint16_t *>(p.out) + row * D + lane * V;
    if (np == 0) {
        if (warp == 0) {
#pragma unroll
            for (int k = 0; k < V; ++k) out[k] = 0;
        }
        return;
    }
    const float *m = p.part_m + row * p.num_partitions;
    const float *l = p.part_l + row * p.num_partitions;
    const float *o = p.part_o + row * p.num_partitions * D + lane * V;
    float M = -INFINITY;
    for (int k = threadIdx.x; k < np; k += W * 32) M = fmaxf(M, __ldcg(m + k));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, off));
    if (lane == 0) s_max[warp] = M;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < W; ++w) M = fmaxf(M, s_max[w]);

    float acc[V];
#pragma unroll
    for (int x = 0; x < V; ++x) acc[x] = 0.f;
    float lsum = 0.f;
    auto fold = [&](float mk, float lk, const float *v) {
        const float wk = (mk == -INFINITY) ? 0.f : lk * fast_exp2(mk - M);  // empty partial: 0
        lsum += wk;
#pragma unroll
        for (int x = 0; x < V; ++x) acc[x] += wk * v[x];
    };
    auto load_o = [&](int k, float *v) {
        const float *src = o + (int64_t)k * D;
        if constexpr (V == 4) {
            const float4 t = __ldcg(reinterpret_cast<const float4 *>(src));
            v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
        } else {
            const float2 t = __ldcg(reinterpret_cast<const float2 *>(src));
            v[0] = t.x; v[1] = t.y;
        }
    };
    int k = warp;
    for (; k + (U - 1) * W < np; k += U * W) {
        float mk[U], lk[U], v[U][V];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            mk[u] = __ldcg(m + k + u * W);
            lk[u] = __ldcg(l + k + u * W);
            load_o(k + u * W, v[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) fold(mk[u], lk[u], v[u]);
    }
    for (; k < np; k += W) {
        float v[V];
        load_o(k, v);
        fold(__ldcg(m + k), __ldcg(l + k), v);
    }
#pragma unroll
    for (int x = 0; x < V; ++x) s_acc[warp][lane * V + x] = acc[x];
    if (lane == 0) s_l[warp] = lsum;
    __syncthreads();
    if (warp != 0) return;
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) tot += s_l[w];
    const float inv = tot > 0.f ? 1.0f / tot : 0.f;
    float r[V];
#pragma unroll
    for (int x = 0; x < V; ++x) {
        float a = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) a += s_acc[w][lane * V + x];
        r[x] = a * inv;
    }
    if constexpr (V == 4) {
        *reinterpret_cast<uint2 *>(out) =
            make_uint2(narrow2<BF16>(r[0], r[1]), narrow2<BF16>(r[2], r[3]));
    } else {
        *reinterpret_cast<uint32_t *>(out) = narrow2<BF16>(r[0], r[1]);
    }
}

// ------------------------------------------------------------------ host side
using DecodeKernel = void (*)(const DecodeParams);
using ReduceKernel = void (*)(const ReduceParams);

struct DecodeEntry {
    DecodeKernel fn;
    int smem;
};

template <bool BF16, int D, int GP>
DecodeEntry decode_entry() {
    return {paged_decode_kernel<BF16, D, GP>, DecodeShape<D, GP>::SMEM_BYTES};
}

static int group_pad(int G) { return G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : 8; }

static bool pick_decode(pa_dtype dt, int D, int GP, DecodeEntry *e) {
    const bool bf = dt == PA_BF16;
#define PA_CASE(BFV, DV, GV)                          \
    if (bf == BFV && D == DV && GP == GV) {            \
        *e = decode_entry<BFV, DV, GV>();              \
        return true;                                   \
    }
    PA_CASE(false, 64, 1) PA_CASE(false, 64, 2) PA_CASE(false, 64, 4) PA_CASE(false, 64, 8)
    PA_CASE(false, 128, 1) PA_CASE(false, 128, 2) PA_CASE(false, 128, 4) PA_CASE(false, 128, 8)
    PA_CASE(true, 64, 1) PA_CASE(true, 64, 2) PA_CASE(true, 64, 4) PA_CASE(true, 64, 8)
    PA_CASE(true, 128, 1) PA_CASE(true, 128, 2) PA_CASE(true, 128, 4) PA_CASE(true, 128, 8)
#undef PA_CASE
    return false;
}

static ReduceKernel pick_reduce(pa_dtype dt, int D) {
    if (dt == PA_BF16) return D == 64 ? split_reduce_kernel<true, 64> : split_reduce_kernel<true, 128>;
    return D == 64 ? split_reduce_kernel<false, 64> : split_reduce_kernel<false, 128>;
}

static int ilog2_exact(int x) {
    int k = 0;
    while ((1 << k) < x) ++k;
    return (1 << k) == x ? k : -1;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WorkspaceLayout {
    size_t m_off, l_off, o_off, c_off, f_off, bytes;
};

// m, l, O partials, then the fused combine's arrival counters (one 64-bit
// word per (sequence, KV head)) and ready flags (one 32-bit word per
// (sequence, KV head, slot)).
static WorkspaceLayout workspace_layout(int S, int Hq, int D, int NP, int Hkv) {
    const size_t rows = (size_t)S * Hq * NP;
    WorkspaceLayout w;
    w.m_off = 0;
    w.l_off = align256(rows * sizeof(float));
    w.o_off = w.l_off + align256(rows * sizeof(float));
    w.c_off = w.o_off + align256(rows * D * sizeof(float));
    w.f_off = w.c_off + align256((size_t)S * Hkv * sizeof(unsigned long long));
    w.bytes = w.f_off + align256((size_t)S * Hkv * NP * sizeof(unsigned int));
    return w;
}

// Tag of a decode call in the fused-combine flags: never 0 (a cleared flag)
// nor all ones (a workspace filled with 0xFF bytes).
static unsigned int next_epoch() {
    static std::atomic<unsigned int> epoch{0x9e3779b9u};
    for (;;) {
        const unsigned int e = epoch.fetch_add(1) + 1;
        if (e != 0u && e != 0xffffffffu) return e;
    }
}


// Occupancy of a decode instantiation (CTAs per SM), cached per kernel/device.
static int decode_ctas_per_sm(const DecodeEntry &e) {
    int n = 0;
    if (!ensure_smem_attr(reinterpret_cast<const void *>(e.fn), e.smem)) return 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, e.fn, kDecodeThreads, e.smem) !=
        cudaSuccess)
        return 1;
    return n > 0 ? n : 1;
}

// Automatic partition size: aim for the largest work item to be at most
// 1/share_div of one CTA slot's share of the whole job (the share taken at
// the maximum length), in multiples of 256 positions and at least
// min_tokens, and run single pass when that would not split anything.
// share_div is 4 and min_tokens 512, for 16-bit and E4M3 pools alike (a
// tile's softmax, not its bytes, sets the pace of a short item): coarse
// enough that a work item's prologue, ring fill and partial writes stay
// small next to its tiles (the Llama-shaped batch runs single pass), fine
// enough to split a few long sequences over the GPU.
static int auto_partition(int S, int Hkv, int max_seq_len, int ctas_per_sm, int block_size,
                          double share_div, int min_tokens) {
    if (max_seq_len <= 0) return -1;
    const int slots = sm_count() * ctas_per_sm;
    const double units = (double)S * Hkv;
    double target = (double)max_seq_len * units / (share_div * (slots > 0 ? slots : 1));
    int P = (int)std::ceil(target / 256.0) * 256;
    if (P < min_tokens) P = min_tokens;
    if (P % block_size) P = (P / block_size + 1) * block_size;
    if (P >= max_seq_len) return -1;
    return P;
}

struct ResolvedDecode {
    DecodeEntry entry;
    bool tc;  // tensor-core kernel (pa_decode_tc.cu) instead of the CUDA-core one
    bool bf16;
    int head_dim;
    int P;    // -1 single pass, else the positions of a partial (a chunk, see resolve)
    int NP;   // partials per row
    int part_tokens;  // the partition size asked for (or chosen when automatic)
    bool fp8 = false;  // E4M3 pools: the E4M3 variants of the tensor-core kernel
    int span = 1;      // partitions per CTA (tensor-core kernel); grid.x = ceil(NP / span)
};

// Scales of E4M3 pools (element = scale * code value).
struct KvFp8 {
    float k_scale;
    float v_scale;
};

// Process-wide choice of decode kernel: 0 automatic, 1 CUDA cores, 2 tensor cores.
static std::atomic<int> g_decode_impl{0};
// Process-wide partitions per tensor-core CTA: 0 automatic, else forced.
static std::atomic<int> g_decode_span{0};

// Automatic choice: the tensor-core kernel wherever it applies (measured
// faster on every workload shape here; the CUDA-core kernel is bound by
// instruction issue at 5..8 heads per KV head).
static bool use_tensor_cores(int head_dim, int group) {
    const int impl = g_decode_impl.load(std::memory_order_relaxed);
    if (!tc_supported(head_dim, group)) return false;
    return impl != 1;
}

static pa_status resolve(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                         int block_size, int max_seq_len, int partition_tokens, pa_dtype dtype,
                         ResolvedDecode *r, bool fp8 = false, bool merge_span = true) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_seq_len < 0)
        return PA_ERR_INVALID;
    if (num_seqs > 65535 || num_kv_heads > 65535) return PA_ERR_INVALID;  // grid y and z
    if ((int64_t)num_seqs * num_q_heads > 0x7fffffff) return PA_ERR_INVALID;  // combine grid
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID;
    if (num_q_heads % num_kv_heads) return PA_ERR_INVALID;
    const int G = num_q_heads / num_kv_heads;
    if (G > 8 || (head_dim != 64 && head_dim != 128) || (block_size != 16 && block_size != 32))
        return PA_ERR_UNSUPPORTED;
    if (!pick_decode(dtype, head_dim, group_pad(G), &r->entry)) return PA_ERR_UNSUPPORTED;
    r->tc = use_tensor_cores(head_dim, G);
    r->fp8 = fp8;
    if (fp8 && !fp8_supported(head_dim, G)) return PA_ERR_UNSUPPORTED;
    r->bf16 = dtype == PA_BF16;
    r->head_dim = head_dim;
    int P = partition_tokens;
    if (P == 0) {
        const int per_sm = r->fp8  ? fp8_ctas_per_sm(dtype == PA_BF16, head_dim, G)
                           : r->tc ? tc_ctas_per_sm(dtype == PA_BF16, head_dim)
                                   : decode_ctas_per_sm(r->entry);
        P = auto_partition(num_seqs, num_kv_heads, max_seq_len, per_sm, block_size, 4.0, 512);
    }
    if (P < -1) return PA_ERR_INVALID;
    if (P > 0 && (P % block_size != 0 || P % kUnit != 0)) return PA_ERR_INVALID;
    r->P = P;
    r->NP = (P > 0) ? (max_seq_len + P - 1) / P : 1;
    if (r->NP < 1) r->NP = 1;
    r->span = 1;
    if ((r->tc || r->fp8) && P > 0 && P % 128 == 0) {
        // One CTA computes several consecutive partitions (each still its own
        // partial) when partitions are short: a CTA's prologue and pipeline
        // fill are then paid once per ~2048 positions, as long as a CTA's
        // span stays within a quarter of one CTA slot's share of the job (the
        // share taken at the maximum length, an upper bound), so that short,
        // latency-bound batches keep one partition a CTA.
        const int forced = g_decode_span.load(std::memory_order_relaxed);
        int R = forced > 0 ? forced : 2048 / P;
        if (R > r->NP) R = r->NP;
        if (forced <= 0) {
            const int slots = sm_count() * (r->fp8 ? fp8_ctas_per_sm(dtype == PA_BF16, head_dim, G)
                                                   : tc_ctas_per_sm(dtype == PA_BF16, head_dim));
            const double share =
                (double)num_seqs * num_kv_heads * max_seq_len / (slots > 0 ? slots : 1);
            while (R > 1 && 4.0 * R * P > share) --R;
        }
        r->span = R > 1 ? R : 1;
    }
    r->part_tokens = P;
    if (merge_span && r->span > 1) {
        // Decode (the output, not the partials, is the result): a CTA's span
        // of consecutive partitions reaches HBM as one partial.  The online
        // softmax runs on across their boundaries; its rescale is the
        // cross-partition combine ([P3] section 4, step 3) applied as each
        // partition arrives, so the CTA leaves the combine of its span, and
        // the launch sees chunks of span * P positions with one partial each
        // (pa_decode_partitions keeps one partial per partition).
        r->P = P * r->span;
        r->NP = (max_seq_len + r->P - 1) / r->P;
        if (r->NP < 1) r->NP = 1;
        r->span = 1;
    }
    return PA_OK;
}

static pa_status launch_decode(const ResolvedDecode &r, DecodeParams prm, int num_seqs,
                               int num_kv_heads, cudaStream_t stream) {
    if (num_seqs == 0) return PA_OK;
    if (num_kv_heads > 65535 || num_seqs > 65535) return PA_ERR_INVALID;
    if (prm.ws_parts == 0) prm.ws_parts = prm.num_partitions;  // plain launch: own workspace
    // CTAs along x: split-KV chunks of each sequence (spans of partitions)
    const int span = (r.tc || r.fp8) && !prm.prefix_parts ? r.span : 1;
    const int chunks = (r.NP + span - 1) / span;
    prm.compact = prm.mode == 0 && prm.prefix_parts == 0 && num_seqs <= kCompactMaxSeqs &&
                  (int64_t)chunks * num_kv_heads * num_seqs < (1ll << 31);
    if (!prm.out && (prm.mode == 0 || prm.counters || prm.prefix_parts)) return PA_ERR_INVALID;
    if (prm.counters) {
        // ready flags only when every CTA is resident at once (a waiting
        // combiner must never hold a slot a partner needs)
        const int per_sm = r.fp8 ? fp8_ctas_per_sm(r.bf16, r.head_dim, prm.group)
                           : r.tc ? tc_ctas_per_sm(r.bf16, r.head_dim)
                                  : 0;
        prm.one_wave = (r.tc || r.fp8) &&
                       (int64_t)chunks * num_kv_heads * num_seqs <= (int64_t)sm_count() * per_sm;
    }
    if (r.fp8) {
        if (prm.prefix_parts) return PA_ERR_UNSUPPORTED;  // no cascade over E4M3 pools
        prm.span = span;
        return launch_decode_fp8(prm, r.bf16, r.head_dim, chunks, num_kv_heads, num_seqs, stream);
    }
    if (r.tc) {
        prm.span = span;  // cascade tails: one partition a CTA
        return launch_decode_tc(prm, r.bf16, r.head_dim, chunks, num_kv_heads, num_seqs, stream);
    }
    if (!ensure_smem_attr(reinterpret_cast<const void *>(r.entry.fn), r.entry.smem))
        return PA_ERR_CUDA;
    const dim3 grid = decode_grid(prm, chunks, num_kv_heads, num_seqs);
    if (launch_pdl(r.entry.fn, grid, dim3(kDecodeThreads), (size_t)r.entry.smem, stream, prm) !=
        cudaSuccess)
        return PA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

static pa_status fill_common(DecodeParams *prm, const void *q, const void *k_pool,
                             const void *v_pool, int num_blocks, const int32_t *block_tables,
                             int max_blocks_per_seq, const int32_t *seq_lens, int max_seq_len,
                             int num_seqs, int num_q_heads, int num_kv_heads, int block_size,
                             float scale) {
    if (num_blocks <= 0 || max_blocks_per_seq < 0 || !std::isfinite(scale)) return PA_ERR_INVALID;
    if (num_seqs > 0 && (!q || !k_pool || !v_pool || !block_tables || !seq_lens))
        return PA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool)) return PA_ERR_INVALID;
    std::memset(prm, 0, sizeof *prm);
    prm->q = static_cast<const uint16_t *>(q);
    prm->k_pool = static_cast<const uint16_t *>(k_pool);
    prm->v_pool = static_cast<const uint16_t *>(v_pool);
    prm->block_tables = block_tables;
    prm->seq_lens = seq_lens;
    prm->num_seqs = num_seqs;
    prm->num_blocks = num_blocks;
    prm->max_blocks_per_seq = max_blocks_per_seq;
    prm->max_seq_len = max_seq_len;
    prm->num_q_heads = num_q_heads;
    prm->num_kv_heads = num_kv_heads;
    prm->group = num_q_heads / num_kv_heads;
    prm->block_size = block_size;
    prm->log2_block = ilog2_exact(block_size);
    prm->scale_log2 = scale * kLog2e;
    prm->err = error_word();
    return prm->err ? PA_OK : PA_ERR_CUDA;
}

// Fixed scratch of pa_decode_static_scratch, for callers that cannot
// allocate.  Every GPU that loads the library holds it until exit.
static __device__ __align__(256) unsigned char g_static_scratch[PA_STATIC_SCRATCH_BYTES];

// Device address of this device's copy of g_static_scratch, looked up once
// per device (with that device current); nullptr if the lookup fails.
static void *static_scratch_address() {
    static std::mutex mu;
    static void *addr[128] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress((void **)&ptr, g_static_scratch) != cudaSuccess) return nullptr;
        addr[dev] = ptr;
    }
    return addr[dev];
}

// Shared body of pa_decode and pa_decode_step (k_new == nullptr: no fused write).
static pa_status decode_impl(void *out, const void *q, const void *k_new, const void *v_new,
                             const int64_t *slot_mapping, const void *k_pool, const void *v_pool,
                             int num_blocks, const int32_t *block_tables, int max_blocks_per_seq,
                             const int32_t *seq_lens, int max_seq_len, int num_seqs,
                             int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                             float scale, int partition_tokens, void *workspace,
                             size_t workspace_bytes, pa_dtype dtype, void *stream,
                             const KvFp8 *fp8 = nullptr) {
    ResolvedDecode r;
    if (fp8 && (!(fp8->k_scale > 0.f) || !(fp8->v_scale > 0.f) || !std::isfinite(fp8->k_scale) ||
                !std::isfinite(fp8->v_scale)))
        return PA_ERR_INVALID;
    pa_status st = resolve(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                           max_seq_len, partition_tokens, dtype, &r, fp8 != nullptr);
    if (st != PA_OK) return st;
    if (num_seqs > 0 && (!out || !aligned16(out))) return PA_ERR_INVALID;
    DecodeParams prm;
    st = fill_common(&prm, q, k_pool, v_pool, num_blocks, block_tables, max_blocks_per_seq,
                     seq_lens, max_seq_len, num_seqs, num_q_heads, num_kv_heads, block_size,
                     scale);
    if (st != PA_OK) return st;
    prm.out = out;
    prm.mode = 0;
    if (fp8) {
        prm.scale_log2 *= fp8->k_scale;  // K elements are k_scale * codes
        prm.k_inv = 1.0f / fp8->k_scale;
        prm.v_inv = 1.0f / fp8->v_scale;
        prm.v_scale = fp8->v_scale;
    }
    if (k_new) {
        if (num_seqs > 0 && (!v_new || !slot_mapping || !aligned16(k_new) || !aligned16(v_new)))
            return PA_ERR_INVALID;
        prm.k_new = static_cast<const uint16_t *>(k_new);
        prm.v_new = static_cast<const uint16_t *>(v_new);
        prm.slot_mapping = slot_mapping;
    }
    cudaStream_t s = as_stream(stream);
    if (r.P <= 0) {
        prm.partition_tokens = kSinglePassTokens;
        prm.num_partitions = 1;
        return launch_decode(r, prm, num_seqs, num_kv_heads, s);
    }
    const WorkspaceLayout w = workspace_layout(num_seqs, num_q_heads, head_dim, r.NP, num_kv_heads);
    if (!workspace || workspace_bytes < w.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return PA_ERR_INVALID;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    prm.part_m = reinterpret_cast<float *>(ws + w.m_off);
    prm.part_l = reinterpret_cast<float *>(ws + w.l_off);
    prm.part_o = reinterpret_cast<float *>(ws + w.o_off);
    prm.partition_tokens = r.P;
    prm.num_partitions = r.NP;
    const bool fuse = r.NP <= kFuseMaxParts;
    if (fuse) {
        // one CTA of each (sequence, KV head) combines its partials
        prm.counters = reinterpret_cast<unsigned long long *>(ws + w.c_off);
        prm.flags = reinterpret_cast<unsigned int *>(ws + w.f_off);
        prm.epoch = next_epoch();
    }
    st = launch_decode(r, prm, num_seqs, num_kv_heads, s);
    if (st != PA_OK || num_seqs == 0 || fuse) return st;
    ReduceParams rp;
    rp.out = out;
    rp.part_m = prm.part_m;
    rp.part_l = prm.part_l;
    rp.part_o = prm.part_o;
    rp.seq_lens = seq_lens;
    rp.err = prm.err;
    rp.num_seqs = num_seqs;
    rp.num_q_heads = num_q_heads;
    rp.max_seq_len = max_seq_len < max_blocks_per_seq * block_size
                         ? max_seq_len
                         : max_blocks_per_seq * block_size;
    rp.partition_tokens = r.P;
    rp.num_partitions = r.NP;
    rp.skip_single = 1;
    const int64_t rows = (int64_t)num_seqs * num_q_heads;
    if (rows > 0x7fffffff) return PA_ERR_INVALID;
    if (launch_pdl(pick_reduce(dtype, head_dim), dim3((unsigned)rows), dim3(kReduceWarps * 32), 0, s,
                   rp) != cudaSuccess)
        return PA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// Shared-prefix (cascade) decode: chunking of the prefix pass and the tail
// launch (positions [prefix_len, L) of each sequence).
struct CascadePlan {
    ResolvedDecode tail;   // the tail launch (positions [prefix_len, L))
    CascadeChunks chunks;  // the prefix pass
    int prefix_slots;      // merged prefix partials per row
    int ws_parts;          // prefix slots + the tail's partitions
};
static pa_status cascade_plan(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                              int block_size, int max_seq_len, int prefix_len, pa_dtype dtype,
                              CascadePlan *c) {
    if (prefix_len <= 0 || max_seq_len < prefix_len || block_size <= 0 ||
        prefix_len % block_size)
        return PA_ERR_INVALID;
    pa_status st = resolve(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                           max_seq_len - prefix_len, 0, dtype, &c->tail);
    if (st != PA_OK) return st;
    const int G = num_q_heads / num_kv_heads;
    c->chunks = cascade_chunks(prefix_len, num_seqs * G, num_kv_heads, head_dim, dtype == PA_BF16);
    c->prefix_slots = c->chunks.num_chunks / c->chunks.cluster;
    c->ws_parts = c->prefix_slots + c->tail.NP;
    return c->ws_parts <= kCombineMaxParts ? PA_OK : PA_ERR_UNSUPPORTED;
}

}  // namespace pa

using namespace pa;

extern "C" {

int pa_decode_auto_partition(int num_seqs, int num_kv_heads, int max_seq_len, int head_dim,
                             int block_size, int group_size, pa_dtype dtype) {
    ResolvedDecode r;
    if (group_size < 1 || resolve(num_seqs, num_kv_heads * group_size, num_kv_heads, head_dim,
                                  block_size, max_seq_len, 0, dtype, &r) != PA_OK)
        return -1;
    return r.part_tokens;
}

int pa_decode_partial_tokens(int num_seqs, int num_kv_heads, int max_seq_len, int head_dim,
                             int block_size, int group_size, int partition_tokens, pa_dtype dtype,
                             int fp8) {
    ResolvedDecode r;
    if (group_size < 1 || resolve(num_seqs, num_kv_heads * group_size, num_kv_heads, head_dim,
                                  block_size, max_seq_len, partition_tokens, dtype, &r,
                                  fp8 != 0) != PA_OK)
        return -2;
    return r.P > 0 ? r.P : -1;
}

int pa_decode_fp8_auto_partition(int num_seqs, int num_kv_heads, int max_seq_len, int head_dim,
                                 int block_size, int group_size, pa_dtype dtype) {
    ResolvedDecode r;
    if (group_size < 1 || resolve(num_seqs, num_kv_heads * group_size, num_kv_heads, head_dim,
                                  block_size, max_seq_len, 0, dtype, &r, true) != PA_OK)
        return -1;
    return r.part_tokens;
}

int pa_set_decode_impl(int impl) {
    if (impl < 0 || impl > 2) return -1;
    return g_decode_impl.exchange(impl);
}

int pa_get_decode_impl(void) { return g_decode_impl.load(); }

int pa_set_decode_span(int span) {
    if (span < 0) return -1;
    return g_decode_span.exchange(span);
}

int pa_decode_ctas_per_sm(int head_dim, int group_size, pa_dtype dtype) {
    DecodeEntry e;
    if (group_size < 1 || group_size > 8 || !pick_decode(dtype, head_dim, group_pad(group_size), &e))
        return 0;
    if (use_tensor_cores(head_dim, group_size)) return tc_ctas_per_sm(dtype == PA_BF16, head_dim);
    return decode_ctas_per_sm(e);
}

size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                int block_size, int max_seq_len, int partition_tokens,
                                pa_dtype dtype) {
    ResolvedDecode r;
    if (resolve(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_seq_len,
                partition_tokens, dtype, &r, false, false) != PA_OK)
        return 0;
    if (r.P <= 0) return 0;
    return workspace_layout(num_seqs, num_q_heads, head_dim, r.NP, num_kv_heads).bytes;
}

pa_status pa_decode(void *out, const void *q, const void *k_pool, const void *v_pool,
                    int num_blocks, const int32_t *block_tables, int max_blocks_per_seq,
                    const int32_t *seq_lens, int max_seq_len, int num_seqs, int num_q_heads,
                    int num_kv_heads, int head_dim, int block_size, float scale,
                    int partition_tokens, void *workspace, size_t workspace_bytes,
                    pa_dtype dtype, void *stream) {
    return decode_impl(out, q, nullptr, nullptr, nullptr, k_pool, v_pool, num_blocks,
                       block_tables, max_blocks_per_seq, seq_lens, max_seq_len, num_seqs,
                       num_q_heads, num_kv_heads, head_dim, block_size, scale, partition_tokens,
                       workspace, workspace_bytes, dtype, stream);
}

size_t pa_decode_fp8_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                    int head_dim, int block_size, int max_seq_len,
                                    int partition_tokens, pa_dtype dtype) {
    ResolvedDecode r;
    if (resolve(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_seq_len,
                partition_tokens, dtype, &r, true) != PA_OK)
        return 0;
    if (r.P <= 0) return 0;
    return workspace_layout(num_seqs, num_q_heads, head_dim, r.NP, num_kv_heads).bytes;
}

pa_status pa_decode_fp8(void *out, const void *q, const void *k_new, const void *v_new,
                        const int64_t *slot_mapping, void *k_pool, void *v_pool, int num_blocks,
                        const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *seq_lens, int max_seq_len, int num_seqs, int num_q_heads,
                        int num_kv_heads, int head_dim, int block_size, float scale,
                        float k_scale, float v_scale, int partition_tokens, void *workspace,
                        size_t workspace_bytes, pa_dtype dtype, void *stream) {
    const KvFp8 fp8 = {k_scale, v_scale};
    return decode_impl(out, q, k_new, v_new, slot_mapping, k_pool, v_pool, num_blocks,
                       block_tables, max_blocks_per_seq, seq_lens, max_seq_len, num_seqs,
                       num_q_heads, num_kv_heads, head_dim, block_size, scale, partition_tokens,
                       workspace, workspace_bytes, dtype, stream, &fp8);
}

pa_status pa_decode_step(void *out, const void *q, const void *k_new, const void *v_new,
                         const int64_t *slot_mapping, void *k_pool, void *v_pool, int num_blocks,
                         const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *seq_lens, int max_seq_len, int num_seqs, int num_q_heads,
                         int num_kv_heads, int head_dim, int block_size, float scale,
                         int partition_tokens, void *workspace, size_t workspace_bytes,
                         pa_dtype dtype, void *stream) {
    if (num_seqs > 0 && !k_new) return PA_ERR_INVALID;
    return decode_impl(out, q, k_new, v_new, slot_mapping, k_pool, v_pool, num_blocks,
                       block_tables, max_blocks_per_seq, seq_lens, max_seq_len, num_seqs,
                       num_q_heads, num_kv_heads, head_dim, block_size, scale, partition_tokens,
                       workspace, workspace_bytes, dtype, stream);
}


size_t pa_decode_cascade_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                        int head_dim, int block_size, int max_seq_len,
                                        int prefix_len, pa_dtype dtype) {
    if (prefix_len == 0)
        return pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                        block_size, max_seq_len, 0, dtype);
    CascadePlan c;
    if (cascade_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_seq_len,
                     prefix_len, dtype, &c) != PA_OK)
        return 0;
    return workspace_layout(num_seqs, num_q_heads, head_dim, c.ws_parts, num_kv_heads).bytes;
}

pa_status pa_decode_cascade(void *out, const void *q, const void *k_new, const void *v_new,
                            const int64_t *slot_mapping, void *k_pool, void *v_pool,
                            int num_blocks, const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *seq_lens, int max_seq_len, int num_seqs,
                            int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                            float scale, int prefix_len, void *workspace, size_t workspace_bytes,
                            pa_dtype dtype, void *stream) {
    if (prefix_len == 0)
        return decode_impl(out, q, k_new, v_new, slot_mapping, k_pool, v_pool, num_blocks,
                           block_tables, max_blocks_per_seq, seq_lens, max_seq_len, num_seqs,
                           num_q_heads, num_kv_heads, head_dim, block_size, scale, 0, workspace,
                           workspace_bytes, dtype, stream);
    CascadePlan c;
    pa_status st = cascade_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                max_seq_len, prefix_len, dtype, &c);
    if (st != PA_OK) return st;
    if (prefix_len > max_blocks_per_seq * block_size) return PA_ERR_INVALID;
    if (num_seqs > 0 && (!out || !aligned16(out))) return PA_ERR_INVALID;
    DecodeParams prm;
    st = fill_common(&prm, q, k_pool, v_pool, num_blocks, block_tables, max_blocks_per_seq,
                     seq_lens, max_seq_len, num_seqs, num_q_heads, num_kv_heads, block_size,
                     scale);
    if (st != PA_OK) return st;
    prm.out = out;
    if (k_new) {
        if (num_seqs > 0 && (!v_new || !slot_mapping || !aligned16(k_new) || !aligned16(v_new)))
            return PA_ERR_INVALID;
        prm.k_new = static_cast<const uint16_t *>(k_new);
        prm.v_new = static_cast<const uint16_t *>(v_new);
        prm.slot_mapping = slot_mapping;
    }
    const WorkspaceLayout w =
        workspace_layout(num_seqs, num_q_heads, head_dim, c.ws_parts, num_kv_heads);
    if (num_seqs > 0 &&
        (!workspace || workspace_bytes < w.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255)))
        return PA_ERR_INVALID;
    if (num_seqs == 0) return PA_OK;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    prm.part_m = reinterpret_cast<float *>(ws + w.m_off);
    prm.part_l = reinterpret_cast<float *>(ws + w.l_off);
    prm.part_o = reinterpret_cast<float *>(ws + w.o_off);
    cudaStream_t s = as_stream(stream);

    CascadeParams cp;
    cp.q = prm.q;
    cp.block_tables = block_tables;
    cp.seq_lens = seq_lens;
    cp.part_m = prm.part_m;
    cp.part_l = prm.part_l;
    cp.part_o = prm.part_o;
    cp.err = prm.err;
    cp.num_seqs = num_seqs;
    cp.num_q_heads = num_q_heads;
    cp.num_kv_heads = num_kv_heads;
    cp.group = prm.group;
    cp.num_blocks = num_blocks;
    cp.max_blocks_per_seq = max_blocks_per_seq;
    cp.block_size = block_size;
    cp.log2_block = prm.log2_block;
    cp.prefix_len = prefix_len;
    cp.chunk_tokens = c.chunks.chunk_tokens;
    cp.num_chunks = c.chunks.num_chunks;
    cp.cluster = c.chunks.cluster;
    cp.ws_parts = c.ws_parts;
    cp.scale_log2 = prm.scale_log2;
    st = launch_cascade_prefix(cp, k_pool, v_pool, dtype == PA_BF16, head_dim, s);
    if (st != PA_OK) return st;

    // one tail partition: the tail kernel merges the prefix's partials and
    // writes the output; several: partials, and the last CTA merges
    prm.mode = c.tail.NP > 1 ? 1 : 0;
    prm.len_offset = prefix_len;
    prm.table_offset = prefix_len / block_size;
    prm.ws_parts = c.ws_parts;
    prm.part_base = c.prefix_slots;
    prm.prefix_parts = c.prefix_slots;
    prm.late_wait = cp.num_chunks > 0;  // the prefix pass was launched just before
    prm.partition_tokens = c.tail.P > 0 ? c.tail.P : kSinglePassTokens;
    prm.num_partitions = c.tail.NP;
    if (c.tail.NP > 1) {
        prm.counters = reinterpret_cast<unsigned long long *>(ws + w.c_off);
        prm.flags = reinterpret_cast<unsigned int *>(ws + w.f_off);
        prm.epoch = next_epoch();
    }
    return launch_decode(c.tail, prm, num_seqs, num_kv_heads, s);
}

pa_status pa_decode_partitions(const void *q, const void *k_pool, const void *v_pool,
                               int num_blocks, const int32_t *block_tables,
                               int max_blocks_per_seq, const int32_t *seq_lens, int max_seq_len,
                               int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                               int block_size, float scale, int partition_tokens,
                               void *workspace, size_t workspace_bytes, pa_dtype dtype,
                               void *stream) {
    if (partition_tokens <= 0) return PA_ERR_INVALID;
    ResolvedDecode r;
    pa_status st = resolve(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                           max_seq_len, partition_tokens, dtype, &r, false, false);
    if (st != PA_OK) return st;
    DecodeParams prm;
    st = fill_common(&prm, q, k_pool, v_pool, num_blocks, block_tables, max_blocks_per_seq,
                     seq_lens, max_seq_len, num_seqs, num_q_heads, num_kv_heads, block_size,
                     scale);
    if (st != PA_OK) return st;
    const WorkspaceLayout w = workspace_layout(num_seqs, num_q_heads, head_dim, r.NP, num_kv_heads);
    if (num_seqs > 0 &&
        (!workspace || workspace_bytes < w.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255)))
        return PA_ERR_INVALID;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    prm.part_m = reinterpret_cast<float *>(ws + w.m_off);
    prm.part_l = reinterpret_cast<float *>(ws + w.l_off);
    prm.part_o = reinterpret_cast<float *>(ws + w.o_off);
    prm.partition_tokens = r.P;
    prm.num_partitions = r.NP;
    prm.mode = 1;
    return launch_decode(r, prm, num_seqs, num_kv_heads, as_stream(stream));
}

pa_status pa_split_kv_reduce(void *out, const void *workspace, size_t workspace_bytes,
                             const int32_t *seq_lens, int max_seq_len, int num_seqs,
                             int num_q_heads, int head_dim, int partition_tokens, pa_dtype dtype,
                             void *stream) {
    if (num_seqs < 0 || num_q_heads <= 0 || max_seq_len < 0 || partition_tokens <= 0 ||
        partition_tokens % kUnit)
        return PA_ERR_INVALID;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PA_OK;
    const int NP = max_seq_len > 0 ? (max_seq_len + partition_tokens - 1) / partition_tokens : 1;
    const WorkspaceLayout w = workspace_layout(num_seqs, num_q_heads, head_dim, NP, 0);
    if (!out || !seq_lens || !workspace || workspace_bytes < w.bytes ||
        (reinterpret_cast<uintptr_t>(workspace) & 255) || !aligned16(out))
        return PA_ERR_INVALID;
    ReduceParams rp;
    const uint8_t *ws = static_cast<const uint8_t *>(workspace);
    rp.out = out;
    rp.part_m = reinterpret_cast<const float *>(ws + w.m_off);
    rp.part_l = reinterpret_cast<const float *>(ws + w.l_off);
    rp.part_o = reinterpret_cast<const float *>(ws + w.o_off);
    rp.seq_lens = seq_lens;
    rp.err = error_word();
    if (!rp.err) return PA_ERR_CUDA;
    rp.num_seqs = num_seqs;
    rp.num_q_heads = num_q_heads;
    rp.max_seq_len = max_seq_len;
    rp.partition_tokens = partition_tokens;
    rp.num_partitions = NP;
    rp.skip_single = 0;
    const int64_t rows = (int64_t)num_seqs * num_q_heads;
    if (rows > 0x7fffffff) return PA_ERR_INVALID;
    pick_reduce(dtype, head_dim)<<<(unsigned)rows, kReduceWarps * 32, 0, as_stream(stream)>>>(rp);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// Same computation as pa_decode; the split-KV partials go to the library's
// fixed device array instead of a caller workspace (see pa.h).
pa_status pa_decode_static_scratch(void *out, const void *q, const void *k_pool,
                                   const void *v_pool, int num_blocks,
                                   const int32_t *block_tables, int max_blocks_per_seq,
                                   const int32_t *seq_lens, int max_seq_len, int num_seqs,
                                   int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, float scale, int partition_tokens,
                                   pa_dtype dtype, void *stream) {
    ResolvedDecode r;
    pa_status st = resolve(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                           max_seq_len, partition_tokens, dtype, &r);
    if (st != PA_OK) return st;
    const size_t need =
        r.P > 0 ? workspace_layout(num_seqs, num_q_heads, head_dim, r.NP, num_kv_heads).bytes : 0;
    if (need > PA_STATIC_SCRATCH_BYTES) return PA_ERR_TOO_LARGE;
    void *scratch = nullptr;
    if (need > 0) {
        scratch = static_scratch_address();
        if (!scratch) return PA_ERR_CUDA;
    }
    return pa_decode(out, q, k_pool, v_pool, num_blocks, block_tables, max_blocks_per_seq,
                     seq_lens, max_seq_len, num_seqs, num_q_heads, num_kv_heads, head_dim,
                     block_size, scale, r.P > 0 ? r.P : -1, scratch,
                     need > 0 ? (size_t)PA_STATIC_SCRATCH_BYTES : 0, dtype, stream);
}

}  // extern "C"
