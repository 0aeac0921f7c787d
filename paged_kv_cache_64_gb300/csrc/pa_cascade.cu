// Shared-prefix ("cascade") decode for GB300 (sm_103a): the prefix pass.
//
// Sequences forked from one prompt point the first entries of their block
// tables at the same physical blocks ([P1] "The same trick for the cache":
// sequences that begin with the same tokens share blocks; [P3] §5
// copy-on-write forking: the children's tables copy the parent's pointers).
// Plain paged decode reads those blocks once per sequence.  The cascade splits
// every sequence's positions at prefix_len (a whole number of blocks):
//   - the shared prefix [0, prefix_len) is attended ONCE per KV head, by the
//     query rows of all sequences together, as dense products on the tensor
//     cores (this file);
//   - each tail [prefix_len, L) by the paged decode kernels;
// and the partial results are merged by the split-KV log-sum-exp combine
// ([P3] §4 "Parallel Partitioning Across GPU Warps", step 3), which is exact:
// the softmax over the union of the two position ranges.
//
// One CTA per (128-row tile of query rows, chunk of prefix positions, KV
// head).  Query row r of tile t is head (128 t + r) % G of sequence
// (128 t + r) / G within the KV head's group.  Per tile of 128 positions:
//
//   S[128 rows x 128 pos] = Q[128 x d] . K_tile^T      (M=128, N=128, K=d)
//   O[128 rows x d]      += P[128 x 128 pos] . V_tile  (M=128, N=d,   K=128)
//
// Q, K and P are K-major operands, V an MN-major one (its rows exactly as
// the TMA copies land them); S (two buffers) and O live in TMEM.  Roles
// (10 warps):
//   warp 0      producer: TMA copies of 16-row boxes through the prefix's
//               block-table entries into a 2-stage K/V ring;
//   warp 1      allocates TMEM; lane 0 issues every MMA and commits;
//   warps 2..9  softmax / epilogue in two warpgroups; thread r of each owns
//               query row r (TMEM lane r): group 0 positions 0..63 of every
//               score tile and dims [0, d/2) of O, group 1 the rest.  Each
//               half row is in the thread's registers; the two halves meet
//               through shared memory, row maxima every tile and row sums at
//               the end.
// The CTAs of consecutive chunks form a thread-block cluster (up to 8); at
// the end they merge their chunks' partials through distributed shared
// memory, and the cluster leaves one (m, l, O) partial per row in workspace
// slot blockIdx.y / cluster (m the true base-2 maximum, l relative to it, O
// normalised), as the split-KV partition kernels do.
#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "pa_common.cuh"
#include "pa_decode.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {

constexpr int kCsTile = 128;   // positions per tile: N of q.K^T, K of P.V
constexpr int kCsRows = 128;   // query rows per CTA: M of both products
constexpr int kCsWarps = 10;   // producer, MMA issuer, two softmax warpgroups
constexpr int kCsThreads = kCsWarps * 32;
constexpr int kCsCols = 512;   // TMEM columns: S x2 (128 each) and O (d)
constexpr int kCsS0 = 0, kCsO = 256;
constexpr int kCsMaxCluster = 8;  // chunks merged through distributed shared memory

enum CsBar { kCsFull0 = 0, kCsFull1, kCsEmpty0, kCsEmpty1, kCsQReady, kCsSFull0, kCsSFull1,
             kCsPReady0, kCsPReady1, kCsODone, kNumCsBars };

template <int D>
struct CsShape {
    static constexpr int KH = D / 64;               // 64-dim (128-byte) slabs along d
    static constexpr int SLAB = kCsRows * 128;      // 128 rows x 128 bytes
    static constexpr int Q_BYTES = KH * SLAB;
    static constexpr int P_BYTES = 2 * SLAB;        // 128 rows x 128 positions
    static constexpr int KV_BYTES = KH * SLAB;      // K (or V) of one tile
    static constexpr int STAGE = 2 * KV_BYTES;      // K then V
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_P = OFF_Q + Q_BYTES;
    static constexpr int OFF_STAGE = OFF_P + P_BYTES;
    // the two softmax groups' row maxima (two buffers, by tile parity) and,
    // at the end, their row sums
    static constexpr int OFF_XCH = OFF_STAGE + 2 * STAGE;
    static constexpr int XCH_FLOATS = 2 * 2 * kCsRows + 2 * kCsRows;
    static constexpr int OFF_BAR = OFF_XCH + XCH_FLOATS * 4;
    static constexpr int OFF_MISC = OFF_BAR + kNumCsBars * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack to align the base to 1 KiB
    static_assert(OFF_P % 1024 == 0 && OFF_STAGE % 1024 == 0 && STAGE % 1024 == 0, "atoms");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(kCsRows * (D + 4) * 4 + 2 * kCsRows * 4 <= 2 * STAGE, "merge staging in the ring");
    static_assert(3 * kCsRows * 4 <= P_BYTES, "merge weights in the P tile");
};

// Named barrier 1 over the 256 softmax threads (warps 2-9); true on every
// thread if any of them passed true.  Orders their shared-memory accesses
// like bar.sync.
__device__ __forceinline__ bool softmax_bar256_or(bool v) {
    int any;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.s32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, 1, 256, pi;\n\t"
        "selp.s32 %0, 1, 0, po;\n\t}"
        : "=r"(any)
        : "r"((int)v)
        : "memory");
    return any != 0;
}

// Cluster merge, last step, in the CTA of rank `rank`: rows
// [rank * R, rank * R + R) of the tile (R = 128 / CL) summed over the CL
// chunks' weighted O rows that the cluster's CTAs pushed into this CTA's
// shared memory (slot [c][row][D + 4]), with the weights already in
// wts[R][CL]; written as one partial per row.  256 threads.
template <int D, int CL>
__device__ __forceinline__ void owner_sum(const CascadeParams &p, const float *ost,
                                          const float *wts, const float *rowM, const float *rowL,
                                          uint32_t rank, int t, int mt, int kvh, int slot) {
    constexpr int R = kCsRows / CL;
    constexpr int ITEMS = R * (D / 4) / 256;  // float4 outputs per thread
    static_assert(R * (D / 4) % 256 == 0, "whole items per thread");
    const int G = p.group;
    const int rows_total = p.num_seqs * G;
#pragma unroll 4
    for (int i = 0; i < ITEMS; ++i) {
        const int idx = t + 256 * i;
        const int jl = idx / (D / 4), q4 = idx % (D / 4);
        const int gr = mt * kCsRows + (int)rank * R + jl;
        if (gr >= rows_total) continue;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int c = 0; c < CL; ++c) {
            if (wts[jl * CL + c] == 0.f) continue;  // empty or failed chunk pushed nothing
            const float4 v = *reinterpret_cast<const float4 *>(ost + (c * R + jl) * (D + 4) + q4 * 4);
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        const int64_t row =
            ((int64_t)(gr / G) * p.num_q_heads + (int64_t)kvh * G + gr % G) * p.ws_parts + slot;
        *reinterpret_cast<float4 *>(p.part_o + row * D + q4 * 4) = acc;
        if (q4 == 0) {
            p.part_m[row] = rowM[jl];
            p.part_l[row] = rowL[jl];
        }
    }
}

template <bool BF16, int D>
__global__ void __launch_bounds__(kCsThreads, 1)
    cascade_prefix_kernel(const CascadeParams p, const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v) {
    using S = CsShape<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + S::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::OFF_MISC + 8);

    const int mt = blockIdx.x, chunk = blockIdx.y, kvh = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.group;
    const int rows_total = p.num_seqs * G;
    const int cstart = chunk * p.chunk_tokens;
    // trailing chunks of the last cluster may lie past the prefix: empty
    const int cend = max(cstart, min(cstart + p.chunk_tokens, p.prefix_len));
    const int nunits = (cend - cstart) / kUnit;  // whole blocks, so whole 16-position units
    const int ntiles = (cend - cstart + kCsTile - 1) / kCsTile;

    if (threadIdx.x == 0) {  // descriptors are kernel parameters: fetch them early
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    pdl_wait();  // inputs may come from the previous kernel on the stream
    if (threadIdx.x == 0) {
        const int counts[kNumCsBars] = {1, 1, 1, 1, 8, 1, 1, 8, 8, 1};
        for (int b = 0; b < kNumCsBars; ++b) mbar_init(&bar[b], counts[b]);
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kCsCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // The tail pass may start now: it reads this launch's partials only after
    // its own wait for the launch to complete, and everything else it reads
    // or writes (the sequences' own blocks past the prefix, their newest
    // tokens, its partial slots) is disjoint from what this launch touches.
    // Its CTAs take the SMs this grid leaves free.  Not before this CTA holds
    // its TMEM: a tail CTA on the same SM could otherwise take columns first
    // and then wait for this launch to complete.
    pdl_trigger();
    // staging of the chunk's partial for the cluster merge, in the K/V ring
    float *ost = reinterpret_cast<float *>(smem + S::OFF_STAGE);  // [128][D + 4]
    float *cm = ost + kCsRows * (D + 4);
    float *cl = cm + kCsRows;
    float keep_inv = 0.f;    // 1 / l of the thread's row (softmax threads)
    bool keep_have = false;  // the chunk's O is in TMEM

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        const int32_t *prefix_table = p.block_tables;  // sequence 0's row
        bool ok = true;
        // block-table lookups 32 units (4 tiles) at a time, one round ahead:
        // lane i holds the first row of unit 32 r + i in the 2-D view
        // [NB*Hkv*B, d] of the pool
        auto unit_row = [&](int u) -> int {
            if (u >= nunits) return 0;
            const int pos = cstart + u * kUnit;
            int phys = prefix_table[pos >> p.log2_block];
            if ((unsigned)phys >= (unsigned)p.num_blocks) {
                record_error(p.err, PA_ERR_BAD_INDEX);
                phys = 0;
            }
            return (phys * p.num_kv_heads + kvh) * p.block_size + (pos & (p.block_size - 1));
        };
        int rows_cur = unit_row(lane), rows_next = unit_row(32 + lane);
        for (int t = 0; t < ntiles; ++t) {
            const int st = t & 1;
            if (t > 0 && (t & 3) == 0) {
                rows_cur = rows_next;
                rows_next = unit_row(32 * ((t >> 2) + 1) + lane);
            }
            if (t >= 2) {
                const bool done = mbar_wait(&bar[kCsEmpty0 + st], ((t >> 1) - 1) & 1);
                if (!__all_sync(kFullMask, done)) {
                    ok = false;
                    break;
                }
            }
            const int u0 = t * (kCsTile / kUnit);
            const int nu = (nunits - u0 < kCsTile / kUnit) ? nunits - u0 : kCsTile / kUnit;
            uint8_t *kbuf = smem + S::OFF_STAGE + st * S::STAGE;
            uint8_t *vbuf = kbuf + S::KV_BYTES;
            if (nu < kCsTile / kUnit) {
                // positions past the prefix: P is 0 there, and V must be
                // finite (0 * NaN would poison the product), so zero its rows
#pragma unroll
                for (int h = 0; h < S::KH; ++h) {
                    uint4 *z = reinterpret_cast<uint4 *>(vbuf + h * S::SLAB + nu * 2048);
                    for (int i = lane; i < (kCsTile / kUnit - nu) * 128; i += 32)
                        z[i] = make_uint4(0, 0, 0, 0);
                }
                fence_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&bar[kCsFull0 + st], nu * S::KH * 2048 * 2);
            // lane j < nu copies unit j of the tile: one instruction issues
            // the tile's copies
            const int r0 = __shfl_sync(kFullMask, rows_cur, ((t & 3) * 8 + lane) & 31);
            if (lane < nu) {
#pragma unroll
                for (int h = 0; h < S::KH; ++h) {
                    tma_load_2d(kbuf + h * S::SLAB + lane * 2048, &tmap_k, 64 * h, r0,
                                &bar[kCsFull0 + st]);
                    tma_load_2d(vbuf + h * S::SLAB + lane * 2048, &tmap_v, 64 * h, r0,
                                &bar[kCsFull0 + st]);
                }
            }
            __syncwarp();
        }
        if (!ok && lane == 0) {
            record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
        }
        // The prefix is only shared if every sequence of this tile reaches it
        // through the same entries and is at least as long.  The (sequence,
        // block) pairs of this tile and chunk are dealt to the KV heads' CTAs
        // and their lanes, four loads in flight per lane.
        {
            const int s_lo = mt * kCsRows / G;
            int s_hi = ((mt + 1) * kCsRows + G - 1) / G;
            if (s_hi > p.num_seqs) s_hi = p.num_seqs;
            const int b_lo = cstart >> p.log2_block, nb = (cend - cstart) >> p.log2_block;
            const int npairs = (s_hi - s_lo) * nb;
            const int stride = 32 * p.num_kv_heads;
            bool bad = false;
            for (int i0 = kvh * 32 + lane; i0 < npairs; i0 += 4 * stride) {
                int got[4], want[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int i = i0 + j * stride;
                    got[j] = want[j] = 0;
                    if (i < npairs) {
                        const int s = s_lo + i / nb, b = b_lo + i % nb;
                        got[j] = p.block_tables[(int64_t)s * p.max_blocks_per_seq + b];
                        want[j] = prefix_table[b];
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) bad |= got[j] != want[j];
            }
            if (chunk == 0 && kvh == 0)
                for (int s = s_lo + lane; s < s_hi; s += 32) bad |= p.seq_lens[s] < p.prefix_len;
            if (bad) record_error(p.err, PA_ERR_BAD_INDEX);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc_qk = f16_idesc(BF16, false, false, kCsRows, kCsTile);
            constexpr uint32_t idesc_pv = f16_idesc(BF16, false, true, kCsRows, D);
            const uint32_t sbase = smem_addr(smem);
            auto issue_qk = [&](int t) -> bool {
                const int st = t & 1;
                if (!mbar_wait(&bar[kCsFull0 + st], (t >> 1) & 1)) return false;
                tc_fence_after();
                const uint32_t kb = sbase + S::OFF_STAGE + st * S::STAGE;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * S::SLAB + (ks & 3) * 32;
                    tc_mma(tmem + kCsS0 + 128 * st, sw128_desc(sbase + S::OFF_Q + off, 16, 1024),
                           sw128_desc(kb + off, 16, 1024), idesc_qk, ks > 0);
                }
                tc_commit(&bar[kCsSFull0 + st]);
                return true;
            };
            auto issue_pv = [&](int t) {
                const int st = t & 1;
                tc_fence_after();
                const uint32_t vb = sbase + S::OFF_STAGE + st * S::STAGE + S::KV_BYTES;
#pragma unroll
                for (int ks = 0; ks < kCsTile / 16; ++ks) {
                    const uint32_t poff = (ks >> 2) * S::SLAB + (ks & 3) * 32;
                    tc_mma(tmem + kCsO, sw128_desc(sbase + S::OFF_P + poff, 16, 1024),
                           sw128_desc(vb + ks * 2048, S::SLAB, 1024), idesc_pv, (t > 0) || (ks > 0));
                }
                tc_commit(&bar[kCsEmpty0 + st]);
                tc_commit(&bar[kCsODone]);
            };
            bool ok = ntiles == 0 || mbar_wait(&bar[kCsQReady], 0);
            // Whichever is ready first: q.K^T of tile nq once its K has landed
            // (its S buffer was released with tile nq-2's P, seen before P.V of
            // nq-2 was issued), or P.V of tile nv once its P is written.  A
            // P.V never waits behind a later tile's copies.
            int nq = 0, nv = 0;
            unsigned long long since = global_timer_ns();
            unsigned spins = 0;
            while (ok && nv < ntiles) {
                bool moved = false;
                if (nq < ntiles && nq <= nv + 1 &&
                    mbar_test_wait(&bar[kCsFull0 + (nq & 1)], (nq >> 1) & 1)) {
                    ok = issue_qk(nq);  // landed: returns at once
                    ++nq;
                    moved = true;
                }
                if (ok && nv < nq && mbar_test_wait(&bar[kCsPReady0 + (nv & 1)], (nv >> 1) & 1)) {
                    issue_pv(nv);
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
        // Two warpgroups share the rows: thread r of each owns TMEM lane r
        // (query row r of the tile); group sg takes positions [64 sg,
        // 64 sg + 64) of each S row and dims [sg d/2, (sg + 1) d/2) of each O
        // row.  The groups exchange their row maxima every tile and their row
        // sums at the end, through shared memory at a named barrier that also
        // ORs the threads' failures (so that all 256 take the same branches).
        const int sg = (warp - 2) >> 2;          // softmax group
        const int quad = warp & 3;               // TMEM lane quadrant this warp may access
        const int r = quad * 32 + lane;          // query row of the tile = TMEM lane
        const int st_id = threadIdx.x - 64;      // 0..255
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        float *xmax = reinterpret_cast<float *>(smem + S::OFF_XCH);  // [tile parity][group][row]
        float *xsum = xmax + 4 * kCsRows;                            // [group][row]
        constexpr int kHalf = kCsTile / 2;       // positions of a group
        constexpr int kOHalf = D / 2;            // O dims of a group

        // Q tile (128 rows x d, K-major, 128-byte swizzle), rows past the last
        // sequence zero.  Unscaled: the scale is applied to S in fp32.
        // all of the thread's loads in flight before the first store
        constexpr int kQPer = kCsRows * (D / 8) / 256;
        uint4 qv[kQPer];
#pragma unroll
        for (int i = 0; i < kQPer; ++i) {
            const int ci = st_id + 256 * i;
            const int rr = ci / (D / 8), c = ci % (D / 8);
            const int gr = mt * kCsRows + rr;
            qv[i] = make_uint4(0, 0, 0, 0);
            if (gr < rows_total)
                qv[i] = *reinterpret_cast<const uint4 *>(
                    p.q + ((int64_t)(gr / G) * p.num_q_heads + (int64_t)kvh * G + gr % G) * D + c * 8);
        }
#pragma unroll
        for (int i = 0; i < kQPer; ++i) {
            const int ci = st_id + 256 * i;
            const int rr = ci / (D / 8), c = ci % (D / 8);
            *reinterpret_cast<uint4 *>(smem + S::OFF_Q + sw128_offset(rr, c * 8, S::SLAB)) = qv[i];
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kCsQReady]);

        float m_run = -INFINITY, m_true = -INFINITY, l_run = 0.f;
        bool failed = false, fail_local = false;
        for (int t = 0; t < ntiles; ++t) {
            const int b = t & 1;
            const bool landed = __all_sync(kFullMask, mbar_wait(&bar[kCsSFull0 + b], (t >> 1) & 1));
            float s[kHalf];
            if (landed) {
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < kHalf / 32; ++c)
                    tmem_ld32(tmem + lane_addr + kCsS0 + 128 * b + kHalf * sg + 32 * c, s + 32 * c);
            } else {
#pragma unroll
                for (int j = 0; j < kHalf; ++j) s[j] = 0.f;
            }
            const int nvalid = (cend - cstart - t * kCsTile < kCsTile) ? cend - cstart - t * kCsTile
                                                                        : kCsTile;
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < kHalf; ++j) {
                s[j] = (kHalf * sg + j < nvalid) ? s[j] * p.scale_log2 : -INFINITY;  // NaN-safe select
                mx = fmaxf(mx, s[j]);
            }
            xmax[(2 * b + sg) * kCsRows + r] = mx;
            if (softmax_bar256_or(!landed || fail_local)) {  // every thread breaks, or none
                failed = true;
                break;
            }
            mx = fmaxf(mx, xmax[(2 * b + 1 - sg) * kCsRows + r]);  // the row's tile maximum
            m_true = fmaxf(m_true, mx);
            float alpha = 1.f;
            const bool need = mx > m_run + kLazyRescale;  // the same in both groups' threads
            if (need) {  // first tile: alpha = 2^-inf = 0 on an empty sum
                alpha = fast_exp2(m_run - mx);
                m_run = mx;
                l_run *= alpha;
            }
            uint32_t pk[kHalf / 2];
#pragma unroll
            for (int j = 0; j < kHalf / 2; ++j) {
                const float a = fast_exp2(s[2 * j] - m_run), c = fast_exp2(s[2 * j + 1] - m_run);
                l_run += a + c;
                pk[j] = narrow2<BF16>(a, c);
            }
            if (t >= 1) {
                // the previous tile's P.V must be done before P is rewritten or
                // O rescaled (a failure is everyone's at the next exchange)
                const bool done = __all_sync(kFullMask, mbar_wait(&bar[kCsODone], (t - 1) & 1));
                if (!done) {
                    fail_local = true;
                } else {
                    tc_fence_after();
                    if (__any_sync(kFullMask, need)) {
#pragma unroll
                        for (int c = 0; c < kOHalf / 32; ++c) {
                            float o[32];
                            tmem_ld32(tmem + lane_addr + kCsO + kOHalf * sg + 32 * c, o);
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] *= alpha;
                            tmem_st32(tmem + lane_addr + kCsO + kOHalf * sg + 32 * c, o);
                        }
                        tmem_wait_st();
                    }
                }
            }
            // P row r, the group's 64 positions, in the K-major operand layout
#pragma unroll
            for (int j = 0; j < kHalf / 8; ++j) {  // 16-byte chunk j of slab sg
                const uint32_t off = sg * S::SLAB + (r >> 3) * 1024 + (r & 7) * 128 +
                                     ((j ^ (r & 7)) << 4);
                *reinterpret_cast<uint4 *>(smem + S::OFF_P + off) =
                    make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[kCsPReady0 + b]);
        }
        // the row's sum over both groups' positions (and any failure, everyone's)
        xsum[sg * kCsRows + r] = l_run;
        failed |= softmax_bar256_or(failed || fail_local);
        l_run += xsum[(1 - sg) * kCsRows + r];
        if (!failed && ntiles > 0) {
            const bool done = mbar_wait(&bar[kCsODone], (ntiles - 1) & 1);
            failed = !__all_sync(kFullMask, done);
        }
        if (failed && lane == 0) {
            record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
        }
        // This chunk's partial of row r, staged in shared memory for the
        // cluster merge: m the true maximum, l relative to it, O normalised.
        // The K/V ring is free: every copy has landed and every MMA is done.
        // A failed or empty chunk contributes l = 0.
        keep_have = !failed && ntiles > 0;  // warp-uniform
        keep_inv = keep_have ? 1.0f / l_run : 0.f;
        if (sg == 0) {
            cm[r] = keep_have ? m_true : -INFINITY;
            cl[r] = keep_have ? l_run * fast_exp2(m_run - m_true) : 0.f;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0 && ntiles > 0) {
        // let copies and MMAs still in flight finish before shared memory and
        // TMEM are released (each wait is bounded)
        const int last = ntiles - 1;
        (void)mbar_wait(&bar[kCsFull0 + (last & 1)], (last >> 1) & 1);
        (void)mbar_wait(&bar[kCsEmpty0 + (last & 1)], (last >> 1) & 1);
    }

    // ---------------------------------------------------------- cluster merge
    // The cluster's CTAs hold consecutive chunks of the same rows (split-KV
    // step 3 through distributed shared memory).  Every CTA reads the CL
    // (m, l) pairs of each row, scales its own O row by its weight and pushes
    // it into the shared memory of the CTA that owns the row (rank r / R);
    // each owner sums what it received and writes one partial per row to
    // slot blockIdx.y / cluster.  The K/V ring is free by now: every copy
    // has landed and every MMA is done.
    const int CL = p.cluster;
    const int R = kCsRows / CL;
    const uint32_t rank = cluster_ctarank();
    float *wts = reinterpret_cast<float *>(smem + S::OFF_P);  // [R][CL] (R * CL = 128)
    float *rowM = wts + kCsRows;
    float *rowL = rowM + kCsRows;
    __syncwarp();
    cluster_sync();  // every chunk's (m, l) is visible
    if (warp >= 2) {
        const int sg = (warp - 2) >> 2;        // softmax group: pushes O dims [sg d/2, (sg + 1) d/2)
        const int r = (warp & 3) * 32 + lane;  // row of the tile = TMEM lane
        float mc[kCsMaxCluster], lc[kCsMaxCluster];
#pragma unroll
        for (int c = 0; c < kCsMaxCluster; ++c) {
            mc[c] = -INFINITY;
            lc[c] = 0.f;
            if (c < CL) {
                mc[c] = ld_cluster_f32(map_cluster(smem_addr(cm + r), c));
                lc[c] = ld_cluster_f32(map_cluster(smem_addr(cl + r), c));
            }
        }
        float M = -INFINITY;
#pragma unroll
        for (int c = 0; c < kCsMaxCluster; ++c) M = fmaxf(M, (lc[c] > 0.f) ? mc[c] : -INFINITY);
        float w[kCsMaxCluster], L = 0.f;
#pragma unroll
        for (int c = 0; c < kCsMaxCluster; ++c) {
            w[c] = (lc[c] > 0.f) ? lc[c] * fast_exp2(mc[c] - M) : 0.f;
            L += w[c];
        }
        const float invL = L > 0.f ? 1.0f / L : 0.f;
        float w_self = 0.f;
#pragma unroll
        for (int c = 0; c < kCsMaxCluster; ++c) {
            w[c] *= invL;
            if (c == (int)rank) w_self = w[c];
        }
        if (sg == 0 && r / R == (int)rank) {  // this CTA owns row r
            const int jl = r % R;
#pragma unroll
            for (int c = 0; c < kCsMaxCluster; ++c)
                if (c < CL) wts[jl * CL + c] = w[c];
            rowM[jl] = M;
            rowL[jl] = L;
        }
        if (keep_have) {
            tc_fence_after();
            const float sc = w_self * keep_inv;  // normalise, then weigh
            const uint32_t dst = map_cluster(
                smem_addr(ost + ((int)rank * R + r % R) * (D + 4)), (uint32_t)(r / R));
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                float o[32];
                const int col = (D / 2) * sg + 32 * c;
                tmem_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + kCsO + col, o);
                if (w_self != 0.f) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        st_cluster_f4(dst + (col + 4 * i) * 4,
                                      make_float4(o[4 * i] * sc, o[4 * i + 1] * sc,
                                                  o[4 * i + 2] * sc, o[4 * i + 3] * sc));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kCsCols);
    }
    __syncwarp();
    cluster_sync();  // every pushed row has landed
    if (warp >= 2) {
        const int t = threadIdx.x - 64;
        const int slot = blockIdx.y / CL;
        switch (CL) {
            case 1: owner_sum<D, 1>(p, ost, wts, rowM, rowL, rank, t, mt, kvh, slot); break;
            case 2: owner_sum<D, 2>(p, ost, wts, rowM, rowL, rank, t, mt, kvh, slot); break;
            case 4: owner_sum<D, 4>(p, ost, wts, rowM, rowL, rank, t, mt, kvh, slot); break;
            default: owner_sum<D, 8>(p, ost, wts, rowM, rowL, rank, t, mt, kvh, slot); break;
        }
    }
}

// ------------------------------------------------------------------ host side
using CsKernel = void (*)(const CascadeParams, const CUtensorMap, const CUtensorMap);

static CsKernel pick_cascade(bool bf16, int D, int *smem) {
    if (D == 128) {
        *smem = CsShape<128>::SMEM_BYTES;
        return bf16 ? cascade_prefix_kernel<true, 128> : cascade_prefix_kernel<false, 128>;
    }
    *smem = CsShape<64>::SMEM_BYTES;
    return bf16 ? cascade_prefix_kernel<true, 64> : cascade_prefix_kernel<false, 64>;
}

// Clusters of `cl` CTAs of this kernel that can be resident at once on the
// current device (0 if the query fails), cached per (kernel, size).
static int active_clusters(CsKernel k, int smem, int cl) {
    static std::mutex mu;
    static std::map<std::pair<const void *, int>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const auto key = std::make_pair(reinterpret_cast<const void *>(k), dev * 16 + cl);
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    if (!ensure_smem_attr(reinterpret_cast<const void *>(k), smem)) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, (unsigned)cl, 1);
    cfg.blockDim = dim3(kCsThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)cl;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void *>(k), &cfg) != cudaSuccess)
        n = 0;
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = n;
    return n;
}

CascadeChunks cascade_chunks(int prefix_len, int num_rows, int num_kv_heads, int head_dim,
                             bool bf16) {
    const int ntiles = (prefix_len + kCsTile - 1) / kCsTile;
    const int per_chunk = ((num_rows + kCsRows - 1) / kCsRows) * num_kv_heads;
    const int sms = sm_count();
    int n = per_chunk > 0 ? (sms > 0 ? sms : 1) / per_chunk : 1;
    if (n > ntiles) n = ntiles;
    if (n < 1) n = 1;
    const int tiles_per_chunk = (ntiles + n - 1) / n;
    n = (ntiles + tiles_per_chunk - 1) / tiles_per_chunk;
    CascadeChunks c;
    c.chunk_tokens = tiles_per_chunk * kCsTile;
    // Clusters of 1, 2, 4 or 8 consecutive chunks (portable sizes that divide
    // the grid; chunks added to fill the last cluster are empty): the largest
    // that still lets the whole grid be resident at once, as one CTA per
    // cluster-free SM would be.
    int smem = 0;
    CsKernel k = pick_cascade(bf16, head_dim, &smem);
    c.cluster = 1;
    c.num_chunks = n;
    for (int cl = kCsMaxCluster; cl >= 2; cl /= 2) {
        if (cl >= 2 * n) continue;  // more empty chunks than real ones
        const int nc = (n + cl - 1) / cl * cl;
        const int ctas = nc * per_chunk;
        const int fit = active_clusters(k, smem, cl) * cl;
        const int plain = sms > 0 ? sms : 1;
        const bool one_wave = n * per_chunk <= plain;
        if (fit >= (ctas < plain ? ctas : plain) && (!one_wave || ctas <= fit)) {
            c.cluster = cl;
            c.num_chunks = nc;
            break;
        }
    }
    return c;
}

pa_status launch_cascade_prefix(const CascadeParams &cp, const void *k_pool, const void *v_pool,
                                bool bf16, int head_dim, cudaStream_t stream) {
    if (cp.num_seqs == 0 || cp.num_chunks == 0) return PA_OK;
    const int mtiles = (cp.num_seqs * cp.group + kCsRows - 1) / kCsRows;
    if (cp.num_chunks > 65535 || cp.num_kv_heads > 65535) return PA_ERR_INVALID;
    int smem = 0;
    CsKernel k = pick_cascade(bf16, head_dim, &smem);
    if (!ensure_smem_attr(reinterpret_cast<const void *>(k), smem)) return PA_ERR_CUDA;
    const int64_t rows = (int64_t)cp.num_blocks * cp.num_kv_heads * cp.block_size;
    CUtensorMap mk, mv;
    if (!pool_tensor_map(&mk, k_pool, rows, head_dim, bf16) ||
        !pool_tensor_map(&mv, v_pool, rows, head_dim, bf16))
        return PA_ERR_CUDA;
    if (cp.cluster < 1 || cp.cluster > kCsMaxCluster || cp.num_chunks % cp.cluster)
        return PA_ERR_INVALID;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)mtiles, (unsigned)cp.num_chunks, (unsigned)cp.num_kv_heads);
    cfg.blockDim = dim3(kCsThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = (unsigned)cp.cluster;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, k, cp, mk, mv) != cudaSuccess) return PA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
