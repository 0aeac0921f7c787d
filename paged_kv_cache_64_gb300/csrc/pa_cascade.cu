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
// (6 warps):
//   warp 0      producer: TMA copies of 16-row boxes through the prefix's
//               block-table entries into a 2-stage K/V ring;
//   warp 1      allocates TMEM; lane 0 issues every MMA and commits;
//   warps 2..5  softmax / epilogue, one query row (TMEM lane) per thread:
//               the whole 128-position score row is in the thread's
//               registers, so row max and sum need no shuffles.
// Each CTA leaves, for each of its rows, the (m, l, O) partial of its chunk
// in workspace slot `chunk` (m the true base-2 maximum, l relative to it, O
// normalised), as the split-KV partition kernels do.
#include <cmath>
#include <cstdint>

#include "pa_common.cuh"
#include "pa_decode.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {

constexpr int kCsTile = 128;   // positions per tile: N of q.K^T, K of P.V
constexpr int kCsRows = 128;   // query rows per CTA: M of both products
constexpr int kCsWarps = 6;
constexpr int kCsThreads = kCsWarps * 32;
constexpr int kCsCols = 512;   // TMEM columns: S x2 (128 each) and O (d)
constexpr int kCsS0 = 0, kCsO = 256;

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
    static constexpr int OFF_BAR = OFF_STAGE + 2 * STAGE;
    static constexpr int OFF_MISC = OFF_BAR + kNumCsBars * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack to align the base to 1 KiB
    static_assert(OFF_P % 1024 == 0 && OFF_STAGE % 1024 == 0 && STAGE % 1024 == 0, "atoms");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

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
    const int cend = (cstart + p.chunk_tokens < p.prefix_len) ? cstart + p.chunk_tokens : p.prefix_len;
    const int nunits = (cend - cstart) / kUnit;  // whole blocks, so whole 16-position units
    const int ntiles = (cend - cstart + kCsTile - 1) / kCsTile;

    pdl_wait();  // inputs may come from the previous kernel on the stream
    if (threadIdx.x == 0) {
        const int counts[kNumCsBars] = {1, 1, 1, 1, 4, 1, 1, 4, 4, 1};
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

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        const int32_t *prefix_table = p.block_tables;  // sequence 0's row
        bool ok = true;
        for (int t = 0; t < ntiles; ++t) {
            const int st = t & 1;
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
            int row0 = 0;  // first row of the unit in the 2-D view [NB*Hkv*B, d]
            if (lane < nu) {
                const int pos = cstart + (u0 + lane) * kUnit;
                int phys = prefix_table[pos >> p.log2_block];
                if ((unsigned)phys >= (unsigned)p.num_blocks) {
                    record_error(p.err, PA_ERR_BAD_INDEX);
                    phys = 0;
                }
                row0 = (phys * p.num_kv_heads + kvh) * p.block_size + (pos & (p.block_size - 1));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&bar[kCsFull0 + st], nu * S::KH * 2048 * 2);
            for (int j = 0; j < nu; ++j) {
                const int r0 = __shfl_sync(kFullMask, row0, j);
                if (lane == 0) {
#pragma unroll
                    for (int h = 0; h < S::KH; ++h) {
                        tma_load_2d(kbuf + h * S::SLAB + j * 2048, &tmap_k, 64 * h, r0,
                                    &bar[kCsFull0 + st]);
                        tma_load_2d(vbuf + h * S::SLAB + j * 2048, &tmap_v, 64 * h, r0,
                                    &bar[kCsFull0 + st]);
                    }
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
            bool ok = mbar_wait(&bar[kCsQReady], 0) && issue_qk(0);
            for (int t = 0; t < ntiles && ok; ++t) {
                // q.K^T of the next tile runs while the softmax works on this one
                if (t + 1 < ntiles && !issue_qk(t + 1)) {
                    ok = false;
                    break;
                }
                const int st = t & 1;
                if (!mbar_wait(&bar[kCsPReady0 + st], (t >> 1) & 1)) {
                    ok = false;
                    break;
                }
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
            }
            if (!ok) {
                record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
            }
        }
    } else {
        // ---------------------------------------------------------- softmax / epilogue
        const int quad = warp & 3;               // TMEM lane quadrant this warp may access
        const int r = quad * 32 + lane;          // query row of the tile = TMEM lane
        const int st_id = threadIdx.x - 64;      // 0..127
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;

        // Q tile (128 rows x d, K-major, 128-byte swizzle), rows past the last
        // sequence zero.  Unscaled: the scale is applied to S in fp32.
        // all of the thread's loads in flight before the first store
        constexpr int kQPer = kCsRows * (D / 8) / 128;
        uint4 qv[kQPer];
#pragma unroll
        for (int i = 0; i < kQPer; ++i) {
            const int ci = st_id + 128 * i;
            const int rr = ci / (D / 8), c = ci % (D / 8);
            const int gr = mt * kCsRows + rr;
            qv[i] = make_uint4(0, 0, 0, 0);
            if (gr < rows_total)
                qv[i] = *reinterpret_cast<const uint4 *>(
                    p.q + ((int64_t)(gr / G) * p.num_q_heads + (int64_t)kvh * G + gr % G) * D + c * 8);
        }
#pragma unroll
        for (int i = 0; i < kQPer; ++i) {
            const int ci = st_id + 128 * i;
            const int rr = ci / (D / 8), c = ci % (D / 8);
            *reinterpret_cast<uint4 *>(smem + S::OFF_Q + sw128_offset(rr, c * 8, S::SLAB)) = qv[i];
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kCsQReady]);

        float m_run = -INFINITY, m_true = -INFINITY, l_run = 0.f;
        bool failed = false;
        for (int t = 0; t < ntiles; ++t) {
            const int b = t & 1;
            const bool landed = mbar_wait(&bar[kCsSFull0 + b], (t >> 1) & 1);
            if (!__all_sync(kFullMask, landed)) {
                failed = true;
                break;
            }
            tc_fence_after();
            float s[kCsTile];
#pragma unroll
            for (int c = 0; c < kCsTile / 32; ++c)
                tmem_ld32(tmem + lane_addr + kCsS0 + 128 * b + 32 * c, s + 32 * c);
            const int nvalid = (cend - cstart - t * kCsTile < kCsTile) ? cend - cstart - t * kCsTile
                                                                        : kCsTile;
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < kCsTile; ++j) {
                s[j] = (j < nvalid) ? s[j] * p.scale_log2 : -INFINITY;  // select: NaN-safe
                mx = fmaxf(mx, s[j]);
            }
            m_true = fmaxf(m_true, mx);
            float alpha = 1.f;
            const bool need = mx > m_run + kLazyRescale;
            if (need) {  // first tile: alpha = 2^-inf = 0 on an empty sum
                alpha = fast_exp2(m_run - mx);
                m_run = mx;
                l_run *= alpha;
            }
            uint32_t pk[kCsTile / 2];
#pragma unroll
            for (int j = 0; j < kCsTile / 2; ++j) {
                const float a = fast_exp2(s[2 * j] - m_run), c = fast_exp2(s[2 * j + 1] - m_run);
                l_run += a + c;
                pk[j] = narrow2<BF16>(a, c);
            }
            if (t >= 1) {
                // the previous tile's P.V must be done before P is rewritten or
                // O rescaled
                const bool done = mbar_wait(&bar[kCsODone], (t - 1) & 1);
                if (!__all_sync(kFullMask, done)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                if (__any_sync(kFullMask, need)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        tmem_ld32(tmem + lane_addr + kCsO + 32 * c, o);
            #pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        tmem_st32(tmem + lane_addr + kCsO + 32 * c, o);
                    }
                    tmem_wait_st();
                }
            }
            // P row r (128 positions) in the K-major operand layout
#pragma unroll
            for (int c = 0; c < kCsTile / 8; ++c) {
                const uint32_t off = (c >> 3) * S::SLAB + (r >> 3) * 1024 + (r & 7) * 128 +
                                     (((c & 7) ^ (r & 7)) << 4);
                *reinterpret_cast<uint4 *>(smem + S::OFF_P + off) =
                    make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[kCsPReady0 + b]);
        }
        if (!failed) {
            const bool done = mbar_wait(&bar[kCsODone], (ntiles - 1) & 1);
            failed = !__all_sync(kFullMask, done);
        }
        if (failed) {
            if (lane == 0) {
                record_error(p.err, PA_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
            }
        } else {
            tc_fence_after();
            const int gr = mt * kCsRows + r;
            const bool row_valid = gr < rows_total;
            const int64_t row =
                ((int64_t)(gr / G) * p.num_q_heads + (int64_t)kvh * G + gr % G) * p.ws_parts + chunk;
            const float inv = 1.0f / l_run;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float o[32];
                tmem_ld32(tmem + lane_addr + kCsO + 32 * c, o);
                    if (row_valid) {
                    float4 *dst = reinterpret_cast<float4 *>(p.part_o + row * D + 32 * c);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv,
                                             o[4 * i + 3] * inv);
                }
            }
            if (row_valid) {
                p.part_m[row] = m_true;
                p.part_l[row] = l_run * fast_exp2(m_run - m_true);
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
        (void)mbar_wait(&bar[kCsFull0 + (last & 1)], (last >> 1) & 1);
        (void)mbar_wait(&bar[kCsEmpty0 + (last & 1)], (last >> 1) & 1);
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kCsCols);
    }
}

// ------------------------------------------------------------------ host side
int cascade_chunk_tokens(int prefix_len, int num_rows, int num_kv_heads) {
    const int ntiles = (prefix_len + kCsTile - 1) / kCsTile;
    const int per_chunk = ((num_rows + kCsRows - 1) / kCsRows) * num_kv_heads;
    const int sms = sm_count();
    int n = per_chunk > 0 ? (sms > 0 ? sms : 1) / per_chunk : 1;
    if (n < 1) n = 1;
    if (n > ntiles) n = ntiles;
    if (n < 1) n = 1;
    const int tiles_per_chunk = (ntiles + n - 1) / n;
    return tiles_per_chunk * kCsTile;
}

using CsKernel = void (*)(const CascadeParams, const CUtensorMap, const CUtensorMap);

static CsKernel pick_cascade(bool bf16, int D, int *smem) {
    if (D == 128) {
        *smem = CsShape<128>::SMEM_BYTES;
        return bf16 ? cascade_prefix_kernel<true, 128> : cascade_prefix_kernel<false, 128>;
    }
    *smem = CsShape<64>::SMEM_BYTES;
    return bf16 ? cascade_prefix_kernel<true, 64> : cascade_prefix_kernel<false, 64>;
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
    dim3 grid((unsigned)mtiles, (unsigned)cp.num_chunks, (unsigned)cp.num_kv_heads);
    if (launch_pdl(k, grid, dim3(kCsThreads), (size_t)smem, stream, cp, mk, mv) != cudaSuccess)
        return PA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
