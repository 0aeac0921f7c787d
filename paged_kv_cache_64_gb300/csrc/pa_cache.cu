// pa_cache_write (reshape_and_cache), pa_copy_blocks (copy-on-write block
// duplication), the per-device error word and pa_check_error.
//
// Both kernels are pure 16-byte-vector copies: one thread moves one 16-byte
// piece per iteration, consecutive threads move consecutive pieces, so every
// warp reads and writes whole 512-byte runs.  They are bound by HBM (copy
// bytes), and tiny next to decode.
#include <cmath>
#include <cstdint>
#include <mutex>
#include <set>
#include <utility>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

// One error word per device, shared by every kernel of the library.
__device__ int g_error_word;

int *error_word() {
    static std::mutex mu;
    static int *ptrs[128] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<int *>(p);
    }
    return ptrs[dev];
}

int sm_count() {
    static std::mutex mu;
    static int counts[128] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!counts[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        counts[dev] = n;
    }
    return counts[dev];
}

bool ensure_smem_attr(const void *kernel, int bytes) {
    static std::mutex mu;
    static std::set<std::pair<const void *, int>> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({kernel, dev})) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess)
        return false;
    // Prefer the largest shared-memory carveout so several CTAs fit per SM.
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return false;
    done.insert({kernel, dev});
    return true;
}

// ---------------------------------------------------------------- cache write
// Piece index i covers token t, K-or-V, KV head h, 16-byte piece c of the
// head_dim vector:  i = ((t * 2 + kv) * num_kv_heads + h) * pieces + c.
__global__ void cache_write_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                                   const int64_t *__restrict__ slot_mapping, int num_tokens,
                                   uint4 *__restrict__ k_pool, uint4 *__restrict__ v_pool,
                                   int64_t num_slots, int num_kv_heads, int pieces, int block_size,
                                   int *err) {
    asm volatile("griddepcontrol.wait;" ::: "memory");  // programmatic dependent launch
    const int64_t per_token = 2ll * num_kv_heads * pieces;
    const int64_t total = per_token * num_tokens;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / per_token;
        const int64_t r = i - t * per_token;
        const int is_v = (int)(r / ((int64_t)num_kv_heads * pieces));
        const int64_t r2 = r - (int64_t)is_v * num_kv_heads * pieces;
        const int h = (int)(r2 / pieces);
        const int c = (int)(r2 - (int64_t)h * pieces);
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) {
            record_error(err, PA_ERR_BAD_INDEX);
            continue;
        }
        const int64_t blk = slot / block_size;
        const int64_t off = slot - blk * block_size;
        const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * pieces + c;
        const int64_t src = ((int64_t)t * num_kv_heads + h) * pieces + c;
        if (is_v)
            v_pool[dst] = v_new[src];
        else
            k_pool[dst] = k_new[src];
    }
}

// ---------------------------------------------------------------- copy blocks
constexpr int kMaxLayersPerLaunch = 64;

struct PoolPtrs {
    uint4 *k[kMaxLayersPerLaunch];
    uint4 *v[kMaxLayersPerLaunch];
};

// grid.y: pair, grid.z: layer * 2 + (0 = K, 1 = V); x covers the block's
// 16-byte pieces.
// FP8 cache write: token t's K/V (16-bit, [T][Hkv][d]) quantised to E4M3
// codes with the pools' scales (code = nearest(x * inv_scale), fp32) and
// stored at its slot.  One work item is 16 elements: 32 bytes read, 16
// written.
template <bool BF16>
__global__ void cache_write_fp8_kernel(const uint4 *__restrict__ k_new,
                                       const uint4 *__restrict__ v_new,
                                       const int64_t *__restrict__ slot_mapping, int num_tokens,
                                       uint4 *__restrict__ k_pool, uint4 *__restrict__ v_pool,
                                       int64_t num_slots, int num_kv_heads, int chunks,
                                       int block_size, float k_inv, float v_inv, int *err) {
    asm volatile("griddepcontrol.wait;" ::: "memory");  // programmatic dependent launch
    const int64_t per_token = 2ll * num_kv_heads * chunks;
    const int64_t total = per_token * num_tokens;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / per_token;
        const int64_t r = i - t * per_token;
        const int is_v = (int)(r / ((int64_t)num_kv_heads * chunks));
        const int64_t r2 = r - (int64_t)is_v * num_kv_heads * chunks;
        const int h = (int)(r2 / chunks);
        const int c = (int)(r2 - (int64_t)h * chunks);
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) {
            record_error(err, PA_ERR_BAD_INDEX);
            continue;
        }
        const int64_t blk = slot / block_size;
        const int64_t off = slot - blk * block_size;
        const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * chunks + c;
        const int64_t src = (((int64_t)t * num_kv_heads + h) * chunks + c) * 2;
        const uint4 *in = is_v ? v_new : k_new;
        const uint4 q = quantize16_e4m3<BF16>(in[src], in[src + 1], is_v ? v_inv : k_inv);
        (is_v ? v_pool : k_pool)[dst] = q;
    }
}

constexpr int kCopyPer = 4;  // 16-byte pieces a thread copies per round

__global__ void copy_blocks_kernel(const PoolPtrs pools, const int64_t *__restrict__ mapping,
                                   int num_blocks, int64_t pieces, int *err) {
    const int pair = blockIdx.y;
    const int layer = blockIdx.z >> 1;
    const int64_t src = mapping[2 * pair];
    const int64_t dst = mapping[2 * pair + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && blockIdx.x == 0) record_error(err, PA_ERR_BAD_INDEX);
        return;
    }
    uint4 *pool = (blockIdx.z & 1) ? pools.v[layer] : pools.k[layer];
    const uint4 *s = pool + src * pieces;
    uint4 *d = pool + dst * pieces;
    // kCopyPer pieces a thread, all loaded before any is stored (the pairs
    // are independent, so no store of this launch feeds one of its loads):
    // one memory round trip instead of one per piece
    const int64_t stride = (int64_t)gridDim.x * blockDim.x * kCopyPer;
    for (int64_t i0 = blockIdx.x * (int64_t)blockDim.x * kCopyPer + threadIdx.x; i0 < pieces;
         i0 += stride) {
        uint4 v[kCopyPer];
#pragma unroll
        for (int k = 0; k < kCopyPer; ++k) {
            const int64_t i = i0 + (int64_t)k * blockDim.x;
            if (i < pieces) v[k] = s[i];
        }
#pragma unroll
        for (int k = 0; k < kCopyPer; ++k) {
            const int64_t i = i0 + (int64_t)k * blockDim.x;
            if (i < pieces) d[i] = v[k];
        }
    }
}

// Waits on a barrier that never completes; the bounded wait must give up.
__global__ void wait_timeout_kernel(int *err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0)) record_error(err, PA_ERR_DEVICE_TIMEOUT);
}

}  // namespace pa

using namespace pa;

extern "C" {

int pa_version(void) { return 100; }

const char *pa_status_string(pa_status s) {
    switch (s) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID: return "invalid argument";
        case PA_ERR_OUT_OF_BLOCKS: return "out of blocks";
        case PA_ERR_UNSUPPORTED: return "unsupported shape";
        case PA_ERR_CUDA: return "CUDA error";
        case PA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case PA_ERR_BAD_INDEX: return "out-of-range index met on the device";
        case PA_ERR_NOT_FOUND: return "unknown or duplicate sequence id";
        case PA_ERR_TOO_LARGE: return "split-KV partials exceed the fixed static scratch";
    }
    return "unknown status";
}

pa_status pa_cache_write_fp8(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                             int num_tokens, void *k_pool, void *v_pool, int num_blocks,
                             int num_kv_heads, int head_dim, int block_size, float k_scale,
                             float v_scale, pa_dtype dtype, void *stream) {
    if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 || block_size <= 0)
        return PA_ERR_INVALID;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID;
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
        return PA_ERR_INVALID;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !slot_mapping || !k_pool || !v_pool) return PA_ERR_INVALID;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool))
        return PA_ERR_INVALID;
    int *err = error_word();
    if (!err) return PA_ERR_CUDA;
    const int chunks = head_dim / 16;
    const int64_t total = 2ll * num_tokens * num_kv_heads * chunks;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = 16ll * (sm_count() > 0 ? sm_count() : 148);
    if (blocks > cap) blocks = cap;
    const float k_inv = 1.0f / k_scale, v_inv = 1.0f / v_scale;
    auto kern = dtype == PA_BF16 ? cache_write_fp8_kernel<true> : cache_write_fp8_kernel<false>;
    kern<<<(unsigned)blocks, threads, 0, as_stream(stream)>>>(
        static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), slot_mapping,
        num_tokens, static_cast<uint4 *>(k_pool), static_cast<uint4 *>(v_pool),
        (int64_t)num_blocks * block_size, num_kv_heads, chunks, block_size, k_inv, v_inv, err);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_cache_write(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                         int num_tokens, void *k_pool, void *v_pool, int num_blocks,
                         int num_kv_heads, int head_dim, int block_size, pa_dtype dtype,
                         void *stream) {
    if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 || block_size <= 0)
        return PA_ERR_INVALID;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !slot_mapping || !k_pool || !v_pool) return PA_ERR_INVALID;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool))
        return PA_ERR_INVALID;
    int *err = error_word();
    if (!err) return PA_ERR_CUDA;
    const int pieces = head_dim * 2 / 16;
    const int64_t total = 2ll * num_tokens * num_kv_heads * pieces;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = 16ll * (sm_count() > 0 ? sm_count() : 148);
    if (blocks > cap) blocks = cap;
    cache_write_kernel<<<(unsigned)blocks, threads, 0, as_stream(stream)>>>(
        static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), slot_mapping,
        num_tokens, static_cast<uint4 *>(k_pool), static_cast<uint4 *>(v_pool),
        (int64_t)num_blocks * block_size, num_kv_heads, pieces, block_size, err);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_copy_blocks(void *const *k_pools, void *const *v_pools, int num_layers,
                         const int64_t *block_mapping, int num_pairs, int num_blocks,
                         size_t block_bytes, void *stream) {
    if (num_layers < 1 || num_layers > 1024 || num_pairs < 0 || num_blocks <= 0 ||
        block_bytes == 0 || block_bytes % 16 != 0 || !k_pools || !v_pools)
        return PA_ERR_INVALID;
    if (num_pairs == 0) return PA_OK;
    if (!block_mapping || num_pairs > 65535) return PA_ERR_INVALID;
    for (int l = 0; l < num_layers; ++l)
        if (!k_pools[l] || !v_pools[l] || !aligned16(k_pools[l]) || !aligned16(v_pools[l]))
            return PA_ERR_INVALID;
    int *err = error_word();
    if (!err) return PA_ERR_CUDA;
    const int64_t pieces = (int64_t)(block_bytes / 16);
    const int threads = 256;
    int64_t bx = (pieces + threads * kCopyPer - 1) / (threads * kCopyPer);
    if (bx < 1) bx = 1;
    if (bx > 65535) bx = 65535;
    for (int l0 = 0; l0 < num_layers; l0 += kMaxLayersPerLaunch) {
        const int nl = num_layers - l0 < kMaxLayersPerLaunch ? num_layers - l0
                                                             : kMaxLayersPerLaunch;
        PoolPtrs p{};
        for (int i = 0; i < nl; ++i) {
            p.k[i] = static_cast<uint4 *>(k_pools[l0 + i]);
            p.v[i] = static_cast<uint4 *>(v_pools[l0 + i]);
        }
        dim3 grid((unsigned)bx, (unsigned)num_pairs, (unsigned)(2 * nl));
        copy_blocks_kernel<<<grid, threads, 0, as_stream(stream)>>>(p, block_mapping, num_blocks,
                                                                    pieces, err);
        if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    }
    return PA_OK;
}

pa_status pa_selftest_wait_timeout(void *stream) {
    int *err = error_word();
    if (!err) return PA_ERR_CUDA;
    wait_timeout_kernel<<<1, 32, 0, as_stream(stream)>>>(err);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_check_error(void *stream) {
    int *err = error_word();
    if (!err) return PA_ERR_CUDA;
    if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return PA_ERR_CUDA;
    int value = 0;
    if (cudaMemcpy(&value, err, sizeof value, cudaMemcpyDeviceToHost) != cudaSuccess)
        return PA_ERR_CUDA;
    if (value != 0) {
        const int zero = 0;
        if (cudaMemcpy(err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return PA_ERR_CUDA;
    }
    return static_cast<pa_status>(value);
}

}  // extern "C"
