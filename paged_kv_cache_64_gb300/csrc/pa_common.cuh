// Shared device helpers for the paged KV-cache kernels (sm_103a).
//
// Inline PTX for the Blackwell async-copy path: mbarrier init / arrive /
// bounded parity wait, and the 1-D bulk copy (cp.async.bulk, the TMA engine's
// untiled form) from global into shared memory that completes a transaction
// count on an mbarrier.  Plus packed fp32x2 math and 16-bit -> fp32 widening.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

constexpr unsigned kFullMask = 0xffffffffu;
// A bounded device wait gives up after this long and reports
// PA_ERR_DEVICE_TIMEOUT instead of hanging.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ void record_error(int *err, int code) {
    if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make initialised barriers visible to the async proxy (bulk-copy engine).
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Non-blocking test of the same (never suspends the thread): for issue loops
// that poll several barriers.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase with the given parity to complete; false after
// kWaitLimitNs without completion.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// 1-D bulk copy global -> shared; completion is signalled as `bytes`
// transaction bytes on `bar`.  Addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// 2^x on the special-function unit (PTX ex2.approx, flush-to-zero):
// 2^-inf = +0, which is what masked scores rely on.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Widen two packed 16-bit values (low half first) to fp32.
template <bool BF16>
__device__ __forceinline__ float2 widen2(uint32_t w) {
    if constexpr (BF16) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    } else {
        __half2 h;
        memcpy(&h, &w, sizeof h);
        return __half22float2(h);
    }
}

// Round two fp32 values to nearest-even 16-bit and pack (low half first).
template <bool BF16>
__device__ __forceinline__ uint32_t narrow2(float a, float b) {
    uint32_t w;
    if constexpr (BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        memcpy(&w, &h, sizeof w);
    } else {
        __half2 h = __floats2half2_rn(a, b);
        memcpy(&w, &h, sizeof w);
    }
    return w;
}

// FP8 KV cache (OCP E4M3 codes, one scale per pool).  Two fp32 values to
// two codes, nearest with ties to even, saturating at +-448 (PTX
// cvt.rn.satfinite.e4m3x2.f32; the first value in the low byte).
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// 16 16-bit values (two uint4, low element first) times `inv` in fp32, as
// 16 E4M3 codes.
template <bool BF16>
__device__ __forceinline__ uint4 quantize16_e4m3(uint4 a, uint4 b, float inv) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 x = widen2<BF16>(w[2 * i]), y = widen2<BF16>(w[2 * i + 1]);
        c[i] = e4m3x2_from_f32(x.x * inv, x.y * inv) |
               (e4m3x2_from_f32(y.x * inv, y.y * inv) << 16);
    }
    return make_uint4(c[0], c[1], c[2], c[3]);
}

}  // namespace pa
