// Inline-PTX helpers for sm_103a: mbarriers, TMA tensor loads, proxy fences,
// the global timer, and the error-free float transformations used by the
// mat-vec epilogue.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace xq {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier ---------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Makes the barrier initialisation visible to other threads and to the async
// (TMA) proxy.  The proxy fence is required: a TMA completion that reaches a
// barrier whose initialisation the async proxy has not been ordered after
// raised an illegal-address exception on GB300.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t phase) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(phase)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Status bits of the device status word.
constexpr uint32_t kStatusWaitTimeout = 1u;
// A wait that has not completed after this long is treated as lost.
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

// Bounded wait on phase `phase` of `bar`.  Returns false (and sets the status
// word) if the phase has not completed within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t phase,
                                                  uint32_t *status) {
    if (mbar_try_wait(bar, phase)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, phase)) return true;
        if ((it & 63u) == 0u && global_timer_ns() - t0 > kWaitLimitNs) {
            atomicOr(status, kStatusWaitTimeout);
            return false;
        }
    }
}

// ---- TMA ------------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 2-D tiled tensor load global -> shared, completion counted on `bar` in bytes.
// x is the innermost coordinate in elements (bytes here); it must be a multiple
// of 16 bytes, which every caller guarantees (x = 144 * chunk).
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *tmap, int32_t x,
                                            int32_t y, uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Orders this thread's preceding generic-proxy shared-memory accesses (after a
// warp barrier, those of the whole warp) before its following async-proxy ones.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ---- integer dot ------------------------------------------------------------------
// Four int8 x int8 products summed into c (signed x signed; a nibble byte
// 0..15 reads the same as signed).
__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) {
    return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

__device__ __forceinline__ float f16_bits_to_f32(uint32_t bits16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

// ---- error-free transformations (Ogita, Rump & Oishi, "Accurate Sum and Dot
// Product", SIAM J. Sci. Comput. 26(6), 2005: TwoSum and TwoProduct with FMA) --
// Explicit _rn intrinsics keep the compiler from contracting or reassociating.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ void two_prod(float a, float b, float &p, float &e) {
    p = __fmul_rn(a, b);
    e = __fmaf_rn(a, b, -p);
}

// acc (hi, lo) += v (a value with its own small correction term v_lo).
__device__ __forceinline__ void acc_add(float &hi, float &lo, float v, float v_lo) {
    float s, e;
    two_sum(hi, v, s, e);
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(e, v_lo));
}

}  // namespace xq
