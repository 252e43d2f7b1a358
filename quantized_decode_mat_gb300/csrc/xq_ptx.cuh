// Inline-PTX helpers for sm_103a: asynchronous shared-memory staging copies,
// the integer dot, and the error-free float transformations used by the
// mat-vec epilogue.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace xq {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- asynchronous 16-byte copies global -> shared (cp.async, sm_80+) ----------
// dst: shared address; src: 16-byte aligned global address; src_size 16 copies,
// 0 zero-fills the destination without reading global memory.  Bypasses L1.
__device__ __forceinline__ void cp_async_16_zfill(uint32_t dst, const void *src,
                                                  uint32_t src_size) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_size)
                 : "memory");
}

// The same without the source-size operand (a full 16-byte copy).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most n (0..7) of this thread's committed groups are pending.
__device__ __forceinline__ void cp_async_wait_pending(int n) {
    switch (n) {
        case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
        case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
        case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
        case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
        case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
        case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
        case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
        default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
    }
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---- integer dot ------------------------------------------------------------------
// Four int8 x int8 products summed into c (signed x signed; a nibble byte
// 0..15 reads the same as signed).
__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) {
    return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

// Four (unsigned byte x signed byte) products summed into c.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Four (unsigned byte x unsigned byte) products summed into c.
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
    uint32_t d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"((uint32_t)c));
    return (int)d;
}

// Byte permute in prmt's generic mode: the low three bits of selector nibble
// i pick byte i of the result from the eight bytes of (a, b); bit 3 set
// replicates the sign (top) bit of that byte over the whole result byte.
// (__byte_perm keeps only the low three bits of each nibble, which costs a
// masking operation per call when the selector is not a constant.)
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// ---- programmatic dependent launch (sm_90+) ------------------------------------------
// Wait until the grid launched before this one on the stream has completed and
// its memory writes are visible; returns at once when this grid was launched
// without the programmatic-serialization attribute.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Let the next grid on the stream (if launched with that attribute) start its
// prologue; it still waits for this grid's completion before it reads inputs.
__device__ __forceinline__ void grid_dependency_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier of the two warps of warp pair `pair` (barrier ids 2..;
// 0 is __syncthreads and 1 the RMSNorm workgroup's).
__device__ __forceinline__ void pair_barrier(int pair) {
    asm volatile("bar.sync %0, 64;" ::"r"(2 + pair) : "memory");
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

// acc (hi, lo) += v (a value with its own small correction term v_lo).  The
// result is symmetric in its two operands: TwoSum's sum and error term are,
// and the correction terms are added to each other before the error term, so
// a sum over a fixed pairing tree has the same bits whichever side of each
// pair holds the accumulator (a lane's own value or one received from
// another lane).
__device__ __forceinline__ void acc_add(float &hi, float &lo, float v, float v_lo) {
    float s, e;
    two_sum(hi, v, s, e);
    hi = s;
    lo = __fadd_rn(__fadd_rn(lo, v_lo), e);
}

}  // namespace xq
