// RMSNorm scale of one activation vector, in the summation order of the
// workgroup reduction in "25 - Writing XPU Kernels" 25.2.3: a workgroup of
// 256 items (eight waves of 32); item t adds x_t^2, x_{t+256}^2, ... in that
// order; each wave combines its 32 partials by an xor butterfly over item
// offsets 16, 8, 4, 2, 1; the eight wave partials are added to 0 from wave 0
// upward; scale = 1 / sqrt(total / n + 1e-5).  Every operation is one f32
// rounding with nothing contracted, so the scale is one defined value and
// the q8 codes of y = x * scale are decided the same way on every run.
//
// One warp evaluates that workgroup: lane j carries items 8j .. 8j+7, so
// each 256-value chunk is two 16-byte loads per lane and wave v is lanes
// 4v .. 4v+3.  The butterfly's offsets 16 and 8 are then lane offsets 2 and
// 1, and offsets 4, 2, 1 pair registers of one lane.  Each addition joins
// the same two partials as in the workgroup (f32 addition commutes), so the
// result is bit-identical, with no shared memory and no barrier.
#pragma once

#include <stdint.h>

namespace xq {

// All 32 lanes must call; every lane returns the scale.  x: 16-byte aligned,
// n a multiple of 256 and at most 2^24.
__device__ __forceinline__ float rms_scale_warp(const float *__restrict__ x, int64_t n, int lane) {
    float s[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) s[r] = 0.0f;
    const float4 *p = reinterpret_cast<const float4 *>(x) + 2 * lane;
#pragma unroll 8
    for (int64_t k = 0; k < n; k += 256, p += 64) {
        const float4 u = __ldg(p), v = __ldg(p + 1);
        s[0] = __fadd_rn(s[0], __fmul_rn(u.x, u.x));
        s[1] = __fadd_rn(s[1], __fmul_rn(u.y, u.y));
        s[2] = __fadd_rn(s[2], __fmul_rn(u.z, u.z));
        s[3] = __fadd_rn(s[3], __fmul_rn(u.w, u.w));
        s[4] = __fadd_rn(s[4], __fmul_rn(v.x, v.x));
        s[5] = __fadd_rn(s[5], __fmul_rn(v.y, v.y));
        s[6] = __fadd_rn(s[6], __fmul_rn(v.z, v.z));
        s[7] = __fadd_rn(s[7], __fmul_rn(v.w, v.w));
    }
    // item offsets 16 and 8: lanes 2 and 1 apart
#pragma unroll
    for (int r = 0; r < 8; ++r) s[r] = __fadd_rn(s[r], __shfl_xor_sync(0xffffffffu, s[r], 2));
#pragma unroll
    for (int r = 0; r < 8; ++r) s[r] = __fadd_rn(s[r], __shfl_xor_sync(0xffffffffu, s[r], 1));
    // item offsets 4, 2, 1: registers r ^ 4, r ^ 2, r ^ 1 (only item 0's chain)
    const float t0 = __fadd_rn(s[0], s[4]), t1 = __fadd_rn(s[1], s[5]);
    const float t2 = __fadd_rn(s[2], s[6]), t3 = __fadd_rn(s[3], s[7]);
    const float wave = __fadd_rn(__fadd_rn(t0, t2), __fadd_rn(t1, t3));
    // the eight wave partials (lanes 0, 4, ..., 28) from wave 0 upward
    float total = 0.0f;
#pragma unroll
    for (int v = 0; v < 8; ++v) total = __fadd_rn(total, __shfl_sync(0xffffffffu, wave, 4 * v));
    const float mean = __fdiv_rn(total, (float)n);  // n <= 2^24 converts exactly
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, 1e-5f)));
}

// The same scale evaluated by the workgroup itself: 256 threads, thread t is
// item t (t = threadIdx.x), the wave butterfly is a shuffle butterfly and the
// eight wave partials meet in s_wave (8 floats of shared memory).  Each thread
// loads 32 of its rows before adding any, so a vector of n values takes
// ceil(n / 8192) L2 round trips (one warp alone needs one per 8 rows); a row
// past the end adds an exact zero (the partial sums are never negative).
// Every thread of the block must call (with named: threads 0..255 only, which
// then meet at barrier 1 instead of the block barrier); every calling thread
// returns the scale.
__device__ __forceinline__ float rms_scale_block(const float *__restrict__ x, int64_t n,
                                                 float *s_wave, bool named = false) {
    const int t = threadIdx.x;
    const int64_t rows = n / 256;
    float s = 0.0f;
    for (int64_t k = 0; k < rows; k += 32) {
        const float *p = x + k * 256 + t;
        float v[32];
        if (k + 32 <= rows) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __ldg(p + j * 256);
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = k + j < rows ? __ldg(p + j * 256) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) s = __fadd_rn(s, __fmul_rn(v[j], v[j]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, off));
    if ((t & 31) == 0) s_wave[t >> 5] = s;
    if (named)
        asm volatile("bar.sync 1, 256;" ::: "memory");
    else
        __syncthreads();
    float total = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) total = __fadd_rn(total, s_wave[w]);
    const float mean = __fdiv_rn(total, (float)n);
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, 1e-5f)));
}

}  // namespace xq
